// int32 / uint32 sum scans (wraparound mod 2^32), all tile-shape variants.
#include "sc_scan_launch.cuh"

namespace scg {

#define SHAPE(i) SC_SHAPE_ARGS(kShapeSumU32[i])

template <>
cudaError_t launch_scan<OpSumU32>(const ScanParams& p, bool exclusive, bool segmented, int variant, cudaStream_t s) {
    if (segmented) {
        switch (variant) {
        case 0: return launch_shape<OpSumU32, SHAPE(0)>(p, exclusive, true, s);
        case 5: return launch_shape<OpSumU32, SHAPE(5)>(p, exclusive, true, s);
        case 8: return launch_shape<OpSumU32, SHAPE(8)>(p, exclusive, true, s);
        case 9: return launch_shape<OpSumU32, SHAPE(9)>(p, exclusive, true, s);
        case 10: return launch_shape<OpSumU32, SHAPE(10)>(p, exclusive, true, s);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (variant) {
    case 0: return launch_shape<OpSumU32, SHAPE(0)>(p, exclusive, false, s);
    case 1: return launch_shape_plain<OpSumU32, SHAPE(1)>(p, exclusive, s);
    case 2: return launch_shape_plain<OpSumU32, SHAPE(2)>(p, exclusive, s);
    case 3: return launch_shape_plain<OpSumU32, SHAPE(3)>(p, exclusive, s);
    case 4: return launch_shape_plain<OpSumU32, SHAPE(4)>(p, exclusive, s);
    case 5: return launch_shape_plain<OpSumU32, SHAPE(5)>(p, exclusive, s);
    case 6: return launch_shape_plain<OpSumU32, SHAPE(6)>(p, exclusive, s);
    case 7: return launch_shape_plain<OpSumU32, SHAPE(7)>(p, exclusive, s);
    case 8: return launch_shape_plain<OpSumU32, SHAPE(8)>(p, exclusive, s);
    case 9: return launch_shape_plain<OpSumU32, SHAPE(9)>(p, exclusive, s);
    case 10: return launch_shape_plain<OpSumU32, SHAPE(10)>(p, exclusive, s);
    case 11: return launch_shape_plain<OpSumU32, SHAPE(11)>(p, exclusive, s);
    case 12: return launch_shape_plain<OpSumU32, SHAPE(12)>(p, exclusive, s);
    case 13: return launch_shape_plain<OpSumU32, SHAPE(13)>(p, exclusive, s);
    case 14: return launch_shape_plain<OpSumU32, SHAPE(14)>(p, exclusive, s);
    default: return cudaErrorInvalidValue;
    }
}

bool segmented_shape(int variant) {
    return variant == 0 || variant == 5 || variant == 8 || variant == 9 || variant == 10;
}

#undef SHAPE
}  // namespace scg
