// int32 / uint32 sum scans (wraparound mod 2^32), all tile-shape variants.
#include "sc_scan_launch.cuh"

namespace scg {

#define SHAPE(i) kShapeSumU32[i].nt, kShapeSumU32[i].ipt, kShapeSumU32[i].load

template <>
cudaError_t launch_scan<OpSumU32>(const ScanParams& p, bool exclusive, bool segmented, int variant, cudaStream_t s) {
    if (segmented) {
        if (variant != 0) return cudaErrorInvalidValue;
        return launch_shape<OpSumU32, SHAPE(0)>(p, exclusive, true, s);
    }
    switch (variant) {
    case 0: return launch_shape<OpSumU32, SHAPE(0)>(p, exclusive, false, s);
    case 1: return launch_shape_plain<OpSumU32, SHAPE(1)>(p, exclusive, s);
    case 2: return launch_shape_plain<OpSumU32, SHAPE(2)>(p, exclusive, s);
    case 3: return launch_shape_plain<OpSumU32, SHAPE(3)>(p, exclusive, s);
    case 4: return launch_shape_plain<OpSumU32, SHAPE(4)>(p, exclusive, s);
    default: return cudaErrorInvalidValue;
    }
}

#undef SHAPE
}  // namespace scg
