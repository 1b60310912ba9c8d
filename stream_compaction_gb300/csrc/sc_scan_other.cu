// float32 sum (float-float inter-tile carry), int32 max and affine-map composition scans.
#include "sc_scan_launch.cuh"

namespace scg {

template <>
cudaError_t launch_scan<OpSumF32>(const ScanParams& p, bool exclusive, bool segmented, int variant, cudaStream_t s) {
    if (variant != 0) return cudaErrorInvalidValue;
    return launch_shape<OpSumF32, SC_SHAPE_ARGS(kShapeSumF32)>(p, exclusive, segmented, s);
}

template <>
cudaError_t launch_scan<OpMaxI32>(const ScanParams& p, bool exclusive, bool segmented, int variant, cudaStream_t s) {
    if (variant != 0) return cudaErrorInvalidValue;
    return launch_shape<OpMaxI32, SC_SHAPE_ARGS(kShapeMaxI32)>(p, exclusive, segmented, s);
}

template <>
cudaError_t launch_scan<OpAffineU32>(const ScanParams& p, bool exclusive, bool segmented, int variant, cudaStream_t s) {
    if (variant != 0) return cudaErrorInvalidValue;
    return launch_shape<OpAffineU32, SC_SHAPE_ARGS(kShapeAffine)>(p, exclusive, segmented, s);
}

}  // namespace scg
