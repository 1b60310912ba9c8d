// One operator of the sc_ops_*.cu groups: the one-tile-per-CTA kernel (plain
// or segmented, shape by element size) or the persistent kernel (shape 0).
#pragma once
#include "sc_scan_launch.cuh"
#include "sc_scan_tma.cuh"

namespace scg {

template <class Op>
cudaError_t launch_op(const ScanParams& p, bool exclusive, bool segmented, unsigned tma_grid, cudaStream_t s) {
    if (tma_grid) {
        if (segmented) return cudaErrorInvalidValue;
        return launch_cfg<Op, typename DefaultCfg<Op>::type>(p, exclusive, tma_grid, s, false);
    }
    if constexpr (sizeof(typename Op::T) == 8)
        return launch_shape<Op, SC_SHAPE_ARGS(kShapeExtra8)>(p, exclusive, segmented, s);
    else
        return launch_shape<Op, SC_SHAPE_ARGS(kShapeExtra4)>(p, exclusive, segmented, s);
}

}  // namespace scg

// The dispatcher of one group: SC_OPS_GROUP(name, (oid, Op), ...).
#define SC_OPS_CASE(oid, Op) \
    case oid: return launch_op<Op>(p, exclusive, segmented, tma_grid, s);
