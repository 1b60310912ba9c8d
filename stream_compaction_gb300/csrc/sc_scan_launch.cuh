// Launch one scan tile shape (inclusive/exclusive x plain/segmented).
#pragma once
#include "sc_scan.cuh"
#include "sc_shapes.h"

namespace scg {

template <class Op, int NT, int IPT, int kLoad, int kLb, int kMinB, int kStats>
cudaError_t launch_shape(const ScanParams& p, bool exclusive, bool segmented, cudaStream_t s) {
    const dim3 grid(p.lb.num_tiles);
    if (segmented) {
        if (exclusive) scan_kernel<Op, NT, IPT, true, true, kLoad, kLb, kMinB><<<grid, NT, 0, s>>>(p);
        else scan_kernel<Op, NT, IPT, false, true, kLoad, kLb, kMinB><<<grid, NT, 0, s>>>(p);
    } else {
        if (exclusive) scan_kernel<Op, NT, IPT, true, false, kLoad, kLb, kMinB><<<grid, NT, 0, s>>>(p);
        else scan_kernel<Op, NT, IPT, false, false, kLoad, kLb, kMinB><<<grid, NT, 0, s>>>(p);
    }
    return cudaGetLastError();
}

// Plain scans only (tuning variants have no segmented form).
template <class Op, int NT, int IPT, int kLoad, int kLb, int kMinB, int kStats>
cudaError_t launch_shape_plain(const ScanParams& p, bool exclusive, cudaStream_t s) {
    const dim3 grid(p.lb.num_tiles);
    if (exclusive) scan_kernel<Op, NT, IPT, true, false, kLoad, kLb, kMinB, kStats != 0><<<grid, NT, 0, s>>>(p);
    else scan_kernel<Op, NT, IPT, false, false, kLoad, kLb, kMinB, kStats != 0><<<grid, NT, 0, s>>>(p);
    return cudaGetLastError();
}

#define SC_SHAPE_ARGS(sh) sh.nt, sh.ipt, sh.load, sh.lb, sh.minb, sh.stats

}  // namespace scg
