// Hierarchical scan-then-propagate comparison variant, restated for sm_103a.
//
// This is the multi-kernel design of "Lecture 7: Parallel pattern -- prefix
// sum / scan" (UIUC ECE408 notes), section 6 "Hierarchical Scan" (scan each
// segment and record its total; scan the totals; add each segment's offset
// back), made recursive on the totals as in "CUDA programming: parallel
// prefix-sum scan explained" (m.youleyou.com), so that any n is handled.  It
// moves every element through global memory twice (about 4 passes of 4 bytes
// for 32-bit data instead of 2) and exists to be timed beside the single-pass
// kernel on the same inputs.  The tile pass reuses the register / warp-shuffle
// block scan of the single-pass kernel; no look-back is involved.
#include "sc_device.cuh"
#include "sc_launch.h"

namespace scg {

template <class Op>
struct HierShape;
template <> struct HierShape<OpSumU32> { static constexpr int IPT = 16; };
template <> struct HierShape<OpSumF32> { static constexpr int IPT = 16; };
template <> struct HierShape<OpMaxI32> { static constexpr int IPT = 16; };
template <> struct HierShape<OpAffineU32> { static constexpr int IPT = 8; };

int hier_tile_elems(int op_id) {
    switch (op_id) {
    case 0: case 1: case 2: return kHierNT * 16;
    case 3: return kHierNT * 8;
    default: return 0;
    }
}

// Pass 1 (and every recursion level): scan each tile on its own, write the
// tile-local scan and the tile's total.
template <class Op, int NT, int IPT, bool kExcl>
__global__ void __launch_bounds__(NT) hier_tile_kernel(const HierParams p) {
    using T = typename Op::T;
    constexpr int NW = NT / 32;
    constexpr int TILE = NT * IPT;
    constexpr int NV = IPT / Vec<T>::kPer;
    __shared__ uint4 s_buf[NT * NV];
    __shared__ T s_wagg[NW];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long tile = blockIdx.x;
    const long long tile_start = tile * TILE;
    const long long valid = min((long long)TILE, p.n - tile_start);
    const T* tin = static_cast<const T*>(p.in) + tile_start;
    T* tout = static_cast<T*>(p.out) + tile_start;
    uint4* wbuf = s_buf + warp * 32 * NV;
    const bool full = valid == TILE && p.vec_ok;

    T v[IPT];
    if (full) load_full_tile<T, IPT, LOAD_XPOSE>(tin, v, wbuf);
    else load_partial_tile<T, IPT>(tin, v, valid, Op::identity());
#pragma unroll
    for (int k = 1; k < IPT; ++k) v[k] = Op::op(v[k - 1], v[k]);
    T x = v[IPT - 1];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const T y = shfl_up_v(x, d);
        if (lane >= d) x = Op::op(y, x);
    }
    T carry = shfl_up_v(x, 1);
    if (lane == 0) carry = Op::identity();
    if (lane == 31) s_wagg[warp] = x;
    __syncthreads();
    T wcarry = Op::identity();
    for (int w = 0; w < warp; ++w) wcarry = Op::op(wcarry, s_wagg[w]);
    if (tid == NT - 1) static_cast<T*>(p.totals)[tile] = Op::op(wcarry, x);
    carry = Op::op(wcarry, carry);
    if constexpr (kExcl) {
#pragma unroll
        for (int k = IPT - 1; k >= 1; --k) v[k] = Op::op(carry, v[k - 1]);
        v[0] = carry;
    } else {
#pragma unroll
        for (int k = 0; k < IPT; ++k) v[k] = Op::op(carry, v[k]);
    }
    if (full) store_full_tile<T, IPT, LOAD_XPOSE>(tout, v, wbuf);
    else store_partial_tile<T, IPT>(tout, v, valid);
}

// Pass 3: y = offset[tile] (+) y for every element of tiles 1.. (the offset of
// tile 0 is the identity).  Elementwise, so the tile is walked in coalesced
// 16-byte vectors without any transpose.
template <class Op, int NT, int IPT>
__global__ void __launch_bounds__(NT) hier_add_kernel(const HierParams p) {
    using T = typename Op::T;
    constexpr int TILE = NT * IPT;
    constexpr int PER = Vec<T>::kPer;
    constexpr int NV = IPT / PER;
    const long long tile = blockIdx.x + 1;
    const long long tile_start = tile * TILE;
    const long long valid = min((long long)TILE, p.n - tile_start);
    const T off = static_cast<const T*>(p.offsets)[tile];
    T* t = static_cast<T*>(p.out) + tile_start;
    if (valid == TILE && p.vec_ok) {
        uint4* t4 = reinterpret_cast<uint4*>(t);
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            uint4 r = t4[j * NT + threadIdx.x];
            T e[PER];
            unpack(r, e);
#pragma unroll
            for (int q = 0; q < PER; ++q) e[q] = Op::op(off, e[q]);
            st_stream(t4 + j * NT + threadIdx.x, pack(e));
        }
    } else {
        for (long long i = threadIdx.x; i < valid; i += NT) t[i] = Op::op(off, t[i]);
    }
}

template <class Op>
cudaError_t launch_hier_tiles(const HierParams& p, bool exclusive, unsigned ntiles, cudaStream_t s) {
    constexpr int IPT = HierShape<Op>::IPT;
    if (exclusive) hier_tile_kernel<Op, kHierNT, IPT, true><<<ntiles, kHierNT, 0, s>>>(p);
    else hier_tile_kernel<Op, kHierNT, IPT, false><<<ntiles, kHierNT, 0, s>>>(p);
    return cudaGetLastError();
}

template <class Op>
cudaError_t launch_hier_add(const HierParams& p, unsigned ntiles, cudaStream_t s) {
    constexpr int IPT = HierShape<Op>::IPT;
    if (ntiles > 1) hier_add_kernel<Op, kHierNT, IPT><<<ntiles - 1, kHierNT, 0, s>>>(p);
    return cudaGetLastError();
}

template cudaError_t launch_hier_tiles<OpSumU32>(const HierParams&, bool, unsigned, cudaStream_t);
template cudaError_t launch_hier_tiles<OpSumF32>(const HierParams&, bool, unsigned, cudaStream_t);
template cudaError_t launch_hier_tiles<OpMaxI32>(const HierParams&, bool, unsigned, cudaStream_t);
template cudaError_t launch_hier_tiles<OpAffineU32>(const HierParams&, bool, unsigned, cudaStream_t);
template cudaError_t launch_hier_add<OpSumU32>(const HierParams&, unsigned, cudaStream_t);
template cudaError_t launch_hier_add<OpSumF32>(const HierParams&, unsigned, cudaStream_t);
template cudaError_t launch_hier_add<OpMaxI32>(const HierParams&, unsigned, cudaStream_t);
template cudaError_t launch_hier_add<OpAffineU32>(const HierParams&, unsigned, cudaStream_t);

}  // namespace scg
