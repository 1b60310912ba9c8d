// Fused stream compaction: predicate -> flag scan -> look-back on counts ->
// order-preserving, coalesced scatter, all in one pass over the input.
//
// The method is the two-phase compaction of "Lecture 7: Parallel pattern --
// prefix sum / scan" (UIUC ECE408 notes), section 2 "Applications of Scan",
// and of "Chapter 9 Parallel Patterns: Prefix Sum - Scan Algorithms" (PMPP
// notes), sections 9.6 and 4.2: flag each element, exclusive-scan the flags to
// get each kept element's output slot, write kept elements to their slots.
// Here the flags never leave registers: each tile counts its kept elements,
// takes its output offset from the look-back over tile counts, packs its kept
// elements contiguously in shared memory and writes them out as one
// contiguous run (the "one contiguous, coalesced write" the notes point out).
#include "sc_device.cuh"
#include "sc_launch.h"

namespace scg {

__device__ __forceinline__ bool keep(int32_t x, const PredParams& q) {
    const bool in = x >= (int32_t)q.lo && x <= (int32_t)q.hi;
    return in != (q.invert != 0);
}
__device__ __forceinline__ bool keep(uint32_t x, const PredParams& q) {
    const bool in = x >= (uint32_t)q.lo && x <= (uint32_t)q.hi;
    return in != (q.invert != 0);
}
// Floats: q.lo holds a 4-bit mask of the outcomes that keep x:
// bit 0 x > tf, bit 1 x == tf, bit 2 x < tf, bit 3 unordered (x is NaN).
__device__ __forceinline__ bool keep(float x, const PredParams& q) {
    const unsigned m = (unsigned)q.lo;
    const unsigned outcome = (x > q.tf) ? 1u : (x == q.tf) ? 2u : (x < q.tf) ? 4u : 8u;
    return (m & outcome) != 0u;
}

template <class T, class CntOp, int NT, int IPT, int kLoad>
__global__ void __launch_bounds__(NT) compact_kernel(const CompactParams p) {
    using C = typename CntOp::C;
    constexpr int NW = NT / 32;
    constexpr int TILE = NT * IPT;
    constexpr int NV = IPT / Vec<T>::kPer;

    __shared__ uint4 s_buf[NT * NV];  // load transpose, then the packed kept elements
    __shared__ uint32_t s_wcnt[NW];
    __shared__ C s_prefix;
    __shared__ unsigned s_tile;
    __shared__ int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_tile = p.lb.static_ids ? blockIdx.x : (unsigned)(atomicAdd(p.lb.counter, 1ull) - p.lb.counter_base);
        s_abort = 0;
    }
    __syncthreads();
    const long long tile = s_tile;
    const long long tile_start = tile * TILE;
    const long long valid = min((long long)TILE, p.n - tile_start);
    const T* tin = static_cast<const T*>(p.in) + tile_start;
    const bool full = valid == TILE && p.vec_ok;

    T v[IPT];
    if (full) load_full_tile<T, IPT, kLoad>(tin, v, s_buf + warp * 32 * NV);
    else load_partial_tile<T, IPT>(tin, v, valid, T(0));

    // flags in a register bitmask
    uint32_t bits = 0;
    const long long base = (long long)tid * IPT;
#pragma unroll
    for (int k = 0; k < IPT; ++k)
        if (base + k < valid && keep(v[k], p.pred)) bits |= 1u << k;
    const uint32_t cnt = __popc(bits);

    // warp exclusive scan of the counts
    uint32_t x = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    const uint32_t lane_excl = x - cnt;
    if (lane == 31) s_wcnt[warp] = x;
    __syncthreads();  // also: every warp is done with its load transpose
    uint32_t wexcl = 0, tcnt = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const uint32_t c = s_wcnt[w];
        if (w < warp) wexcl += c;
        tcnt += c;
    }

    // pack kept elements at their tile-local slots (the exclusive flag scan)
    T* stage = reinterpret_cast<T*>(s_buf);
    uint32_t pos = wexcl + lane_excl;
#pragma unroll
    for (int k = 0; k < IPT; ++k)
        if ((bits >> k) & 1u) stage[pos++] = v[k];

    if (warp == 0) {
        const C agg = CntOp::lift(tcnt);
        C prefix = CntOp::c_identity();
        bool ok = true;
        if (tile == p.lb.stall_tile) {
            ok = false;
        } else if (tile == 0) {
            if (lane == 0) StatusIO<C>::publish(p.lb, tile, ST_PREFIX, agg);
        } else {
            if (lane == 0) StatusIO<C>::publish(p.lb, tile, ST_AGGREGATE, agg);
            ok = lookback_prefix<CntOp>(p.lb, tile, prefix);
            if (lane == 0) StatusIO<C>::publish(p.lb, tile, ok ? ST_PREFIX : ST_POISON, CntOp::c_op(prefix, agg));
        }
        if (lane == 0) {
            s_prefix = prefix;
            if (!ok) s_abort = 1;
            if (ok && tile == (long long)p.lb.num_tiles - 1) *p.count = (long long)(prefix + agg);
        }
    }
    __syncthreads();
    if (s_abort) return;

    // one contiguous run out[prefix .. prefix + tcnt): consecutive threads write
    // consecutive elements
    T* dst = static_cast<T*>(p.out) + (long long)s_prefix;
    for (uint32_t i = tid; i < tcnt; i += NT) dst[i] = stage[i];
}

template <class T>
cudaError_t launch_compact(const CompactParams& p, bool wide_count, cudaStream_t s) {
    constexpr int NT = CompactConfig::NT, IPT = CompactConfig::IPT;
    const dim3 grid(p.lb.num_tiles);
    if (wide_count) compact_kernel<T, OpCountU64, NT, IPT, LOAD_XPOSE><<<grid, NT, 0, s>>>(p);
    else compact_kernel<T, OpCountU32, NT, IPT, LOAD_XPOSE><<<grid, NT, 0, s>>>(p);
    return cudaGetLastError();
}

template cudaError_t launch_compact<int32_t>(const CompactParams&, bool, cudaStream_t);
template cudaError_t launch_compact<uint32_t>(const CompactParams&, bool, cudaStream_t);
template cudaError_t launch_compact<float>(const CompactParams&, bool, cudaStream_t);

}  // namespace scg
