// Single-pass device-wide scan: one launch, each CTA scans one tile and takes
// its carry from its predecessors through the decoupled look-back.
//
// Per tile:  dynamic tile id (atomic counter, so a tile only ever waits on
// tiles whose CTAs are already running) -> 16-byte vector loads -> serial scan
// of the thread's items in registers -> Kogge-Stone warp scan with
// __shfl_up_sync -> block combine over warp totals -> publish the tile
// aggregate, look back, publish the inclusive prefix -> outputs -> 16-byte
// stores.  Each element is read once and written once.
//
// The pages' multi-kernel designs pay one extra global round trip of the data
// for the carry ("Lecture 7" notes, section 6 "Hierarchical Scan", which also
// names the single-kernel decoupled look-back with atomic flags as the
// alternative); the thread-serial register stage and the warp shuffle stage
// follow the optimisation notes of the same page and of PMPP chapter 9
// (section 9.7, warp-level optimisation).
#pragma once
#include "sc_device.cuh"

namespace scg {

// Segment heads inside the thread's IPT items (bit k: item k starts a segment).
template <int IPT>
__device__ __forceinline__ uint32_t head_bits(long long first_index, long long seg_len) {
    const long long r = first_index % seg_len;
    long long k = r == 0 ? 0 : seg_len - r;
    uint32_t hm = 0;
    for (; k < IPT; k += seg_len) hm |= 1u << k;
    return hm;
}

// Segment heads inside the thread's IPT items from a head-flag array (one
// byte per element, nonzero = head); one vector load when the flags are full
// and aligned, else byte loads up to n.
template <int IPT>
__device__ __forceinline__ uint32_t head_bits_flags(const unsigned char* heads, long long first, long long n) {
    uint32_t hm = 0;
    const unsigned char* f = heads + first;
    if constexpr (IPT == 16 || IPT == 8) {
        if (first + IPT <= n && (reinterpret_cast<uintptr_t>(f) % IPT) == 0) {
            uint32_t w[IPT / 4];
            if constexpr (IPT == 16) {
                const uint4 q = __ldg(reinterpret_cast<const uint4*>(f));
                w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
            } else {
                const uint2 q = __ldg(reinterpret_cast<const uint2*>(f));
                w[0] = q.x; w[1] = q.y;
            }
#pragma unroll
            for (int j = 0; j < IPT / 4; ++j)
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    if ((w[j] >> (8 * b)) & 0xffu) hm |= 1u << (4 * j + b);
            return hm;
        }
    }
#pragma unroll
    for (int k = 0; k < IPT; ++k)
        if (first + k < n && f[k]) hm |= 1u << k;
    return hm;
}

// Sleep for the test hook that slows one tile down (bounded by ns itself).
__device__ __forceinline__ void hook_delay(unsigned ns) {
    const unsigned long long t0 = global_ns();
    for (int i = 0; i < (1 << 20) && global_ns() - t0 < ns; ++i) __nanosleep(1000);
}

// Instrumented variants (kStats) add, per tile, the time spent in each phase
// to 8 counters: [0] tiles, [1] ns until the tile id is known, [2] ns loading
// and scanning the tile, [3] ns in the look-back, [4] look-back windows read,
// [5] polls that found a predecessor not yet published, [6] ns from the
// prefix to the end of the stores, [7] ns of the whole tile.
template <class Op, int NT, int IPT, bool kExcl, bool kSeg, int kLoad, int kLb = 1, int kMinB = 1, bool kStats = false>
__global__ void __launch_bounds__(NT, kMinB) scan_kernel(const ScanParams p) {
    using T = typename Op::T;
    using C = typename Op::C;
    constexpr int NW = NT / 32;
    constexpr int TILE = NT * IPT;
    constexpr int NV = IPT / Vec<T>::kPer;
    static_assert(IPT <= 32 && IPT % Vec<T>::kPer == 0, "items per thread");

    __shared__ uint4 s_buf[kLoad == LOAD_XPOSE ? NT * NV : 1];
    __shared__ T s_wagg[NW];
    __shared__ int s_whead[NW];
    __shared__ C s_prefix;
    __shared__ unsigned s_tile;
    __shared__ int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned long long t0 = 0, t1 = 0, t2 = 0, t3 = 0, t4 = 0;
    unsigned windows = 0, polls = 0;
    if (kStats && tid == 0) t0 = global_ns();
    if (tid == 0) {
        s_tile = p.lb.static_ids ? blockIdx.x : (unsigned)(atomicAdd(p.lb.counter, 1ull) - p.lb.counter_base);
        s_abort = 0;
    }
    __syncthreads();
    if (kStats && tid == 0) t1 = global_ns();
    const long long tile = s_tile;
    const long long tile_start = tile * TILE;
    const long long valid = min((long long)TILE, p.n - tile_start);
    const T* tin = static_cast<const T*>(p.in) + tile_start;
    T* tout = static_cast<T*>(p.out) + tile_start;
    uint4* wbuf = s_buf + (kLoad == LOAD_XPOSE ? warp * 32 * NV : 0);
    const bool full = valid == TILE && p.vec_ok;

    T v[IPT];
    if (full) load_full_tile<T, IPT, kLoad>(tin, v, wbuf);
    else load_partial_tile<T, IPT>(tin, v, valid, Op::identity());

    uint32_t hm = 0;
    if constexpr (kSeg) {
        const long long first = tile_start + (long long)tid * IPT;
        hm = p.heads ? head_bits_flags<IPT>(p.heads, first, p.n) : head_bits<IPT>(first, p.seg_len);
    }

    // thread-serial inclusive scan (restarting at segment heads)
#pragma unroll
    for (int k = 1; k < IPT; ++k) v[k] = (kSeg && ((hm >> k) & 1u)) ? v[k] : Op::op(v[k - 1], v[k]);

    // warp scan of the thread aggregates; with segments a lane only combines
    // values from lanes at or after the newest head at or before it
    T x = v[IPT - 1];
    uint32_t wmask = 0;
    int hl = -1;
    if constexpr (kSeg) {
        wmask = __ballot_sync(0xffffffffu, hm != 0u);
        const uint32_t le = wmask & lanemask_le();
        hl = le ? 31 - __clz(le) : -1;
    }
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const T y = shfl_up_v(x, d);
        if (lane >= d && (!kSeg || lane - d >= hl)) x = Op::op(y, x);
    }
    T lane_carry = shfl_up_v(x, 1);
    if (lane == 0) lane_carry = Op::identity();
    const bool lane_open = kSeg ? ((wmask & lanemask_lt()) == 0u) : true;
    if (lane == 31) {
        s_wagg[warp] = x;
        s_whead[warp] = kSeg ? (wmask != 0u) : 0;
    }
    __syncthreads();
    if (kStats && tid == 0) t2 = global_ns();

    // block combine: carry from the warps before this one
    T wcarry = Op::identity();
    bool wopen = true;
    for (int w = 0; w < warp; ++w) {
        if (kSeg && s_whead[w]) { wcarry = s_wagg[w]; wopen = false; }
        else wcarry = Op::op(wcarry, s_wagg[w]);
    }

    if (warp == 0) {
        // tile aggregate (segmented: the fold from the tile's last head)
        T tagg = Op::identity();
        bool thead = false;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            if (kSeg && s_whead[w]) { tagg = s_wagg[w]; thead = true; }
            else tagg = Op::op(tagg, s_wagg[w]);
        }
        const C agg = Op::lift(tagg);
        C prefix = Op::c_identity();
        bool ok = true;
        if (tile == p.lb.stall_tile) {
            ok = false;  // test hook: this tile never publishes
        } else {
            if (tile == p.lb.delay_tile && lane == 0) hook_delay(p.lb.delay_ns);
            __syncwarp();
            const bool first_is_head =
                kSeg && (p.heads ? (p.heads[tile_start] != 0) : (tile_start % p.seg_len == 0));
            if (tile == 0 || first_is_head) {
                if (!kSeg && p.carry_in) prefix = *static_cast<const C*>(p.carry_in);
                if (lane == 0) StatusIO<C>::publish(p.lb, tile, ST_PREFIX, kSeg ? agg : Op::c_op(prefix, agg));
            } else {
                const bool complete = kSeg && thead;  // aggregate already starts at a head
                if (lane == 0) StatusIO<C>::publish(p.lb, tile, complete ? ST_PREFIX : ST_AGGREGATE, agg);
                ok = lookback_prefix<Op, kLb>(p.lb, tile, prefix, kStats ? &windows : nullptr,
                                              kStats ? &polls : nullptr);
                if (ok && !complete && lane == 0) StatusIO<C>::publish(p.lb, tile, ST_PREFIX, Op::c_op(prefix, agg));
                if (!ok && lane == 0) StatusIO<C>::publish(p.lb, tile, ST_POISON, agg);
            }
            if (ok && lane == 0 && p.carry_out && tile == (long long)p.lb.num_tiles - 1)
                *static_cast<C*>(p.carry_out) = Op::c_op(prefix, agg);
        }
        if (lane == 0) {
            s_prefix = prefix;
            if (!ok) s_abort = 1;
        }
    }
    __syncthreads();
    if (kStats && tid == 0) t3 = global_ns();
    if (s_abort) return;

    // carry into the thread's first item: tile prefix (+) warp carry (+) lane carry,
    // each applied only while no segment head intervenes
    T carry = lane_carry;
    if (lane_open) {
        carry = Op::op(wcarry, carry);
        if (wopen) carry = Op::op(Op::lower(s_prefix), carry);
    }
    const int fh = kSeg ? (hm ? __ffs(hm) - 1 : IPT) : IPT;  // first head in this thread
    if constexpr (kExcl) {
#pragma unroll
        for (int k = IPT - 1; k >= 1; --k) {
            const T e = (kSeg && ((hm >> k) & 1u)) ? Op::identity() : v[k - 1];
            v[k] = (k < fh) ? Op::op(carry, e) : e;
        }
        v[0] = (kSeg && (hm & 1u)) ? Op::identity() : carry;
    } else {
#pragma unroll
        for (int k = 0; k < IPT; ++k)
            if (k < fh) v[k] = Op::op(carry, v[k]);
    }

    if (full) store_full_tile<T, IPT, kLoad>(tout, v, wbuf);
    else store_partial_tile<T, IPT>(tout, v, valid);
    if constexpr (kStats) {
        __syncthreads();
        if (tid == 0) {
            t4 = global_ns();
            unsigned long long* st = p.lb.stats;
            atomicAdd(st + 0, 1ull);
            atomicAdd(st + 1, t1 - t0);
            atomicAdd(st + 2, t2 - t1);
            atomicAdd(st + 3, t3 - t2);
            atomicAdd(st + 4, (unsigned long long)windows);
            atomicAdd(st + 5, (unsigned long long)polls);
            atomicAdd(st + 6, t4 - t3);
            atomicAdd(st + 7, t4 - t0);
        }
    }
}

}  // namespace scg
