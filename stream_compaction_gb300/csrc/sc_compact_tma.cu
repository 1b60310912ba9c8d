// Persistent, warp-specialised fused stream compaction (the default path for
// 16-byte-aligned inputs of at least one full tile).
//
// The method is the two-phase compaction of "Lecture 7: Parallel pattern --
// prefix sum / scan" (UIUC ECE408 notes), section 2 "Applications of Scan",
// and of "Chapter 9 Parallel Patterns: Prefix Sum - Scan Algorithms" (PMPP
// notes), sections 9.6 and 4.2: flag every element, exclusive-scan the flags
// to find each kept element's output slot, write kept elements there.  The
// flags never reach memory and the scan of the flags is the same chained,
// decoupled look-back over chunk counts as the persistent scan uses:
//
//   producer A      chunk ids from the atomic counter, fresh tiles by TMA;
//   compute warps   pass 1: each warp evaluates the predicate on its part of a
//                   fresh tile, keeps one 32-bit flag mask per 128-byte row
//                   in shared memory and counts the kept elements (the stage
//                   is freed at once);
//                   pass 2 (kLag tiles later, the tile re-loaded from L2):
//                   each warp packs its kept elements in order inside its own
//                   part of the stage (the row masks + popcount give
//                   consecutive slots), then writes them as one contiguous
//                   run: the 16-byte aligned middle by a bulk copy, up to
//                   3 + 3 edge elements by plain stores;
//   bookkeeping     tile counts, chunk counts, chunk aggregates published;
//   look-back       chunk prefixes; the last chunk also writes the count;
//   producer B      the pass-2 re-loads.
//
// Each input element is read from HBM once and each kept element written
// once.
#include <atomic>
#include <type_traits>

#include "sc_launch.h"
#include "sc_persist.cuh"
#include "sc_scan.cuh"

namespace scg {

// Integers: lo <= x <= hi as one unsigned range check, xor invert (an empty
// interval is stored with lo > hi, which the host encodes as span < 0: never).
__device__ __forceinline__ bool keep_elem(int32_t x, const PredParams& q) {
    const uint32_t d = (uint32_t)x - (uint32_t)(int32_t)q.lo;
    const bool in = q.hi >= q.lo && d <= (uint32_t)((int32_t)q.hi - (int32_t)q.lo);
    return in != (q.invert != 0);
}
__device__ __forceinline__ bool keep_elem(uint32_t x, const PredParams& q) {
    const uint32_t d = x - (uint32_t)q.lo;
    const bool in = q.hi >= q.lo && d <= (uint32_t)q.hi - (uint32_t)q.lo;
    return in != (q.invert != 0);
}
// Floats: q.lo holds a 4-bit mask of the outcomes that keep x:
// bit 0 x > tf, bit 1 x == tf, bit 2 x < tf, bit 3 unordered (x is NaN).
__device__ __forceinline__ bool keep_elem(float x, const PredParams& q) {
    const unsigned m = (unsigned)q.lo;
    const unsigned outcome = (x > q.tf) ? 1u : (x == q.tf) ? 2u : (x < q.tf) ? 4u : 8u;
    return (m & outcome) != 0u;
}

namespace {

using namespace persist;

constexpr int kTileBytes = 32768;       // 256 rows of 128 bytes
constexpr int kRows = kTileBytes / 128;
constexpr int kSA = 3;                  // pass-1 stages: fresh tiles from HBM
constexpr int kSB = 3;                  // pass-2 stages: the same tiles again, from L2
constexpr int kChunk = 2;               // tiles per counter tick and per look-back status
constexpr int kLag = 6;                 // pass 2 of tile k follows pass 1 of tile k + kLag
constexpr int kLbWarps = 3;
constexpr int kChunkSlots = 6;
constexpr int kRing = 64;
constexpr int kR1 = 32;
constexpr int TILE = kTileBytes / 4;    // 8192 four-byte elements
constexpr int kLbPer = 8;
constexpr unsigned kSentinel = 0xffffffffu;
constexpr unsigned kVoid = 0xfffffffeu;
constexpr int kCtrlBytes = 16384;
constexpr int kSmemBytes = (kSA + kSB) * kTileBytes + 1024 + kCtrlBytes;
constexpr int kMaxComputeWarps = 16;
constexpr int kMaskRing = 8;            // tiles whose row masks are kept (pass 1 -> pass 2)
static_assert(kMaskRing > kLag, "row masks outlive the lag");

// Compute-warp count of a compaction shape: each warp owns kRowsPerWarp rows
// (128 bytes each) of a tile in both passes.
template <int CW>
struct CompactShape {
    static constexpr int kComputeWarps = CW;
    static constexpr int kCompute = 32 * CW;
    static constexpr int kBookWarp = CW + kLbWarps;
    static constexpr int kProducerA = kBookWarp + 1;
    static constexpr int kProducerB = kProducerA + 1;
    static constexpr int kThreads = 32 * (kProducerB + 1);
    static constexpr int kRowsPerWarp = kRows / CW;
    static constexpr int kWarpBytes = kRowsPerWarp * 128;
    static constexpr int kThreadsPerRow = kCompute / kRows;       // pass 1: 1 (8 warps) or 2 (16 warps)
    static constexpr int kChunksPerThread = 8 / kThreadsPerRow;   // 16-byte chunks per thread in pass 1
    static_assert(kRows % CW == 0 && kCompute % kRows == 0 && CW <= kMaxComputeWarps, "compaction shape");
    static_assert(kRowsPerWarp % 8 == 0, "a warp's rows start on a swizzle period");
};

static_assert(kChunkSlots % kLbWarps == 0, "a look-back warp owns fixed chunk slots");
static_assert(kR1 > kLag && kLag >= kSB, "pass-1-done ring covers the lag");
static_assert(kRing >= kSA + kLag + kSB + 4, "tile ring outlives every reader");
static_assert(kChunkSlots * kChunk >= kLag + 2 * kChunk, "chunk ring covers the lag");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

struct Ctrl {
    unsigned long long a_full[kSA], a_empty[kSA];
    unsigned long long b_full[kSB], b_empty[kSB];
    unsigned long long p1done[kR1], wready[kR1];
    unsigned long long agg[kChunkSlots], pre[kChunkSlots];
    unsigned tile[kRing];
    unsigned long long offset[kRing];        // count of kept elements in the chunk's earlier tiles
    unsigned wcnt[kRing][kMaxComputeWarps];  // kept elements per warp part, from pass 1
    unsigned rowmask[kMaskRing][kRows];      // pass 1's flags, one bit per element of each 32-element row
    unsigned long long chunk_agg[kChunkSlots], chunk_prefix[kChunkSlots];
    long long chunk_id[kChunkSlots];
    int end_k;
    int consumed_a;
    int consumed_b;
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t r;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(a) : "memory");
    return r;
}
__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

template <class T>
__device__ __forceinline__ uint32_t bits_of(T v) { return to_bits32(v); }
template <class T>
__device__ __forceinline__ T from_bits(uint32_t b) { T v; from_bits32(b, v); return v; }

}  // namespace

template <class T, class CntOp, int CW>
__global__ void __launch_bounds__(CompactShape<CW>::kThreads, 1)
    compact_tma_kernel(const __grid_constant__ CUtensorMap tm_in, const CompactParams p, const long long n_full_tiles) {
    using C = typename CntOp::C;
    using Sh = CompactShape<CW>;
    constexpr int kComputeWarps = Sh::kComputeWarps, kBookWarp = Sh::kBookWarp;
    constexpr int kProducerA = Sh::kProducerA, kProducerB = Sh::kProducerB;
    constexpr int kRowsPerWarp = Sh::kRowsPerWarp, kWarpBytes = Sh::kWarpBytes;
    constexpr int kThreadsPerRow = Sh::kThreadsPerRow, kChunksPerThread = Sh::kChunksPerThread;
    constexpr int kPerThread = kChunksPerThread * 4;  // pass-1 elements per thread
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + (kSA + kSB) * kTileBytes);
    const uint32_t stageA = smem_u32(smem);
    const uint32_t stageB = stageA + kSA * kTileBytes;
    auto B = [](const unsigned long long& b) { return smem_u32(&b); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long num_tiles = p.n / TILE + (p.n % TILE != 0);
    const long long num_chunks = p.lb.num_tiles;
    const unsigned long long wait_limit = p.lb.timeout_ns + 500000000ull;
    const volatile int* end_k = &ctl->end_k;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSA; ++i) {
            mbar_init(B(ctl->a_full[i]), 1);
            mbar_init(B(ctl->a_empty[i]), kComputeWarps);
        }
        for (int i = 0; i < kSB; ++i) {
            mbar_init(B(ctl->b_full[i]), 1);
            mbar_init(B(ctl->b_empty[i]), kComputeWarps);
        }
        for (int i = 0; i < kR1; ++i) {
            mbar_init(B(ctl->p1done[i]), 1);
            mbar_init(B(ctl->wready[i]), kComputeWarps);
        }
        for (int i = 0; i < kChunkSlots; ++i) {
            mbar_init(B(ctl->agg[i]), 1);
            mbar_init(B(ctl->pre[i]), 1);
        }
        ctl->end_k = 0x7fffffff;
        ctl->consumed_a = -1;
        ctl->consumed_b = -1;
        fence_mbar_init();
    }
    __syncthreads();

    // ---------------------------------------------- producer A: fresh tiles
    if (warp == kProducerA) {
        if (lane != 0) return;
        unsigned long long* ctr = p.lb.counter;
        const unsigned long long base = p.lb.counter_base;
        unsigned long long a0 = atomicAdd(ctr, 1ull);  // chunk ids one chunk ahead of use
        const uint64_t keep_l2 = l2_policy_evict_last();
        int issued = -1;
        long long c = 0;
        for (int k = 0;; ++k) {
            const int s = k % kSA;
            if (k >= kSA && !bar_wait(B(ctl->a_empty[s]), ((k / kSA) - 1) & 1, wait_limit)) {
                raise_error(p.lb.error, DEV_LOOKBACK_TIMEOUT);
                break;
            }
            const int pos = k % kChunk;
            if (pos == 0) {
                c = (long long)(a0 - base);
                a0 = atomicAdd(ctr, 1ull);
            }
            const bool done = c >= num_chunks;
            const long long t = c * kChunk + pos;
            ctl->tile[k % kRing] = done ? kSentinel : (t < num_tiles ? (unsigned)t : kVoid);
            if (done) vstore(&ctl->end_k, k);
            issued = k;
            if (!done && t < n_full_tiles) {
                mbar_arrive_expect_tx(B(ctl->a_full[s]), kTileBytes);
                tma_load_2d_hint(stageA + s * kTileBytes, &tm_in, 0, (int)(t * kRows), B(ctl->a_full[s]), keep_l2);
            } else {
                mbar_arrive(B(ctl->a_full[s]));
            }
            if (done) break;
        }
        for (int k = vload(&ctl->consumed_a) + 1; k <= issued; ++k)
            bar_wait(B(ctl->a_full[k % kSA]), (k / kSA) & 1, wait_limit);
        asm volatile("" ::"l"(a0));
        return;
    }

    // ------------------------------------- producer B: re-loads for pass 2
    if (warp == kProducerB) {
        if (lane != 0) return;
        const uint64_t drop = l2_policy_evict_first();
        int issued = -1;
        for (int j = 0;; ++j) {
            const int s = j % kSB;
            if (*end_k <= j) break;
            if (j >= kSB && !bar_wait(B(ctl->b_empty[s]), ((j / kSB) - 1) & 1, wait_limit, end_k, j)) break;
            if (!bar_wait(B(ctl->p1done[j % kR1]), (j / kR1) & 1, wait_limit, end_k, j)) break;
            const unsigned tu = ctl->tile[j % kRing];
            issued = j;
            if (tu != kVoid && (long long)tu < n_full_tiles) {
                mbar_arrive_expect_tx(B(ctl->b_full[s]), kTileBytes);
                tma_load_2d_hint(stageB + s * kTileBytes, &tm_in, 0, (int)((long long)tu * kRows), B(ctl->b_full[s]),
                                 drop);
            } else {
                mbar_arrive(B(ctl->b_full[s]));
            }
        }
        for (int j = vload(&ctl->consumed_b) + 1; j <= issued; ++j)
            bar_wait(B(ctl->b_full[j % kSB]), (j / kSB) & 1, wait_limit);
        return;
    }

    // ------------------------------------------------------- bookkeeping
    if (warp == kBookWarp) {
        C run = CntOp::c_identity();
        for (int k = 0;; ++k) {
            if (!warp_bar_wait(B(ctl->wready[k % kR1]), (k / kR1) & 1, wait_limit, end_k, k)) break;
            const unsigned w = lane < kComputeWarps ? ctl->wcnt[k % kRing][lane] : 0u;
            const unsigned tcnt = __reduce_add_sync(0xffffffffu, w);
            const int pos = k % kChunk;
            if (pos == 0) run = CntOp::c_identity();
            if (lane == 0) {
                ctl->offset[k % kRing] = (unsigned long long)run;
                run = CntOp::c_op(run, CntOp::lift(tcnt));
                if (pos == kChunk - 1) {
                    const int q = k / kChunk;
                    const long long c = ((long long)ctl->tile[(k - pos) % kRing]) / kChunk;
                    ctl->chunk_agg[q % kChunkSlots] = (unsigned long long)run;
                    ctl->chunk_id[q % kChunkSlots] = c;
                    const bool stalled = p.lb.stall_tile >= 0 && p.lb.stall_tile / kChunk == c;
                    if (p.lb.delay_tile >= 0 && p.lb.delay_tile / kChunk == c) hook_delay(p.lb.delay_ns);
                    if (!stalled) StatusIO<C>::publish(p.lb, c, c == 0 ? ST_PREFIX : ST_AGGREGATE, run);
                    mbar_arrive(B(ctl->agg[q % kChunkSlots]));
                }
                mbar_arrive(B(ctl->p1done[k % kR1]));
            }
            run = __shfl_sync(0xffffffffu, run, 0);
        }
        return;
    }

    // ------------------------------------------------------------ look-back
    if (warp >= kComputeWarps) {
        const int lw = warp - kComputeWarps;
        for (int q = lw;; q += kLbWarps) {
            const int k0 = q * kChunk;
            if (!warp_bar_wait(B(ctl->agg[q % kChunkSlots]), (q / kChunkSlots) & 1, wait_limit, end_k, k0)) break;
            const long long c = ctl->chunk_id[q % kChunkSlots];
            C prefix = CntOp::c_identity();
            bool ok = true;
            if (c != 0) {
                ok = lookback_prefix_adaptive<CntOp, kLbPer>(p.lb, c, prefix);
                if (!ok && lane == 0) StatusIO<C>::publish(p.lb, c, ST_POISON, CntOp::c_identity());
            }
            if (lane == 0) {
                const C agg = (C)ctl->chunk_agg[q % kChunkSlots];
                const bool stalled = p.lb.stall_tile >= 0 && p.lb.stall_tile / kChunk == c;
                if (ok && c != 0 && !stalled) StatusIO<C>::publish(p.lb, c, ST_PREFIX, CntOp::c_op(prefix, agg));
                if (ok && c == num_chunks - 1) *p.count = (long long)CntOp::c_op(prefix, agg);
                ctl->chunk_prefix[q % kChunkSlots] = (unsigned long long)prefix;
                mbar_arrive(B(ctl->pre[q % kChunkSlots]));
            }
            __syncwarp();
        }
        return;
    }

    // -------------------------------------------------------------- compute
    const int ctid = threadIdx.x;
    bool ok = true;
    int pending = -1;  // stage whose bulk copy may still be reading (lane 0 of each warp)
    T* const out = static_cast<T*>(p.out);

    auto wait = [&](uint32_t b, uint32_t parity) {
        const bool good = warp_bar_wait(b, parity, wait_limit);
        if (!good) {
            if (lane == 0 && ok) raise_error(p.lb.error, DEV_LOOKBACK_TIMEOUT);
            ok = false;
        }
        return good;
    };
    // Lane 0: once the previous run's bulk copy has read the stage, free it.
    auto release_pending = [&]() {
        if (lane == 0 && pending >= 0) {
            bulk_wait_read_all();
            mbar_arrive(B(ctl->b_empty[pending]));
            pending = -1;
        }
    };

    // pass 1: kept elements in this warp's part of fresh tile k
    // (thread = kChunksPerThread 16-byte chunks of one row)
    const int p1_row = ctid / kThreadsPerRow;
    const int p1_c0 = (ctid % kThreadsPerRow) * kChunksPerThread;
    auto pass1 = [&](int k, int s, unsigned tu) {
        uint32_t mine = 0;  // this thread's flags, already at their bit positions in the row
        if (tu != kVoid) {
            const long long t = tu;
            if (t < n_full_tiles) {
                const uint32_t row = stageA + s * kTileBytes + p1_row * 128;
#pragma unroll
                for (int j = 0; j < kChunksPerThread; ++j) {
                    T e[4];
                    unpack(lds128(row + (((p1_c0 + j) ^ (p1_row & 7)) << 4)), e);
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        if (keep_elem(e[w], p.pred)) mine |= 1u << ((p1_c0 + j) * 4 + w);
                }
            } else {
                const long long first = t * TILE + (long long)ctid * kPerThread;
                const T* in = static_cast<const T*>(p.in) + first;
                const long long valid = p.n - first;
#pragma unroll 4
                for (int w = 0; w < kPerThread; ++w)
                    if (w < valid && keep_elem(in[w], p.pred)) mine |= 1u << (p1_c0 * 4 + w);
            }
        }
        uint32_t rowm = mine;
        if constexpr (kThreadsPerRow == 2) rowm |= __shfl_xor_sync(0xffffffffu, mine, 1);
        if (ctid % kThreadsPerRow == 0) ctl->rowmask[k % kMaskRing][p1_row] = rowm;
        const unsigned wsum = __reduce_add_sync(0xffffffffu, (unsigned)__popc(mine));
        if (lane == 0) ctl->wcnt[k % kRing][warp] = wsum;
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(B(ctl->a_empty[s]));
            mbar_arrive(B(ctl->wready[k % kR1]));
        }
    };

    // pass 2: pack this warp's kept elements of tile j in order and write them out.
    // Element ranks come from pass 1's row masks: rank = kept elements of the
    // warp's part before it.  Rank r goes to slot r - h of the warp's part of
    // the stage, where h (0..3) is the number of leading elements before the
    // first 16-byte boundary of the output run; those h go to the top slots
    // kW - h .. kW - 1 (slot (r - h) mod kW), which no other rank reaches since
    // ranks stay below kW.  Slots 0 .. mid - 1 then leave by one bulk copy,
    // the head and the tail (< 4 elements) by plain stores.
    constexpr int kSteps = kRowsPerWarp / 4;           // 4 rows (128 elements) per step
    constexpr unsigned kW = kRowsPerWarp * 32;         // slots (elements) of a warp's part
    const uint32_t q_c = lane & 7, q_r = lane >> 3;    // step lane: 16-byte chunk q_c of row 4g + q_r
    const uint32_t lowmask = (1u << (4 * q_c)) - 1u;   // elements of the row before the chunk
    // the chunk's place in shared memory, 128-byte swizzle term (4g + q_r) & 7
    const uint32_t ch_even = q_r * 128 + ((q_c ^ q_r) << 4);
    const uint32_t ch_odd = q_r * 128 + ((q_c ^ (q_r | 4u)) << 4);
    auto pass2 = [&](int j) {
        const int s = j % kSB;
        const int q = j / kChunk;
        const unsigned tu = ctl->tile[j % kRing];
        release_pending();
        if (tu == kVoid) {
            __syncwarp();
            if (lane == 0) mbar_arrive(B(ctl->b_empty[s]));
            return;
        }
        const long long t = tu;
        // output position of this warp's first kept element
        const unsigned wv = lane < kComputeWarps ? ctl->wcnt[j % kRing][lane] : 0u;
        unsigned incl = wv;
#pragma unroll
        for (int d = 1; d < kComputeWarps; d <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += y;
        }
        const unsigned wpre = warp > 0 ? __shfl_sync(0xffffffffu, incl, warp - 1) : 0u;
        const unsigned wcnt = __shfl_sync(0xffffffffu, wv, warp);
        const long long gw = (long long)(ctl->chunk_prefix[q % kChunkSlots] + ctl->offset[j % kRing]) + wpre;
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(out + gw);
        const unsigned h = min(wcnt, (unsigned)(((16u - (unsigned)(a0 & 15u)) & 15u) >> 2));
        const unsigned mid = (wcnt - h) & ~3u;
        const uint32_t region = stageB + s * kTileBytes + warp * kWarpBytes;
        // lane r < kRowsPerWarp: row r's mask and the rank (minus h) of its first kept element
        const uint32_t mr = lane < kRowsPerWarp ? ctl->rowmask[j % kMaskRing][warp * kRowsPerWarp + lane] : 0u;
        unsigned rin = __popc(mr);
#pragma unroll
        for (int d = 1; d < kRowsPerWarp; d <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, rin, d);
            if (lane >= d) rin += y;
        }
        const int rfirst = (int)(rin - __popc(mr)) - (int)h;
        if (t < n_full_tiles) {
            // every lane reads all its chunks before any lane writes: the
            // packing overwrites the part in place
            uint4 v[kSteps];
#pragma unroll
            for (int g = 0; g < kSteps; ++g) v[g] = lds128(region + g * 512 + ((g & 1) ? ch_odd : ch_even));
            __syncwarp();
#pragma unroll
            for (int g = 0; g < kSteps; ++g) {
                const int row = 4 * g + (int)q_r;
                const uint32_t m = __shfl_sync(0xffffffffu, mr, row);
                const int e = __shfl_sync(0xffffffffu, rfirst, row) + __popc(m & lowmask);
                const uint32_t nib = m >> (4 * q_c);
                if (e >= 0) {
                    const uint32_t a = region + 4u * (uint32_t)e;
                    if (nib & 1u) sts32(a, v[g].x);
                    if (nib & 2u) sts32(a + 4u * (nib & 1u), v[g].y);
                    if (nib & 4u) sts32(a + 4u * __popc(nib & 3u), v[g].z);
                    if (nib & 8u) sts32(a + 4u * __popc(nib & 7u), v[g].w);
                } else {  // holds some of the warp's first h kept elements
                    const uint32_t w4[4] = {v[g].x, v[g].y, v[g].z, v[g].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if ((nib >> i) & 1u)
                            sts32(region + 4u * ((uint32_t)(e + __popc(nib & ((1u << i) - 1u))) & (kW - 1u)), w4[i]);
                }
            }
        } else {  // the partial last tile: values from global memory, one row per step
            const uint32_t* in = static_cast<const uint32_t*>(p.in) + t * TILE + (long long)warp * kW;
            const uint32_t below = lanemask_lt();
            for (int jj = 0; jj < kRowsPerWarp; ++jj) {
                const uint32_t m = __shfl_sync(0xffffffffu, mr, jj);
                const int e = __shfl_sync(0xffffffffu, rfirst, jj) + __popc(m & below);
                if ((m >> lane) & 1u) sts32(region + 4u * ((uint32_t)e & (kW - 1u)), in[jj * 32 + lane]);
            }
        }
        fence_proxy_async();
        __syncwarp();
        const unsigned tail = wcnt - h - mid;  // < 4
        if (lane < h) out[gw + lane] = from_bits<T>(lds32(region + 4u * (kW - h + lane)));
        else if (lane >= 4 && lane - 4 < tail) out[gw + h + mid + (lane - 4)] = from_bits<T>(lds32(region + 4u * (mid + lane - 4)));
        if (lane == 0) {
            if (mid > 0) {
                bulk_s2g(out + gw + h, region, mid * 4);
                bulk_commit();
                pending = s;
            } else {
                mbar_arrive(B(ctl->b_empty[s]));
            }
        }
    };

    int k = 0;
    bool draining = true;
    for (;; ++k) {
        const int s = k % kSA;
        if (!wait(B(ctl->a_full[s]), (k / kSA) & 1)) { draining = false; break; }
        if (ctid == 0) vstore(&ctl->consumed_a, k);
        const unsigned tu = ctl->tile[k % kRing];
        if (tu == kSentinel) break;
        pass1(k, s, tu);
        const int j = k - kLag;
        if (j >= 0) {
            if (!wait(B(ctl->b_full[j % kSB]), (j / kSB) & 1)) { draining = false; break; }
            if (ctid == 0) vstore(&ctl->consumed_b, j);
            if (!wait(B(ctl->pre[(j / kChunk) % kChunkSlots]), ((j / kChunk) / kChunkSlots) & 1)) { draining = false; break; }
            pass2(j);
        }
    }
    if (draining)
        for (int j = (k > kLag ? k - kLag : 0); j < k; ++j) {
            if (!wait(B(ctl->b_full[j % kSB]), (j / kSB) & 1)) break;
            if (ctid == 0) vstore(&ctl->consumed_b, j);
            if (!wait(B(ctl->pre[(j / kChunk) % kChunkSlots]), ((j / kChunk) / kChunkSlots) & 1)) break;
            pass2(j);
        }
    if (lane == 0) bulk_wait_all();  // this warp's copies must finish before the CTA's shared memory is released
}

// ----------------------------------------------------------------- host side
namespace {

template <class T, class CntOp, int CW>
cudaError_t launch_ct(const CompactParams& p, unsigned grid, cudaStream_t s) {
    const long long nfull = p.n / TILE;
    CUtensorMap a;
    if (!make_map(&a, p.in, (unsigned long long)nfull * kRows, kRows)) return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> done_mask{0};
    const cudaError_t e = allow_smem(compact_tma_kernel<T, CntOp, CW>, kSmemBytes, done_mask);
    if (e != cudaSuccess) return e;
    compact_tma_kernel<T, CntOp, CW><<<grid, CompactShape<CW>::kThreads, kSmemBytes, s>>>(a, p, nfull);
    return cudaGetLastError();
}

}  // namespace

int compact_tma_tile_elems() { return TILE; }
int compact_tma_chunk_tiles() { return kChunk; }

// shape 0: 16 compute warps (the default, fastest measured), shape 1: 8 compute warps
template <class T>
cudaError_t launch_compact_tma(const CompactParams& p, bool wide_count, unsigned grid, cudaStream_t s, int shape) {
    if (shape == 0)
        return wide_count ? launch_ct<T, OpCountU64, 16>(p, grid, s) : launch_ct<T, OpCountU32, 16>(p, grid, s);
    if (shape == 1)
        return wide_count ? launch_ct<T, OpCountU64, 8>(p, grid, s) : launch_ct<T, OpCountU32, 8>(p, grid, s);
    return cudaErrorInvalidValue;
}

template cudaError_t launch_compact_tma<int32_t>(const CompactParams&, bool, unsigned, cudaStream_t, int);
template cudaError_t launch_compact_tma<uint32_t>(const CompactParams&, bool, unsigned, cudaStream_t, int);
template cudaError_t launch_compact_tma<float>(const CompactParams&, bool, unsigned, cudaStream_t, int);

}  // namespace scg
