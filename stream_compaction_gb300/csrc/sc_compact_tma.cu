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
//   producer A      chunk ids from the atomic counter, fresh tiles by TMA
//                   (kept in L2 for the re-load);
//   compute warps   pass 1 (tile k): each warp evaluates the predicate on its
//                   rows of the fresh tile and keeps, per 128-byte row, a
//                   32-bit flag mask and the rank of the row's first kept
//                   element within the warp's part; it counts its kept
//                   elements and frees the stage at once;
//                   pass 2 (tile k - kLag, re-loaded from L2 by producer B,
//                   run in the same instruction stream as pass 1 of tile k):
//                   each lane moves one 16-byte chunk per step and stores its
//                   kept elements to consecutive output slots; a warp's stores
//                   cover one contiguous run, which L2 merges into whole lines;
//   bookkeeping     tile and warp offsets within a chunk, chunk aggregates
//                   published;
//   look-back       chunk prefixes; the last chunk also writes the count;
//   producer B      the pass-2 re-loads.
//
// Each input element is read from HBM once (and once more from L2) and each
// kept element is written once.
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
constexpr int kStages = 6;              // 32 KiB stages: kSA for fresh tiles from HBM, the rest for the
                                        // pass-2 re-loads of the same tiles from L2 (a kernel parameter)
constexpr int kMaxSB = 4;               // most re-load stages of any split
constexpr int kChunk = 2;               // tiles per counter tick and per look-back status
constexpr int kMaxLag = 8;              // pass 2 of tile k follows pass 1 of tile k + lag (a kernel parameter)
constexpr int kLbWarps = 3;
constexpr int kChunkSlots = 6;
constexpr int kRing = 32;
constexpr int kR1 = 32;
constexpr int TILE = kTileBytes / 4;    // 8192 four-byte elements
constexpr int kLbPer = 8;
constexpr unsigned kSentinel = 0xffffffffu;
constexpr unsigned kVoid = 0xfffffffeu;
constexpr int kCtrlBytes = 30720;
constexpr int kSmemBytes = kStages * kTileBytes + 1024 + kCtrlBytes;
constexpr int kMaxComputeWarps = 16;
constexpr int kMaskRing = 12;           // tiles whose row information is kept (pass 1 -> pass 2)
static_assert(kMaskRing > kMaxLag, "row information outlives the lag");

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
static_assert(kR1 > kMaxLag, "pass-1-done ring covers the lag");
static_assert(kRing >= kStages + kMaxLag + 4, "tile ring outlives every reader");
static_assert(kChunkSlots * kChunk >= kMaxLag + 2 * kChunk, "chunk ring covers the lag");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

struct Ctrl {
    unsigned long long a_full[kStages], a_empty[kStages];   // the first kSA used
    unsigned long long b_full[kStages], b_empty[kStages];   // the first kSB used
    unsigned long long p1done[kR1], wready[kR1];
    unsigned long long agg[kChunkSlots], pre[kChunkSlots];
    // per row of a tile, from pass 1: the flag mask (one bit per element of the
    // 32-element row) and the rank of the row's first kept element within its
    // warp part
    uint2 rowinfo[kMaskRing][kRows];
    unsigned tile[kRing];
    unsigned wcnt[kRing][kMaxComputeWarps];  // kept elements per warp part, from pass 1
    unsigned woff[kRing][kMaxComputeWarps];  // kept elements of the chunk before each warp part
    unsigned long long chunk_agg[kChunkSlots], chunk_prefix[kChunkSlots];
    long long chunk_id[kChunkSlots];
    int end_k;
    int consumed_a;
    int consumed_b;
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

template <class T>
__device__ __forceinline__ T from_bits(uint32_t b) { T v; from_bits32(b, v); return v; }

}  // namespace

__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// kPack: pass 2 packs each warp's kept elements in its own part of the
// re-load stage and writes them out as aligned 16-byte stores (a comparison
// shape); otherwise every kept element is a 4-byte store of its own (the
// default: fewer instructions, and L2 merges the partial sectors), and a warp
// frees its re-load stage as soon as it has read its part into registers.
// kSA_: fresh-tile stages; the other kStages - kSA_ hold the re-loads.
// kLag_: pass 2 of tile k follows pass 1 of tile k + kLag_.
template <class T, class CntOp, int CW, bool kPack, int kSA_, int kLag_>
__global__ void __launch_bounds__(CompactShape<CW>::kThreads, 1)
    compact_tma_kernel(const __grid_constant__ CUtensorMap tm_in, const CompactParams p, const long long n_full_tiles) {
    constexpr int kSA = kSA_, kSB = kStages - kSA_, kLag = kLag_;
    static_assert(kSA >= 2 && kSB >= 2 && kSB <= kMaxSB, "stage split");
    static_assert(kLag <= kMaxLag && kLag >= kSB, "lag");
    static_assert(!kPack || kSB >= 3, "the packed stores keep their stage until the prefix arrives");
    using C = typename CntOp::C;
    using Sh = CompactShape<CW>;
    constexpr int kComputeWarps = Sh::kComputeWarps, kBookWarp = Sh::kBookWarp;
    constexpr int kProducerA = Sh::kProducerA, kProducerB = Sh::kProducerB;
    constexpr int kRowsPerWarp = Sh::kRowsPerWarp, kWarpBytes = Sh::kWarpBytes;
    constexpr int kThreadsPerRow = Sh::kThreadsPerRow, kChunksPerThread = Sh::kChunksPerThread;
    constexpr int kPerThread = kChunksPerThread * 4;  // pass-1 elements per thread
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + kStages * kTileBytes);
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
        ChunkIds ids{p.lb.counter, p.lb.counter_base, num_chunks, (long long)gridDim.x, p.lb.error};
        ids.start();  // chunk ids one chunk ahead of use, except near the end
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
            if (pos == 0) c = ids.take();
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
        unsigned run = 0;  // kept elements of the chunk's earlier tiles (at most kChunk * TILE)
        for (int k = 0;; ++k) {
            if (!warp_bar_wait(B(ctl->wready[k % kR1]), (k / kR1) & 1, wait_limit, end_k, k)) break;
            const unsigned w = lane < kComputeWarps ? ctl->wcnt[k % kRing][lane] : 0u;
            unsigned incl = w;
#pragma unroll
            for (int d = 1; d < kComputeWarps; d <<= 1) {
                const unsigned y = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += y;
            }
            const int pos = k % kChunk;
            if (pos == 0) run = 0;
            if (lane < kComputeWarps) ctl->woff[k % kRing][lane] = run + incl - w;
            run += __shfl_sync(0xffffffffu, incl, kComputeWarps - 1);
            __syncwarp();
            if (lane == 0) {
                if (pos == kChunk - 1) {
                    const int q = k / kChunk;
                    const long long c = ((long long)ctl->tile[(k - pos) % kRing]) / kChunk;
                    const C agg = CntOp::lift(run);
                    ctl->chunk_agg[q % kChunkSlots] = (unsigned long long)agg;
                    ctl->chunk_id[q % kChunkSlots] = c;
                    const bool stalled = p.lb.stall_tile >= 0 && p.lb.stall_tile / kChunk == c;
                    if (p.lb.delay_tile >= 0 && p.lb.delay_tile / kChunk == c) hook_delay(p.lb.delay_ns);
                    if (!stalled) StatusIO<C>::publish(p.lb, c, c == 0 ? ST_PREFIX : ST_AGGREGATE, agg);
                    mbar_arrive(B(ctl->agg[q % kChunkSlots]));
                }
                mbar_arrive(B(ctl->p1done[k % kR1]));
            }
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
    T* const out = static_cast<T*>(p.out);

    auto wait = [&](uint32_t b, uint32_t parity) {
        const bool good = warp_bar_wait(b, parity, wait_limit);
        if (!good) {
            if (lane == 0 && ok) raise_error(p.lb.error, DEV_LOOKBACK_TIMEOUT);
            ok = false;
        }
        return good;
    };

    // pass 1 (tile k, fresh from HBM): thread = kChunksPerThread 16-byte chunks
    // of one row; flags land at their bit positions in the row's mask
    const int p1_row = ctid / kThreadsPerRow;
    const int p1_c0 = (ctid % kThreadsPerRow) * kChunksPerThread;
    auto p1_flags = [&](int s) {
        const uint32_t row = stageA + s * kTileBytes + p1_row * 128;
        uint4 raw[kChunksPerThread];
#pragma unroll
        for (int c = 0; c < kChunksPerThread; ++c) raw[c] = lds128(row + (((p1_c0 + c) ^ (p1_row & 7)) << 4));
        uint32_t mine = 0;
#pragma unroll
        for (int c = 0; c < kChunksPerThread; ++c) {
            T e[4];
            unpack(raw[c], e);
#pragma unroll
            for (int w = 0; w < 4; ++w)
                if (keep_elem(e[w], p.pred)) mine |= 1u << ((p1_c0 + c) * 4 + w);
        }
        return mine;
    };
    auto p1_flags_partial = [&](long long t) {  // the last, partial tile: from global memory
        const long long first = t * TILE + (long long)ctid * kPerThread;
        const T* in = static_cast<const T*>(p.in) + first;
        const long long valid = p.n - first;
        uint32_t mine = 0;
#pragma unroll 4
        for (int w = 0; w < kPerThread; ++w)
            if (w < valid && keep_elem(in[w], p.pred)) mine |= 1u << (p1_c0 * 4 + w);
        return mine;
    };
    // row masks with the rank of each row's first kept element, and the warp's count
    auto p1_publish = [&](int k, uint32_t mine) {
        const unsigned cnt = __popc(mine);
        unsigned incl = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += y;
        }
        uint32_t rowm = mine;
        if constexpr (kThreadsPerRow == 2) rowm |= __shfl_xor_sync(0xffffffffu, mine, 1);
        if (ctid % kThreadsPerRow == 0) ctl->rowinfo[k % kMaskRing][p1_row] = make_uint2(rowm, incl - cnt);
        if (lane == 31) ctl->wcnt[k % kRing][warp] = incl;
    };

    // pass 2 (tile j, re-loaded from L2): write this warp's kept elements to
    // their output slots.  Each lane moves one 16-byte chunk per step and stores
    // its kept elements to consecutive slots; a warp's stores cover one
    // contiguous run, which L2 merges into whole lines.
    constexpr int kSteps = kRowsPerWarp / 4;           // 4 rows (128 elements) per step
    const uint32_t q_c = lane & 7, q_r = lane >> 3;    // step lane: 16-byte chunk q_c of row 4g + q_r
    const uint32_t lowmask = (1u << (4 * q_c)) - 1u;   // elements of the row before the chunk
    // the chunk's place in shared memory, 128-byte swizzle term (4g + q_r) & 7
    const uint32_t ch_even = q_r * 128 + ((q_c ^ q_r) << 4);
    const uint32_t ch_odd = q_r * 128 + ((q_c ^ (q_r | 4u)) << 4);
    auto p2_load = [&](int j, uint4 (&v)[kSteps]) {
        const uint32_t part = stageB + (j % kSB) * kTileBytes + warp * kWarpBytes;
#pragma unroll
        for (int g = 0; g < kSteps; ++g) v[g] = lds128(part + g * 512 + ((g & 1) ? ch_odd : ch_even));
    };
    auto p2_out = [&](int j) {  // output slot of the warp part's first kept element
        return out + (long long)(ctl->chunk_prefix[(j / kChunk) % kChunkSlots] + ctl->woff[j % kRing][warp]);
    };
    // row information of each step's row (read before any store, so that no
    // shared-memory load waits behind a global store)
    auto p2_rows = [&](int j, uint2 (&r)[kSteps]) {
        const uint2* ri = &ctl->rowinfo[j % kMaskRing][warp * kRowsPerWarp + q_r];
#pragma unroll
        for (int g = 0; g < kSteps; ++g) r[g] = ri[4 * g];
    };
    auto p2_store_direct = [&](const uint4 (&v)[kSteps], const uint2 (&r)[kSteps], T* wout) {
#pragma unroll
        for (int g = 0; g < kSteps; ++g) {
            const uint32_t nib = r[g].x >> (4 * q_c);
            T* const o = wout + (r[g].y + __popc(r[g].x & lowmask));
            if (nib & 1u) o[0] = from_bits<T>(v[g].x);
            if (nib & 2u) o[nib & 1u] = from_bits<T>(v[g].y);
            if (nib & 4u) o[__popc(nib & 3u)] = from_bits<T>(v[g].z);
            if (nib & 8u) o[__popc(nib & 7u)] = from_bits<T>(v[g].w);
        }
    };
    // Packed form.  The warp's kept elements form one output run [S, S + K);
    // in 16-byte-aligned coordinates (Q = position + o0, o0 = the output's
    // misalignment in elements) that is [Q0, Q0 + K).  Each kept element is
    // written to slot Q mod kSlots of the warp's own part of the re-load stage
    // (already read into registers; K <= kSlots, so no two share a slot, and
    // the four slots of an aligned group are one aligned 16-byte word); then
    // lane l moves groups Q0/4 + l, Q0/4 + l + 32, ...: a full group is one
    // 16-byte store, the two partial end groups store only their elements of
    // the run (the rest of those groups belongs to the neighbouring runs).
    constexpr uint32_t kSlots = kWarpBytes / 4;
    static_assert((kSlots & (kSlots - 1)) == 0, "slot ring is a power of two");
    const uint32_t o0 = (uint32_t)((reinterpret_cast<uintptr_t>(out) >> 2) & 3u);
    auto p2_store_packed = [&](int j, const uint4 (&v)[kSteps], const uint2 (&r)[kSteps]) {
        const uint32_t part = stageB + (j % kSB) * kTileBytes + warp * kWarpBytes;
        const long long Q0 =
            (long long)(ctl->chunk_prefix[(j / kChunk) % kChunkSlots] + ctl->woff[j % kRing][warp]) + o0;
        const long long Qend = Q0 + ctl->wcnt[j % kRing][warp];
        const uint32_t qlo = (uint32_t)Q0;
        __syncwarp();  // every lane has read its chunks of the part before any slot is overwritten
#pragma unroll
        for (int g = 0; g < kSteps; ++g) {
            const uint32_t nib = r[g].x >> (4 * q_c);
            const uint32_t q = qlo + r[g].y + __popc(r[g].x & lowmask);
            if (nib & 1u) sts32(part + ((q & (kSlots - 1)) << 2), v[g].x);
            if (nib & 2u) sts32(part + (((q + (nib & 1u)) & (kSlots - 1)) << 2), v[g].y);
            if (nib & 4u) sts32(part + (((q + __popc(nib & 3u)) & (kSlots - 1)) << 2), v[g].z);
            if (nib & 8u) sts32(part + (((q + __popc(nib & 7u)) & (kSlots - 1)) << 2), v[g].w);
        }
        __syncwarp();  // every slot written before any lane reads a group
        T* const obase = out - o0;  // 16-byte aligned; indexed only at positions q >= Q0 >= o0
        for (long long A = (Q0 >> 2) + lane; 4 * A < Qend; A += 32) {
            const long long q = 4 * A;
            const uint4 w = lds128(part + (((uint32_t)q & (kSlots - 1)) << 2));
            if (q >= Q0 && q + 4 <= Qend) {
                *reinterpret_cast<uint4*>(obase + q) = w;
            } else {
                if (q >= Q0 && q < Qend) obase[q] = from_bits<T>(w.x);
                if (q + 1 >= Q0 && q + 1 < Qend) obase[q + 1] = from_bits<T>(w.y);
                if (q + 2 >= Q0 && q + 2 < Qend) obase[q + 2] = from_bits<T>(w.z);
                if (q + 3 >= Q0 && q + 3 < Qend) obase[q + 3] = from_bits<T>(w.w);
            }
        }
        fence_proxy_async();  // these shared-memory accesses come before the stage's next TMA fill
    };
    auto p2_store = [&](int j, const uint4 (&v)[kSteps], const uint2 (&r)[kSteps]) {
        if constexpr (kPack) p2_store_packed(j, v, r);
        else p2_store_direct(v, r, p2_out(j));
    };
    // Direct stores: the warp's part of a full re-loaded tile is in registers
    // after p2_load, so the stage is freed at once (producer B can re-load into
    // it while this warp waits for the prefix and stores).
    auto release_b = [&](int j) {
        if constexpr (!kPack) {
            __syncwarp();
            if (lane == 0) mbar_arrive(B(ctl->b_empty[j % kSB]));
        }
    };

    // general forms (first kLag tiles, the partial tile, void tiles, the drain)
    auto pass1 = [&](int k, int s, unsigned tu) {
        uint32_t mine = 0;
        if (tu != kVoid) mine = (long long)tu < n_full_tiles ? p1_flags(s) : p1_flags_partial((long long)tu);
        p1_publish(k, mine);
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(B(ctl->a_empty[s]));
            mbar_arrive(B(ctl->wready[k % kR1]));
        }
    };
    auto pass2 = [&](int j) {
        const unsigned tu = ctl->tile[j % kRing];
        if (tu != kVoid) {
            T* const wout = p2_out(j);
            const long long t = tu;
            if (t < n_full_tiles) {
                uint4 v[kSteps];
                uint2 r[kSteps];
                p2_load(j, v);
                p2_rows(j, r);
                release_b(j);
                p2_store(j, v, r);
            } else {
                const T* in = static_cast<const T*>(p.in) + t * TILE + (long long)warp * (kRowsPerWarp * 32);
                const uint2* ri = &ctl->rowinfo[j % kMaskRing][warp * kRowsPerWarp];
                const uint32_t below = lanemask_lt();
                for (int jj = 0; jj < kRowsPerWarp; ++jj) {
                    const uint2 r = ri[jj];
                    if ((r.x >> lane) & 1u) wout[r.y + __popc(r.x & below)] = in[jj * 32 + lane];
                }
            }
        }
        __syncwarp();
        if (lane == 0 && (kPack || tu == kVoid || (long long)tu >= n_full_tiles)) mbar_arrive(B(ctl->b_empty[j % kSB]));
    };
    const auto pre_bar = [&](int j) { return B(ctl->pre[(j / kChunk) % kChunkSlots]); };
    const auto pre_par = [&](int j) { return (uint32_t)(((j / kChunk) / kChunkSlots) & 1); };

    int k = 0;
    bool draining = true;
    for (;; ++k) {
        const int s = k % kSA;
        if (!wait(B(ctl->a_full[s]), (k / kSA) & 1)) { draining = false; break; }
        if (ctid == 0) vstore(&ctl->consumed_a, k);
        const unsigned tu = ctl->tile[k % kRing];
        if (tu == kSentinel) break;
        const int j = k - kLag;
        if (j < 0) {
            pass1(k, s, tu);
            continue;
        }
        if (!wait(B(ctl->b_full[j % kSB]), (j / kSB) & 1)) { draining = false; break; }
        if (ctid == 0) vstore(&ctl->consumed_b, j);
        const unsigned tj = ctl->tile[j % kRing];
        if ((long long)tu < n_full_tiles && (long long)tj < n_full_tiles) {
            // the common case, both tiles full, in one instruction stream: pass
            // 2's loads first, so that their latency hides behind pass 1's
            // arithmetic; pass 1 never waits for a prefix, so this CTA's chunk
            // aggregates (which other chunks' look-backs wait for) are not held up
            uint4 v[kSteps];
            uint2 r[kSteps];
            p2_load(j, v);
            p2_rows(j, r);
            release_b(j);
            p1_publish(k, p1_flags(s));
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(B(ctl->wready[k % kR1]));
                mbar_arrive(B(ctl->a_empty[s]));
            }
            if (!wait(pre_bar(j), pre_par(j))) { draining = false; break; }
            p2_store(j, v, r);
            __syncwarp();
            if (kPack && lane == 0) mbar_arrive(B(ctl->b_empty[j % kSB]));
        } else {
            pass1(k, s, tu);
            if (!wait(pre_bar(j), pre_par(j))) { draining = false; break; }
            pass2(j);
        }
    }
    if (draining)
        for (int j = (k > kLag ? k - kLag : 0); j < k; ++j) {
            if (!wait(B(ctl->b_full[j % kSB]), (j / kSB) & 1)) break;
            if (ctid == 0) vstore(&ctl->consumed_b, j);
            if (!wait(pre_bar(j), pre_par(j))) break;
            pass2(j);
        }
}

// ----------------------------------------------------------------- host side
namespace {

template <class T, class CntOp, int CW, bool kPack, int SA, int Lag>
cudaError_t launch_ct(const CompactParams& p, unsigned grid, cudaStream_t s) {
    const long long nfull = p.n / TILE;
    CUtensorMap a;
    if (!make_map(&a, p.in, (unsigned long long)nfull * kRows, kRows)) return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> done_mask{0};
    const cudaError_t e = allow_smem(compact_tma_kernel<T, CntOp, CW, kPack, SA, Lag>, kSmemBytes, done_mask);
    if (e != cudaSuccess) return e;
    compact_tma_kernel<T, CntOp, CW, kPack, SA, Lag><<<grid, CompactShape<CW>::kThreads, kSmemBytes, s>>>(a, p, nfull);
    return cudaGetLastError();
}

template <class T, int CW, bool kPack, int SA, int Lag = kMaxLag>
cudaError_t launch_ct_count(const CompactParams& p, bool wide_count, unsigned grid, cudaStream_t s) {
    return wide_count ? launch_ct<T, OpCountU64, CW, kPack, SA, Lag>(p, grid, s)
                      : launch_ct<T, OpCountU32, CW, kPack, SA, Lag>(p, grid, s);
}

}  // namespace

int compact_tma_tile_elems() { return TILE; }
int compact_tma_chunk_tiles() { return kChunk; }

// shape 0: 8 compute warps, one 4-byte store per kept element (the default,
// fastest measured); shape 1: 16 compute warps, the same stores; shape 2: 8
// compute warps, kept elements packed into aligned 16-byte stores (measured on
// GB300 at 2^27 int32, x > 0: store sectors 33.8 M -> 9.0 M, but 76 M -> 104 M
// instructions and 171 -> 189 us: the compute warps' instruction stream, not
// the store path, bounds this kernel); shapes 3 and 4: as shape 0 with 4
// fresh-tile and 2 re-load stages, or 2 and 4; shapes 5 and 6: as shape 0
// with a pass-2 lag of 6 or 4 tiles instead of 8
template <class T>
cudaError_t launch_compact_tma(const CompactParams& p, bool wide_count, unsigned grid, cudaStream_t s, int shape) {
    if (shape == 0) return launch_ct_count<T, 8, false, 3>(p, wide_count, grid, s);
    if (shape == 1) return launch_ct_count<T, 16, false, 3>(p, wide_count, grid, s);
    if (shape == 2) return launch_ct_count<T, 8, true, 3>(p, wide_count, grid, s);
    if (shape == 3) return launch_ct_count<T, 8, false, 4>(p, wide_count, grid, s);
    if (shape == 4) return launch_ct_count<T, 8, false, 2>(p, wide_count, grid, s);
    if (shape == 5) return launch_ct_count<T, 8, false, 3, 6>(p, wide_count, grid, s);
    if (shape == 6) return launch_ct_count<T, 8, false, 3, 4>(p, wide_count, grid, s);
    return cudaErrorInvalidValue;
}

template cudaError_t launch_compact_tma<int32_t>(const CompactParams&, bool, unsigned, cudaStream_t, int);
template cudaError_t launch_compact_tma<uint32_t>(const CompactParams&, bool, unsigned, cudaStream_t, int);
template cudaError_t launch_compact_tma<float>(const CompactParams&, bool, unsigned, cudaStream_t, int);

}  // namespace scg
