// Persistent, warp-specialised single-pass scan (the default path for
// 16-byte-aligned arrays of more than 2^22 elements).  The kernel and its
// launch helpers; sc_scan_tma.cu instantiates it for the first operators,
// sc_ops_*.cu for the others.
//
// Why: measured on GB300, a tile's decoupled look-back takes several
// microseconds under full HBM load (each status probe is an L2 round trip of
// about 1 us, and predecessors are often not yet published), which is most of
// a one-tile-per-CTA kernel's lifetime; the CTA holds its registers the whole
// time, so too few loads are in flight.  Here one CTA per SM keeps rings of
// shared-memory stages filled by TMA and takes the look-back off the critical
// path:
//
//   producer A       chunk ids (kChunk tiles each) from the atomic counter,
//                    requested one chunk ahead -> 2-D TMA loads (128-byte
//                    swizzle, L2 evict-last) of fresh tiles into ring A;
//   compute warps    pass 1 of fresh tile k: each warp's total of its part,
//                    the stage freed at once;
//                    pass 2 of tile j = k - kLag, re-loaded from L2 into ring
//                    B: serial register scan, warp shuffle scan, combine with
//                    the earlier warps' totals and the tile's prefix (for
//                    costly operators: the carry first, from thread totals
//                    kept from pass 1, then one serial scan seeded with it),
//                    results written back to the stage; both passes in one
//                    instruction stream;
//   bookkeeping      per tile: its total and its offset in the chunk; per
//                    chunk: the aggregate, published for later look-backs;
//   look-back warps  once a chunk's aggregate is published, its decoupled
//                    look-back (chunks round-robin over the warps); publishes
//                    the chunk's inclusive prefix and hands the exclusive one
//                    to the compute warps;
//   producer B       the pass-2 re-loads (L2 evict-first);
//   store warps      TMA store of each finished stage (evict-first), then
//                    the stage is freed.
//
// Each element is read from HBM once (and once more from L2) and written once.
// Scan definitions as in "Lecture 7: Parallel pattern -- prefix sum / scan"
// (UIUC ECE408 notes), section 1; the single-kernel look-back is the
// alternative that section 6 of the same notes names for the hierarchical
// design.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "sc_device.cuh"
#include "sc_launch.h"
#include "sc_scan.cuh"
#include "sc_persist.cuh"
#include "sc_tma.cuh"

namespace scg {

namespace {

using namespace persist;

// Shape of the persistent kernel: tile bytes, fresh / re-load ring depths,
// compute warps, pass-1 to pass-2 lag (tiles) and tiles per chunk.
// P1First: each compute iteration finishes pass 1 of its fresh tile (reads,
// warp totals published, stage freed) before it waits for the pass-2 tile and
// its prefix, so chunk aggregates never wait behind an older chunk's prefix
// (otherwise both tiles' reads come first and the two scan chains interleave).
// LbWarps: look-back warps; MinBlocks: CTAs resident per SM (each then gets
// its share of the SM's shared memory and registers).
template <int TileBytes, int SA, int SB, int CW, int Lag, int Chunk, bool P1First = false, int LbWarps = 3,
          int MinBlocks = 1>
struct TmaCfg {
    static constexpr bool kP1First = P1First;
    // counter ticks per CTA beyond the chunks: the id that ends its loop (see
    // ChunkIds); the host advances the counter's base by exactly this
    static constexpr int kIdsPerCta = 1;
    static constexpr int kMinBlocks = MinBlocks;
    static constexpr int kTileBytes = TileBytes;  // rows of 128 bytes
    static constexpr int kSA = SA;                // pass-1 stages: fresh tiles from HBM
    static constexpr int kSB = SB;                // pass-2 stages: the same tiles again, from L2
    static constexpr int kChunk = Chunk;          // tiles per counter tick and per look-back status
    static constexpr int kLag = Lag;              // pass 2 of tile k follows pass 1 of tile k + kLag
    static constexpr int kComputeWarps = CW;
    // chunk bookkeeping ring: covers the lag, a multiple of the look-back warps
    static constexpr int kChunkSlots =
        ((((Lag + 2 * Chunk + Chunk - 1) / Chunk > 6 ? (Lag + 2 * Chunk + Chunk - 1) / Chunk : 6) + LbWarps - 1) /
         LbWarps) * LbWarps;
    static constexpr int kRing = 64;              // per-tile bookkeeping ring
    static constexpr int kR1 = 32;                // pass-1-done barrier ring
    static constexpr int kLbWarps = LbWarps;
    static constexpr int kStoreWarps = SB % 2 == 0 ? 2 : 1;
    static constexpr int kBookWarp = kComputeWarps + kLbWarps;
    static constexpr int kProducerA = kBookWarp + 1;
    static constexpr int kProducerB = kProducerA + 1;
    static constexpr int kStoreWarp0 = kProducerB + 1;
    static constexpr int kThreads = 32 * (kStoreWarp0 + kStoreWarps);
    static constexpr int kCompute = 32 * kComputeWarps;
    static constexpr int kRows = kTileBytes / 128;
    static constexpr int kBytesPerThread = kTileBytes / kCompute;
    static constexpr int kThreadsPerRow = 128 / kBytesPerThread;
    // control block: 16 KiB, or what the stages leave of the CTA's share of
    // shared memory (227 KiB for one CTA per SM; 228 KiB less 1 KiB reserved
    // per CTA, shared, for more)
    static constexpr int kSmemCap = MinBlocks == 1 ? 232448 : 233472 / MinBlocks - 1024;
    static constexpr int kCtrlBytes =
        (kSA + kSB) * kTileBytes + 1024 + 16384 <= kSmemCap ? 16384 : (kSmemCap - 1024 - (kSA + kSB) * kTileBytes) / 128 * 128;
    static constexpr int kSmemBytes = (kSA + kSB) * kTileBytes + 1024 + kCtrlBytes;

    // Parity waits on an mbarrier are exact only if the waiter is at most one
    // phase behind.  Each ring below is waited on in order by one thread or
    // warp (or by warps that always own the same slots), and its producer
    // cannot run a full ring ahead of its consumer; these constraints keep
    // that true.
    static_assert(kChunkSlots % kLbWarps == 0, "a look-back warp owns fixed chunk slots");
    static_assert(kSB % kStoreWarps == 0, "a store warp owns fixed pass-2 stages");
    static_assert(kR1 > kLag && kLag >= kSB, "pass-1-done ring covers the lag");
    static_assert(kRing >= kSA + kLag + kSB + 4, "tile ring outlives every reader");
    static_assert(kChunkSlots * kChunk >= kLag + 2 * kChunk, "chunk ring covers the lag");
    static_assert(kBytesPerThread % 16 == 0 && kBytesPerThread <= 128, "16-byte chunks within one row");
    static_assert(kRows <= 256, "one TMA box per stage");
    static_assert(kSmemBytes <= kSmemCap, "shared memory per CTA");

    struct Ctrl {
        unsigned long long a_full[kSA], a_empty[kSA];
        unsigned long long b_full[kSB], b_empty[kSB], written[kSB];
        unsigned long long p1done[kR1];
        unsigned long long wready[kR1];                   // all compute warps wrote their pass-1 totals
        unsigned long long agg[kChunkSlots], pre[kChunkSlots];
        unsigned tile[kRing];
        unsigned seg_r[kRing];                            // batched rows: the tile's first index mod the row length
        unsigned long long offset[kRing];                 // carry-typed: fold of the chunk's earlier tiles
        unsigned long long wtot[kRing][kComputeWarps];    // element-typed warp totals from pass 1
        unsigned long long chunk_agg[kChunkSlots], chunk_prefix[kChunkSlots];
        long long chunk_id[kChunkSlots];
        int ok;
        int end_k;                                        // iteration that carried the end-of-work sentinel
        int consumed_a;                                   // last pass-1 fill the compute warps waited for
        int consumed_b;                                   // last pass-2 fill the compute warps waited for
    };
    static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");
};

// The shapes compiled in.  0 is the default of every operator but the
// float32 sum (32 KiB tiles, 3 + 3 stages, 8 compute warps, pass-2 lag of 5
// tiles, 2-tile chunks, pass 1 first: the fastest of the shapes measured on
// GB300 for uint32 sums of 2^27-2^30 elements, with look-back statuses in
// lines of their own); the others are uint32-sum variants kept for on-GPU
// comparison.  The float32 sum's look-back (float-float statuses) takes
// longer, so its default waits one tile more before pass 2 (CfgSumF32:
// measured at 2^26 / 2^27 / 2^28 elements 0.76 / 0.83 / 0.87 of the copy peak
// at lag 5, 0.79 / 0.85 / 0.89 at lag 6, 0.79 / 0.86 / 0.89 at lag 7 (on the
// final code: lag 7 +1 % at 2^26, -1.2 % at 2^28 against lag 6; lag 6 without
// pass 1 first -1 %), 0.77 / 0.81 / 0.83 at lag 8; the uint32 sum at lag 6:
// 0.85 / 0.90 / 0.93 against 0.84 / 0.91 / 0.96 at lag 5).
using Cfg0 = TmaCfg<32768, 3, 3, 8, 5, 2, true>;
using Cfg1 = TmaCfg<16384, 6, 6, 16, 12, 4>;
using Cfg2 = TmaCfg<32768, 3, 3, 16, 6, 2>;
using Cfg3 = TmaCfg<16384, 6, 6, 8, 12, 4>;
using Cfg4 = TmaCfg<32768, 3, 3, 8, 8, 2>;
// the former default (lag 6, both tiles' reads first), pass 1 first at lag 6,
// 16 compute warps, 1-tile chunks
using Cfg5 = TmaCfg<32768, 3, 3, 8, 6, 2>;
using Cfg6 = TmaCfg<32768, 3, 3, 8, 6, 2, true>;
using Cfg7 = TmaCfg<32768, 3, 3, 16, 6, 2, true>;
using Cfg8 = TmaCfg<32768, 3, 3, 8, 6, 1>;
using Cfg9 = TmaCfg<32768, 3, 3, 16, 5, 2, true>;
using CfgSumF32 = TmaCfg<32768, 3, 3, 8, 6, 2, true>;
// The default shape of an operator (same tile, chunk and thread count as Cfg0,
// which the host sizes launches by).
template <class Op> struct DefaultCfg { using type = Cfg0; };
template <> struct DefaultCfg<OpSumF32> { using type = CfgSumF32; };
static_assert(CfgSumF32::kTileBytes == Cfg0::kTileBytes && CfgSumF32::kChunk == Cfg0::kChunk &&
                  CfgSumF32::kThreads == Cfg0::kThreads && CfgSumF32::kSmemBytes == Cfg0::kSmemBytes,
              "the host sizes every default launch by Cfg0");
constexpr int kNumCfgs = 10;

// For operators with costly combines, pass 1 keeps each compute thread's
// total of a tile in shared memory for pass 2 (kLag + 2 tiles deep) where the
// shape leaves room for it; pass 2 then needs one combine per element instead
// of two.  Measured on GB300: float64 sum 531 -> 413 us and float32 max
// 144 -> 122 us (2^26); for cheap integer operators it cost 1-1.5 %, so they
// keep the two-combine form.
template <class Op, class Cfg>
struct ThreadTotals {
    static constexpr int kSlots = Cfg::kLag + 2;
    static constexpr int kBytes = kSlots * Cfg::kCompute * (int)sizeof(typename Op::T);
    static constexpr bool kKeep = HeavyCombine<Op>::value && Cfg::kSmemBytes + kBytes <= 232448;
    static constexpr int kSmemBytes = Cfg::kSmemBytes + (kKeep ? kBytes : 0);
};

constexpr int kLbPer = 8;               // at most 8 status words per lane: 256-chunk windows
constexpr unsigned kSentinel = 0xffffffffu;  // end of work
constexpr unsigned kVoid = 0xfffffffeu;      // past the last tile, inside the last chunk


}  // namespace

// Instrumented builds (kStats) add to 8 counters: [0] tiles, [1] ns the compute
// warps waited for fresh tiles, [2] ns they waited for chunk prefixes or
// re-loaded tiles, [3] ns in look-backs, [4] look-back windows read,
// [5] look-back polls that found a predecessor not yet published, [6] ns
// look-back warps waited for chunk aggregates, [7] ns the fresh-tile producer
// waited for a free stage.
template <class Op, bool kExcl, bool kStats, class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, Cfg::kMinBlocks)
    scan_tma_kernel(const __grid_constant__ CUtensorMap tm_in, const __grid_constant__ CUtensorMap tm_out,
                    const ScanParams p, const long long n_full_tiles) {
    using T = typename Op::T;
    using C = typename Op::C;
    using Ctrl = typename Cfg::Ctrl;
    constexpr int kTileBytes = Cfg::kTileBytes, kSA = Cfg::kSA, kSB = Cfg::kSB, kChunk = Cfg::kChunk;
    constexpr int kLag = Cfg::kLag, kComputeWarps = Cfg::kComputeWarps, kChunkSlots = Cfg::kChunkSlots;
    constexpr int kRing = Cfg::kRing, kR1 = Cfg::kR1, kLbWarps = Cfg::kLbWarps, kStoreWarps = Cfg::kStoreWarps;
    constexpr int kBookWarp = Cfg::kBookWarp, kProducerA = Cfg::kProducerA, kProducerB = Cfg::kProducerB;
    constexpr int kStoreWarp0 = Cfg::kStoreWarp0, kCompute = Cfg::kCompute, kRows = Cfg::kRows;
    constexpr int kBytesPerThread = Cfg::kBytesPerThread, kThreadsPerRow = Cfg::kThreadsPerRow;
    constexpr int IPT = kBytesPerThread / sizeof(T);
    constexpr int TILE = kCompute * IPT;
    constexpr int NV = kBytesPerThread / 16;  // 16-byte chunks per compute thread
    using TT = ThreadTotals<Op, Cfg>;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + (kSA + kSB) * kTileBytes);
    // each compute thread's pass-1 total, kept for its pass 2 (TT::kSlots tiles)
    T* ttot = reinterpret_cast<T*>(smem + (kSA + kSB) * kTileBytes + Cfg::kCtrlBytes);
    const uint32_t stageA = smem_u32(smem);
    const uint32_t stageB = stageA + kSA * kTileBytes;
    auto B = [](const unsigned long long& b) { return smem_u32(&b); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long num_tiles = p.n / TILE + (p.n % TILE != 0);
    const long long num_chunks = p.lb.num_tiles;  // the look-back runs over chunks
    const unsigned long long wait_limit = p.lb.timeout_ns + 500000000ull;
    unsigned long long* st = p.lb.stats;
    const volatile int* end_k = &ctl->end_k;
    if (threadIdx.x == 0) {  // fetch both tensor maps while the barriers are set up
        prefetch_tensormap(&tm_in);
        prefetch_tensormap(&tm_out);
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSA; ++i) {
            mbar_init(B(ctl->a_full[i]), 1);
            mbar_init(B(ctl->a_empty[i]), kComputeWarps);  // every compute warp has read the stage
        }
        for (int i = 0; i < kSB; ++i) {
            mbar_init(B(ctl->b_full[i]), 1);
            mbar_init(B(ctl->b_empty[i]), 1);
            mbar_init(B(ctl->written[i]), kComputeWarps);  // one arrival per compute warp
        }
        for (int i = 0; i < kR1; ++i) {
            mbar_init(B(ctl->p1done[i]), 1);
            mbar_init(B(ctl->wready[i]), kComputeWarps);
        }
        for (int i = 0; i < kChunkSlots; ++i) { mbar_init(B(ctl->agg[i]), 1); mbar_init(B(ctl->pre[i]), 1); }
        ctl->ok = 1;
        ctl->end_k = 0x7fffffff;
        ctl->consumed_a = -1;
        ctl->consumed_b = -1;
        fence_mbar_init();
    }
    __syncthreads();

    // ---------------------------------------------- producer A: fresh tiles
    if (warp == kProducerA) {
        if (lane != 0) return;
        // chunk ids requested one chunk ahead of use (except near the end):
        // early enough to hide the atomic's latency, late enough that chunks
        // are published in about the order in which they were handed out
        ChunkIds ids{p.lb.counter, p.lb.counter_base, num_chunks, (long long)gridDim.x, p.lb.error};
        ids.start();
        // fresh tiles stay in L2 until their pass-2 re-load
        const uint64_t keep = l2_policy_evict_last();
        int issued = -1;
        long long c = 0;
        unsigned long long waited = 0;
        for (int k = 0;; ++k) {
            const int s = k % kSA;
            if (k >= kSA) {
                const unsigned long long w0 = kStats ? global_ns() : 0;
                if (!bar_wait(B(ctl->a_empty[s]), ((k / kSA) - 1) & 1, wait_limit)) {
                    raise_error(p.lb.error, DEV_LOOKBACK_TIMEOUT);
                    break;
                }
                if (kStats) waited += global_ns() - w0;
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
                tma_load_2d_hint(stageA + s * kTileBytes, &tm_in, 0, (int)(t * kRows), B(ctl->a_full[s]), keep);
            } else {
                mbar_arrive(B(ctl->a_full[s]));  // sentinel, void slot, or the ragged last tile
            }
            if (done) break;
        }
        // Every TMA load must land before the CTA may exit; fills up to
        // consumed_a were waited for by the compute warps, each later one is
        // its stage's newest phase.
        for (int k = vload(&ctl->consumed_a) + 1; k <= issued; ++k)
            bar_wait(B(ctl->a_full[k % kSA]), (k / kSA) & 1, wait_limit);
        if (kStats) atomicAdd(st + 7, waited);
        return;
    }

    // ------------------------------------- producer B: re-loads for pass 2
    if (warp == kProducerB) {
        if (lane != 0) return;
        const uint64_t drop = l2_policy_evict_first();  // last use of the input tile
        int issued = -1;
        for (int j = 0;; ++j) {
            const int s = j % kSB;
            if (*end_k <= j) break;
            if (j >= kSB && !bar_wait(B(ctl->b_empty[s]), ((j / kSB) - 1) & 1, wait_limit, end_k, j)) break;
            // after pass 1 of tile j, so the tile is in L2 and its id is known
            if (!bar_wait(B(ctl->p1done[j % kR1]), (j / kR1) & 1, wait_limit, end_k, j)) break;
            const unsigned tu = ctl->tile[j % kRing];
            issued = j;
            if (tu != kVoid && (long long)tu < n_full_tiles) {
                mbar_arrive_expect_tx(B(ctl->b_full[s]), kTileBytes);
                tma_load_2d_hint(stageB + s * kTileBytes, &tm_in, 0, (int)((long long)tu * kRows), B(ctl->b_full[s]),
                                 drop);
            } else {
                mbar_arrive(B(ctl->b_full[s]));  // void slot or the ragged last tile
            }
        }
        for (int j = vload(&ctl->consumed_b) + 1; j <= issued; ++j)
            bar_wait(B(ctl->b_full[j % kSB]), (j / kSB) & 1, wait_limit);
        return;
    }

    // --------------------------------------------------------------- stores
    // Store warp w issues the TMA store of tiles j = w, w + kStoreWarps, ...
    // once the compute warps have written them, and frees the stage as soon as
    // the store has read it.
    if (warp >= kStoreWarp0) {
        if (lane != 0) return;
        const uint64_t stream = l2_policy_evict_first();  // outputs are not read again here
        for (int j = warp - kStoreWarp0;; j += kStoreWarps) {
            const int s = j % kSB;
            if (*end_k <= j || !bar_wait(B(ctl->written[s]), (j / kSB) & 1, wait_limit, end_k, j)) break;
            const unsigned tu = ctl->tile[j % kRing];
            if (tu != kVoid && (long long)tu < n_full_tiles) {
                tma_store_2d_hint(&tm_out, 0, (int)((long long)tu * kRows), stageB + s * kTileBytes, stream);
                bulk_commit();
                bulk_wait_read_all();
            }
            mbar_arrive(B(ctl->b_empty[s]));
        }
        bulk_wait_all();  // stores must finish before the CTA's shared memory is released
        return;
    }

    // ------------------------------------------------------- bookkeeping
    // Per fresh tile, in order: the tile total from the compute warps' totals,
    // the tile's offset inside its chunk, and at the end of each chunk the
    // chunk aggregate (published for the look-backs of later chunks).
    if (warp == kBookWarp) {
        C run = Op::c_identity();
        for (int k = 0;; ++k) {
            if (!warp_bar_wait(B(ctl->wready[k % kR1]), (k / kR1) & 1, wait_limit, end_k, k)) break;
            T wv = lane < kComputeWarps ? unpack_bits<T>(ctl->wtot[k % kRing][lane]) : Op::identity();
#pragma unroll
            for (int d = 1; d < kComputeWarps; d <<= 1) {  // ordered: lane 0 ends with warps 0..15
                const T y = shfl_down_v(wv, d);
                if (lane + d < kComputeWarps) wv = Op::op(wv, y);
            }
            const int pos = k % kChunk;
            if (pos == 0) run = Op::c_identity();
            if (lane == 0) {
                ctl->offset[k % kRing] = pack_bits(run);
                run = Op::c_op(run, Op::lift(wv));
                if (pos == kChunk - 1) {
                    const int q = k / kChunk;
                    const long long c = ((long long)ctl->tile[(k - pos) % kRing]) / kChunk;
                    ctl->chunk_agg[q % kChunkSlots] = pack_bits(run);
                    ctl->chunk_id[q % kChunkSlots] = c;
                    const bool stalled = p.lb.stall_tile >= 0 && p.lb.stall_tile / kChunk == c;
                    if (p.lb.delay_tile >= 0 && p.lb.delay_tile / kChunk == c) hook_delay(p.lb.delay_ns);
                    if (!stalled) {
                        if (c == 0) {
                            C c0 = Op::c_identity();
                            if (p.carry_in) c0 = *static_cast<const C*>(p.carry_in);
                            StatusIO<C>::publish(p.lb, c, ST_PREFIX, Op::c_op(c0, run));
                        } else {
                            StatusIO<C>::publish(p.lb, c, ST_AGGREGATE, run);
                        }
                    }
                    mbar_arrive(B(ctl->agg[q % kChunkSlots]));
                }
                mbar_arrive(B(ctl->p1done[k % kR1]));
            }
            run = shfl_idx_v(run, 0);
        }
        return;
    }

    // ------------------------------------------------------------ look-back
    if (warp >= kComputeWarps) {
        const int lw = warp - kComputeWarps;
        unsigned long long t_lb = 0, t_agg = 0;
        unsigned windows = 0, polls = 0;
        for (int q = lw;; q += kLbWarps) {
            const int k0 = q * kChunk;
            const unsigned long long w0 = kStats ? global_ns() : 0;
            if (!warp_bar_wait(B(ctl->agg[q % kChunkSlots]), (q / kChunkSlots) & 1, wait_limit, end_k, k0)) break;
            const unsigned long long w1 = kStats ? global_ns() : 0;
            const long long c = ctl->chunk_id[q % kChunkSlots];
            C prefix = Op::c_identity();
            bool ok = true;
            if (c == 0) {
                if (p.carry_in) prefix = *static_cast<const C*>(p.carry_in);
            } else {
                unsigned wnd = 0, pl = 0;
                ok = lookback_prefix_adaptive<Op, kLbPer>(p.lb, c, prefix, kStats ? &wnd : nullptr,
                                                          kStats ? &pl : nullptr);
                windows += wnd;
                polls += pl;
                if (!ok && lane == 0) StatusIO<C>::publish(p.lb, c, ST_POISON, Op::c_identity());
            }
            if (kStats) {
                t_agg += w1 - w0;
                t_lb += global_ns() - w1;
            }
            if (lane == 0) {
                const C agg = unpack_bits<C>(ctl->chunk_agg[q % kChunkSlots]);
                const bool stalled = p.lb.stall_tile >= 0 && p.lb.stall_tile / kChunk == c;
                if (ok && c != 0 && !stalled) StatusIO<C>::publish(p.lb, c, ST_PREFIX, Op::c_op(prefix, agg));
                if (ok && p.carry_out && c == num_chunks - 1) *static_cast<C*>(p.carry_out) = Op::c_op(prefix, agg);
                ctl->chunk_prefix[q % kChunkSlots] = pack_bits(prefix);
                mbar_arrive(B(ctl->pre[q % kChunkSlots]));
            }
            __syncwarp();
        }
        if (kStats && lane == 0) {
            atomicAdd(st + 3, t_lb);
            atomicAdd(st + 4, (unsigned long long)windows);
            atomicAdd(st + 5, (unsigned long long)polls);
            atomicAdd(st + 6, t_agg);
        }
        return;
    }

    // -------------------------------------------------------------- compute
    const int ctid = threadIdx.x;  // 0 .. kCompute-1
    const int row = ctid / kThreadsPerRow;
    // Swizzled byte offsets of this thread's 16-byte chunks: with the TMA's
    // 128-byte swizzle, chunk c of row r sits at chunk position c ^ (r & 7),
    // which keeps every quarter-warp's 16-byte accesses on distinct banks.
    uint32_t off[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) off[j] = row * 128 + ((((ctid % kThreadsPerRow) * NV + j) ^ (row & 7)) << 4);
    bool ok = true;                // this warp has not timed out
    unsigned long long t_fresh = 0, t_wait2 = 0, ntiles = 0;

    // Compute warps run independently (no block-wide barrier).  A warp that
    // times out records the error and stops; the other roles' waits are
    // bounded too.
    auto wait = [&](uint32_t b, uint32_t parity, unsigned long long* acc) {
        const unsigned long long w0 = (kStats && ctid == 0) ? global_ns() : 0;
        const bool good = warp_bar_wait(b, parity, wait_limit);
        if (!good) {
            if (lane == 0 && ok) raise_error(p.lb.error, DEV_LOOKBACK_TIMEOUT);
            ok = false;
        }
        if (kStats && ctid == 0) *acc += global_ns() - w0;
        return good;
    };

    // One loop iteration does pass 1 of fresh tile k and pass 2 of tile
    // j = k - kLag in a single instruction stream: all waits first, then both
    // tiles' shared-memory loads, then the two independent scan chains, which
    // the compiler interleaves.  A warp thus overlaps the latency of the two.
    auto fetch = [&](uint32_t sbase, long long t, T (&v)[IPT]) {
        if (t < n_full_tiles) {
#pragma unroll
            for (int i = 0; i < NV; ++i) unpack(lds128(sbase + off[i]), &v[i * Vec<T>::kPer]);
        } else {
            load_partial_tile<T, IPT>(static_cast<const T*>(p.in) + t * TILE, v, p.n - t * TILE, Op::identity());
        }
    };
    // pass 1 body: this warp's total of the fresh tile, published to the
    // bookkeeping warp (the same blocked partition pass 2 scans)
    auto finish1 = [&](int k, int s, unsigned tu, T (&v)[IPT]) {
        T acc = Op::identity();
        if (tu != kVoid) {
            if constexpr (TT::kKeep && IPT % 4 == 0) {
                // costly combines: four independent in-order chains, then their
                // totals in order (the same number of combines, a quarter of
                // the dependency depth)
                T part[4];
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    part[g] = v[g * (IPT / 4)];
#pragma unroll
                    for (int w = 1; w < IPT / 4; ++w) part[g] = Op::op(part[g], v[g * (IPT / 4) + w]);
                }
                acc = Op::op(Op::op(part[0], part[1]), Op::op(part[2], part[3]));
            } else {
                acc = v[0];
#pragma unroll
                for (int w = 1; w < IPT; ++w) acc = Op::op(acc, v[w]);
            }
            if constexpr (TT::kKeep) ttot[(k % TT::kSlots) * kCompute + ctid] = acc;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {  // ordered reduction: lane 0 ends with lanes 0..31
                const T y = shfl_down_v(acc, d);
                if (lane + d < 32) acc = Op::op(acc, y);
            }
        }
        if (lane == 0) ctl->wtot[k % kRing][warp] = pack_bits(acc);
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(B(ctl->a_empty[s]));  // this warp is done reading the stage
            mbar_arrive(B(ctl->wready[k % kR1]));
        }
        if (kStats && ctid == 0 && tu != kVoid) ++ntiles;
    };
    // pass 2 body: full scan of this warp's part of tile j with its prefix,
    // written back for the store warps
    auto finish2 = [&](int j, unsigned tu, T (&v)[IPT]) {
        const int s = j % kSB;
        const int q = j / kChunk;
        if (tu != kVoid) {
            const long long t = tu;
            const bool full = t < n_full_tiles;
            // carry into this warp: chunk prefix (+) tile offset in the chunk (+)
            // the warp totals before this warp, recorded in pass 1
            T wv = lane < kComputeWarps ? unpack_bits<T>(ctl->wtot[j % kRing][lane]) : Op::identity();
#pragma unroll
            for (int d = 1; d < kComputeWarps; d <<= 1) {
                const T y = shfl_up_v(wv, d);
                if (lane >= d) wv = Op::op(y, wv);
            }
            const T wpre = shfl_idx_v(wv, warp > 0 ? warp - 1 : 0);
            const C cp = Op::c_op(unpack_bits<C>(ctl->chunk_prefix[q % kChunkSlots]), unpack_bits<C>(ctl->offset[j % kRing]));
            T base = Op::lower(cp);
            if (warp > 0) base = Op::op(base, wpre);
            if constexpr (TT::kKeep) {
                // the thread's total from pass 1 gives its carry first; then one
                // serial pass seeded with the carry: one combine per element
                T x = ttot[(j % TT::kSlots) * kCompute + ctid];
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const T y = shfl_up_v(x, d);
                    if (lane >= d) x = Op::op(y, x);
                }
                T run = shfl_up_v(x, 1);
                run = lane == 0 ? base : Op::op(base, run);
                if constexpr (kExcl) {
#pragma unroll
                    for (int w = 0; w < IPT; ++w) {
                        const T xw = v[w];
                        v[w] = run;
                        run = Op::op(run, xw);
                    }
                } else {
                    v[0] = Op::op(run, v[0]);
#pragma unroll
                    for (int w = 1; w < IPT; ++w) v[w] = Op::op(v[w - 1], v[w]);
                }
            } else {
#pragma unroll
                for (int w = 1; w < IPT; ++w) v[w] = Op::op(v[w - 1], v[w]);
                T x = v[IPT - 1];
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const T y = shfl_up_v(x, d);
                    if (lane >= d) x = Op::op(y, x);
                }
                T carry = shfl_up_v(x, 1);
                carry = lane == 0 ? base : Op::op(base, carry);
                if constexpr (kExcl) {
#pragma unroll
                    for (int w = IPT - 1; w >= 1; --w) v[w] = Op::op(carry, v[w - 1]);
                    v[0] = carry;
                } else {
#pragma unroll
                    for (int w = 0; w < IPT; ++w) v[w] = Op::op(carry, v[w]);
                }
            }
            if (full) {
                const uint32_t sb = stageB + s * kTileBytes;
#pragma unroll
                for (int i = 0; i < NV; ++i) sts128(sb + off[i], pack(&v[i * Vec<T>::kPer]));
                fence_proxy_async();  // before the store warp's TMA reads this stage
            } else {
                store_partial_tile<T, IPT>(static_cast<T*>(p.out) + t * TILE, v, p.n - t * TILE);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(B(ctl->written[s]));
    };
    auto wait2 = [&](int j) -> bool {
        const int q = j / kChunk;
        if (!wait(B(ctl->b_full[j % kSB]), (j / kSB) & 1, &t_wait2)) return false;
        if (ctid == 0) vstore(&ctl->consumed_b, j);
        return wait(B(ctl->pre[q % kChunkSlots]), (q / kChunkSlots) & 1, &t_wait2);
    };

    int k = 0;
    bool draining = ok;
    for (;; ++k) {
        const int s = k % kSA;
        if (!wait(B(ctl->a_full[s]), (k / kSA) & 1, &t_fresh)) { draining = false; break; }
        if (ctid == 0) vstore(&ctl->consumed_a, k);
        const unsigned tu1 = ctl->tile[k % kRing];
        if (tu1 == kSentinel) break;
        const int j = k - kLag;
        unsigned tu2 = kVoid;
        T v1[IPT], v2[IPT];
        if constexpr (Cfg::kP1First) {
            if (tu1 != kVoid) fetch(stageA + s * kTileBytes, tu1, v1);
            finish1(k, s, tu1, v1);
        }
        if (j >= 0) {
            if (!wait2(j)) { draining = false; break; }
            tu2 = ctl->tile[j % kRing];
        }
        if (!Cfg::kP1First && tu1 != kVoid) fetch(stageA + s * kTileBytes, tu1, v1);
        if (j >= 0 && tu2 != kVoid) fetch(stageB + (j % kSB) * kTileBytes, tu2, v2);
        if (!Cfg::kP1First) finish1(k, s, tu1, v1);
        if (j >= 0) finish2(j, tu2, v2);
    }
    if (draining)
        for (int j = (k > kLag ? k - kLag : 0); j < k; ++j) {
            if (!wait2(j)) break;
            const unsigned tu2 = ctl->tile[j % kRing];
            T v2[IPT];
            if (tu2 != kVoid) fetch(stageB + (j % kSB) * kTileBytes, tu2, v2);
            finish2(j, tu2, v2);
        }
    if (kStats && ctid == 0) {
        atomicAdd(st + 0, ntiles);
        atomicAdd(st + 1, t_fresh);
        atomicAdd(st + 2, t_wait2);
    }
}

// ----------------------------------------------------------------- host side
namespace {

template <class Op, bool kExcl, bool kStats, class Cfg>
cudaError_t launch_one(const ScanParams& p, unsigned grid, cudaStream_t s) {
    using T = typename Op::T;
    const long long tile = Cfg::kTileBytes / sizeof(T);
    const long long nfull = p.n / tile;
    CUtensorMap a, b;
    const unsigned long long rows = (unsigned long long)nfull * Cfg::kRows;
    if (!make_map(&a, p.in, rows, Cfg::kRows) || !make_map(&b, p.out, rows, Cfg::kRows)) return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> done_mask{0};
    constexpr int smem = ThreadTotals<Op, Cfg>::kSmemBytes;
    const cudaError_t e = allow_smem(scan_tma_kernel<Op, kExcl, kStats, Cfg>, smem, done_mask);
    if (e != cudaSuccess) return e;
    scan_tma_kernel<Op, kExcl, kStats, Cfg><<<grid, Cfg::kThreads, smem, s>>>(a, b, p, nfull);
    return cudaGetLastError();
}

template <class Op, class Cfg>
cudaError_t launch_cfg(const ScanParams& p, bool exclusive, unsigned grid, cudaStream_t s, bool stats) {
    if (stats) {
        if constexpr (std::is_same<Op, OpSumU32>::value)
            return exclusive ? launch_one<Op, true, true, Cfg>(p, grid, s) : launch_one<Op, false, true, Cfg>(p, grid, s);
        return cudaErrorInvalidValue;
    }
    return exclusive ? launch_one<Op, true, false, Cfg>(p, grid, s) : launch_one<Op, false, false, Cfg>(p, grid, s);
}

template <class Cfg>
void cfg_info(TmaShape* sh) {
    sh->tile_bytes = Cfg::kTileBytes;
    sh->chunk_tiles = Cfg::kChunk;
    sh->compute_threads = Cfg::kCompute;
    sh->threads = Cfg::kThreads;
    sh->ctas_per_sm = Cfg::kMinBlocks;
    sh->ids_per_cta = Cfg::kIdsPerCta;
}

}  // namespace

}  // namespace scg
