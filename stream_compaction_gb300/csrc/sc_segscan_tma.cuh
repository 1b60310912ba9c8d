// Persistent, warp-specialised scan segmented by head flags (one byte per
// element, nonzero = a segment starts there), or by rows of a fixed length
// (batched rows: the heads are the multiples of the row length, computed from
// the element index): the same pipeline as the persistent scan
// (sc_scan_tma.cuh) with the heads carried along.
//
// "Lecture 7: Parallel pattern -- prefix sum / scan" (UIUC ECE408 notes),
// section 2, names the segmented scan (the running value restarts at every
// head); a segmented scan is a plain scan of (value, flag) pairs under
//
//   (v1, f1) (+) (v2, f2) = (f2 ? v2 : v1 (+) v2,  f1 | f2),
//
// which is associative, so the decoupled look-back carries such pairs.  A
// chunk that holds a head publishes its aggregate as its inclusive prefix at
// once (what came before it no longer matters), so look-backs stop there.
//
//   producer A       chunk ids; per fresh tile a 2-D TMA load of the values
//                    and a 1-D bulk copy of its head flags (one byte each);
//   compute warps    pass 1: each thread turns its flags into a bit mask
//                    (kept in shared memory for pass 2) and folds its items
//                    into a (value, flag) total; warps fold those in order;
//                    pass 2 (tile re-loaded from L2): the carry into each
//                    thread from the chunk prefix, the tile's offset in the
//                    chunk, the earlier warps and a warp scan of the thread
//                    totals, then a serial scan that restarts at heads;
//   bookkeeping, look-back warps, producer B, store warps as in the plain
//   persistent scan, with (value, flag) pairs as carries.
//
// Each value is read from HBM once (and once more from L2) and written once;
// each flag is read once.  Operators with 4-byte elements whose (value, flag)
// pair fits 8 bytes: those whose carry is the element, and the float32 sum.
#pragma once
#include "sc_scan_tma.cuh"

namespace scg {

namespace {

// Pair forms of a 4-byte operator.  E: the in-tile pair (x = the element's
// bits, y = the flag), combined in the element type; C: the carry pair that
// travels between tiles.  make() builds an E from a value, value() reads an
// E back, lift() / lower() convert between E and C, flag() reads C's flag.
template <class Op>
struct SegPairOp {
    using T = typename Op::T;
    using E = uint2;
    using C = uint2;
    static_assert(sizeof(T) == 4 && std::is_same<typename Op::C, T>::value, "4-byte operators with C == T");
    __device__ __forceinline__ static E make(T v, bool f) { return make_uint2(to_bits32(v), f ? 1u : 0u); }
    __device__ __forceinline__ static T value(E e) { T v; from_bits32(e.x, v); return v; }
    __device__ __forceinline__ static E e_identity() { return make(Op::identity(), false); }
    __device__ __forceinline__ static E e_op(E a, E b) {
        if (b.y) return b;
        return make_uint2(to_bits32(Op::op(value(a), value(b))), a.y);  // the flag passes through as is
    }
    __device__ __forceinline__ static C lift(E e) { return e; }
    __device__ __forceinline__ static E lower(C c) { return c; }
    __device__ __forceinline__ static bool flag(C c) { return c.y != 0u; }
    __device__ __forceinline__ static C c_identity() { return e_identity(); }
    __device__ __forceinline__ static C c_op(C a, C b) { return e_op(a, b); }
};

// The float32 sum: a float-float carry (high, low) whose low part's lowest
// mantissa bit holds the flag (a change of at most 2^-48 of the carry, below
// its 2^-44 precision), so that the pair stays 8 bytes.
// Inside a tile the float32 sum's pairs are float32 (as in the plain scan);
// between tiles its carry is a float-float pair.
template <>
struct SegPairOp<OpSumF32> {
    using T = float;
    using E = uint2;
    using C = float2;
    __device__ __forceinline__ static E make(T v, bool f) { return make_uint2(__float_as_uint(v), f ? 1u : 0u); }
    __device__ __forceinline__ static T value(E e) { return __uint_as_float(e.x); }
    __device__ __forceinline__ static E e_identity() { return make(0.0f, false); }
    __device__ __forceinline__ static E e_op(E a, E b) {
        if (b.y) return b;
        return make_uint2(__float_as_uint(__fadd_rn(value(a), value(b))), a.y);
    }
    __device__ __forceinline__ static C tag(float2 v, bool f) {
        return make_float2(v.x, __uint_as_float((__float_as_uint(v.y) & ~1u) | (f ? 1u : 0u)));
    }
    __device__ __forceinline__ static float2 plain(C c) {
        return make_float2(c.x, __uint_as_float(__float_as_uint(c.y) & ~1u));
    }
    __device__ __forceinline__ static bool flag(C c) { return (__float_as_uint(c.y) & 1u) != 0u; }
    __device__ __forceinline__ static C lift(E e) { return tag(make_float2(value(e), 0.0f), e.y != 0u); }
    __device__ __forceinline__ static E lower(C c) { return make(OpSumF32::lower(plain(c)), flag(c)); }
    __device__ __forceinline__ static C c_identity() { return tag(make_float2(0.0f, 0.0f), false); }
    __device__ __forceinline__ static C c_op(C a, C b) {
        if (flag(b)) return b;
        return tag(OpSumF32::c_op(plain(a), plain(b)), flag(a));
    }
    // look-back: a chunk that holds a head publishes its inclusive prefix at
    // once, so the aggregates after the newest prefix carry no flag and fold
    // as a float32 sum (as OpSumF32's)
    static constexpr bool kLowFold = true;
    using L = float;
    __device__ __forceinline__ static L low(C c) { return c.x; }
    __device__ __forceinline__ static L low_identity() { return 0.0f; }
    __device__ __forceinline__ static L low_op(L a, L b) { return __fadd_rn(a, b); }
    __device__ __forceinline__ static C with_low(C prefix, L s) { return c_op(prefix, tag(make_float2(s, 0.0f), false)); }
};

// 1-D bulk copy global -> shared, completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load_1d_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                                  uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Head flags of 16 consecutive elements (one byte each) as 16 bits.
__device__ __forceinline__ uint32_t head_bits16(const uint4& q) {
    uint32_t m = 0;
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // 0x01 in every nonzero byte, then the four bytes' low bits gathered
        // into bits 24..27 by one multiplication (no carries between them)
        const uint32_t b = (__vcmpne4(w[i], 0u) >> 7) & 0x01010101u;
        m |= ((b * 0x01020408u) >> 24) << (4 * i);
    }
    return m;
}

// pass-2 lag 5 with pass 1 first, as the plain persistent scan
using SegCfg = TmaCfg<32768, 3, 2, 8, 5, 2, true>;      // 3 fresh-tile stages + flags, 2 re-load stages
using SegRowsCfg = TmaCfg<32768, 3, 3, 8, 5, 2, true>;  // heads at multiples of a row length: no flags to hold

}  // namespace

// kPeriodic: the heads are the multiples of p.seg_len (batched rows), computed
// from the element index; otherwise p.heads holds one flag byte per element.
template <class Op, bool kExcl, class Cfg, bool kPeriodic>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    segscan_tma_kernel(const __grid_constant__ CUtensorMap tm_in, const __grid_constant__ CUtensorMap tm_out,
                       const ScanParams p, const long long n_full_tiles) {
    using T = typename Op::T;
    using PO = SegPairOp<Op>;
    using C = typename PO::C;  // carries between tiles
    using E = typename PO::E;  // pairs inside a tile
    using Ctrl = typename Cfg::Ctrl;
    constexpr int kTileBytes = Cfg::kTileBytes, kSA = Cfg::kSA, kSB = Cfg::kSB, kChunk = Cfg::kChunk;
    constexpr int kLag = Cfg::kLag, kComputeWarps = Cfg::kComputeWarps, kChunkSlots = Cfg::kChunkSlots;
    constexpr int kRing = Cfg::kRing, kR1 = Cfg::kR1, kLbWarps = Cfg::kLbWarps, kStoreWarps = Cfg::kStoreWarps;
    constexpr int kBookWarp = Cfg::kBookWarp, kProducerA = Cfg::kProducerA, kProducerB = Cfg::kProducerB;
    constexpr int kStoreWarp0 = Cfg::kStoreWarp0, kCompute = Cfg::kCompute, kRows = Cfg::kRows;
    constexpr int kBytesPerThread = Cfg::kBytesPerThread;
    constexpr int IPT = kBytesPerThread / sizeof(T);
    constexpr int TILE = kCompute * IPT;
    constexpr int NV = kBytesPerThread / 16;
    constexpr int kMaskSlots = kLag + 2;
    static_assert(IPT == 32 && Cfg::kThreadsPerRow == 1, "one 128-byte row and 32 flags per compute thread");

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + (kSA + kSB) * kTileBytes);
    const uint32_t stageA = smem_u32(smem);
    const uint32_t stageB = stageA + kSA * kTileBytes;
    const uint32_t headsA = stageA + (kSA + kSB) * kTileBytes + Cfg::kCtrlBytes;  // kSA buffers of TILE bytes
    uint32_t* hmask = reinterpret_cast<uint32_t*>(smem + (kSA + kSB) * kTileBytes + Cfg::kCtrlBytes + kSA * TILE);
    auto B = [](const unsigned long long& b) { return smem_u32(&b); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long num_tiles = p.n / TILE + (p.n % TILE != 0);
    const long long num_chunks = p.lb.num_tiles;
    // batched rows no longer than 2^31 elements: head positions in 32-bit arithmetic
    const bool short_rows = kPeriodic && p.seg_len <= 0x7fffffffLL;
    const unsigned long long wait_limit = p.lb.timeout_ns + 500000000ull;
    const volatile int* end_k = &ctl->end_k;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSA; ++i) {
            mbar_init(B(ctl->a_full[i]), 1);
            mbar_init(B(ctl->a_empty[i]), kComputeWarps);
        }
        for (int i = 0; i < kSB; ++i) {
            mbar_init(B(ctl->b_full[i]), 1);
            mbar_init(B(ctl->b_empty[i]), 1);
            mbar_init(B(ctl->written[i]), kComputeWarps);
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
        ChunkIds ids{p.lb.counter, p.lb.counter_base, num_chunks, (long long)gridDim.x, p.lb.error};
        ids.start();  // chunk ids one chunk ahead of use, except near the end
        const uint64_t keep = l2_policy_evict_last();   // values stay in L2 for the re-load
        const uint64_t drop = l2_policy_evict_first();  // flags are read once
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
            // batched rows: the row position of the tile's first element, once per tile
            if (kPeriodic && short_rows && !done && t < num_tiles) ctl->seg_r[k % kRing] = (unsigned)((t * TILE) % p.seg_len);
            if (done) vstore(&ctl->end_k, k);
            issued = k;
            if (!done && t < n_full_tiles) {
                mbar_arrive_expect_tx(B(ctl->a_full[s]), kTileBytes + (kPeriodic ? 0 : TILE));
                tma_load_2d_hint(stageA + s * kTileBytes, &tm_in, 0, (int)(t * kRows), B(ctl->a_full[s]), keep);
                if (!kPeriodic) bulk_load_1d_hint(headsA + s * TILE, p.heads + t * TILE, TILE, B(ctl->a_full[s]), drop);
            } else {
                mbar_arrive(B(ctl->a_full[s]));  // sentinel, void slot, or the ragged last tile
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

    // --------------------------------------------------------------- stores
    if (warp >= kStoreWarp0) {
        if (lane != 0) return;
        const uint64_t stream = l2_policy_evict_first();
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
        bulk_wait_all();
        return;
    }

    // ------------------------------------------------------- bookkeeping
    // Per fresh tile: its (value, flag) total from the warp totals and its
    // offset inside the chunk; per chunk the aggregate, published as the
    // chunk's inclusive prefix at once when it holds a head.
    if (warp == kBookWarp) {
        C run = PO::c_identity();
        for (int k = 0;; ++k) {
            if (!warp_bar_wait(B(ctl->wready[k % kR1]), (k / kR1) & 1, wait_limit, end_k, k)) break;
            E wv = lane < kComputeWarps ? unpack_bits<E>(ctl->wtot[k % kRing][lane]) : PO::e_identity();
#pragma unroll
            for (int d = 1; d < kComputeWarps; d <<= 1) {  // ordered: lane 0 ends with warps 0..kComputeWarps-1
                const E y = shfl_down_v(wv, d);
                if (lane + d < kComputeWarps) wv = PO::e_op(wv, y);
            }
            const int pos = k % kChunk;
            if (pos == 0) run = PO::c_identity();
            if (lane == 0) {
                ctl->offset[k % kRing] = pack_bits(run);
                run = PO::c_op(run, PO::lift(wv));
                if (pos == kChunk - 1) {
                    const int q = k / kChunk;
                    const long long c = ((long long)ctl->tile[(k - pos) % kRing]) / kChunk;
                    ctl->chunk_agg[q % kChunkSlots] = pack_bits(run);
                    ctl->chunk_id[q % kChunkSlots] = c;
                    const bool stalled = p.lb.stall_tile >= 0 && p.lb.stall_tile / kChunk == c;
                    if (p.lb.delay_tile >= 0 && p.lb.delay_tile / kChunk == c) hook_delay(p.lb.delay_ns);
                    if (!stalled)
                        StatusIO<C>::publish(p.lb, c, (c == 0 || PO::flag(run)) ? ST_PREFIX : ST_AGGREGATE, run);
                    mbar_arrive(B(ctl->agg[q % kChunkSlots]));
                }
                mbar_arrive(B(ctl->p1done[k % kR1]));
            }
            run = shfl_idx_v(run, 0);
        }
        return;
    }

    // ------------------------------------------------------------ look-back
    // Every chunk needs its exclusive prefix (its elements before its first
    // head take it); a chunk without a head then publishes its inclusive one.
    if (warp >= kComputeWarps) {
        const int lw = warp - kComputeWarps;
        for (int q = lw;; q += kLbWarps) {
            const int k0 = q * kChunk;
            if (!warp_bar_wait(B(ctl->agg[q % kChunkSlots]), (q / kChunkSlots) & 1, wait_limit, end_k, k0)) break;
            const long long c = ctl->chunk_id[q % kChunkSlots];
            C prefix = PO::c_identity();
            bool ok = true;
            if (c != 0) {
                ok = lookback_prefix_adaptive<PO, kLbPer>(p.lb, c, prefix);
                if (!ok && lane == 0) StatusIO<C>::publish(p.lb, c, ST_POISON, PO::c_identity());
            }
            if (lane == 0) {
                const C agg = unpack_bits<C>(ctl->chunk_agg[q % kChunkSlots]);
                const bool stalled = p.lb.stall_tile >= 0 && p.lb.stall_tile / kChunk == c;
                if (ok && c != 0 && !PO::flag(agg) && !stalled)
                    StatusIO<C>::publish(p.lb, c, ST_PREFIX, PO::c_op(prefix, agg));
                ctl->chunk_prefix[q % kChunkSlots] = pack_bits(prefix);
                mbar_arrive(B(ctl->pre[q % kChunkSlots]));
            }
            __syncwarp();
        }
        return;
    }

    // -------------------------------------------------------------- compute
    const int ctid = threadIdx.x;  // 0 .. kCompute-1: row ctid of every tile
    uint32_t off[NV];  // swizzled 16-byte chunks of the thread's row (128-byte TMA swizzle)
#pragma unroll
    for (int j = 0; j < NV; ++j) off[j] = ctid * 128 + ((j ^ (ctid & 7)) << 4);
    bool ok = true;

    auto wait = [&](uint32_t b, uint32_t parity) {
        const bool good = warp_bar_wait(b, parity, wait_limit);
        if (!good) {
            if (lane == 0 && ok) raise_error(p.lb.error, DEV_LOOKBACK_TIMEOUT);
            ok = false;
        }
        return good;
    };
    auto fetch = [&](uint32_t sbase, long long t, T (&v)[IPT]) {
        if (t < n_full_tiles) {
#pragma unroll
            for (int i = 0; i < NV; ++i) unpack(lds128(sbase + off[i]), &v[i * Vec<T>::kPer]);
        } else {
            load_partial_tile<T, IPT>(static_cast<const T*>(p.in) + t * TILE, v, p.n - t * TILE, Op::identity());
        }
    };
    // batched rows: the thread's offset inside a tile, mod the row length
    const uint32_t row_len = short_rows ? (uint32_t)p.seg_len : 0u;
    const uint32_t rc = short_rows ? (uint32_t)(ctid * IPT) % row_len : 0u;
    // head bits of the thread's items of tile t in ring slot `slot` (batched rows)
    auto heads_periodic = [&](int slot, long long t) -> uint32_t {
        if constexpr (kPeriodic) {
            if (!short_rows) return head_bits<IPT>(t * TILE + (long long)ctid * IPT, p.seg_len);
            uint32_t r = ctl->seg_r[slot % kRing] + rc;  // < 2 * row_len <= 2^32 - 2
            if (r >= row_len) r -= row_len;
            uint32_t hm = 0;
            for (uint32_t k = r == 0 ? 0u : row_len - r; k < (uint32_t)IPT; k += row_len) hm |= 1u << k;
            return hm;
        } else {
            return 0u;
        }
    };
    // the head bits of this thread's items of tile t (fresh tile in stage s, ring slot k)
    auto heads_of = [&](int s, int k, long long t) -> uint32_t {
        if constexpr (kPeriodic) return heads_periodic(k, t);
        if (t < n_full_tiles) {
            const uint32_t hb = headsA + s * TILE + ctid * IPT;
            return head_bits16(lds128(hb)) | (head_bits16(lds128(hb + 16)) << 16);
        }
        const long long first = t * TILE + (long long)ctid * IPT;
        uint32_t m = 0;
        for (int w = 0; w < IPT; ++w)
            if (first + w < p.n && p.heads[first + w] != 0) m |= 1u << w;
        return m;
    };
    // the thread's (value, flag) total: the fold since its last head
    auto thread_total = [&](const T (&v)[IPT], uint32_t hm) {
        T acc = v[0];
#pragma unroll
        for (int w = 1; w < IPT; ++w) acc = ((hm >> w) & 1u) ? v[w] : Op::op(acc, v[w]);
        return PO::make(acc, hm != 0u);
    };

    // pass 1: head mask kept for pass 2, warp total published to the bookkeeping warp
    auto finish1 = [&](int k, int s, unsigned tu, const T (&v)[IPT]) {
        E tot = PO::e_identity();
        if (tu != kVoid) {
            const uint32_t hm = heads_of(s, k, (long long)tu);
            if (!kPeriodic) hmask[(k % kMaskSlots) * kCompute + ctid] = hm;
            tot = thread_total(v, hm);
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {  // ordered: lane 0 ends with lanes 0..31
                const E y = shfl_down_v(tot, d);
                if (lane + d < 32) tot = PO::e_op(tot, y);
            }
        }
        if (lane == 0) ctl->wtot[k % kRing][warp] = pack_bits(tot);
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(B(ctl->a_empty[s]));  // values and flags of the stage read
            mbar_arrive(B(ctl->wready[k % kR1]));
        }
    };
    // pass 2: carry into the thread, then the serial scan restarting at heads
    auto finish2 = [&](int j, unsigned tu, T (&v)[IPT]) {
        const int s = j % kSB;
        const int q = j / kChunk;
        if (tu != kVoid) {
            const long long t = tu;
            const uint32_t hm = kPeriodic ? heads_periodic(j, t) : hmask[(j % kMaskSlots) * kCompute + ctid];
            E wv = lane < kComputeWarps ? unpack_bits<E>(ctl->wtot[j % kRing][lane]) : PO::e_identity();
#pragma unroll
            for (int d = 1; d < kComputeWarps; d <<= 1) {
                const E y = shfl_up_v(wv, d);
                if (lane >= d) wv = PO::e_op(y, wv);
            }
            const E wpre = shfl_idx_v(wv, warp > 0 ? warp - 1 : 0);
            // the tile's prefix in carry precision, then the element type
            E base = PO::lower(
                PO::c_op(unpack_bits<C>(ctl->chunk_prefix[q % kChunkSlots]), unpack_bits<C>(ctl->offset[j % kRing])));
            if (warp > 0) base = PO::e_op(base, wpre);
            E x = thread_total(v, hm);
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const E y = shfl_up_v(x, d);
                if (lane >= d) x = PO::e_op(y, x);
            }
            E cin = shfl_up_v(x, 1);
            cin = lane == 0 ? base : PO::e_op(base, cin);
            T run = PO::value(cin);
            if constexpr (kExcl) {
#pragma unroll
                for (int w = 0; w < IPT; ++w) {
                    const T xw = v[w];
                    const bool h = (hm >> w) & 1u;
                    v[w] = h ? Op::identity() : run;
                    run = h ? xw : Op::op(run, xw);
                }
            } else {
#pragma unroll
                for (int w = 0; w < IPT; ++w) {
                    run = ((hm >> w) & 1u) ? v[w] : Op::op(run, v[w]);
                    v[w] = run;
                }
            }
            if (t < n_full_tiles) {
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
        if (!wait(B(ctl->b_full[j % kSB]), (j / kSB) & 1)) return false;
        if (ctid == 0) vstore(&ctl->consumed_b, j);
        return wait(B(ctl->pre[q % kChunkSlots]), (q / kChunkSlots) & 1);
    };

    int k = 0;
    bool draining = ok;
    for (;; ++k) {
        const int s = k % kSA;
        if (!wait(B(ctl->a_full[s]), (k / kSA) & 1)) { draining = false; break; }
        if (ctid == 0) vstore(&ctl->consumed_a, k);
        const unsigned tu1 = ctl->tile[k % kRing];
        if (tu1 == kSentinel) break;
        const int j = k - kLag;
        unsigned tu2 = kVoid;
        if (!Cfg::kP1First && j >= 0) {
            if (!wait2(j)) { draining = false; break; }
            tu2 = ctl->tile[j % kRing];
        }
        T v1[IPT], v2[IPT];
        if constexpr (Cfg::kP1First) {
            if (tu1 != kVoid) fetch(stageA + s * kTileBytes, tu1, v1);
            finish1(k, s, tu1, v1);
            if (j >= 0) {
                if (!wait2(j)) { draining = false; break; }
                tu2 = ctl->tile[j % kRing];
                if (tu2 != kVoid) fetch(stageB + (j % kSB) * kTileBytes, tu2, v2);
                finish2(j, tu2, v2);
            }
            continue;
        }
        if (tu1 != kVoid) fetch(stageA + s * kTileBytes, tu1, v1);
        if (j >= 0 && tu2 != kVoid) fetch(stageB + (j % kSB) * kTileBytes, tu2, v2);
        finish1(k, s, tu1, v1);
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
}

// ----------------------------------------------------------------- host side
namespace {

template <class Op, bool kExcl, class Cfg, bool kPeriodic>
cudaError_t launch_seg_cfg(const ScanParams& p, unsigned grid, cudaStream_t s) {
    using T = typename Op::T;
    const long long tile = Cfg::kTileBytes / sizeof(T);
    const long long nfull = p.n / tile;
    CUtensorMap a, b;
    const unsigned long long rows = (unsigned long long)nfull * Cfg::kRows;
    if (nfull < 1 || !make_map(&a, p.in, rows, Cfg::kRows) || !make_map(&b, p.out, rows, Cfg::kRows))
        return cudaErrorInvalidValue;
    // stages and control block, then (flags only) kSA flag buffers and the pass-2 mask ring
    constexpr int smem =
        Cfg::kSmemBytes + (kPeriodic ? 0 : Cfg::kSA * Cfg::kCompute * 32 + (Cfg::kLag + 2) * Cfg::kCompute * 4);
    static_assert(smem <= 232448, "shared memory per CTA");
    static std::atomic<unsigned long long> done_mask{0};
    const cudaError_t e = allow_smem(segscan_tma_kernel<Op, kExcl, Cfg, kPeriodic>, smem, done_mask);
    if (e != cudaSuccess) return e;
    segscan_tma_kernel<Op, kExcl, Cfg, kPeriodic><<<grid, Cfg::kThreads, smem, s>>>(a, b, p, nfull);
    return cudaGetLastError();
}

// Head flags (p.heads) or batched rows (heads at multiples of p.seg_len).
template <class Op, bool kExcl>
cudaError_t launch_seg_one(const ScanParams& p, unsigned grid, cudaStream_t s) {
    static_assert(SegCfg::kTileBytes == SegRowsCfg::kTileBytes && SegCfg::kChunk == SegRowsCfg::kChunk,
                  "both shapes share the host's tile and chunk sizes");
    if (p.heads) return launch_seg_cfg<Op, kExcl, SegCfg, false>(p, grid, s);
    if (p.seg_len <= 0) return cudaErrorInvalidValue;
    return launch_seg_cfg<Op, kExcl, SegRowsCfg, true>(p, grid, s);
}

}  // namespace

}  // namespace scg
