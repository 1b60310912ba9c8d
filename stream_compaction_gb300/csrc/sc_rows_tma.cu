// Batched rows of at most 8192 elements.  When the row length divides the
// 8192-element tile, every tile holds whole rows, so a tile's scan needs
// nothing from any other tile -- no look-back, no second read; the CTAs take
// tiles blockIdx.x, blockIdx.x + gridDim.x, ...  Otherwise (kRagged) a tile
// may start inside a row, but every full tile holds a row start (any 8192
// consecutive indices hold a multiple of a row length <= 8192), so the carry
// into tile t + 1 is the fold of tile t since its last row start: each CTA
// takes a contiguous range of tiles and carries that fold from one tile to
// the next in registers; only its first tile reads back the part of its row
// that lies before it.  A persistent CTA per SM streams tiles through a ring
// of shared-memory stages:
//
//   producer warp   2-D TMA loads of the CTA's tiles (blockIdx.x +
//                   i * gridDim.x, or its contiguous range) into the ring;
//   compute warps   each thread scans its 32 items as (value, head) pairs
//                   (heads at the multiples of the row length), a warp scan
//                   of the pairs, then the CTA's warp totals through shared
//                   memory (one mbarrier phase per tile, bounded waits);
//                   results are written back into the stage;
//   store warp      TMA store of each finished stage; a stage is freed once
//                   its store has read it, with up to kRowsStoresInFlight
//                   newer stores still reading theirs.
//
// Each element is read once and written once.  The segmented form of the
// scan is that of "Lecture 7: Parallel pattern -- prefix sum / scan" (UIUC
// ECE408 notes), section 2 (a scan that restarts at segment heads); rows of a
// row-major matrix are segments of equal length.
#include "sc_segscan_tma.cuh"

namespace scg {

namespace {

using namespace persist;

constexpr int kRowsTileBytes = 32768;            // 256 rows of 128 bytes
constexpr int kRowsStages = 6;
constexpr int kRowsStoresInFlight = 3;           // TMA stores that may still read their stage
static_assert(kRowsStoresInFlight < kRowsStages, "a stage is freed before the producer needs it again");
constexpr int kRowsComputeWarps = 8;
constexpr int kRowsCompute = 32 * kRowsComputeWarps;
constexpr int kRowsProducer = kRowsComputeWarps;  // warp index
constexpr int kRowsStore = kRowsComputeWarps + 1;
constexpr int kRowsThreads = 32 * (kRowsComputeWarps + 2);
constexpr int kRowsTileRows = kRowsTileBytes / 128;

struct RowsCtrl {
    unsigned long long full[kRowsStages], empty[kRowsStages], written[kRowsStages];
    unsigned long long totals[kRowsStages];      // every compute warp wrote its total of the stage's tile
    uint2 wtot[kRowsStages][kRowsComputeWarps];  // (value bits, head flag) of each warp's part
    uint32_t red[kRowsComputeWarps];             // ragged rows: the first tile's read-back, per warp
};
constexpr int kRowsSmem = kRowsStages * kRowsTileBytes + 1024 + (int)sizeof(RowsCtrl);
static_assert(kRowsSmem <= 232448, "shared memory per CTA");

}  // namespace

template <class Op, bool kExcl, bool kRagged>
__global__ void __launch_bounds__(kRowsThreads, 1)
    rows_tma_kernel(const __grid_constant__ CUtensorMap tm_in, const __grid_constant__ CUtensorMap tm_out,
                    const ScanParams p, const long long n_full_tiles) {
    using T = typename Op::T;
    using PO = SegPairOp<Op>;
    using E = typename PO::E;
    constexpr int IPT = 32;
    constexpr int TILE = kRowsCompute * IPT;  // 8192 four-byte elements
    static_assert(sizeof(T) == 4 && TILE * 4 == kRowsTileBytes, "4-byte elements, one 128-byte row per thread");

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    RowsCtrl* ctl = reinterpret_cast<RowsCtrl*>(smem + kRowsStages * kRowsTileBytes);
    const uint32_t stage0 = smem_u32(smem);
    auto B = [](const unsigned long long& b) { return smem_u32(&b); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long num_tiles = p.n / TILE + (p.n % TILE != 0);
    // this CTA's tiles: blockIdx.x, blockIdx.x + gridDim.x, ...; ragged rows:
    // a contiguous range [t_begin, t_begin + my_tiles)
    long long my_tiles, t_begin = blockIdx.x;
    if constexpr (kRagged) {
        const long long q = num_tiles / gridDim.x, rem = num_tiles % gridDim.x;
        my_tiles = q + ((long long)blockIdx.x < rem);
        t_begin = (long long)blockIdx.x * q + min((long long)blockIdx.x, rem);
    } else {
        my_tiles = num_tiles > blockIdx.x ? (num_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    }
    auto tile_of = [&](long long i) -> long long { return kRagged ? t_begin + i : t_begin + i * gridDim.x; };
    const unsigned long long wait_limit = p.lb.timeout_ns + 500000000ull;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRowsStages; ++i) {
            mbar_init(B(ctl->full[i]), 1);
            mbar_init(B(ctl->empty[i]), 1);
            mbar_init(B(ctl->written[i]), kRowsComputeWarps);
            mbar_init(B(ctl->totals[i]), kRowsComputeWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    // ------------------------------------------------------------- producer
    if (warp == kRowsProducer) {
        if (lane != 0) return;
        const uint64_t once = l2_policy_evict_first();  // read once
        long long issued = -1;
        for (long long i = 0; i < my_tiles; ++i) {
            const int s = (int)(i % kRowsStages);
            if (i >= kRowsStages &&
                !bar_wait(B(ctl->empty[s]), (uint32_t)(((i / kRowsStages) - 1) & 1), wait_limit)) {
                raise_error(p.lb.error, DEV_LOOKBACK_TIMEOUT);
                break;
            }
            const long long t = tile_of(i);
            issued = i;
            if (t < n_full_tiles) {
                mbar_arrive_expect_tx(B(ctl->full[s]), kRowsTileBytes);
                tma_load_2d_hint(stage0 + s * kRowsTileBytes, &tm_in, 0, (int)(t * kRowsTileRows), B(ctl->full[s]),
                                 once);
            } else {
                mbar_arrive(B(ctl->full[s]));  // the ragged last tile: plain loads by the compute warps
            }
        }
        // every load must land before the CTA exits: wait for the stages'
        // newest fills (the store warp waits on each stage's later phases)
        for (long long i = issued - kRowsStages + 1 < 0 ? 0 : issued - kRowsStages + 1; i <= issued; ++i)
            bar_wait(B(ctl->full[i % kRowsStages]), (uint32_t)((i / kRowsStages) & 1), wait_limit);
        return;
    }

    // --------------------------------------------------------------- stores
    if (warp == kRowsStore) {
        if (lane != 0) return;
        const uint64_t once = l2_policy_evict_first();
        for (long long i = 0; i < my_tiles; ++i) {
            const int s = (int)(i % kRowsStages);
            if (!bar_wait(B(ctl->written[s]), (uint32_t)((i / kRowsStages) & 1), wait_limit)) {
                raise_error(p.lb.error, DEV_LOOKBACK_TIMEOUT);
                break;
            }
            const long long t = tile_of(i);
            if (t < n_full_tiles)
                tma_store_2d_hint(&tm_out, 0, (int)(t * kRowsTileRows), stage0 + s * kRowsTileBytes, once);
            bulk_commit();  // one group per tile (empty for the ragged tile, stored by the compute warps)
            bulk_wait_read<kRowsStoresInFlight>();
            if (i >= kRowsStoresInFlight) mbar_arrive(B(ctl->empty[(i - kRowsStoresInFlight) % kRowsStages]));
        }
        bulk_wait_all();
        return;
    }

    // -------------------------------------------------------------- compute
    const int ctid = threadIdx.x;  // row ctid of every tile (32 items)
    uint32_t off[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) off[j] = ctid * 128 + ((j ^ (ctid & 7)) << 4);
    // Heads of the thread's items from rr, the offset of its first item inside
    // its row; r0, that of the tile's first element.  Rows dividing the tile:
    // both the same in every tile.  Ragged: both advance by 8192 mod cols.
    const uint32_t cols = (uint32_t)p.seg_len;
    const uint32_t adv = (uint32_t)(TILE % cols);
    uint32_t rr = (uint32_t)(((kRagged ? (unsigned long long)t_begin * TILE : 0ull) + (unsigned)(ctid * IPT)) % cols);
    uint32_t r0 = kRagged ? (uint32_t)(((unsigned long long)t_begin * TILE) % cols) : 0u;
    auto heads = [&]() {
        uint32_t hm = 0;
        for (uint32_t k = rr == 0 ? 0u : cols - rr; k < (uint32_t)IPT; k += cols) hm |= 1u << k;
        return hm;
    };
    uint32_t hm = heads();
    // ragged rows: the fold of the current row up to the tile's start
    T carry = Op::identity();
    if constexpr (kRagged) {
        if (r0 != 0 && my_tiles > 0) {
            // the CTA's first tile: read back its row's first r0 elements, in
            // order (a contiguous part per thread, then warps, then the CTA)
            const T* src = static_cast<const T*>(p.in) + (t_begin * TILE - (long long)r0);
            const uint32_t per = (r0 + kRowsCompute - 1) / kRowsCompute;
            T acc = Op::identity();
            for (uint32_t j = ctid * per; j < min(r0, (uint32_t)(ctid + 1) * per); ++j) acc = Op::op(acc, src[j]);
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {  // ordered: lane 0 ends with lanes 0..31
                const T y = shfl_down_v(acc, d);
                if (lane + d < 32) acc = Op::op(acc, y);
            }
            if (lane == 0) ctl->red[warp] = to_bits32(acc);
            named_bar_sync(1, kRowsCompute);
            T c = Op::identity();
#pragma unroll
            for (int w = 0; w < kRowsComputeWarps; ++w) {
                T x;
                from_bits32(ctl->red[w], x);
                c = Op::op(c, x);
            }
            carry = c;
        }
    }
    for (long long i = 0; i < my_tiles; ++i) {
        const int s = (int)(i % kRowsStages);
        const long long t = tile_of(i);
        const bool full = t < n_full_tiles;
        if (!warp_bar_wait(B(ctl->full[s]), (uint32_t)((i / kRowsStages) & 1), wait_limit)) {
            if (lane == 0) raise_error(p.lb.error, DEV_LOOKBACK_TIMEOUT);
            break;
        }
        const uint32_t sb = stage0 + s * kRowsTileBytes;
        T v[IPT];
        if (full) {
#pragma unroll
            for (int j = 0; j < 8; ++j) unpack(lds128(sb + off[j]), &v[j * 4]);
        } else {
            load_partial_tile<T, IPT>(static_cast<const T*>(p.in) + t * TILE, v, p.n - t * TILE, Op::identity());
        }
        // the thread's (value, head) total, then the warp's inclusive scan of them
        T acc = v[0];
#pragma unroll
        for (int w = 1; w < IPT; ++w) acc = ((hm >> w) & 1u) ? v[w] : Op::op(acc, v[w]);
        E x = PO::make(acc, hm != 0u);
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const E y = shfl_up_v(x, d);
            if (lane >= d) x = PO::e_op(y, x);
        }
        if (lane == 31) ctl->wtot[s][warp] = x;
        __syncwarp();
        if (lane == 0) mbar_arrive(B(ctl->totals[s]));
        if (!warp_bar_wait(B(ctl->totals[s]), (uint32_t)((i / kRowsStages) & 1), wait_limit)) {
            if (lane == 0) raise_error(p.lb.error, DEV_LOOKBACK_TIMEOUT);
            break;
        }
        // carry into the thread: the tile's carry (ragged rows), the earlier
        // warps' totals, this warp's earlier lanes
        E wv = lane < kRowsComputeWarps ? ctl->wtot[s][lane] : PO::e_identity();
#pragma unroll
        for (int d = 1; d < kRowsComputeWarps; d <<= 1) {
            const E y = shfl_up_v(wv, d);
            if (lane >= d) wv = PO::e_op(y, wv);
        }
        E cin = shfl_up_v(x, 1);
        const E wpre = shfl_idx_v(wv, warp > 0 ? warp - 1 : 0);
        const E total = shfl_idx_v(wv, kRowsComputeWarps - 1);  // the whole tile's (fold since its last head, head)
        // the tile's first element starts a row unless r0 != 0 (ragged rows only)
        const bool tcarry = kRagged && r0 != 0;
        const E tp = tcarry ? PO::make(carry, false) : PO::e_identity();
        E before = warp > 0 ? wpre : tp;  // everything before this warp
        if (tcarry && warp > 0) before = PO::e_op(tp, wpre);
        if (lane == 0) cin = before;
        else if (warp > 0 || tcarry) cin = PO::e_op(before, cin);
        // the carry applies to the items before the thread's first head
        T run = PO::value(cin);
        if constexpr (kRagged) {
            // the next tile's carry: this tile's fold since its last head (a
            // full tile always holds one); then the next tile's row offsets
            carry = PO::value(total);
            r0 += adv;
            if (r0 >= cols) r0 -= cols;
            rr += adv;
            if (rr >= cols) rr -= cols;
        }
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
        if (full) {
#pragma unroll
            for (int j = 0; j < 8; ++j) sts128(sb + off[j], pack(&v[j * 4]));
            fence_proxy_async();  // before the store warp's TMA reads this stage
        } else {
            store_partial_tile<T, IPT>(static_cast<T*>(p.out) + t * TILE, v, p.n - t * TILE);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(B(ctl->written[s]));
        if constexpr (kRagged) hm = heads();
    }
}

// ----------------------------------------------------------------- host side
namespace {

template <class Op, bool kExcl, bool kRagged>
cudaError_t launch_rows_one(const ScanParams& p, unsigned grid, cudaStream_t s) {
    const long long tile = kRowsTileBytes / 4;
    const long long nfull = p.n / tile;
    CUtensorMap a, b;
    const unsigned long long rows = (unsigned long long)nfull * kRowsTileRows;
    if (nfull < 1 || !make_map(&a, p.in, rows, kRowsTileRows) || !make_map(&b, p.out, rows, kRowsTileRows))
        return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> done_mask{0};
    const cudaError_t e = allow_smem(rows_tma_kernel<Op, kExcl, kRagged>, kRowsSmem, done_mask);
    if (e != cudaSuccess) return e;
    rows_tma_kernel<Op, kExcl, kRagged><<<grid, kRowsThreads, kRowsSmem, s>>>(a, b, p, nfull);
    return cudaGetLastError();
}

template <class Op>
cudaError_t launch_rows_op(const ScanParams& p, bool exclusive, unsigned grid, cudaStream_t s) {
    if (kRowsTileBytes / 4 % p.seg_len == 0)
        return exclusive ? launch_rows_one<Op, true, false>(p, grid, s) : launch_rows_one<Op, false, false>(p, grid, s);
    return exclusive ? launch_rows_one<Op, true, true>(p, grid, s) : launch_rows_one<Op, false, true>(p, grid, s);
}

}  // namespace

int rows_tma_tile_elems() { return kRowsTileBytes / 4; }
bool rows_tma_supported(int oid) { return oid == OID_SUM_U32 || oid == OID_MAX_I32 || oid == OID_SUM_F32; }

cudaError_t launch_rows_tma(int oid, const ScanParams& p, bool exclusive, unsigned grid, cudaStream_t s) {
    switch (oid) {
    case OID_SUM_U32: return launch_rows_op<OpSumU32>(p, exclusive, grid, s);
    case OID_MAX_I32: return launch_rows_op<OpMaxI32>(p, exclusive, grid, s);
    case OID_SUM_F32: return launch_rows_op<OpSumF32>(p, exclusive, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace scg
