// Kernel launchers (host side), one set per translation unit.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "sc_params.h"

namespace scg {

struct OpSumU32;
struct OpSumF32;
struct OpMaxI32;
struct OpAffineU32;

// Tile shape of the fused compaction: 256 threads x 16 items.
struct CompactConfig {
    static constexpr int NT = 256;
    static constexpr int IPT = 16;
    static constexpr int TILE = NT * IPT;
};

// Single-pass scan tile shapes.  Variant 0 is the default of every operator;
// the uint32 sum also carries alternative shapes (selected through the tuning
// hook) so that tile size, block size and loader can be compared on the GPU
// without a rebuild.
struct ScanShape {
    int nt;     // threads per CTA
    int ipt;    // items per thread
    int load;   // LOAD_DIRECT / LOAD_XPOSE
    int lb;     // look-back status words read per lane per round trip
    int minb;   // minimum resident CTAs per SM requested from the compiler
    int stats;  // 1: instrumented (phase timers), for measurement only
};

constexpr int kNumSumU32Variants = 15;

// Operator ids: one per (element type, operator) pair with distinct bits.
// int32 and uint32 share the sum, product and bitwise operators (the same
// bits), as do int64 and uint64.
enum ScanOpId : int {
    OID_SUM_U32 = 0, OID_SUM_F32 = 1, OID_MAX_I32 = 2, OID_AFFINE_U32 = 3,
    // the rest run through launch_scan_extra
    OID_PROD_U32 = 4, OID_AND_U32, OID_OR_U32, OID_XOR_U32, OID_MIN_I32, OID_MAX_U32, OID_MIN_U32,
    OID_SUM_U64, OID_PROD_U64, OID_AND_U64, OID_OR_U64, OID_XOR_U64, OID_MAX_I64, OID_MIN_I64, OID_MAX_U64,
    OID_MIN_U64, OID_MAX_F32, OID_MIN_F32, OID_SUM_F64, OID_MAX_F64, OID_MIN_F64, OID_MAXCOUNT_I32,
    OID_COUNT
};
constexpr int kFirstExtraOid = OID_PROD_U32;

// Epoch bits of the one-word float-float look-back status (float32 sums):
// calls with that carry run with epochs below 2^kFloat2EpochBits.
constexpr unsigned kFloat2EpochBits = 7;

// Element bytes of an operator id (4, or 8 for 64-bit types and pairs).
constexpr int oid_elem_bytes(int oid) {
    return (oid == OID_AFFINE_U32 || oid == OID_MAXCOUNT_I32 || (oid >= OID_SUM_U64 && oid <= OID_MIN_U64) ||
            oid == OID_SUM_F64 || oid == OID_MAX_F64 || oid == OID_MIN_F64)
               ? 8
               : 4;
}

// Tile size (elements) of operator `op_id` in the given variant; 0 if that
// variant does not exist.
int scan_tile_elems(int op_id, int variant);
// Persistent scans segmented by head flags (sc_segscan_tma.cu): tile
// elements, tiles per look-back chunk, the operators compiled, the launch.
int segscan_tma_tile_elems();
int segscan_tma_chunk_tiles();
bool segscan_tma_supported(int op_id);
cudaError_t launch_segscan_tma(int op_id, const ScanParams& p, bool exclusive, unsigned grid, cudaStream_t s);
cudaError_t launch_segscan_tma_bits(int op_id, const ScanParams& p, bool exclusive, unsigned grid, cudaStream_t s);
cudaError_t launch_segscan_tma_order(int op_id, const ScanParams& p, bool exclusive, unsigned grid, cudaStream_t s);
// Batched rows of at most one tile (sc_rows_tma.cu): a persistent kernel with
// no look-back (rows dividing the tile: every tile holds whole rows; other
// lengths: a contiguous range of tiles per CTA, the open row carried from tile
// to tile, out != in); the int32/uint32 sum, int32 max and float32 sum on
// 16-byte aligned arrays of at least one tile.
int rows_tma_tile_elems();
bool rows_tma_supported(int op_id);
cudaError_t launch_rows_tma(int op_id, const ScanParams& p, bool exclusive, unsigned grid, cudaStream_t s);
// Whether the uint32-sum shape `variant` has a segmented form (the others
// fall back to shape 0 for segmented scans and batched rows).
bool segmented_shape(int variant);
ScanShape scan_shape(int op_id, int variant);

// Scans of the operators from kFirstExtraOid on: the one-tile-per-CTA kernel
// (tma_grid == 0; plain or segmented) or the persistent kernel (shape 0) on
// tma_grid CTAs.  One translation unit per group of operators (sc_ops_*.cu).
cudaError_t launch_scan_extra(int oid, const ScanParams& p, bool exclusive, bool segmented, unsigned tma_grid,
                              cudaStream_t s);
cudaError_t launch_ops_int32_bits(int oid, const ScanParams&, bool, bool, unsigned, cudaStream_t);
cudaError_t launch_ops_int32_order(int oid, const ScanParams&, bool, bool, unsigned, cudaStream_t);
cudaError_t launch_ops_int64_bits(int oid, const ScanParams&, bool, bool, unsigned, cudaStream_t);
cudaError_t launch_ops_int64_order(int oid, const ScanParams&, bool, bool, unsigned, cudaStream_t);
cudaError_t launch_ops_float_a(int oid, const ScanParams&, bool, bool, unsigned, cudaStream_t);
cudaError_t launch_ops_float_b(int oid, const ScanParams&, bool, bool, unsigned, cudaStream_t);

template <class Op>
cudaError_t launch_scan(const ScanParams& p, bool exclusive, bool segmented, int variant, cudaStream_t s);
template <> cudaError_t launch_scan<OpSumU32>(const ScanParams&, bool, bool, int, cudaStream_t);
template <> cudaError_t launch_scan<OpSumF32>(const ScanParams&, bool, bool, int, cudaStream_t);
template <> cudaError_t launch_scan<OpMaxI32>(const ScanParams&, bool, bool, int, cudaStream_t);
template <> cudaError_t launch_scan<OpAffineU32>(const ScanParams&, bool, bool, int, cudaStream_t);

// Persistent TMA-pipelined scan (16-byte aligned arrays of at least one full
// tile, no segments).  Its look-back runs over chunks of chunk_tiles tiles:
// p.lb.num_tiles holds the number of chunks, and the counter advances by
// num_chunks + grid * tma_ids_per_cta() per launch.  Shape 0 is the default of
// every operator; shapes 1 .. tma_num_cfgs()-1 exist for the uint32 sum only.
// stats: instrumented build (uint32 sum, shape 0).
struct TmaShape {
    int tile_bytes;
    int chunk_tiles;
    int compute_threads;
    int threads;
    int ctas_per_sm;  // the grid is at most this many CTAs per SM
    int ids_per_cta;  // counter ticks per CTA beyond the chunks (see tma_ids_per_cta)
};
int tma_num_cfgs();
int tma_ids_per_cta();
bool tma_shape(int cfg, TmaShape* sh);
template <class Op>
cudaError_t launch_scan_tma(const ScanParams& p, bool exclusive, unsigned grid, cudaStream_t s, bool stats, int cfg);

template <class T>
cudaError_t launch_compact(const CompactParams& p, bool wide_count, cudaStream_t s);

// Persistent TMA-pipelined compaction (16-byte aligned input of at least one
// full tile): look-back over chunks of compact_tma_chunk_tiles() tiles of
// compact_tma_tile_elems() elements; p.lb.num_tiles holds the number of
// chunks; the counter advances by num_chunks + grid * tma_ids_per_cta().
int compact_tma_tile_elems();
int compact_tma_chunk_tiles();
template <class T>
cudaError_t launch_compact_tma(const CompactParams& p, bool wide_count, unsigned grid, cudaStream_t s, int shape);

// Histogram of int32 bins into uint64 counts (which the caller has zeroed);
// entries outside [0, nbins) are skipped.
cudaError_t launch_histogram(const int32_t* bins, long long n, int nbins, unsigned long long* counts, int num_sms,
                             cudaStream_t s);

// One radix-sort pass of uint32 keys by (k >> shift) & mask over tiles of
// radix_tile_keys() keys: the tiles' digit counts into counts[d * ntiles + t],
// then (after an exclusive scan of the counts in place) the placement.
int radix_tile_keys();
cudaError_t launch_radix_count(const uint32_t* keys, long long n, int shift, uint32_t mask, uint32_t* counts,
                               long long ntiles, cudaStream_t s);
// variant: 0 the default ranking, 1..radix_num_variants()-1 the ranking with
// variant - 1 digit bits matched by __match_any_sync (the rest by ballots).
int radix_num_variants();
cudaError_t launch_radix_place(const uint32_t* in, uint32_t* out, long long n, int shift, uint32_t mask,
                               const uint32_t* offsets, long long ntiles, unsigned int* error, int variant,
                               cudaStream_t s);

// The current look-back test hooks (sc_debug_set_lookback) copied into lb.
void lookback_hooks(LookbackCtl* lb);
// Status stride (LookbackCtl::stride_words) for `units` tiles or chunks whose
// statuses live in `area` bytes.
unsigned lookback_stride_words(size_t area, long long units);

// Hierarchical (scan-then-propagate) comparison variant.
constexpr int kHierNT = 256;
int hier_tile_elems(int op_id);
template <class Op>
cudaError_t launch_hier_tiles(const HierParams& p, bool exclusive, unsigned ntiles, cudaStream_t s);
template <class Op>
cudaError_t launch_hier_add(const HierParams& p, unsigned ntiles, cudaStream_t s);

}  // namespace scg
