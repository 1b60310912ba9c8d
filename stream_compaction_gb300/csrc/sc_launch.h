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

// Tile size (elements) of operator `op_id` (0 sum u32, 1 sum f32, 2 max i32,
// 3 affine) in the given variant; 0 if that variant does not exist.
int scan_tile_elems(int op_id, int variant);
ScanShape scan_shape(int op_id, int variant);

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

// Hierarchical (scan-then-propagate) comparison variant.
constexpr int kHierNT = 256;
int hier_tile_elems(int op_id);
template <class Op>
cudaError_t launch_hier_tiles(const HierParams& p, bool exclusive, unsigned ntiles, cudaStream_t s);
template <class Op>
cudaError_t launch_hier_add(const HierParams& p, unsigned ntiles, cudaStream_t s);

}  // namespace scg
