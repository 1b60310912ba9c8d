// Persistent scans segmented by head flags: the compiled operators (the
// kernel is in sc_segscan_tma.cuh).
#include "sc_segscan_tma.cuh"

namespace scg {

int segscan_tma_tile_elems() { return SegCfg::kTileBytes / 4; }
int segscan_tma_chunk_tiles() { return SegCfg::kChunk; }
bool segscan_tma_supported(int oid) { return oid == OID_SUM_U32 || oid == OID_MAX_I32; }

cudaError_t launch_segscan_tma(int oid, const ScanParams& p, bool exclusive, unsigned grid, cudaStream_t s) {
    switch (oid) {
    case OID_SUM_U32:
        return exclusive ? launch_seg_one<OpSumU32, true>(p, grid, s) : launch_seg_one<OpSumU32, false>(p, grid, s);
    case OID_MAX_I32:
        return exclusive ? launch_seg_one<OpMaxI32, true>(p, grid, s) : launch_seg_one<OpMaxI32, false>(p, grid, s);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace scg
