// Persistent scans segmented by head flags: the compiled operators (the
// kernel is in sc_segscan_tma.cuh).
#include "sc_segscan_tma.cuh"

namespace scg {

int segscan_tma_tile_elems() { return SegCfg::kTileBytes / 4; }
int segscan_tma_chunk_tiles() { return SegCfg::kChunk; }
// every operator with 4-byte elements whose carry is the element, and the
// float32 sum (float-float carry with the flag in its low bit)
bool segscan_tma_supported(int oid) {
    return oid == OID_SUM_U32 || oid == OID_SUM_F32 || oid == OID_MAX_I32 ||
           (oid >= OID_PROD_U32 && oid <= OID_MIN_U32) || oid == OID_MAX_F32 || oid == OID_MIN_F32;
}

cudaError_t launch_segscan_tma(int oid, const ScanParams& p, bool exclusive, unsigned grid, cudaStream_t s) {
    switch (oid) {
    case OID_SUM_U32:
        return exclusive ? launch_seg_one<OpSumU32, true>(p, grid, s) : launch_seg_one<OpSumU32, false>(p, grid, s);
    case OID_MAX_I32:
        return exclusive ? launch_seg_one<OpMaxI32, true>(p, grid, s) : launch_seg_one<OpMaxI32, false>(p, grid, s);
    case OID_SUM_F32:
        return exclusive ? launch_seg_one<OpSumF32, true>(p, grid, s) : launch_seg_one<OpSumF32, false>(p, grid, s);
    case OID_PROD_U32: case OID_AND_U32: case OID_OR_U32: case OID_XOR_U32:
        return launch_segscan_tma_bits(oid, p, exclusive, grid, s);
    case OID_MIN_I32: case OID_MAX_U32: case OID_MIN_U32: case OID_MAX_F32: case OID_MIN_F32:
        return launch_segscan_tma_order(oid, p, exclusive, grid, s);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace scg
