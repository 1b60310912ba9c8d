// Persistent scans segmented by head flags: 32-bit min / max operators
// (integers in their own order, floats with NaN propagation; the kernel is in
// sc_segscan_tma.cuh).
#include "sc_segscan_tma.cuh"

namespace scg {

cudaError_t launch_segscan_tma_order(int oid, const ScanParams& p, bool exclusive, unsigned grid, cudaStream_t s) {
#define SC_SEG_CASE(ID, OP) \
    case ID: return exclusive ? launch_seg_one<OP, true>(p, grid, s) : launch_seg_one<OP, false>(p, grid, s);
    switch (oid) {
        SC_SEG_CASE(OID_MIN_I32, OpMinI32)
        SC_SEG_CASE(OID_MAX_U32, OpMaxU32)
        SC_SEG_CASE(OID_MIN_U32, OpMinU32)
        SC_SEG_CASE(OID_MAX_F32, OpMaxF32)
        SC_SEG_CASE(OID_MIN_F32, OpMinF32)
    default: return cudaErrorInvalidValue;
    }
#undef SC_SEG_CASE
}

}  // namespace scg
