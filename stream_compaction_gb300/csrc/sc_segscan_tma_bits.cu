// Persistent scans segmented by head flags: 32-bit product and bitwise
// operators (the kernel is in sc_segscan_tma.cuh).
#include "sc_segscan_tma.cuh"

namespace scg {

cudaError_t launch_segscan_tma_bits(int oid, const ScanParams& p, bool exclusive, unsigned grid, cudaStream_t s) {
#define SC_SEG_CASE(ID, OP) \
    case ID: return exclusive ? launch_seg_one<OP, true>(p, grid, s) : launch_seg_one<OP, false>(p, grid, s);
    switch (oid) {
        SC_SEG_CASE(OID_PROD_U32, OpProdU32)
        SC_SEG_CASE(OID_AND_U32, OpAndU32)
        SC_SEG_CASE(OID_OR_U32, OpOrU32)
        SC_SEG_CASE(OID_XOR_U32, OpXorU32)
    default: return cudaErrorInvalidValue;
    }
#undef SC_SEG_CASE
}

}  // namespace scg
