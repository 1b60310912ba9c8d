// Scans of the int32/uint32 product, and, or, xor (wraparound on the bits).
#include "sc_ops_common.cuh"

namespace scg {

cudaError_t launch_ops_int32_bits(int oid, const ScanParams& p, bool exclusive, bool segmented, unsigned tma_grid,
                                  cudaStream_t s) {
    switch (oid) {
    SC_OPS_CASE(OID_PROD_U32, OpProdU32)
    SC_OPS_CASE(OID_AND_U32, OpAndU32)
    SC_OPS_CASE(OID_OR_U32, OpOrU32)
    SC_OPS_CASE(OID_XOR_U32, OpXorU32)
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace scg
