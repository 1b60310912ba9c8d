// Scans of the int64/uint64 sum, product, and, or, xor (wraparound on the bits).
#include "sc_ops_common.cuh"

namespace scg {

cudaError_t launch_ops_int64_bits(int oid, const ScanParams& p, bool exclusive, bool segmented, unsigned tma_grid,
                                  cudaStream_t s) {
    switch (oid) {
    SC_OPS_CASE(OID_SUM_U64, OpSumU64)
    SC_OPS_CASE(OID_PROD_U64, OpProdU64)
    SC_OPS_CASE(OID_AND_U64, OpAndU64)
    SC_OPS_CASE(OID_OR_U64, OpOrU64)
    SC_OPS_CASE(OID_XOR_U64, OpXorU64)
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace scg
