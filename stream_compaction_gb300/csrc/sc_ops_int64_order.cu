// Scans of the int64 and uint64 max and min.
#include "sc_ops_common.cuh"

namespace scg {

cudaError_t launch_ops_int64_order(int oid, const ScanParams& p, bool exclusive, bool segmented, unsigned tma_grid,
                                   cudaStream_t s) {
    switch (oid) {
    SC_OPS_CASE(OID_MAX_I64, OpMaxI64)
    SC_OPS_CASE(OID_MIN_I64, OpMinI64)
    SC_OPS_CASE(OID_MAX_U64, OpMaxU64)
    SC_OPS_CASE(OID_MIN_U64, OpMinU64)
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace scg
