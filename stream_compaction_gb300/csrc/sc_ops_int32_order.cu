// Scans of the int32 min, uint32 max and min.
#include "sc_ops_common.cuh"

namespace scg {

cudaError_t launch_ops_int32_order(int oid, const ScanParams& p, bool exclusive, bool segmented, unsigned tma_grid,
                                   cudaStream_t s) {
    switch (oid) {
    SC_OPS_CASE(OID_MIN_I32, OpMinI32)
    SC_OPS_CASE(OID_MAX_U32, OpMaxU32)
    SC_OPS_CASE(OID_MIN_U32, OpMinU32)
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace scg
