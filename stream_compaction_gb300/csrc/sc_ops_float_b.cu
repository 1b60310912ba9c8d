// Scans of the float64 max and min, (max, count) pairs.
#include "sc_ops_common.cuh"

namespace scg {

cudaError_t launch_ops_float_b(int oid, const ScanParams& p, bool exclusive, bool segmented, unsigned tma_grid,
                               cudaStream_t s) {
    switch (oid) {
    SC_OPS_CASE(OID_MAX_F64, OpMaxF64)
    SC_OPS_CASE(OID_MIN_F64, OpMinF64)
    SC_OPS_CASE(OID_MAXCOUNT_I32, OpMaxCount)
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace scg
