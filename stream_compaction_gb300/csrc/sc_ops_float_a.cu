// Scans of the float32 max and min, float64 sum.
#include "sc_ops_common.cuh"

namespace scg {

cudaError_t launch_ops_float_a(int oid, const ScanParams& p, bool exclusive, bool segmented, unsigned tma_grid,
                               cudaStream_t s) {
    switch (oid) {
    SC_OPS_CASE(OID_MAX_F32, OpMaxF32)
    SC_OPS_CASE(OID_MIN_F32, OpMinF32)
    SC_OPS_CASE(OID_SUM_F64, OpSumF64)
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace scg
