// Persistent single-pass scan: the compiled shapes and the instantiations for
// the int32/uint32 sum, float32 sum, int32 max and affine composition (the
// kernel itself is in sc_scan_tma.cuh).
#include "sc_scan_tma.cuh"

namespace scg {

int tma_num_cfgs() { return kNumCfgs; }
int tma_ids_per_cta() { return 1; }  // the id that ends the CTA's loop (ChunkIds)

bool tma_shape(int cfg, TmaShape* sh) {
    switch (cfg) {
    case 0: cfg_info<Cfg0>(sh); return true;
    case 1: cfg_info<Cfg1>(sh); return true;
    case 2: cfg_info<Cfg2>(sh); return true;
    case 3: cfg_info<Cfg3>(sh); return true;
    case 4: cfg_info<Cfg4>(sh); return true;
    case 5: cfg_info<Cfg5>(sh); return true;
    case 6: cfg_info<Cfg6>(sh); return true;
    case 7: cfg_info<Cfg7>(sh); return true;
    case 8: cfg_info<Cfg8>(sh); return true;
    case 9: cfg_info<Cfg9>(sh); return true;
    default: return false;
    }
}

template <class Op>
cudaError_t launch_scan_tma(const ScanParams& p, bool exclusive, unsigned grid, cudaStream_t s, bool stats, int cfg) {
    if (cfg == 0) return stats ? launch_cfg<Op, Cfg0>(p, exclusive, grid, s, true)
                               : launch_cfg<Op, typename DefaultCfg<Op>::type>(p, exclusive, grid, s, false);
    if constexpr (std::is_same<Op, OpSumU32>::value) {
        if (stats) return cudaErrorInvalidValue;
        switch (cfg) {
        case 1: return launch_cfg<Op, Cfg1>(p, exclusive, grid, s, false);
        case 2: return launch_cfg<Op, Cfg2>(p, exclusive, grid, s, false);
        case 3: return launch_cfg<Op, Cfg3>(p, exclusive, grid, s, false);
        case 4: return launch_cfg<Op, Cfg4>(p, exclusive, grid, s, false);
        case 5: return launch_cfg<Op, Cfg5>(p, exclusive, grid, s, false);
        case 6: return launch_cfg<Op, Cfg6>(p, exclusive, grid, s, false);
        case 7: return launch_cfg<Op, Cfg7>(p, exclusive, grid, s, false);
        case 8: return launch_cfg<Op, Cfg8>(p, exclusive, grid, s, false);
        case 9: return launch_cfg<Op, Cfg9>(p, exclusive, grid, s, false);
        default: break;
        }
    }
    return cudaErrorInvalidValue;
}

template cudaError_t launch_scan_tma<OpSumU32>(const ScanParams&, bool, unsigned, cudaStream_t, bool, int);
template cudaError_t launch_scan_tma<OpSumF32>(const ScanParams&, bool, unsigned, cudaStream_t, bool, int);
template cudaError_t launch_scan_tma<OpMaxI32>(const ScanParams&, bool, unsigned, cudaStream_t, bool, int);
template cudaError_t launch_scan_tma<OpAffineU32>(const ScanParams&, bool, unsigned, cudaStream_t, bool, int);

}  // namespace scg
