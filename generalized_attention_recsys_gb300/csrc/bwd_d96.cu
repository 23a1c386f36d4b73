// Backward instantiations for head dims (d_qk, d_v) = (96, 96).
#include "bwd_kernel.cuh"

namespace gdpa {

cudaError_t launch_bwd_d96(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                            cudaStream_t stream) {
  if (dtype == DT_FP16) return launch_bwd_cfg<96, 96, DT_FP16>(tq, tk, tv, tdo, tdq, a, grid, stream);
  return launch_bwd_cfg<96, 96, DT_BF16>(tq, tk, tv, tdo, tdq, a, grid, stream);
}

}  // namespace gdpa
