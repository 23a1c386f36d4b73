// Backward instantiations for head dims (d_qk, d_v) = (64, 64).
#include "bwd_kernel.cuh"

namespace gdpa {

cudaError_t launch_bwd_d64(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                            cudaStream_t stream) {
  if (dtype == DT_FP16) return launch_bwd_cfg<64, 64, DT_FP16>(tq, tk, tv, tdo, tdq, a, grid, stream);
  return launch_bwd_cfg<64, 64, DT_BF16>(tq, tk, tv, tdo, tdq, a, grid, stream);
}

}  // namespace gdpa
