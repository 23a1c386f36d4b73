// Backward instantiations for head dims (d_qk, d_v) = (192, 128): dK and dQ
// in two column parts (see bwd_kernel.cuh).
#include "bwd_kernel.cuh"

namespace gdpa {

cudaError_t launch_bwd_d192(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                            cudaStream_t stream) {
  if (dtype == DT_FP16) return launch_bwd_cfg<192, 128, DT_FP16>(tq, tk, tv, tdo, tdq, a, grid, stream);
  return launch_bwd_cfg<192, 128, DT_BF16>(tq, tk, tv, tdo, tdq, a, grid, stream);
}

}  // namespace gdpa
