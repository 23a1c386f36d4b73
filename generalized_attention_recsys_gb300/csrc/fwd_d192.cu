// Forward instantiations for head dims (d_qk, d_v) = (192, 128).
#include "fwd_kernel.cuh"

namespace gdpa {

cudaError_t launch_fwd_d192(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& a, int grid, cudaStream_t stream) {
  switch (dtype) {
    case DT_BF16: return launch_fwd_cfg<192, 128, DT_BF16>(tq, tk, tv, a, grid, stream);
    case DT_FP16: return launch_fwd_cfg<192, 128, DT_FP16>(tq, tk, tv, a, grid, stream);
    default:
      if (a.sf_q != nullptr) return launch_fwd_mx<192, 128>(tq, tk, tv, a, grid, stream);  // MXFP8
      return launch_fwd_cfg<192, 128, DT_E4M3>(tq, tk, tv, a, grid, stream);
  }
}

}  // namespace gdpa
