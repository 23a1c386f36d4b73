// Kernel argument blocks and the launchers each instantiation unit exports.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"

namespace gdpa {

// Launches `kernel` with programmatic dependent launch allowed (see
// pdl_wait in common.cuh): its blocks may start, and run up to pdl_wait,
// while the previous kernel on the stream is still finishing.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}


namespace {
// Sets a kernel's dynamic shared-memory limit once per device (attributes
// are per device). Internal linkage on purpose: a static local of a function
// template would be one object for every loaded copy of this library (the
// dynamic linker unifies such symbols), so a second copy would skip setting
// the attribute for its own kernels.
inline cudaError_t set_smem_limit_once(const void* kern, int bytes) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> g(mu);
  for (const auto& d : done)
    if (d.first == kern && d.second == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.emplace_back(kern, dev);
  return e;
}
}  // namespace

struct FwdArgs {
  Problem pb;
  int act;
  float scale;
  const float* descale;  // e4m3: (q, k, v) per-tensor scales; else NULL
  // MXFP8 (e4m3 codes with E8M0 block scales; NULL otherwise): q [total_q, h_q, d_qk / 32] and
  // k [total_k, h_kv, d_qk / 32] per 32 head-dim elements, v [ceil(total_k / 32), h_kv, d_v] per 32 keys
  const uint8_t* sf_q;
  const uint8_t* sf_k;
  const uint8_t* sf_v;
  // MXFP8: the same scales rearranged into 512-byte TMEM-copy atoms (workspace, written by a
  // kernel before the forward): per work item and 4-block group of q; per 32-key group (the
  // tile of 128 keys starting there) and kv head for k (4-block groups) and for v
  const uint8_t* atoms_q;
  const uint8_t* atoms_k;
  const uint8_t* atoms_v;
  void* out;             // [total_q, h_q, dv]; bf16 for bf16/e4m3 inputs, f16 for f16
  float* lse;            // [h_q, total_q] (softmax)
  const WorkList* work;
  int* status;  // device status word; a bounded wait that gave up writes 5 (timeout)
#ifdef GDPA_TEST_HOOKS
  int test_skip_step;  // test-only builds: CTA 0's activation warps skip the P-full arrive of this step
#endif
};

// How the backward produces dQ.
//   DQ_ACCUMULATE: TMA reduce-adds into an fp32 accumulator, converted after.
//   DQ_SLICES:     deterministic mode: each key block's dQ tile into its own
//                  fp32 slice, added in key-block order after.
//   DQ_DIRECT:     every sequence has at most one 128-row key block
//                  (max_k <= 128), so each dQ row has exactly one producer
//                  and the kernel writes it in the output type directly.
enum DqMode : int { DQ_ACCUMULATE = 0, DQ_SLICES = 1, DQ_DIRECT = 2 };

struct BwdArgs {
  Problem pb;
  int act;
  float scale;
  const WorkList* work;
  int* status;
  const void* out;   // softmax: forward output [total_q, h_q, dv]
  const float* lse;  // softmax: [h_q, total_q]
  const void* dout;  // [total_q, h_q, dv]
  void* dq;          // [total_q, h_q, dqk]
  void* dk;          // [total_k, h_kv, dqk]
  void* dv;          // [total_k, h_kv, dv]
  float* dq_acc;     // workspace: fp32 [total_q, h_q, dqk]
  float* dq_part;    // deterministic mode: fp32 [ceil(max_k / 128), total_q, h_q, dqk], one slice per
                     // key block; NULL otherwise
  float* drow;       // workspace: softmax rowsum(dO * O), [h_q, total_q]
#ifdef GDPA_TEST_HOOKS
  int test_skip_step;  // test-only builds: CTA 0's elementwise warps skip the dS-full arrive of this step
#endif
  int dq_mode;       // DQ_ACCUMULATE, DQ_SLICES (deterministic) or DQ_DIRECT
  int n_kblocks;     // ceil(max_k / 128): key blocks a sequence may have (checked on the device)
  int d_qk, d_v, dtype;
};

cudaError_t launch_fwd_d64(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const FwdArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_fwd_d96(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const FwdArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_fwd_d128(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_fwd_d192(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& a, int grid, cudaStream_t stream);

// Backward: dQ accumulator clear, (softmax) rowsum(dO * O), the main
// kernel, and the dQ conversion, all on `stream`.
// `before`/`after` (may be NULL) are recorded around the main kernel only.
cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid, cudaStream_t stream,
                       cudaEvent_t before, cudaEvent_t after);

}  // namespace gdpa
