// Backward launcher: for softmax computes rowsum(dO * O) (and, with direct dQ,
// zeroes the dq rows no work item writes), runs the main kernel, then
// converts the fp32 dQ accumulator (cleared by the work-list launch); in
// deterministic mode it adds the per-key-block dQ slices in a fixed order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "act.cuh"
#include "args.h"

namespace gdpa {

cudaError_t launch_bwd_d64(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                           cudaStream_t stream);
cudaError_t launch_bwd_d96(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                           cudaStream_t stream);
cudaError_t launch_bwd_d128(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                            cudaStream_t stream);
cudaError_t launch_bwd_d192(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                            cudaStream_t stream);

namespace {

__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }

// Softmax: drow[h, t] = sum_d dO[t, h, d] * O[t, h, d]. With direct dQ (zero_dq set),
// the rows of query blocks that no work item visits are zeroed in dq itself
// (every sequence has at most one key block, covering the query blocks that
// query_range gives; the kernel writes the rest).
template <typename T>
__global__ void __launch_bounds__(256) bwd_prep(const T* out, const T* dout, float* drow, int total_q, int h_q,
                                                int d_v, Problem pb, T* zero_dq, int d_qk) {
  pdl_wait();
  pdl_release();
  const size_t tid = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  const size_t nthr = static_cast<size_t>(gridDim.x) * blockDim.x;
  if (zero_dq != nullptr) {
    const size_t row_elems = static_cast<size_t>(h_q) * d_qk;  // one token: every head
    for (int b = static_cast<int>(tid / 32); b < pb.batch; b += static_cast<int>(nthr / 32)) {
      int qs, lq, ks, lk;
      seq_bounds(pb.cu_q, b, pb.max_q, qs, lq);
      seq_bounds(pb.cu_k, b, pb.max_k, ks, lk);
      int r0 = 0, r1 = 0;  // covered rows [r0, r1)
      int rmin, rmax;
      if (lq > 0 && lk > 0 && query_range(0, lk - 1, lq, lk, pb.causal, pb.window, rmin, rmax)) {
        r0 = (rmin / kTileQ) * kTileQ;
        r1 = min(lq, (rmax / kTileQ + 1) * kTileQ);
      }
      // [0, r0) and [r1, lq) are contiguous token ranges
      for (int part = 0; part < 2; ++part) {
        const int a0 = part == 0 ? 0 : r1, a1 = part == 0 ? r0 : lq;
        if (a1 <= a0) continue;
        T* base = zero_dq + static_cast<size_t>(qs + a0) * row_elems;
        const size_t n = static_cast<size_t>(a1 - a0) * row_elems;  // multiple of 8 elements (16 bytes)
        for (size_t i = (tid & 31) * 8; i < n; i += 32 * 8)
          *reinterpret_cast<uint4*>(base + i) = make_uint4(0, 0, 0, 0);
      }
    }
  }
  if (drow == nullptr) return;
  const size_t warp = tid / 32, nwarps = nthr / 32;
  const int lane = threadIdx.x & 31;
  const size_t rows = static_cast<size_t>(total_q) * h_q;
  for (size_t r = warp; r < rows; r += nwarps) {
    const T* o = out + r * d_v;
    const T* g = dout + r * d_v;
    float sum = 0.f;
    for (int d = lane; d < d_v; d += 32) sum += to_f(o[d]) * to_f(g[d]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) {
      const size_t t = r / h_q, h = r - t * h_q;
      drow[h * total_q + t] = sum;
    }
  }
}

template <typename T>
__device__ __forceinline__ void store4(T* dst, float4 v);
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(dst) = u;
}
template <>
__device__ __forceinline__ void store4<__half>(__half* dst, float4 v) {
  __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(dst) = u;
}

// Deterministic mode: dQ of each (token, head) row is the sum, in key-block
// order, of the slices written by the key blocks whose backward work item
// covered the row's 128-row query block (the same query_range test the work
// items use, so only written slices are read). One warp per row.
template <typename T>
__global__ void __launch_bounds__(256) bwd_post_ordered(const float* part, Problem pb, int d, int n_slices, T* dq) {
  pdl_wait();
  pdl_release();
  const int lane = threadIdx.x & 31;
  const size_t nwarps = static_cast<size_t>(gridDim.x) * (blockDim.x / 32);
  const size_t rows = static_cast<size_t>(pb.total_q) * pb.h_q;
  for (size_t r = blockIdx.x * static_cast<size_t>(blockDim.x / 32) + threadIdx.x / 32; r < rows; r += nwarps) {
    const int t = static_cast<int>(r / pb.h_q);
    int b;  // the sequence holding token t
    if (pb.cu_q == nullptr) {
      b = t / pb.max_q;
    } else {
      int lo = 0, hi = pb.batch - 1;  // last b with cu_q[b] <= t
      while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (pb.cu_q[mid] <= t) lo = mid;
        else hi = mid - 1;
      }
      b = lo;
    }
    int qs, lq, ks, lk;
    seq_bounds(pb.cu_q, b, pb.max_q, qs, lq);
    seq_bounds(pb.cu_k, b, pb.max_k, ks, lk);
    const int qb = (t - qs) / kTileQ;
    float acc[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // columns lane, lane + 32, ... (d <= 192)
    // the workspace holds n_slices; a longer key sequence (max_k understated)
    // was reported by the main kernel, which wrote no slice beyond them
    const int nkv = min(lk > 0 ? (lk + kTileK - 1) / kTileK : 0, n_slices);
    for (int j = 0; j < nkv; ++j) {
      const int k0 = j * kTileK, k1 = min(k0 + kTileK, lk) - 1;
      int rmin, rmax;
      if (!query_range(k0, k1, lq, lk, pb.causal, pb.window, rmin, rmax)) continue;
      if (qb < rmin / kTileQ || qb > rmax / kTileQ) continue;
      const float* src = part + (static_cast<size_t>(j) * pb.total_q * pb.h_q + r) * d;
#pragma unroll
      for (int m = 0; m < 6; ++m)
        if (lane + 32 * m < d) acc[m] += src[lane + 32 * m];
    }
#pragma unroll
    for (int m = 0; m < 6; ++m)
      if (lane + 32 * m < d) dq[r * d + lane + 32 * m] = from_f<T>(acc[m]);
  }
}

template <typename T>
__global__ void __launch_bounds__(256) bwd_post(const float4* acc, size_t n4, T* dq) {
  pdl_wait();
  pdl_release();
  const size_t tid = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  const size_t nthr = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = tid; i < n4; i += nthr) store4<T>(dq + 4 * i, acc[i]);
}

}  // namespace

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tdq, const BwdArgs& a, int grid, cudaStream_t stream, cudaEvent_t before,
                       cudaEvent_t after) {
  // (the accumulating mode's accumulator was cleared by the work-list launch)
  const bool direct = a.dq_mode == DQ_DIRECT;
  const size_t n4_post = a.dq_mode == DQ_ACCUMULATE ? static_cast<size_t>(a.pb.total_q) * a.pb.h_q * a.d_qk / 4 : 0;
  const int eg = grid * 8;  // elementwise kernels: 8 blocks of 256 per SM
  float* drow = a.act == ACT_SOFTMAX ? a.drow : nullptr;
  cudaError_t e = cudaSuccess;
  if (drow == nullptr && !direct) {
    // nothing to prepare
  } else if (a.dtype == DT_FP16) {
    e = launch_pdl(bwd_prep<__half>, dim3(eg), dim3(256), 0, stream, static_cast<const __half*>(a.out),
                   static_cast<const __half*>(a.dout), drow, a.pb.total_q, a.pb.h_q, a.d_v, a.pb,
                   direct ? static_cast<__half*>(a.dq) : nullptr, a.d_qk);
  } else {
    e = launch_pdl(bwd_prep<__nv_bfloat16>, dim3(eg), dim3(256), 0, stream,
                   static_cast<const __nv_bfloat16*>(a.out), static_cast<const __nv_bfloat16*>(a.dout), drow,
                   a.pb.total_q, a.pb.h_q, a.d_v, a.pb, direct ? static_cast<__nv_bfloat16*>(a.dq) : nullptr,
                   a.d_qk);
  }
  if (e != cudaSuccess) return e;
  if (before) cudaEventRecord(before, stream);
  switch (a.d_qk) {
    case 64: e = launch_bwd_d64(a.dtype, tq, tk, tv, tdo, tdq, a, grid, stream); break;
    case 96: e = launch_bwd_d96(a.dtype, tq, tk, tv, tdo, tdq, a, grid, stream); break;
    case 128: e = launch_bwd_d128(a.dtype, tq, tk, tv, tdo, tdq, a, grid, stream); break;
    case 192: e = launch_bwd_d192(a.dtype, tq, tk, tv, tdo, tdq, a, grid, stream); break;
    default: return cudaErrorNotSupported;
  }
  if (e != cudaSuccess) return e;
  if (after) cudaEventRecord(after, stream);
  if (direct) return cudaSuccess;  // dQ is already in place
  if (a.dq_mode == DQ_SLICES) {
    if (a.dtype == DT_FP16)
      return launch_pdl(bwd_post_ordered<__half>, dim3(eg), dim3(256), 0, stream, static_cast<const float*>(a.dq_part),
                        a.pb, a.d_qk, a.n_kblocks, static_cast<__half*>(a.dq));
    return launch_pdl(bwd_post_ordered<__nv_bfloat16>, dim3(eg), dim3(256), 0, stream,
                      static_cast<const float*>(a.dq_part), a.pb, a.d_qk, a.n_kblocks,
                      static_cast<__nv_bfloat16*>(a.dq));
  }
  if (a.dtype == DT_FP16)
    return launch_pdl(bwd_post<__half>, dim3(eg), dim3(256), 0, stream, reinterpret_cast<const float4*>(a.dq_acc),
                      n4_post, static_cast<__half*>(a.dq));
  return launch_pdl(bwd_post<__nv_bfloat16>, dim3(eg), dim3(256), 0, stream,
                    reinterpret_cast<const float4*>(a.dq_acc), n4_post, static_cast<__nv_bfloat16*>(a.dq));
}

}  // namespace gdpa
