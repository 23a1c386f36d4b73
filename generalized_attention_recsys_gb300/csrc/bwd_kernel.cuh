// GDPA backward on sm_103a.
//
// For every sequence b, query head h and its kv head g (gdpa/README.md,
// "Features": forward and backward kernels; the gradients of
// O = where(M, act(scale * Q K^T), 0) V):
//   dV_g += P^T dO,  dP = dO V^T,  dS = scale * where(M, dP * act'(Z), 0),
//   dQ_h = dS K_g,   dK_g += dS^T Q_h.
// Softmax mode (Dao-AILab/flash-attention overview): P = exp(Z - lse),
// dS = scale * P * (dP - rowsum(dO * O)).
//
// A work item is one 128-row key block of one kv head. Its K and V tiles stay
// in shared memory while the CTA walks every query head of the kv head's
// group and every 128-row query block that sees the key block, so dK and dV
// accumulate in TMEM without atomics (GQA/MQA heads summed in place). dQ is
// reduced across key blocks into an fp32 workspace with TMA bulk tensor
// reduce-adds (one 32 x 32 box per warp and chunk) and converted at the end.
//
// All products are computed transposed so that TMEM lanes are key rows:
//   S^T  = K Q^T      (A = K   smem K-major,  B = Q   smem K-major)
//   dP^T = V dO^T     (A = V   smem K-major,  B = dO  smem K-major)
//   dV  += P^T dO     (A = P^T TMEM,          B = dO  smem MN-major)
//   dK  += dS^T Q     (A = dS^T smem K-major, B = Q   smem MN-major)
//   dQ   = dS K       (A = dS^T smem read MN-major, B = K smem MN-major)
// TMEM (512 columns): S^T [0,128) with P^T written over it, dP^T [128,256)
// reused for dQ once dP^T has been read, dV [256,256+dv), dK [384,384+dqk).
//
// d_qk = 192 (with d_v = 128): 192-column dK and dQ accumulators do not fit
// beside S^T, dP^T and dV, so dK and dQ are computed in column parts, [0,128)
// and [128,192), each part its own work item: both recompute S^T, P^T, dP^T
// and dS^T (the activation and its derivative), part 0 also computes dV. The
// two parts of a key block are neighbours in the work order, so they run at
// the same time on two CTAs and read K, V, Q and dO from L2 once. Shared
// memory then holds one Q stage: the next Q tile loads after dK has read the
// current one, and each step issues dQ and dK before the next S^T.
//
// Warp roles (128 * (NG + 2) threads): warp 0 TMA for K/V, warp 1 MMA,
// warp 2 TMA for Q, warp 3 TMA for dO, NG elementwise groups of four warps
// (128 / NG query columns of each tile each), then four warps that drain dQ
// from TMEM into the fp32 accumulator.
//
// Shared memory: K, V, two Q stages, one dO stage, the dS^T tile and the dQ
// staging ring (d = 128: 32 + 32 + 64 + 32 + 32 + 32 KB).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "act.cuh"
#include "args.h"
#include "common.cuh"
#include "sm100.cuh"

namespace gdpa {

// DIRECT_DQ_: the dQ drain writes each tile in the output type (one key
// block per sequence); otherwise it adds into fp32 (accumulator or slices).
// Separate instantiations, so neither drain carries the other's registers.
template <int DQK_, int DV_, int DT_, bool DIRECT_DQ_ = false>
struct BwdCfg {
  static constexpr int DQK = DQK_, DV = DV_, DT = DT_;
  static constexpr bool DIRECT_DQ = DIRECT_DQ_;
  static_assert(DT == DT_BF16 || DT == DT_FP16, "backward takes 16-bit inputs");
  static_assert((DQK <= 128 && DV <= 128) || (DQK == 192 && DV == 128), "backward head dims up to 128, or (192, 128)");
  // dK / dQ column parts: [0, PART_COLS0) and, for d_qk = 192, [128, 192)
  static constexpr int NPART = DQK > 128 ? 2 : 1;
  static constexpr int PART_COLS0 = DQK > 128 ? 128 : DQK;
  static constexpr int PART_COLS1 = DQK - PART_COLS0;
  static constexpr int PART_NCH_MAX = PART_COLS0 / 32;  // 32-column chunks of the wider part
  static constexpr int BOX_ELEMS = 64;
  static constexpr int BOX_BYTES = 128 * 128;
  static constexpr int QK_BOXES = (DQK + 63) / 64;
  static constexpr int V_BOXES = (DV + 63) / 64;
  static constexpr int K_BYTES = QK_BOXES * BOX_BYTES;
  static constexpr int V_BYTES = V_BOXES * BOX_BYTES;
  static constexpr int Q_BYTES = K_BYTES;
  static constexpr int DO_BYTES = V_BYTES;
  static constexpr int DS_BYTES = 2 * BOX_BYTES;
  // dO is single-buffered: its next tile loads while S^T, dQ, dK run
  static constexpr int Q_STAGES = DQK > 128 ? 1 : 2;
  static constexpr int DQ_CHUNK_BYTES = 32 * 128;              // 32 query rows x 32 fp32 columns
  static constexpr int DQ_STAGE_BYTES = 4 * 2 * DQ_CHUNK_BYTES;  // per drain warp: a ring of two chunks
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM_BYTES =
      1024 + K_BYTES + V_BYTES + Q_STAGES * Q_BYTES + DO_BYTES + DS_BYTES + DQ_STAGE_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= 232448, "tiles do not fit in shared memory");
  static constexpr int K_STEP = 16;
  static constexpr int S_MMAS = DQK / K_STEP;
  static constexpr int DP_MMAS = DV / K_STEP;
  static constexpr int T_MMAS = kTileQ / K_STEP;  // GEMMs whose K is a 128-row tile
  static constexpr uint32_t FMT = DT == DT_BF16 ? 1u : 0u;
  static constexpr uint32_t IDESC_S = idesc_make(128, 128, FMT, FMT, 0, 0);
  static constexpr uint32_t IDESC_DV = idesc_make(128, DV, FMT, FMT, 0, 1);
  static constexpr uint32_t IDESC_DK0 = idesc_make(128, PART_COLS0, FMT, FMT, 0, 1);
  static constexpr uint32_t IDESC_DQ0 = idesc_make(128, PART_COLS0, FMT, FMT, 1, 1);
  static constexpr uint32_t IDESC_DK1 = idesc_make(128, NPART > 1 ? PART_COLS1 : PART_COLS0, FMT, FMT, 0, 1);
  static constexpr uint32_t IDESC_DQ1 = idesc_make(128, NPART > 1 ? PART_COLS1 : PART_COLS0, FMT, FMT, 1, 1);
  static constexpr int NG = 2;             // elementwise groups (4 warps each), 64 query columns each
  static constexpr int GCOLS = kTileQ / NG;  // query columns per group
  static constexpr int GCHUNKS = GCOLS / 16;
  static constexpr int THREADS = 128 * (NG + 2);
  static constexpr int ACT_WARP0 = 4, DRAIN_WARP0 = 4 + 4 * NG;
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DQ = 128, T_DV = 256, T_DK = 384;

};

struct BwdItem {
  int g, part, k0, q_start, lq, k_start, lk, krows;
  int qlo, nq, nsteps;
};

// Item pos: work-list entry pos / (h_kv npart), then its column part, then the kv head.
__device__ __forceinline__ BwdItem bwd_decode(const BwdArgs& a, int pos, int npart) {
  BwdItem it;
  const Problem& pb = a.pb;
  const int per = pb.h_kv * npart;
  const int e = pos / per;
  const int r = pos - e * per;
  it.part = npart > 1 ? r / pb.h_kv : 0;
  it.g = r - it.part * pb.h_kv;
  const int4 sq = a.work->items[e].seq, bk = a.work->items[e].blk;
  it.q_start = sq.x;
  it.lq = sq.y;
  it.k_start = sq.z;
  it.lk = sq.w;
  it.k0 = bk.x;
  it.krows = bk.y;
  it.qlo = bk.z;
  it.nq = bk.w;
  it.nsteps = it.nq * pb.group;
  return it;
}

// The item's column part, a compile-time 0 when there is only one.
template <class C>
__device__ __forceinline__ int item_part(const BwdItem& it) {
  return C::NPART > 1 ? it.part : 0;
}

// Query head and first row of step s of an item.
__device__ __forceinline__ void bwd_step(const BwdItem& it, const Problem& pb, int s, int& h, int& q0) {
  const int hh = s / it.nq;
  h = it.g * pb.group + hh;
  q0 = (it.qlo + (s - hh * it.nq)) * kTileQ;
}

struct BwdSmem {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2], do_full, do_empty;
  uint64_t s_full, dp_full, p_full, ds_full, dq_full, dq_empty, acc_full, acc_empty;
  uint64_t drain;    // abort path: every MMA the issuing warp issued has completed
  uint32_t tmem_base;
  int abort_flag;
  int drain_failed;  // abort path: a role's in-flight work did not land in time
};

template <int DT>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  return DT == DT_BF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}

// The elementwise step runs in two passes per tile so that the tensor core
// keeps working meanwhile (thread = key row `row`, group w owns query columns
// [64 w, 64 w + 64)):
//   pass 1 (needs S^T only; dP^T is still being computed): P^T = act(Z^T)
//     and G^T = scale * act'(Z^T) (softmax: G^T = P^T), masked entries 0,
//     both packed to 16 bits and written over the S^T columns just read:
//     for query columns [64w + 32c, +32), P^T at TMEM column 64w + 32c and
//     G^T at 64w + 32c + 16.
//   pass 2 (needs dP^T; dV = P^T dO already runs): dS^T = dP^T * G^T
//     (softmax: scale * G^T (dP^T - rowsum(dO O))) into the swizzled smem tile.
template <class C>
__host__ __device__ constexpr uint32_t pt_col(int k) {  // P^T columns of MMA k-step k (query cols 16k..16k+15)
  return 64 * (k / 4) + 32 * ((k % 4) / 2) + 8 * (k % 2);
}

template <class C, int ACT, bool MASKED>
__device__ __forceinline__ void bwd_pass1(uint32_t t_lane, int w, const BwdConsts& k, int c_lo, int c_hi,
                                          const float* lse, int col_base, int col_max) {
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    // chunk c's outputs land only in chunk c's own 32 S^T columns
    const int col0 = 64 * w + 32 * c;
    uint32_t cur[32];
    tmem_ld32(t_lane + C::T_S + col0, cur);
    tmem_ld_wait(cur);
    uint32_t pk[16], gk[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float p0, p1, g0, g1;
      if constexpr (ACT == ACT_SOFTMAX) {
        const f2_t sv = f2(__uint_as_float(cur[e]), __uint_as_float(cur[e + 1]));
        const int i0 = min(col_base + col0 + e, col_max), i1 = min(col_base + col0 + e + 1, col_max);
        const f2_t a = fma2(sv, f2(k.scale * kLog2e), f2(-__ldg(lse + i0) * kLog2e, -__ldg(lse + i1) * kLog2e));
        p0 = g0 = ex2_approx(f2_lo(a));
        p1 = g1 = ex2_approx(f2_hi(a));
      } else if constexpr (act_scalar_grad_form(ACT)) {
        hardswish_grad(__uint_as_float(cur[e]), k, p0, g0);
        hardswish_grad(__uint_as_float(cur[e + 1]), k, p1, g1);
      } else {
        f2_t pv, gv;
        act_pair_grad<ACT>(f2(__uint_as_float(cur[e]), __uint_as_float(cur[e + 1])), k, pv, gv);
        p0 = f2_lo(pv);
        p1 = f2_hi(pv);
        g0 = f2_lo(gv);
        g1 = f2_hi(gv);
      }
      if (MASKED) {
        const bool ok0 = (col0 + e) >= c_lo && (col0 + e) <= c_hi;
        const bool ok1 = (col0 + e + 1) >= c_lo && (col0 + e + 1) <= c_hi;
        p0 = ok0 ? p0 : 0.0f;
        g0 = ok0 ? g0 : 0.0f;
        p1 = ok1 ? p1 : 0.0f;
        g1 = ok1 ? g1 : 0.0f;
      }
      pk[e / 2] = pack16<C::DT>(p0, p1);
      gk[e / 2] = pack16<C::DT>(g0, g1);
    }
    tmem_st16(t_lane + C::T_S + col0, pk);
    tmem_st16(t_lane + C::T_S + col0 + 16, gk);
  }
}

template <int DT>
__device__ __forceinline__ float unpack_lo(uint32_t v) {
  if constexpr (DT == DT_BF16) return __uint_as_float(v << 16);
  else return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
}
template <int DT>
__device__ __forceinline__ float unpack_hi(uint32_t v) {
  if constexpr (DT == DT_BF16) return __uint_as_float(v & 0xFFFF0000u);
  else return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
}

template <class C, bool SOFTMAX>
__device__ __forceinline__ void bwd_pass2(uint32_t t_lane, uint8_t* sDS, int row, int w, float scale,
                                          const float* drow, int col_base, int col_max) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int col0 = 64 * w + 32 * c;
    uint32_t dp[32], g[16];
    tmem_ld32(t_lane + C::T_DP + col0, dp);
    tmem_ld16(t_lane + C::T_S + col0 + 16, g);
    tmem_ld_wait(dp);
    tmem_ld_wait(g);
    uint32_t dk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      f2_t gv = f2(unpack_lo<C::DT>(g[e]), unpack_hi<C::DT>(g[e]));
      f2_t dv = f2(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1]));
      if constexpr (SOFTMAX) {
        const int i0 = min(col_base + col0 + 2 * e, col_max), i1 = min(col_base + col0 + 2 * e + 1, col_max);
        dv = add2(dv, f2(-__ldg(drow + i0), -__ldg(drow + i1)));
        gv = mul2(gv, f2(scale));
      }
      const f2_t ds = mul2(dv, gv);
      dk[e] = pack16<C::DT>(f2_lo(ds), f2_hi(ds));
    }
    // dS^T row `row`, query columns col0..col0+31: box w, 16-byte chunks 4c..4c+3, XOR-swizzled by row
    uint8_t* base = sDS + w * C::BOX_BYTES + row * 128;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(base + (((4 * c + q) ^ (row & 7)) << 4)) =
          make_uint4(dk[4 * q], dk[4 * q + 1], dk[4 * q + 2], dk[4 * q + 3]);
  }
}

// Whether S^T(t+1) is issued before dQ(t). dQ first starts the dQ drain,
// which frees the columns dP^T(t+1) needs, one GEMM earlier; S^T first
// starts the next elementwise pass 1 one GEMM earlier. Measured on the jagged
// self-attention workload (d = 128): dQ first gains 1.5-3.5% for the
// activations whose pass 1 is a few operations (identity, ReLU, ReLU^2,
// LeakyReLU) and loses 2-6% for the others.
__host__ __device__ constexpr bool bwd_s_first(int act) {
  return !(act == ACT_IDENTITY || act == ACT_RELU || act == ACT_RELU2 || act == ACT_LEAKY_RELU);
}

template <class C, bool MASKED>
__device__ __forceinline__ void bwd_pass1_dispatch(int act, uint32_t t_lane, int w, const BwdConsts& k, int c_lo,
                                                   int c_hi, const float* lse, int col_base, int col_max) {
#define GDPA_BWD_CASE(A) \
  case A: bwd_pass1<C, A, MASKED>(t_lane, w, k, c_lo, c_hi, lse, col_base, col_max); break;
  switch (act) {
    GDPA_BWD_CASE(ACT_IDENTITY)
    GDPA_BWD_CASE(ACT_GELU)
    GDPA_BWD_CASE(ACT_GELU_TANH)
    GDPA_BWD_CASE(ACT_FAST_GELU)
    GDPA_BWD_CASE(ACT_RELU)
    GDPA_BWD_CASE(ACT_RELU2)
    GDPA_BWD_CASE(ACT_LEAKY_RELU)
    GDPA_BWD_CASE(ACT_SILU)
    GDPA_BWD_CASE(ACT_HARDSWISH)
    GDPA_BWD_CASE(ACT_FAST_GELU_BF16)
    GDPA_BWD_CASE(ACT_FAST_SILU)
    default: bwd_pass1<C, ACT_SOFTMAX, MASKED>(t_lane, w, k, c_lo, c_hi, lse, col_base, col_max);
  }
#undef GDPA_BWD_CASE
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    gdpa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const BwdArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::K_BYTES;
  uint8_t* sQ = sV + C::V_BYTES;                 // Q_STAGES x Q_BYTES
  uint8_t* sDO = sQ + C::Q_STAGES * C::Q_BYTES;  // one dO tile
  uint8_t* sDS = sDO + C::DO_BYTES;              // 128 key rows x 128 query columns
  uint8_t* sDQ = sDS + C::DS_BYTES;              // dQ staging for the TMA reduce-adds
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(sDQ + C::DQ_STAGE_BYTES);
  static_assert(sizeof(BwdSmem) <= C::BAR_BYTES, "barrier block too large");

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const Problem& pb = args.pb;
  const int G = gridDim.x;
  volatile int* abort_flag = &sm.abort_flag;

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1);
    }
    mbar_init(&sm.do_full, 1);
    mbar_init(&sm.do_empty, 1);
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.dp_full, 1);
    mbar_init(&sm.p_full, 128 * C::NG);
    mbar_init(&sm.ds_full, 128 * C::NG);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_empty, 128);
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_empty, 128 * C::NG);
    mbar_init(&sm.drain, 1);
    sm.drain_failed = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
    prefetch_tmap(&tm_dq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  pdl_wait();  // the work list, the cleared accumulator and the inputs come from earlier kernels
  // read only after the wait: the work list is the previous kernel's output
  const int n_work = args.work->count * pb.h_kv * C::NPART;
  pdl_release();
  // registers: control warpgroup 96, elementwise warpgroups 160, drain warpgroup 96
  // (128 * 96 + 256 * 160 + 128 * 96 = 65536 = 512 * 128 launched)
  static_assert(C::NG == 2 && C::THREADS == 512, "register split assumes two elementwise warpgroups");
  static_assert(128 * 96 + 256 * 160 + 128 * 96 <= C::THREADS * 128, "register split exceeds the launch");

  if (warp < C::ACT_WARP0) regs_dec<96>();  // each role sets its warpgroup's budget first

  if (warp == 0 || warp == 2 || warp == 3) {
    // ------------------------------------------------ TMA producers
    // warp 0 loads each item's K and V, warp 2 streams the Q tile and warp 3
    // the dO tile of every step, so the next item's first tiles load while
    // the current item still holds K and V.
    if (lane == 0) {
      uint32_t kv_cnt = 0, st_it = 0, issued = 0;  // issued: K/V, Q or dO loads of this thread
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int pos = zigzag_pos(round, blockIdx.x, G);
        if (pos >= n_work) break;
        const BwdItem it = bwd_decode(args, pos, C::NPART);
        if (it.nsteps == 0) continue;
        if (warp == 0) {
          ok = mbar_wait(&sm.kv_empty, (kv_cnt++ & 1) ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&sm.kv_full, C::K_BYTES + C::V_BYTES);
          for (int bx = 0; bx < C::QK_BOXES; ++bx)
            tma_load_3d(sK + bx * C::BOX_BYTES, &tm_k, &sm.kv_full, bx * 64, it.g, it.k_start + it.k0);
          for (int bx = 0; bx < C::V_BOXES; ++bx)
            tma_load_3d(sV + bx * C::BOX_BYTES, &tm_v, &sm.kv_full, bx * 64, it.g, it.k_start + it.k0);
          issued = kv_cnt;
          continue;
        }
        for (int s = 0; s < it.nsteps && ok; ++s, ++st_it) {
          int h, q0;
          bwd_step(it, pb, s, h, q0);
          if (warp == 2) {
            const int st = st_it % C::Q_STAGES;
            ok = mbar_wait(&sm.q_empty[st], ((st_it / C::Q_STAGES) & 1) ^ 1, abort_flag);
            if (!ok) break;
            mbar_arrive_expect_tx(&sm.q_full[st], C::Q_BYTES);
            for (int bx = 0; bx < C::QK_BOXES; ++bx)
              tma_load_3d(sQ + st * C::Q_BYTES + bx * C::BOX_BYTES, &tm_q, &sm.q_full[st], bx * 64, h,
                          it.q_start + q0);
            issued = st_it + 1;
          } else {
            ok = mbar_wait(&sm.do_empty, (st_it & 1) ^ 1, abort_flag);
            if (!ok) break;
            mbar_arrive_expect_tx(&sm.do_full, C::DO_BYTES);
            for (int bx = 0; bx < C::V_BOXES; ++bx)
              tma_load_3d(sDO + bx * C::BOX_BYTES, &tm_do, &sm.do_full, bx * 64, h, it.q_start + q0);
            issued = st_it + 1;
          }
        }
      }
      if (*abort_flag) {  // let this thread's last loads land before the tiles go away
        bool landed = true;
        if (warp == 0 && issued > 0) landed = mbar_wait_timed(&sm.kv_full, (issued - 1) & 1, kDrainTimeoutNs);
        if (warp == 2)
          for (uint32_t i = 0; i < issued && i < static_cast<uint32_t>(C::Q_STAGES); ++i) {
            const uint32_t n = issued - 1 - i;
            landed = mbar_wait_timed(&sm.q_full[n % C::Q_STAGES], (n / C::Q_STAGES) & 1, kDrainTimeoutNs) && landed;
          }
        if (warp == 3 && issued > 0) landed = mbar_wait_timed(&sm.do_full, (issued - 1) & 1, kDrainTimeoutNs);
        if (!landed) sm.drain_failed = 1;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (whole warp; one elected lane issues)
    {
      // descriptors of every operand tile, built once; the K steps add byte offsets
      const uint64_t dK_k = sdesc_sw128(smem_u32(sK), 16, 1024);            // K, K-major (A of S^T)
      const uint64_t dK_mn = sdesc_sw128(smem_u32(sK), C::BOX_BYTES, 1024);  // K, MN-major (B of dQ)
      const uint64_t dV_k = sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t dQ_k = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dQ_mn = sdesc_sw128(smem_u32(sQ), C::BOX_BYTES, 1024);
      const uint64_t dDO_k = sdesc_sw128(smem_u32(sDO), 16, 1024);
      const uint64_t dDO_mn = sdesc_sw128(smem_u32(sDO), C::BOX_BYTES, 1024);
      const uint64_t dDS_k = sdesc_sw128(smem_u32(sDS), 16, 1024);
      const uint64_t dDS_mn = sdesc_sw128(smem_u32(sDS), C::BOX_BYTES, 1024);
      auto issue_s = [&](int st) {
#pragma unroll
        for (int k = 0; k < C::S_MMAS; ++k) {
          const uint32_t off = (k / 4) * C::BOX_BYTES + (k % 4) * 32;
          mma_f16_ss_w(tbase + C::T_S, sdesc_at(dK_k, off), sdesc_at(dQ_k, st * C::Q_BYTES + off), C::IDESC_S, k > 0);
        }
      };
      auto issue_dp = [&]() {
#pragma unroll
        for (int k = 0; k < C::DP_MMAS; ++k) {
          const uint32_t off = (k / 4) * C::BOX_BYTES + (k % 4) * 32;
          mma_f16_ss_w(tbase + C::T_DP, sdesc_at(dV_k, off), sdesc_at(dDO_k, off), C::IDESC_S, k > 0);
        }
      };
      auto issue_dv = [&](bool acc) {  // dV += P^T dO (A = P^T from TMEM)
#pragma unroll
        for (int k = 0; k < C::T_MMAS; ++k)
          mma_f16_ts_w(tbase + C::T_DV, tbase + C::T_S + pt_col<C>(k), sdesc_at(dDO_mn, k * 2048), C::IDESC_DV,
                       (acc || k > 0) ? 1u : 0u);
      };
      // dQ and dK of column part `part` (columns from 128 part: 64-column boxes 2 part on)
      auto issue_dq = [&](int part) {  // dQ = dS K
        const uint32_t boff = part * 2 * C::BOX_BYTES;
        const uint32_t idesc = part ? C::IDESC_DQ1 : C::IDESC_DQ0;
#pragma unroll
        for (int k = 0; k < C::T_MMAS; ++k)
          mma_f16_ss_w(tbase + C::T_DQ, sdesc_at(dDS_mn, k * 2048), sdesc_at(dK_mn, boff + k * 2048), idesc, k > 0);
        mma_commit_w(&sm.dq_full);
      };
      auto issue_dk = [&](int st, bool acc, int part) {  // dK += dS^T Q
        const uint32_t boff = part * 2 * C::BOX_BYTES;
        const uint32_t idesc = part ? C::IDESC_DK1 : C::IDESC_DK0;
#pragma unroll
        for (int k = 0; k < C::T_MMAS; ++k) {
          const uint32_t off = (k / 4) * C::BOX_BYTES + (k % 4) * 32;
          mma_f16_ss_w(tbase + C::T_DK, sdesc_at(dDS_k, off), sdesc_at(dQ_mn, st * C::Q_BYTES + boff + k * 2048), idesc,
                       (acc || k > 0) ? 1u : 0u);
        }
      };
      // Issue order per item (steps t = 0..n-1):
      //   S^T(0), dP^T(0), dV(0), then for each t either
      //   S^T(t+1), dQ(t), dK(t), dP^T(t+1), dV(t+1)   (bwd_s_first) or
      //   dQ(t), S^T(t+1), dK(t), dP^T(t+1), dV(t+1).
      // Pass 1 of step t+1 (needs S^T(t+1) only) overlaps dQ(t), dK(t) and
      // dP^T(t+1); pass 2 overlaps dV. S^T(t+1) may overwrite P^T/G^T(t)
      // and dQ(t) the dP^T(t) columns because dV(t) was issued before them
      // and pass 2(t) has finished; dQ's drain overlaps dK, before dP^T(t+1)
      // reuses the dQ columns; the commit after dP^T(t+1) also covers dQ(t)
      // and dK(t), so pass 2(t+1) may overwrite the dS tile they read.
      // With one Q stage, Q(t+1) loads only once dK(t) has read Q(t), so the
      // order is dK(t), dQ(t), S^T(t+1), dP^T(t+1), dV(t+1). Column part 1
      // (d_qk = 192) computes no dV: dP^T is then its dO tile's last reader.
      const bool s_first = bwd_s_first(args.act);
      uint32_t kv_cnt = 0, qd_it = 0, p_cnt = 0, ds_cnt = 0, dqe = 0, acce = 0;
      bool ok = true;
      // every lane waits; the warp goes on only if all of them succeeded
      auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
      };
      auto issue_s_at = [&](uint32_t it_idx) -> bool {
        const int st = it_idx % C::Q_STAGES;
        if (!wait_all(&sm.q_full[st], (it_idx / C::Q_STAGES) & 1)) return false;
        tc_fence_after();
        issue_s(st);
        mma_commit_w(&sm.s_full);
        return true;
      };
      auto issue_dp_dv_at = [&](uint32_t it_idx, bool first, int part) -> bool {
        if (!wait_all(&sm.dq_empty, (dqe++ & 1) ^ 1)) return false;
        if (!wait_all(&sm.do_full, it_idx & 1)) return false;
        tc_fence_after();
        issue_dp();
        mma_commit_w(&sm.dp_full);
        if (part != 0) mma_commit_w(&sm.do_empty);  // no dV: dP^T is the last reader of this dO tile
        if (!wait_all(&sm.p_full, p_cnt++ & 1)) return false;
        // the previous item's dV / dK epilogue has read TMEM before this item's first dV / dK
        if (first && !wait_all(&sm.acc_empty, (acce++ & 1) ^ 1)) return false;
        if (part == 0) {
          tc_fence_after();
          issue_dv(!first);
          mma_commit_w(&sm.do_empty);  // dV is the last reader of this dO tile
        }
        return true;
      };
      for (int round = 0; ok; ++round) {
        const int pos = zigzag_pos(round, blockIdx.x, G);
        if (pos >= n_work) break;
        const BwdItem it = bwd_decode(args, pos, C::NPART);
        if (it.nsteps == 0) continue;
        ok = wait_all(&sm.kv_full, kv_cnt++ & 1);
        if (ok) ok = issue_s_at(qd_it);
        if (ok) ok = issue_dp_dv_at(qd_it, true, item_part<C>(it));
        for (int s = 0; s < it.nsteps && ok; ++s) {
          const int st = qd_it % C::Q_STAGES;
          const bool more = s + 1 < it.nsteps;
          ok = wait_all(&sm.ds_full, ds_cnt++ & 1);
          if (!ok) break;
          if (C::Q_STAGES > 1 && s_first && more && !issue_s_at(qd_it + 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (C::Q_STAGES == 1) {  // dK first: the next Q tile loads while dQ runs
            issue_dk(st, s > 0, item_part<C>(it));
            mma_commit_w(&sm.q_empty[st]);
          }
          issue_dq(item_part<C>(it));
          if (C::Q_STAGES > 1 && !s_first && more && !issue_s_at(qd_it + 1)) {
            ok = false;
            break;
          }
          if (C::Q_STAGES > 1) {
            issue_dk(st, s > 0, item_part<C>(it));
            mma_commit_w(&sm.q_empty[st]);
          }
          if (C::Q_STAGES == 1 && more && !issue_s_at(qd_it + 1)) {
            ok = false;
            break;
          }
          ++qd_it;
          if (!more) {
            mma_commit_w(&sm.acc_full);
            mma_commit_w(&sm.kv_empty);
          } else {
            ok = issue_dp_dv_at(qd_it, false, item_part<C>(it));
          }
        }
      }
      if (*abort_flag) {  // every MMA this warp issued has completed before TMEM goes away
        mma_commit_w(&sm.drain);
        if (!__all_sync(0xffffffffu, mbar_wait_timed(&sm.drain, 0, kDrainTimeoutNs)) && lane == 0)
          sm.drain_failed = 1;
      }
    }
  } else if (warp >= C::ACT_WARP0 && warp < C::DRAIN_WARP0) {
    // ------------------------------------------------ elementwise groups + dK/dV epilogue
    regs_inc<160>();
    const int w = (warp - C::ACT_WARP0) / 4;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // key row within the block
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    using T = typename std::conditional<C::DT == DT_FP16, __half, __nv_bfloat16>::type;
    const bool softmax = args.act == ACT_SOFTMAX;
    const BwdConsts bwd_k = make_bwd_consts(args.scale);
    uint32_t s_cnt = 0, dp_cnt = 0, acc_cnt = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int pos = zigzag_pos(round, blockIdx.x, G);
      if (pos >= n_work) break;
      const BwdItem it = bwd_decode(args, pos, C::NPART);
      const int kk = it.k0 + row;
      const bool row_valid = row < it.krows;
      // the epilogue splits the 32-column chunks of dV (column part 0 only)
      // then of this part's dK columns round-robin over the groups
      const size_t krow = static_cast<size_t>(it.k_start + kk) * pb.h_kv + it.g;
      T* dv_row = reinterpret_cast<T*>(args.dv) + krow * C::DV;
      T* dk_row = reinterpret_cast<T*>(args.dk) + krow * C::DQK + item_part<C>(it) * 128;
      const int n_dv = item_part<C>(it) == 0 ? C::DV / 32 : 0;
      const int nch = n_dv + (item_part<C>(it) == 0 ? C::PART_COLS0 : C::PART_COLS1) / 32;
      if (it.nsteps == 0) {
        if (row_valid)
          for (int ch = w; ch < nch; ch += C::NG) {
            T* d = ch < n_dv ? dv_row + ch * 32 : dk_row + (ch - n_dv) * 32;
            for (int q4 = 0; q4 < 4; ++q4) reinterpret_cast<uint4*>(d)[q4] = make_uint4(0, 0, 0, 0);
          }
        continue;
      }
      int qmin = 1, qmax = 0;
      if (!(row_valid && query_range(kk, kk, it.lq, it.lk, pb.causal, pb.window, qmin, qmax))) {
        qmin = 1;
        qmax = 0;
      }
      for (int s = 0; s < it.nsteps; ++s) {
        int h, q0;
        bwd_step(it, pb, s, h, q0);
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.s_full, s_cnt++ & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const int c_lo = qmin - q0, c_hi = qmax - q0;
        const float* lse = softmax ? args.lse + static_cast<size_t>(h) * pb.total_q : nullptr;
        const float* drow = softmax ? args.drow + static_cast<size_t>(h) * pb.total_q : nullptr;
        const int col_base = it.q_start + q0;
        const int col_max = pb.total_q - 1;
        if (__all_sync(0xffffffffu, c_lo <= C::GCOLS * w && c_hi >= C::GCOLS * w + C::GCOLS - 1))
          bwd_pass1_dispatch<C, false>(args.act, t_lane, w, bwd_k, c_lo, c_hi, lse, col_base, col_max);
        else
          bwd_pass1_dispatch<C, true>(args.act, t_lane, w, bwd_k, c_lo, c_hi, lse, col_base, col_max);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full);
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.dp_full, dp_cnt++ & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        if (softmax)
          bwd_pass2<C, true>(t_lane, sDS, row, w, bwd_k.scale, drow, col_base, col_max);
        else
          bwd_pass2<C, false>(t_lane, sDS, row, w, bwd_k.scale, drow, col_base, col_max);
        fence_async_shared();
        tc_fence_before();
#ifdef GDPA_TEST_HOOKS
        if (!(blockIdx.x == 0 && static_cast<int>(s_cnt - 1) == args.test_skip_step))
#endif
        mbar_arrive(&sm.ds_full);
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(&sm.acc_full, acc_cnt++ & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int ch = w; ch < nch; ch += C::NG) {
        const bool is_dv = ch < n_dv;
        const int cc = is_dv ? ch * 32 : (ch - n_dv) * 32;
        uint32_t o[32];
        tmem_ld32(t_lane + (is_dv ? C::T_DV : C::T_DK) + cc, o);
        tmem_ld_wait(o);
        if (row_valid) {
          uint32_t wv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) wv[e] = pack16<C::DT>(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1]));
          uint4* d4 = reinterpret_cast<uint4*>((is_dv ? dv_row : dk_row) + cc);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) d4[q4] = make_uint4(wv[4 * q4], wv[4 * q4 + 1], wv[4 * q4 + 2], wv[4 * q4 + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.acc_empty);
    }
  } else if (warp >= C::DRAIN_WARP0) {
    // ------------------------------------------------ dQ drain: TMEM -> smem -> TMA reduce-add
    regs_dec<96>();
    // Each warp owns 32 query rows (its TMEM lane quadrant). A 32-column chunk
    // of those rows is staged as a 32 x 32 fp32 box in shared memory
    // (128-byte swizzle) and lane 0 adds it into the fp32 accumulator with
    // one bulk tensor reduce; each warp has two boxes, so chunks move in
    // pairs. Rows past the sequence end are staged as zeros, so adding them
    // into the next sequence's rows changes nothing.
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // query row within the tile
    const uint32_t t_dq = tbase + (static_cast<uint32_t>(quad * 32) << 16) + C::T_DQ;
    uint8_t* stage_base = sDQ + quad * 2 * C::DQ_CHUNK_BYTES;  // this warp's two 32 x 32 fp32 boxes
    constexpr int NPAIR_MAX = (C::PART_NCH_MAX + 1) / 2;
    uint32_t dq_cnt = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int pos = zigzag_pos(round, blockIdx.x, G);
      if (pos >= n_work) break;
      const BwdItem it = bwd_decode(args, pos, C::NPART);
      // this item's dQ columns: [128 part, 128 part + 32 nch)
      const int nch = (item_part<C>(it) == 0 ? C::PART_COLS0 : C::PART_COLS1) / 32, npair = (nch + 1) / 2;
      const int coff = item_part<C>(it) * 128;
      for (int s = 0; s < it.nsteps; ++s) {
        int h, q0;
        bwd_step(it, pb, s, h, q0);
        const bool valid = q0 + row < it.lq;
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.dq_full, dq_cnt++ & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        // a key block the caller's max_k does not allow: its slice (or, with
        // one producer per row, its rows) would lie outside what the workspace
        // and the mode were sized for, so report the violated precondition
        // and write nothing
        const bool kb_ok = it.k0 / kTileK < args.n_kblocks;
        if (!kb_ok && lane == 0 && quad == 0) atomicExch(args.status, 1);
        if (!kb_ok || q0 + quad * 32 >= it.lq) {  // nothing to add for this warp's 32 rows
          tc_fence_before();
          mbar_arrive(&sm.dq_empty);
          continue;
        }
        if constexpr (C::DIRECT_DQ) {
          // the only key block of the sequence: dQ rows in the output type,
          // 32 columns a chunk, written as paired 32-byte stores
          using T = typename std::conditional<C::DT == DT_FP16, __half, __nv_bfloat16>::type;
          T* drow_out = reinterpret_cast<T*>(args.dq) +
                        (static_cast<size_t>(it.q_start + q0 + row) * pb.h_q + h) * C::DQK + coff;
          const bool v8 = (reinterpret_cast<uintptr_t>(args.dq) & 31) == 0;
          const size_t stride = static_cast<size_t>(pb.h_q) * C::DQK * sizeof(T);
#pragma unroll
          for (int pr = 0; pr < NPAIR_MAX; ++pr) {
            if (pr >= npair) break;
            const int c0 = 2 * pr;
            uint32_t a[32], b[32];
            tmem_ld32(t_dq + c0 * 32, a);
            if (c0 + 1 < nch) tmem_ld32(t_dq + (c0 + 1) * 32, b);
            tmem_ld_wait(a);
            if (c0 + 1 < nch) tmem_ld_wait(b);
            if (pr == npair - 1) {
              tc_fence_before();
              mbar_arrive(&sm.dq_empty);  // every TMEM read of this tile is done
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              if (c0 + half >= nch) break;
              const uint32_t(&o)[32] = half == 0 ? a : b;
              uint32_t w[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) w[e] = pack16<C::DT>(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1]));
              T* dst = drow_out + (c0 + half) * 32;
              if (v8) {
                store_rows64_paired(reinterpret_cast<uint8_t*>(dst), stride, lane, w, valid);
              } else if (valid) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                  reinterpret_cast<uint4*>(dst)[q4] = make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
              }
            }
          }
          continue;
        } else {
        if (args.dq_mode == DQ_SLICES) {
          // deterministic mode: this key block's dQ tile goes to its own slice; a
          // later kernel adds the slices in key-block order
          float* dst = args.dq_part + ((static_cast<size_t>(it.k0 / kTileK) * pb.total_q + it.q_start + q0 + row) *
                                           pb.h_q + h) * C::DQK + coff;
#pragma unroll 1
          for (int ch = 0; ch < nch; ++ch) {
            uint32_t o[32];
            tmem_ld32(t_dq + ch * 32, o);
            tmem_ld_wait(o);
            if (ch == nch - 1) {
              tc_fence_before();
              mbar_arrive(&sm.dq_empty);
            }
            if (valid) {
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4)
                reinterpret_cast<uint4*>(dst + ch * 32)[q4] = make_uint4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
            }
          }
          continue;
        }
        // Chunks go through registers two at a time (one staging box each).
        // The TMEM columns are released as soon as the last pair is in
        // registers; every reduce issue and every wait for a box to be read
        // comes after that, off the path of the next dP^T GEMM.
        auto stage = [&](int bi, const uint32_t(&o)[32]) {
          uint8_t* box = stage_base + bi * C::DQ_CHUNK_BYTES;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = valid ? make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(box + lane * 128 + ((c ^ (lane & 7)) << 4)) = v;
          }
        };
        auto reduce_pair = [&](int c0) {  // lane 0: add boxes 0 (and 1) into chunks c0 (and c0 + 1), one bulk group
          tma_reduce_add_3d(&tm_dq, stage_base, coff + c0 * 32, h, it.q_start + q0 + quad * 32);
          if (c0 + 1 < nch) tma_reduce_add_3d(&tm_dq, stage_base + C::DQ_CHUNK_BYTES, coff + (c0 + 1) * 32, h,
                                              it.q_start + q0 + quad * 32);
          bulk_commit_group();
        };
        if (lane == 0) bulk_wait_group_read<0>();  // the previous tile's reduces are done reading both boxes
        __syncwarp();
#pragma unroll
        for (int pr = 0; pr < NPAIR_MAX; ++pr) {
          if (pr >= npair) break;
          const int c0 = 2 * pr;
          uint32_t a[32], b[32];
          tmem_ld32(t_dq + c0 * 32, a);
          if (c0 + 1 < nch) tmem_ld32(t_dq + (c0 + 1) * 32, b);
          tmem_ld_wait(a);
          if (c0 + 1 < nch) tmem_ld_wait(b);
          if (pr == npair - 1) {
            tc_fence_before();
            mbar_arrive(&sm.dq_empty);  // every TMEM read of this tile is done
          }
          if (pr > 0) {  // add the previous pair, then wait until its boxes have been read
            if (lane == 0) {
              reduce_pair(c0 - 2);
              bulk_wait_group_read<0>();
            }
            __syncwarp();
          }
          stage(0, a);
          if (c0 + 1 < nch) stage(1, b);
          fence_async_shared();
          __syncwarp();
        }
        if (lane == 0) reduce_pair(2 * (npair - 1));
        }  // not C::DIRECT_DQ
      }
    }
    if (lane == 0) bulk_wait_group_all();
  }

  // ------------------------------------------------ teardown
  // After an abort each role above has waited (time-bounded) for its own
  // TMA loads, MMAs and bulk reduce-adds in flight; only if one of those
  // waits gave up does the CTA also wait a fixed 1 ms before TMEM and shared
  // memory go away.
  tc_fence_before();
  __syncthreads();
  if (sm.abort_flag) {
    if (sm.drain_failed) {
      const unsigned long long t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 1000000ull) {
      }
    }
    if (threadIdx.x == 0) atomicExch(args.status, 5);
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int DQK, int DV, int DT, bool DIRECT>
cudaError_t launch_bwd_kernel(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                              cudaStream_t stream) {
  using C = BwdCfg<DQK, DV, DT, DIRECT>;
  auto kern = gdpa_bwd_kernel<C>;
  // the per-role register split assumes 128 registers a thread at launch
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || fa.numRegs < 128) return cudaErrorInvalidConfiguration;
  const cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, stream, tq, tk, tv, tdo, tdq, a);
}

template <int DQK, int DV, int DT>
cudaError_t launch_bwd_cfg(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                           cudaStream_t stream) {
  if (a.dq_mode == DQ_DIRECT) return launch_bwd_kernel<DQK, DV, DT, true>(tq, tk, tv, tdo, tdq, a, grid, stream);
  return launch_bwd_kernel<DQK, DV, DT, false>(tq, tk, tv, tdo, tdq, a, grid, stream);
}

}  // namespace gdpa
