// GDPA forward on sm_103a: O = where(M, act(scale * Q K^T), 0) V.
//
// Definition: gdpa/README.md (facebookresearch/ads_model_kernel_library),
// intro paragraph and "Features"; no row normalisation (softmax replaced by
// an activation). GDPA_ACT_SOFTMAX runs online softmax instead (the
// Dao-AILab/flash-attention overview's rescaling scheme) for cross-checking.
//
// One persistent CTA per SM walks a cost-sorted work list in zigzag order
// ("Zigzag tile scheduling", Features). A work item is two 128-row Q tiles
// of one (sequence, head); the CTA keeps both resident and alternates them so
// that the tensor core computes one tile's GEMMs while the activation warps
// work on the other's. Warp roles (320 threads):
//   warp 0     TMA producer: Q tiles, then K/V blocks through a smem ring
//   warp 1     MMA issuer (one thread): S_i = Q_i K^T into TMEM, then
//              O_i += P_i V with P_i read back from TMEM
//   warps 2-5  activation group for Q tile 0, warps 6-9 for Q tile 1:
//              TMEM S -> registers -> mask, scale, act -> P (bf16/f16/e4m3)
//              written over S in TMEM; after the last KV block, the epilogue
//              reads O from TMEM and stores it to global memory.
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+dv),
// O_1 [384,384+dv). P_i aliases the first columns of S_i.
//
// Ordering: the tensor core executes tcgen05.mma in issue order, so S_i of
// the next KV block may be issued right after O_i += P_i V even though it
// overwrites the TMEM columns P_i is read from. A commit after S_i also
// covers the preceding P_i V, which is what lets the softmax path rescale
// O_i when it sees S_i.
//
// Short KV (a single KV block per item, "Outer-loop software pipelining for
// short K/V sequences", Features): nothing in the loop waits for the previous
// item's epilogue except O_i's reuse, so the next item's Q load and S GEMMs
// overlap the current item's activation and epilogue.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "act.cuh"
#include "args.h"
#include "common.cuh"
#include "sm100.cuh"

namespace gdpa {

template <int DQK_, int DV_, int DT_>
struct FwdCfg {
  static constexpr int DQK = DQK_, DV = DV_, DT = DT_;
  static constexpr int ESZ = DT == DT_E4M3 ? 1 : 2;
  static constexpr int BOX_ELEMS = 128 / ESZ;  // elements per 128-byte swizzle row
  static constexpr int BOX_BYTES = 128 * 128;  // one 128-row x 128-byte swizzled box
  static constexpr int QK_BOXES = (DQK + BOX_ELEMS - 1) / BOX_ELEMS;
  static constexpr int V_BOXES = (DV + BOX_ELEMS - 1) / BOX_ELEMS;
  static constexpr int Q_BYTES = QK_BOXES * BOX_BYTES;
  static constexpr int K_BYTES = QK_BOXES * BOX_BYTES;
  static constexpr int V_BYTES = V_BOXES * BOX_BYTES;
  static constexpr int SMEM_LIMIT = 232448;  // 227 KB per block
  static constexpr int BAR_BYTES = 512;
  static constexpr int AVAIL = SMEM_LIMIT - 1024 - BAR_BYTES - 2 * Q_BYTES;
  static constexpr int FIT = AVAIL / (K_BYTES + V_BYTES);
  static constexpr int KST = FIT >= 2 ? (FIT > 4 ? 4 : FIT) : 2;
  static constexpr int VST = FIT >= 2 ? KST : 1;
  static constexpr int SMEM_BYTES = 1024 + 2 * Q_BYTES + KST * K_BYTES + VST * V_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "tiles do not fit in shared memory");
  static constexpr int K_STEP = ESZ == 1 ? 32 : 16;  // K of one MMA instruction
  static_assert(DQK % K_STEP == 0, "head dim must be a multiple of the MMA K step");
  static constexpr int S_MMAS = DQK / K_STEP;
  static constexpr int PV_MMAS = kTileK / K_STEP;
  static constexpr int P_COLS_PER_CHUNK = 32 * ESZ / 4;  // TMEM columns of 32 packed P values
  static constexpr uint32_t FMT = DT == DT_BF16 ? 1u : 0u;
  static constexpr uint32_t IDESC_S = idesc_make(128, 128, FMT, FMT, 0, 0);
  static constexpr uint32_t IDESC_PV = idesc_make(128, DV, FMT, FMT, 0, 1);
  static constexpr int THREADS = 320;
};

struct FwdItem {
  int b, h, g, q_start, lq, k_start, lk;
  int r0[2], rows[2], lo[2], hi[2], n[2];
  int lo_u, hi_u;
};

__device__ __forceinline__ FwdItem fwd_decode(const FwdArgs& a, int pos) {
  FwdItem it;
  const Problem& pb = a.pb;
  const int e = pos / pb.h_q;
  it.h = pos - e * pb.h_q;
  it.g = it.h / pb.group;
  const int2 bb = a.work->items[e];
  it.b = bb.x;
  seq_bounds(pb.cu_q, it.b, pb.max_q, it.q_start, it.lq);
  seq_bounds(pb.cu_k, it.b, pb.max_k, it.k_start, it.lk);
  it.lo_u = 1 << 30;
  it.hi_u = -1;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    it.r0[i] = bb.y * kFwdItemRows + i * kTileQ;
    int rows = it.lq - it.r0[i];
    rows = rows < 0 ? 0 : (rows > kTileQ ? kTileQ : rows);
    it.rows[i] = rows;
    int kmin, kmax;
    if (rows > 0 && key_range(it.r0[i], it.r0[i] + rows - 1, it.lq, it.lk, pb.causal, pb.window, kmin, kmax)) {
      it.lo[i] = kmin / kTileK;
      it.hi[i] = kmax / kTileK;
      it.n[i] = it.hi[i] - it.lo[i] + 1;
      it.lo_u = min(it.lo_u, it.lo[i]);
      it.hi_u = max(it.hi_u, it.hi[i]);
    } else {
      it.lo[i] = 0;
      it.hi[i] = -1;
      it.n[i] = 0;
    }
  }
  return it;
}

__device__ __forceinline__ bool fwd_in(const FwdItem& it, int i, int j) {
  return it.n[i] > 0 && j >= it.lo[i] && j <= it.hi[i];
}

template <class C>
struct FwdSmem {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[C::KST], k_empty[C::KST];
  uint64_t v_full[C::VST], v_empty[C::VST];
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
  uint32_t tmem_base;
  int abort_flag;
};

// ---------------------------------------------------------------- activation of one S tile

// Converts 32 floats to the P storage type and writes them to TMEM.
template <int DT>
__device__ __forceinline__ void store_p_chunk(uint32_t taddr, const float (&p)[32]) {
  if constexpr (DT == DT_E4M3) {
    uint32_t r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = pack_e4m3x4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
    tmem_st8(taddr, r);
  } else {
    uint32_t r[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      r[i] = DT == DT_BF16 ? pack_bf16x2(p[2 * i], p[2 * i + 1]) : pack_f16x2(p[2 * i], p[2 * i + 1]);
    tmem_st16(taddr, r);
  }
}

// P = where(c_lo <= col <= c_hi, act(scale * S), 0) for one 128x128 tile;
// thread = one row (TMEM lane), t_s = this lane's address of S column 0.
// The load of the next 32 columns is in flight while the current ones are
// activated; P chunk c goes to columns already read (P packs 2 or 4 values
// per 32-bit column, so it never overtakes the S columns still to be read).
template <class C, int ACT, bool MASKED>
__device__ __forceinline__ void act_tile(uint32_t t_s, const ActConsts& k, int c_lo, int c_hi) {
  uint32_t sa[32], sb[32];
  tmem_ld32(t_s, sa);
  tmem_ld_wait(sa);
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t(&cur)[32] = (ch & 1) ? sb : sa;
    uint32_t(&nxt)[32] = (ch & 1) ? sa : sb;
    if (ch < 3) tmem_ld32(t_s + (ch + 1) * 32, nxt);
    float p[32];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const f2_t r = act_pair<ACT>(f2(__uint_as_float(cur[2 * e]), __uint_as_float(cur[2 * e + 1])), k);
      float v0 = f2_lo(r), v1 = f2_hi(r);
      if (MASKED) {
        const int c0 = ch * 32 + 2 * e;
        v0 = (c0 >= c_lo && c0 <= c_hi) ? v0 : 0.0f;
        v1 = (c0 + 1 >= c_lo && c0 + 1 <= c_hi) ? v1 : 0.0f;
      }
      p[2 * e] = v0;
      p[2 * e + 1] = v1;
    }
    store_p_chunk<C::DT>(t_s + ch * C::P_COLS_PER_CHUNK, p);
    if (ch < 3) tmem_ld_wait(nxt);
  }
}

template <class C, bool MASKED>
__device__ __forceinline__ void act_tile_dispatch(int act, uint32_t t_s, const ActConsts& k, int c_lo, int c_hi) {
  switch (act) {
    case ACT_IDENTITY: act_tile<C, ACT_IDENTITY, MASKED>(t_s, k, c_lo, c_hi); break;
    case ACT_GELU: act_tile<C, ACT_GELU, MASKED>(t_s, k, c_lo, c_hi); break;
    case ACT_GELU_TANH: act_tile<C, ACT_GELU_TANH, MASKED>(t_s, k, c_lo, c_hi); break;
    case ACT_FAST_GELU: act_tile<C, ACT_FAST_GELU, MASKED>(t_s, k, c_lo, c_hi); break;
    case ACT_RELU: act_tile<C, ACT_RELU, MASKED>(t_s, k, c_lo, c_hi); break;
    case ACT_RELU2: act_tile<C, ACT_RELU2, MASKED>(t_s, k, c_lo, c_hi); break;
    case ACT_LEAKY_RELU: act_tile<C, ACT_LEAKY_RELU, MASKED>(t_s, k, c_lo, c_hi); break;
    case ACT_SILU: act_tile<C, ACT_SILU, MASKED>(t_s, k, c_lo, c_hi); break;
    default: act_tile<C, ACT_HARDSWISH, MASKED>(t_s, k, c_lo, c_hi); break;
  }
}

// Online softmax over one tile (log2 domain). m is a possibly stale running
// max: it is raised, and O rescaled, only when the tile's max exceeds it by
// more than 8 (P then stays below 2^8).
template <class C>
__device__ __forceinline__ void softmax_tile(uint32_t t_s, uint32_t t_o, bool o_live, float scale_log2, int c_lo,
                                             int c_hi, float& m, float& l) {
  float mb = -INFINITY;
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t s[32];
    tmem_ld32(t_s + ch * 32, s);
    tmem_ld_wait(s);
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int c = ch * 32 + e;
      if (c >= c_lo && c <= c_hi) mb = fmaxf(mb, __uint_as_float(s[e]) * scale_log2);
    }
  }
  const bool raise = mb > -INFINITY && (m == -INFINITY || mb > m + 8.0f);
  const float m_new = raise ? mb : m;
  const float alpha = raise && m != -INFINITY ? ex2_approx(m - m_new) : 1.0f;
  if (__any_sync(0xffffffffu, raise && m != -INFINITY) && o_live) {
#pragma unroll 1
    for (int ch = 0; ch < C::DV / 32; ++ch) {
      uint32_t o[32];
      tmem_ld32(t_o + ch * 32, o);
      tmem_ld_wait(o);
      uint32_t w[16];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(__uint_as_float(o[half * 16 + e]) * alpha);
        tmem_st16(t_o + ch * 32 + half * 16, w);
      }
    }
  }
  l *= alpha;
  m = m_new;
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t s[32];
    tmem_ld32(t_s + ch * 32, s);
    tmem_ld_wait(s);
    float p[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int c = ch * 32 + e;
      const float v = (c >= c_lo && c <= c_hi) ? ex2_approx(__uint_as_float(s[e]) * scale_log2 - m) : 0.0f;
      l += v;
      p[e] = v;
    }
    store_p_chunk<C::DT>(t_s + ch * C::P_COLS_PER_CHUNK, p);
  }
}

// ---------------------------------------------------------------- the kernel

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    gdpa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + 2 * C::Q_BYTES;
  uint8_t* sV = sK + C::KST * C::K_BYTES;
  FwdSmem<C>& sm = *reinterpret_cast<FwdSmem<C>*>(sV + C::VST * C::V_BYTES);
  static_assert(sizeof(FwdSmem<C>) <= C::BAR_BYTES, "barrier block too large");

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const Problem& pb = args.pb;
  const int n_work = args.work->count * pb.h_q;
  const int G = gridDim.x;
  volatile int* abort_flag = &sm.abort_flag;

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1);
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i], 128);
      mbar_init(&sm.o_full[i], 1);
      mbar_init(&sm.o_empty[i], 128);
    }
    for (int i = 0; i < C::KST; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 1);
    }
    for (int i = 0; i < C::VST; ++i) {
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 1);
    }
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t k_it = 0, v_it = 0, qe[2] = {0, 0};
      for (int round = 0;; ++round) {
        const int pos = zigzag_pos(round, blockIdx.x, G);
        if (pos >= n_work) break;
        const FwdItem it = fwd_decode(args, pos);
        bool ok = true;
        for (int i = 0; i < 2 && ok; ++i) {
          if (it.n[i] == 0) continue;
          ok = mbar_wait(&sm.q_empty[i], (qe[i]++ & 1) ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&sm.q_full[i], C::Q_BYTES);
          for (int bx = 0; bx < C::QK_BOXES; ++bx)
            tma_load_3d(sQ + i * C::Q_BYTES + bx * C::BOX_BYTES, &tm_q, &sm.q_full[i], bx * C::BOX_ELEMS, it.h,
                        it.q_start + it.r0[i]);
        }
        for (int j = it.lo_u; j <= it.hi_u && ok; ++j) {
          const int ks = k_it % C::KST;
          ok = mbar_wait(&sm.k_empty[ks], ((k_it / C::KST) & 1) ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&sm.k_full[ks], C::K_BYTES);
          for (int bx = 0; bx < C::QK_BOXES; ++bx)
            tma_load_3d(sK + ks * C::K_BYTES + bx * C::BOX_BYTES, &tm_k, &sm.k_full[ks], bx * C::BOX_ELEMS, it.g,
                        it.k_start + j * kTileK);
          ++k_it;
          const int vs = v_it % C::VST;
          ok = mbar_wait(&sm.v_empty[vs], ((v_it / C::VST) & 1) ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&sm.v_full[vs], C::V_BYTES);
          for (int bx = 0; bx < C::V_BOXES; ++bx)
            tma_load_3d(sV + vs * C::V_BYTES + bx * C::BOX_BYTES, &tm_v, &sm.v_full[vs], bx * C::BOX_ELEMS, it.g,
                        it.k_start + j * kTileK);
          ++v_it;
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t k_it = 0, v_it = 0, qf[2] = {0, 0}, pc[2] = {0, 0}, oe[2] = {0, 0};
      const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
      auto issue_s = [&](int i, int ks) {
        const uint32_t a0 = sQa + i * C::Q_BYTES, b0 = sKa + ks * C::K_BYTES;
#pragma unroll
        for (int k = 0; k < C::S_MMAS; ++k) {
          const uint32_t off = (k / 4) * C::BOX_BYTES + (k % 4) * 32;
          if constexpr (C::DT == DT_E4M3)
            mma_f8_ss(tbase + i * 128, sdesc_sw128(a0 + off, 16, 1024), sdesc_sw128(b0 + off, 16, 1024),
                      C::IDESC_S, k > 0);
          else
            mma_f16_ss(tbase + i * 128, sdesc_sw128(a0 + off, 16, 1024), sdesc_sw128(b0 + off, 16, 1024),
                       C::IDESC_S, k > 0);
        }
      };
      auto issue_pv = [&](int i, int vs, bool acc) {
        const uint32_t b0 = sVa + vs * C::V_BYTES;
#pragma unroll
        for (int k = 0; k < C::PV_MMAS; ++k) {
          const uint32_t a_t = tbase + i * 128 + k * (C::K_STEP * C::ESZ / 4);
          const uint64_t bd = sdesc_sw128(b0 + k * C::K_STEP * 128, C::BOX_BYTES, 1024);
          if constexpr (C::DT == DT_E4M3)
            mma_f8_ts(tbase + 256 + i * 128, a_t, bd, C::IDESC_PV, (acc || k > 0) ? 1u : 0u);
          else
            mma_f16_ts(tbase + 256 + i * 128, a_t, bd, C::IDESC_PV, (acc || k > 0) ? 1u : 0u);
        }
      };
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int pos = zigzag_pos(round, blockIdx.x, G);
        if (pos >= n_work) break;
        const FwdItem it = fwd_decode(args, pos);
        if (it.hi_u < it.lo_u) continue;
        for (int i = 0; i < 2 && ok; ++i)
          if (it.n[i] > 0) ok = mbar_wait(&sm.q_full[i], qf[i]++ & 1, abort_flag);
        if (!ok) break;
        bool first_pv[2] = {true, true};
        // prologue: S for the first KV block
        {
          const int ks = k_it % C::KST;
          ok = mbar_wait(&sm.k_full[ks], (k_it / C::KST) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          for (int i = 0; i < 2; ++i) {
            if (!fwd_in(it, i, it.lo_u)) continue;
            issue_s(i, ks);
            mma_commit(&sm.s_full[i]);
            if (it.lo_u == it.hi[i]) mma_commit(&sm.q_empty[i]);
          }
          mma_commit(&sm.k_empty[ks]);
          ++k_it;
        }
        for (int j = it.lo_u; j <= it.hi_u && ok; ++j) {
          const int vs = v_it % C::VST;
          ok = mbar_wait(&sm.v_full[vs], (v_it / C::VST) & 1, abort_flag);
          if (!ok) break;
          const bool has_next = j < it.hi_u;
          const int ks = k_it % C::KST;
          if (has_next) {
            ok = mbar_wait(&sm.k_full[ks], (k_it / C::KST) & 1, abort_flag);
            if (!ok) break;
          }
          tc_fence_after();
          for (int i = 0; i < 2 && ok; ++i) {
            if (fwd_in(it, i, j)) {
              if (first_pv[i]) ok = mbar_wait(&sm.o_empty[i], (oe[i]++ & 1) ^ 1, abort_flag);
              if (ok) ok = mbar_wait(&sm.p_full[i], pc[i]++ & 1, abort_flag);
              if (!ok) break;
              tc_fence_after();
              issue_pv(i, vs, !first_pv[i]);
              first_pv[i] = false;
              if (j == it.hi[i]) mma_commit(&sm.o_full[i]);
            }
            if (has_next && fwd_in(it, i, j + 1)) {
              issue_s(i, ks);
              mma_commit(&sm.s_full[i]);
              if (j + 1 == it.hi[i]) mma_commit(&sm.q_empty[i]);
            }
          }
          if (!ok) break;
          mma_commit(&sm.v_empty[vs]);
          ++v_it;
          if (has_next) {
            mma_commit(&sm.k_empty[ks]);
            ++k_it;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------ activation + epilogue warpgroups
    const int half = (warp - 2) / 4;
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t t_s = t_lane + half * 128;
    const uint32_t t_o = t_lane + 256 + half * 128;
    const bool softmax = args.act == ACT_SOFTMAX;
    float qk_scale = args.scale;
    float v_scale = 1.0f;
    if (C::DT == DT_E4M3 && args.descale != nullptr) {
      qk_scale *= args.descale[0] * args.descale[1];
      v_scale = args.descale[2];
    }
    const float s_scale = softmax ? qk_scale * kLog2e : qk_scale;
    const ActConsts act_k = make_act_consts(qk_scale);
    uint32_t sc = 0, oc = 0;
    using OutT = typename std::conditional<C::DT == DT_FP16, __half, __nv_bfloat16>::type;
    OutT* out = reinterpret_cast<OutT*>(args.out);
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int pos = zigzag_pos(round, blockIdx.x, G);
      if (pos >= n_work) break;
      const FwdItem it = fwd_decode(args, pos);
      if (it.rows[half] == 0) continue;
      const int qrow = it.r0[half] + row;
      const bool row_valid = row < it.rows[half];
      int kmin = 1, kmax = 0;
      if (!(row_valid && key_range(qrow, qrow, it.lq, it.lk, pb.causal, pb.window, kmin, kmax))) {
        kmin = 1;
        kmax = 0;
      }
      OutT* orow = out + (static_cast<size_t>(it.q_start + qrow) * pb.h_q + it.h) * C::DV;
      float m = -INFINITY, l = 0.0f;
      if (it.n[half] > 0) {
        for (int j = it.lo[half]; j <= it.hi[half]; ++j) {
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.s_full[half], sc++ & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
          const int c_lo = kmin - j * kTileK, c_hi = kmax - j * kTileK;
          if (softmax) {
            softmax_tile<C>(t_s, t_o, j > it.lo[half], s_scale, c_lo, c_hi, m, l);
          } else if (__all_sync(0xffffffffu, c_lo <= 0 && c_hi >= kTileK - 1)) {
            act_tile_dispatch<C, false>(args.act, t_s, act_k, c_lo, c_hi);
          } else {
            act_tile_dispatch<C, true>(args.act, t_s, act_k, c_lo, c_hi);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&sm.p_full[half]);
        }
        if (!ok) break;
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.o_full[half], oc++ & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        float f = v_scale;
        if (softmax) f = l > 0.0f ? v_scale / l : 0.0f;
#pragma unroll 1
        for (int ch = 0; ch < C::DV / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(t_o + ch * 32, o);
          tmem_ld_wait(o);
          if (row_valid) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float lo = __uint_as_float(o[2 * e]) * f, hi = __uint_as_float(o[2 * e + 1]) * f;
              w[e] = C::DT == DT_FP16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) dst[q4] = make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
          }
        }
        tc_fence_before();
        mbar_arrive(&sm.o_empty[half]);
      } else if (row_valid) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
        for (int q4 = 0; q4 < C::DV * 2 / 16; ++q4) dst[q4] = make_uint4(0, 0, 0, 0);
      }
      if (softmax && row_valid && args.lse != nullptr) {
        args.lse[static_cast<size_t>(it.h) * pb.total_q + it.q_start + qrow] =
            l > 0.0f ? m * 0.6931471805599453f + __logf(l) : -INFINITY;
      }
    }
  }

  // ------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (sm.abort_flag) {
    // let copies and MMAs already in flight land before the TMEM and smem go away
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
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

template <int DQK, int DV, int DT>
cudaError_t launch_fwd_cfg(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& a,
                           int grid, cudaStream_t stream) {
  using C = FwdCfg<DQK, DV, DT>;
  auto kern = gdpa_fwd_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace gdpa
