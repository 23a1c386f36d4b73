// GDPA forward on sm_103a: O = where(M, act(scale * Q K^T), 0) V.
//
// Definition: gdpa/README.md (facebookresearch/ads_model_kernel_library),
// intro paragraph and "Features"; no row normalisation (softmax replaced by
// an activation). GDPA_ACT_SOFTMAX runs online softmax instead (the
// Dao-AILab/flash-attention overview's rescaling scheme) for cross-checking.
//
// One persistent CTA per SM walks a cost-sorted work list in zigzag order
// ("Zigzag tile scheduling", Features). A work item is one 128-row Q tile of
// one (sequence, head); its KV blocks form "steps", and all roles walk the
// same flattened stream of steps across items. Warp roles (128 + 128 NG
// threads, NG = 2 or 4 activation groups):
//   warp 0       TMA producers: the K ring (lane 0) and Q tiles (lane 1,
//                double-buffered, so one item ahead)
//   warp 1       MMA issuer for S = Q K^T (whole warp; one elected lane issues)
//   warp 2       MMA issuer for O += P V (likewise)
//   warp 3       TMA producer: the V ring
//   warps 4..    NG activation groups of four warps (one per TMEM lane
//                quadrant); group g owns score columns [g 128/NG, +128/NG)
//                of every S tile and, at the end of an item, O columns
//                [g dv/NG, +dv/NG) (softmax: O / l and lse)
// Four groups (sixteen warps, four per SM sub-partition) keep the FMA pipes
// fed where the activation's arithmetic sets the pace; two leave each thread
// more registers elsewhere. The epilogue of an item runs after the next
// item's first step, so the item's last PV has finished by then.
// TMEM (512 columns): S buffers [0,128) and [128,256), P buffers [256,320)
// and [320,384) (bf16/f16 pairs or e4m3 quads per column), O [384,384+dv).
//
// Two issuing threads: one tcgen05.mma costs its issuing thread about as
// long as an N=128 MMA takes to execute, and every barrier wait or commit
// on a single issuer leaves the tensor core idle. With S and PV issued from
// different warps, one issuer's waits overlap the other's MMAs. Because P
// has its own buffers, S of step u+2 is computed into S buffer u%2 as soon
// as the activation groups have read S of step u (signalled by P(u) being
// full), so activation latency hides behind the GEMMs. The two streams are
// not ordered against each other, so the activation groups wait for
// pv_done[u%2] (PV(u-2) has read P buffer u%2) before storing P(u).
//
// Short KV ("Outer-loop software pipelining for short K/V sequences",
// Features): the step stream crosses item boundaries, so with one or two KV
// blocks per item the next items' Q loads and S GEMMs run while the current
// item's activation and epilogue proceed; only the first PV of an item waits
// for the epilogue to release O.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "act.cuh"
#include "args.h"
#include "common.cuh"
#include "sm100.cuh"

namespace gdpa {

// SOFTMAX_: the online-softmax kernel (GDPA_ACT_SOFTMAX); the elementwise
// activations get kernels of their own, so neither carries the other's code.
// Largest n <= cap with n * per <= avail.
__host__ __device__ constexpr int fwd_ring_stages(int avail, int per, int cap) {
  return avail / per > cap ? cap : avail / per;
}

template <int DQK_, int DV_, int DT_, int NG_, bool SOFTMAX_ = false, bool MX_ = false>
struct FwdCfg {
  static constexpr int DQK = DQK_, DV = DV_, DT = DT_, NG = NG_;
  static constexpr bool SOFTMAX = SOFTMAX_;
  // MXFP8: e4m3 codes with one E8M0 scale per 32 elements along each GEMM's K
  // (see FwdArgs::sf_q); the MMAs apply the scales (kind::mxf8f6f4).
  static constexpr bool MX = MX_;
  static_assert(!MX || (DT_ == DT_E4M3 && DQK_ % 32 == 0 && DV_ == 128), "MXFP8: e4m3, d_qk % 32 == 0, d_v = 128");
  // scale-factor atoms (512 bytes: 128 rows x 4 K blocks) per Q / K tile and per V tile
  static constexpr int NQB = (DQK_ / 32 + 3) / 4;
  static constexpr int SF_ATOM = 512;
  static constexpr int SF_RESERVE = MX ? (2 + 4) * NQB * SF_ATOM + 4 * SF_ATOM + SF_ATOM : 0;
  static_assert(!SOFTMAX || NG == 2, "softmax runs with two activation groups");
  static constexpr int ESZ = DT == DT_E4M3 ? 1 : 2;
  static constexpr int BOX_ELEMS = 128 / ESZ;  // elements per 128-byte swizzle row
  static constexpr int BOX_BYTES = 128 * 128;  // one 128-row x 128-byte swizzled box
  static constexpr int QK_BOXES = (DQK + BOX_ELEMS - 1) / BOX_ELEMS;
  static constexpr int V_BOXES = (DV + BOX_ELEMS - 1) / BOX_ELEMS;
  static constexpr int Q_BYTES = QK_BOXES * BOX_BYTES;
  static constexpr int K_BYTES = QK_BOXES * BOX_BYTES;
  static constexpr int V_BYTES = V_BOXES * BOX_BYTES;
  static constexpr int SMEM_LIMIT = 232448;  // 227 KB per block
  // barriers (and, for softmax, the row statistics exchange)
  static constexpr int EXTRA_BYTES = SOFTMAX ? 8192 : 1024;
  static_assert(NG == 2 || NG == 4, "two or four activation groups");
  // two groups come with a separate epilogue warpgroup; four fold the epilogue into the groups
  static constexpr bool SEP_EPI = NG == 2;
  static constexpr int AVAIL = SMEM_LIMIT - 1024 - EXTRA_BYTES - SF_RESERVE;
  // Q double-buffered when two K and two V stages still fit, else single.
  // MXFP8 takes one Q slot where a second would cost the fourth K stage (the
  // scale atoms' room): the deeper K ring measured faster (0.66 against
  // 0.76 ms on 16 x 8192 tokens, GQA 16/2, (192, 128), window 512, FastGELU).
  static constexpr bool MX_ONE_Q = MX && (AVAIL - 2 * Q_BYTES - 2 * V_BYTES) / K_BYTES < 4;
  static constexpr int QST = !MX_ONE_Q && AVAIL - 2 * Q_BYTES >= 2 * (K_BYTES + V_BYTES) ? 2 : 1;
  static_assert(QST <= 4, "at most four Q slots");
  // K needs the deeper ring: S(u) must wait for K(u), whose load can start
  // only once S(u - KST) has released its stage, while V(u) is wanted one
  // GEMM later. Then V takes what is left (at most as many stages as K).
  static constexpr int KST = fwd_ring_stages(AVAIL - QST * Q_BYTES - 2 * V_BYTES, K_BYTES, 4);
  static constexpr int VST = fwd_ring_stages(AVAIL - QST * Q_BYTES - KST * K_BYTES, V_BYTES, KST);
  static_assert(KST >= 2 && VST >= 2, "need at least two K and two V stages");
  // The separate epilogue stages O rows in shared memory (4 warps x 32 rows x
  // 128 bytes) so that its global stores cover whole 128-byte segments,
  // where that still fits beside the rings.
  static constexpr int STAGE_BYTES =
      SEP_EPI && QST * Q_BYTES + KST * K_BYTES + VST * V_BYTES + 16384 <= AVAIL ? 16384 : 0;
  // scale-factor atoms in shared memory: Q slots, K stages, V stages, then the constant P atom
  static constexpr int SF_BYTES = MX ? (QST + KST) * NQB * SF_ATOM + VST * SF_ATOM + SF_ATOM : 0;
  static constexpr int SMEM_BYTES =
      1024 + QST * Q_BYTES + KST * K_BYTES + VST * V_BYTES + STAGE_BYTES + SF_BYTES + EXTRA_BYTES;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "tiles do not fit in shared memory");
  static constexpr int K_STEP = ESZ == 1 ? 32 : 16;  // K of one MMA instruction
  static_assert(DQK % K_STEP == 0, "head dim must be a multiple of the MMA K step");
  static constexpr int S_MMAS = DQK / K_STEP;
  static constexpr int PV_MMAS = kTileK / K_STEP;
  static constexpr int P_COLS_PER_32 = 32 * ESZ / 4;  // TMEM columns of 32 packed P values
  static constexpr uint32_t FMT = DT == DT_BF16 ? 1u : 0u;
  static constexpr uint32_t IDESC_S = idesc_make(128, 128, FMT, FMT, 0, 0);
  static constexpr uint32_t IDESC_PV = idesc_make(128, DV, FMT, FMT, 0, 1);
  static constexpr int THREADS = 128 + 128 * NG + (SEP_EPI ? 128 : 0);
  static constexpr int ACT_WARP0 = 4, EPI_WARP0 = 4 + 4 * NG;
  static constexpr int GCOLS = 128 / NG;            // score columns per activation group
  static constexpr int OCOLS = DV / NG;             // O columns each group writes back
  static_assert(OCOLS % 8 == 0, "value head dim must split into 8-column slices");
  // O slice access width: 8 columns with four groups (96 registers a thread),
  // else the widest that divides the slice and its column offset
  static constexpr int OCH = NG == 4 ? 8 : (OCOLS % 32 == 0 ? 32 : (OCOLS % 16 == 0 ? 16 : 8));
  static constexpr uint32_t T_S = 0, T_P = 256, T_O = 384;  // TMEM column bases
  // MX scale factors in the TMEM columns that e4m3 P leaves free ([288, 320)
  // and [352, 384)): 4 columns per atom
  static constexpr uint32_t T_SFQ = 288, T_SFP = T_SFQ + QST * NQB * 4, T_SFV = T_SFP + 4, T_SFK = 352;
  static_assert(!MX || (T_SFV + VST * 4 <= 320 && T_SFK + KST * NQB * 4 <= 384), "MX scale factors do not fit in TMEM");
};

struct FwdItem {
  int h, g, q_start, lq, k_start, lk;
  int r0, rows, lo, hi, n;
  int pos;  // position in the work order (entry * h_q + head)
};

__device__ __forceinline__ FwdItem fwd_decode(const FwdArgs& a, int pos) {
  FwdItem it;
  const Problem& pb = a.pb;
  const int e = pos / pb.h_q;
  it.h = pos - e * pb.h_q;
  it.g = it.h / pb.group;
  const int4 sq = a.work->items[e].seq, bk = a.work->items[e].blk;
  it.q_start = sq.x;
  it.lq = sq.y;
  it.k_start = sq.z;
  it.lk = sq.w;
  it.r0 = bk.x;
  it.rows = bk.y;
  it.lo = bk.z;
  it.n = bk.w;
  it.hi = it.lo + it.n - 1;
  it.pos = pos;
  return it;
}

// Walks this CTA's items that have KV blocks, block by block. item_idx
// counts such items from 0 (it selects the Q buffer).
struct StepCursor {
  FwdItem it;
  int round, j, item_idx;
  bool active;

  __device__ __forceinline__ void find_item(const FwdArgs& a, int n_work) {
    while (true) {
      const int pos = zigzag_pos(round++, blockIdx.x, gridDim.x);
      if (pos >= n_work) {
        active = false;
        return;
      }
      it = fwd_decode(a, pos);
      if (it.n > 0) {
        j = it.lo;
        active = true;
        return;
      }
    }
  }
  __device__ __forceinline__ void start(const FwdArgs& a, int n_work) {
    round = 0;
    item_idx = 0;
    find_item(a, n_work);
  }
  __device__ __forceinline__ void next_item(const FwdArgs& a, int n_work) {
    ++item_idx;
    find_item(a, n_work);
  }
  __device__ __forceinline__ void advance(const FwdArgs& a, int n_work) {
    if (++j > it.hi) next_item(a, n_work);
  }
};

struct FwdSmem {
  uint64_t q_full[4], q_empty[4];
  uint64_t k_full[4], k_empty[4];
  uint64_t v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2];
  uint64_t o_full, o_empty, pv_done[2];
  uint64_t stat_full, stat_empty;
  uint64_t red_full[2];  // softmax: every group's partial row max of step u is in red[u % 2]
  uint64_t drain[2];     // abort path: MMAs issued by the S / PV warp have completed
  uint32_t tmem_base;
  int abort_flag;
  int drain_failed;      // abort path: a role's in-flight work did not land in time
};

// Softmax only: the row statistics the activation groups exchange.
struct FwdSoftmaxSmem {
  float red[2][4][128];  // per-group partial row max, by step parity (NG <= 4)
  float stat_l[4][128];  // per-group partial row sums at item end
  float stat_m[128];     // final running max at item end (separate epilogue)
};

// ---------------------------------------------------------------- activation groups

// P buffer u % 2 last held P(u - 2); the PV issuer signals pv_done[u % 2]
// once PV(u - 2) has read it. Who waits for that depends on the activation
// (pv_gate_on_s below): for costly activations the S issuer waits before
// issuing S(u), which keeps the poll off the activation warps' critical
// path; for cheap ones the activation warps wait just before their first
// store, so S(u) is not held back.
__host__ __device__ constexpr bool pv_gate_on_s(int act) {
  return act == ACT_GELU || act == ACT_GELU_TANH || act == ACT_SILU || act == ACT_SOFTMAX;
}

struct StepSync {
  uint64_t* pv_done;
  uint32_t u;
  volatile int* abort_flag;
  bool gated;  // the S issuer already waited for PV(u-2) before issuing S(u)
  __device__ __forceinline__ bool wait_p_buffer() const {
    if (u < 2 || gated) return true;
    return __all_sync(0xffffffffu, mbar_wait(pv_done, ((u - 2) >> 1) & 1, abort_flag));
  }
};

// Packs 32 floats into the P storage type (16 words of bf16/f16 pairs or 8
// words of e4m3 quads).
template <int DT>
__device__ __forceinline__ void pack_p_chunk(const float (&p)[32], uint32_t (&r)[16]) {
  if constexpr (DT == DT_E4M3) {
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = pack_e4m3x4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      r[i] = DT == DT_BF16 ? pack_bf16x2(p[2 * i], p[2 * i + 1]) : pack_f16x2(p[2 * i], p[2 * i + 1]);
  }
}

template <int DT>
__device__ __forceinline__ void store_p_chunk(uint32_t taddr, const uint32_t (&r)[16]) {
  if constexpr (DT == DT_E4M3) {
    uint32_t q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = r[i];
    tmem_st8(taddr, q);
  } else {
    tmem_st16(taddr, r);
  }
}

// N-column (32, 16 or 8) TMEM loads and stores of one lane's registers.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 32) tmem_ld32(taddr, r);
  else if constexpr (N == 16) tmem_ld16(taddr, r);
  else tmem_ld8(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 32) {
    tmem_st16(taddr, *reinterpret_cast<const uint32_t(*)[16]>(r));
    tmem_st16(taddr + 16, *reinterpret_cast<const uint32_t(*)[16]>(r + 16));
  } else if constexpr (N == 16) {
    tmem_st16(taddr, r);
  } else {
    tmem_st8(taddr, r);
  }
}

// Bit e set when column cb + e (0 <= e < 32) lies in [lo, hi].
__device__ __forceinline__ uint32_t cols_in_range(int cb, int lo, int hi) {
  const int a = max(lo - cb, 0), b = min(hi - cb, 31);
  if (a > b) return 0u;
  return (0xFFFFFFFFu >> (31 - b)) & (0xFFFFFFFFu << a);
}

__device__ __forceinline__ uint32_t prmt_b32(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Zeroes the masked elements of 32 packed P values (bit e of m: column e
// kept). Bits 4i..4i+3 are moved to the top bit of bytes 0..3 by one multiply
// (the four shifted copies of the nibble do not overlap), and prmt's
// sign-replicating selectors widen each top bit to its byte (e4m3: one column
// per byte) or to both bytes of its half-word (bf16 / f16 pairs).
template <int DT>
__device__ __forceinline__ void mask_p_words(uint32_t (&w)[16], uint32_t m) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t y = ((m >> (4 * i)) & 0xFu) * 0x10204080u;
    if constexpr (DT == DT_E4M3) {
      w[i] &= prmt_b32(y, y, 0xBA98u);
    } else {
      w[2 * i] &= prmt_b32(y, y, 0x9988u);
      w[2 * i + 1] &= prmt_b32(y, y, 0xBBAAu);
    }
  }
}

// P = where(c_lo <= col <= c_hi, act(scale * S), 0) for one group's GCOLS
// columns of an S tile, 32 at a time; thread = one row (TMEM lane). t_s /
// t_p: this lane's address of the group's first S / P column.
template <class C, int ACT, bool MASKED>
__device__ __forceinline__ bool act_quarter(uint32_t t_s, uint32_t t_p, int col0, const ActConsts& k, int c_lo,
                                            int c_hi, const StepSync& sync) {
  uint32_t sv[C::GCOLS / 32][32];
#pragma unroll
  for (int ch = 0; ch < C::GCOLS / 32; ++ch) tmem_ld32(t_s + 32 * ch, sv[ch]);
#pragma unroll
  for (int ch = 0; ch < C::GCOLS / 32; ++ch) tmem_ld_wait(sv[ch]);
#pragma unroll
  for (int ch = 0; ch < C::GCOLS / 32; ++ch) {
    const uint32_t(&sa)[32] = sv[ch];
    uint32_t pk[16];
    if constexpr (ACT == ACT_FAST_GELU_BF16 && C::DT == DT_BF16) {
      // already bf16 pairs: stored as they come
#pragma unroll
      for (int e = 0; e < 16; ++e) pk[e] = fast_gelu_bf16_pair(__uint_as_float(sa[2 * e]), __uint_as_float(sa[2 * e + 1]), k);
    } else if constexpr (ACT == ACT_GELU && C::DT == DT_BF16) {
      // mixed tanh form / polynomial, packed by truncation (constants carry the bias)
#pragma unroll
      for (int e = 0; e < 16; ++e)
        pk[e] = pack_trunc_bf16x2(gelu_mixed_pair<true>(e, f2(__uint_as_float(sa[2 * e]), __uint_as_float(sa[2 * e + 1])), k));
    } else {
    float p[32];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const f2_t sp = f2(__uint_as_float(sa[2 * e]), __uint_as_float(sa[2 * e + 1]));
      f2_t r;
      if constexpr (ACT == ACT_GELU) r = gelu_mixed_pair<false>(e, sp, k);
      else if constexpr (C::DT == DT_E4M3 && (ACT == ACT_FAST_GELU || ACT == ACT_GELU_TANH))
        r = fast_gelu_mixed_pair(e, sp, k);
      else if constexpr (C::DT == DT_E4M3 && ACT == ACT_SILU) r = act_pair<ACT_FAST_SILU>(sp, k);
      else r = act_pair<ACT>(sp, k);
      p[2 * e] = f2_lo(r);
      p[2 * e + 1] = f2_hi(r);
    }
    pack_p_chunk<C::DT>(p, pk);
    }
    if (MASKED) mask_p_words<C::DT>(pk, cols_in_range(col0 + 32 * ch, c_lo, c_hi));
    if (ch == 0 && !sync.wait_p_buffer()) return false;  // first store into the buffer
    store_p_chunk<C::DT>(t_p + ch * C::P_COLS_PER_32, pk);
  }
  return true;
}

// Each kernel configuration compiles only the activations the launcher can
// start it with (four groups: 16-bit GELU, tanh GELU and SiLU; two groups:
// the rest, or every activation for e4m3), so branches it never takes cost
// it no registers.
template <class C, bool MASKED>
__device__ __forceinline__ bool act_quarter_dispatch(int act, uint32_t t_s, uint32_t t_p, int col0,
                                                     const ActConsts& k, int c_lo, int c_hi, const StepSync& sync) {
#define GDPA_ACT_CASE(A) \
  case A: return act_quarter<C, A, MASKED>(t_s, t_p, col0, k, c_lo, c_hi, sync);
  if constexpr (C::NG == 4 && C::DT != DT_E4M3) {
    switch (act) {
      GDPA_ACT_CASE(ACT_GELU)
      GDPA_ACT_CASE(ACT_GELU_TANH)
      default: return act_quarter<C, ACT_SILU, MASKED>(t_s, t_p, col0, k, c_lo, c_hi, sync);
    }
  } else {
    switch (act) {
      GDPA_ACT_CASE(ACT_IDENTITY)
      GDPA_ACT_CASE(ACT_FAST_GELU)
      GDPA_ACT_CASE(ACT_RELU)
      GDPA_ACT_CASE(ACT_RELU2)
      GDPA_ACT_CASE(ACT_LEAKY_RELU)
      GDPA_ACT_CASE(ACT_FAST_GELU_BF16)
      GDPA_ACT_CASE(ACT_FAST_SILU)
      default: break;
    }
    if constexpr (C::DT == DT_E4M3) {
      switch (act) {
        GDPA_ACT_CASE(ACT_GELU)
        GDPA_ACT_CASE(ACT_GELU_TANH)
        GDPA_ACT_CASE(ACT_SILU)
        default: break;
      }
    }
    return act_quarter<C, ACT_HARDSWISH, MASKED>(t_s, t_p, col0, k, c_lo, c_hi, sync);
  }
#undef GDPA_ACT_CASE
}

// ---------------------------------------------------------------- MXFP8 scale factors
//
// Scale-factor atoms (512 bytes, what tcgen05.cp copies to TMEM): atom row l,
// word j, byte b holds the scale of tile row (Q, K) or value column (V)
// l + 32 j and K block 4 g + b of atom g. A kernel before the forward writes
// them into the workspace from the caller's E8M0 tensors (mx_stage_atoms);
// the TMA producers bulk-copy each tile's atoms into its shared-memory slot
// with the tile, completing on the same barrier, and the MMA warps copy them
// to TMEM in order with the tile's MMAs.

// ---------------------------------------------------------------- the kernel

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    gdpa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + C::QST * C::Q_BYTES;
  uint8_t* sV = sK + C::KST * C::K_BYTES;
  uint8_t* sStage = sV + C::VST * C::V_BYTES;  // STAGE_BYTES (may be 0)
  uint8_t* sSFQ = sStage + C::STAGE_BYTES;      // MX scale-factor atoms (SF_BYTES, may be 0)
  uint8_t* sSFK = sSFQ + C::QST * C::NQB * C::SF_ATOM;
  uint8_t* sSFV = sSFK + C::KST * C::NQB * C::SF_ATOM;
  uint8_t* sSFP = sSFV + C::VST * C::SF_ATOM;
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(sStage + C::STAGE_BYTES + C::SF_BYTES);
  static_assert(sizeof(FwdSmem) <= 1024, "barrier block too large");
  static_assert(!C::SOFTMAX || 1024 + sizeof(FwdSoftmaxSmem) <= C::EXTRA_BYTES, "softmax block too large");
  // only softmax configurations reserve room for it
  FwdSoftmaxSmem& ssm = *reinterpret_cast<FwdSoftmaxSmem*>(reinterpret_cast<uint8_t*>(&sm) + 1024);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const Problem& pb = args.pb;
  volatile int* abort_flag = &sm.abort_flag;
  constexpr bool softmax = C::SOFTMAX;

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    constexpr uint32_t kFullCount = 1;
    for (int i = 0; i < C::QST; ++i) {
      mbar_init(&sm.q_full[i], kFullCount);
      mbar_init(&sm.q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i], 128 * C::NG);
    }
    for (int i = 0; i < C::KST; ++i) {
      mbar_init(&sm.k_full[i], kFullCount);
      mbar_init(&sm.k_empty[i], 1);
    }
    for (int i = 0; i < C::VST; ++i) {
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 1);
    }
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.o_empty, C::SEP_EPI ? 128 : 128 * C::NG);
    mbar_init(&sm.stat_full, 128 * C::NG);
    mbar_init(&sm.stat_empty, 128);
    mbar_init(&sm.pv_done[0], 1);
    mbar_init(&sm.pv_done[1], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.red_full[i], 128 * C::NG);
      mbar_init(&sm.drain[i], 1);
    }
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
  }
  if (warp == 3 && lane == 0) prefetch_tmap(&tm_v);
  if constexpr (C::MX) {
    if (warp == 3) {  // P's scale factors: 2^0 for every row and K block
      for (int i = lane; i < C::SF_ATOM / 4; i += 32) reinterpret_cast<uint32_t*>(sSFP)[i] = 0x7F7F7F7Fu;
      fence_async_shared();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  pdl_wait();  // the work list and inputs come from earlier kernels; out may still be read
  // read only after the wait: the work list is the previous kernel's output
  const int n_work = args.work->count * pb.h_q;
  pdl_release();

  if (warp == 0) {
    // ------------------------------------------------ TMA producers: the K ring (lane 0) and Q tiles (lane 1)
    // Separate threads, so that K can run its full ring ahead while a Q slot
    // is still in use (with one KV block per item, Q slots free only one
    // item at a time).
    if (lane == 0) {
      uint32_t k_it = 0;
      StepCursor kc;
      kc.start(args, n_work);
      bool ok = true;
      while (kc.active && ok) {
        const int ks = k_it % C::KST;
        ok = mbar_wait(&sm.k_empty[ks], ((k_it / C::KST) & 1) ^ 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&sm.k_full[ks], C::K_BYTES + (C::MX ? C::NQB * C::SF_ATOM : 0));
        for (int bx = 0; bx < C::QK_BOXES; ++bx)
          tma_load_3d(sK + ks * C::K_BYTES + bx * C::BOX_BYTES, &tm_k, &sm.k_full[ks], bx * C::BOX_ELEMS, kc.it.g,
                      kc.it.k_start + kc.j * kTileK);
        if constexpr (C::MX) {  // the K tile's scale atoms (keyed by its first 32-key group)
          const size_t grp = static_cast<size_t>((kc.it.k_start + kc.j * kTileK) / 32) * pb.h_kv + kc.it.g;
          bulk_load_1d(sSFK + ks * C::NQB * C::SF_ATOM, args.atoms_k + grp * C::NQB * C::SF_ATOM,
                       C::NQB * C::SF_ATOM, &sm.k_full[ks]);
        }
        ++k_it;
        kc.advance(args, n_work);
      }
      if (*abort_flag) {  // let this thread's last loads land before the tiles go away
        for (uint32_t i = 0; i < k_it && i < static_cast<uint32_t>(C::KST); ++i) {
          const uint32_t n = k_it - 1 - i;
          if (!mbar_wait_timed(&sm.k_full[n % C::KST], (n / C::KST) & 1, kDrainTimeoutNs)) sm.drain_failed = 1;
        }
      }
    } else if (lane == 1) {
      uint32_t q_loads = 0;
      StepCursor qc;
      qc.start(args, n_work);
      bool ok = true;
      while (qc.active && ok) {  // one Q tile per item, into the slot that item's predecessors freed
        const int slot = qc.item_idx % C::QST;
        ok = mbar_wait(&sm.q_empty[slot], ((qc.item_idx / C::QST) & 1) ^ 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&sm.q_full[slot], C::Q_BYTES + (C::MX ? C::NQB * C::SF_ATOM : 0));
        for (int bx = 0; bx < C::QK_BOXES; ++bx)
          tma_load_3d(sQ + slot * C::Q_BYTES + bx * C::BOX_BYTES, &tm_q, &sm.q_full[slot], bx * C::BOX_ELEMS,
                      qc.it.h, qc.it.q_start + qc.it.r0);
        if constexpr (C::MX)  // the Q tile's scale atoms (keyed by the work item)
          bulk_load_1d(sSFQ + slot * C::NQB * C::SF_ATOM,
                       args.atoms_q + static_cast<size_t>(qc.it.pos) * C::NQB * C::SF_ATOM, C::NQB * C::SF_ATOM,
                       &sm.q_full[slot]);
        ++q_loads;
        qc.next_item(args, n_work);
      }
      if (*abort_flag) {  // let this thread's last loads land before the tiles go away
        for (uint32_t i = 0; i < q_loads && i < static_cast<uint32_t>(C::QST); ++i) {
          const uint32_t n = q_loads - 1 - i;
          if (!mbar_wait_timed(&sm.q_full[n % C::QST], (n / C::QST) & 1, kDrainTimeoutNs)) sm.drain_failed = 1;
        }
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------ TMA producer: the V ring
    // (its own thread, so that a V stage still in use by PV does not hold
    // back the K loads, which S needs a GEMM earlier)
    if (lane == 0) {
      uint32_t v_it = 0;
      StepCursor vc;
      vc.start(args, n_work);
      bool ok = true;
      while (vc.active && ok) {
        const int vs = v_it % C::VST;
        ok = mbar_wait(&sm.v_empty[vs], ((v_it / C::VST) & 1) ^ 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&sm.v_full[vs], C::V_BYTES + (C::MX ? C::SF_ATOM : 0));
        for (int bx = 0; bx < C::V_BOXES; ++bx)
          tma_load_3d(sV + vs * C::V_BYTES + bx * C::BOX_BYTES, &tm_v, &sm.v_full[vs], bx * C::BOX_ELEMS, vc.it.g,
                      vc.it.k_start + vc.j * kTileK);
        if constexpr (C::MX) {  // the V tile's scale atom
          const size_t grp = static_cast<size_t>((vc.it.k_start + vc.j * kTileK) / 32) * pb.h_kv + vc.it.g;
          bulk_load_1d(sSFV + vs * C::SF_ATOM, args.atoms_v + grp * C::SF_ATOM, C::SF_ATOM, &sm.v_full[vs]);
        }
        ++v_it;
        vc.advance(args, n_work);
      }
      if (*abort_flag) {  // let this thread's last loads land before the tiles go away
        for (uint32_t i = 0; i < v_it && i < static_cast<uint32_t>(C::VST); ++i) {
          const uint32_t n = v_it - 1 - i;
          if (!mbar_wait_timed(&sm.v_full[n % C::VST], (n / C::VST) & 1, kDrainTimeoutNs)) sm.drain_failed = 1;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer: S = Q K^T (whole warp, one lane issues)
    {
      const uint64_t dq0 = sdesc_sw128(smem_u32(sQ), 16, 1024), dk0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      uint32_t k_it = 0, u = 0;
      const bool gate = pv_gate_on_s(args.act);
      StepCursor sc;
      sc.start(args, n_work);
      bool ok = true;
      while (sc.active && ok) {
        const int slot = sc.item_idx % C::QST;
        const int b = u & 1;
        // S buffer b last held S(u-2): the activation groups have read it once P(u-2) is full
        if (u >= 2) {
          ok = mbar_wait(&sm.p_full[b], ((u - 2) >> 1) & 1, abort_flag);
          if (ok && gate) ok = mbar_wait(&sm.pv_done[b], ((u - 2) >> 1) & 1, abort_flag);
        }
        if (ok && sc.j == sc.it.lo) ok = mbar_wait(&sm.q_full[slot], (sc.item_idx / C::QST) & 1, abort_flag);
        const int ks = k_it % C::KST;
        if (ok) ok = mbar_wait(&sm.k_full[ks], (k_it / C::KST) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        const uint64_t a0 = sdesc_at(dq0, slot * C::Q_BYTES), b0 = sdesc_at(dk0, ks * C::K_BYTES);
        const uint32_t d = tbase + C::T_S + b * 128;
        // MX: this Q tile's (first step of its item) and this K stage's scale atoms into TMEM
        // (the atoms came with the tiles, by bulk copy)
        const uint32_t sfq = tbase + C::T_SFQ + slot * C::NQB * 4, sfk = tbase + C::T_SFK + ks * C::NQB * 4;
        if constexpr (C::MX) {
          if (sc.j == sc.it.lo)
            for (int g = 0; g < C::NQB; ++g)
              tmem_cp_atom_w(sfq + g * 4, sdesc_rows16(smem_u32(sSFQ + (slot * C::NQB + g) * C::SF_ATOM)));
          for (int g = 0; g < C::NQB; ++g)
            tmem_cp_atom_w(sfk + g * 4, sdesc_rows16(smem_u32(sSFK + (ks * C::NQB + g) * C::SF_ATOM)));
        }
#pragma unroll
        for (int k = 0; k < C::S_MMAS; ++k) {
          const uint32_t off = (k / 4) * C::BOX_BYTES + (k % 4) * 32;
          if constexpr (C::MX)  // one MMA per 32-element scale block k: atom k / 4, byte k % 4
            mma_mx_ss_w(d, sdesc_at(a0, off), sdesc_at(b0, off), idesc_mx(128, 128, 0, 0, k % 4, k % 4),
                        sfq + (k / 4) * 4, sfk + (k / 4) * 4, k > 0);
          else if constexpr (C::DT == DT_E4M3)
            mma_f8_ss_w(d, sdesc_at(a0, off), sdesc_at(b0, off), C::IDESC_S, k > 0);
          else
            mma_f16_ss_w(d, sdesc_at(a0, off), sdesc_at(b0, off), C::IDESC_S, k > 0);
        }
        mma_commit_w(&sm.s_full[b]);
        mma_commit_w(&sm.k_empty[ks]);
        ++k_it;
        if (sc.j == sc.it.hi) mma_commit_w(&sm.q_empty[slot]);
        ++u;
        sc.advance(args, n_work);
      }
      if (*abort_flag) {  // every MMA this warp issued has completed before TMEM goes away
        mma_commit_w(&sm.drain[0]);
        if (!__all_sync(0xffffffffu, mbar_wait_timed(&sm.drain[0], 0, kDrainTimeoutNs)) && lane == 0)
          sm.drain_failed = 1;
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------ MMA issuer: O += P V (whole warp, one lane issues)
    {
      const uint64_t dv0 = sdesc_sw128(smem_u32(sV), C::BOX_BYTES, 1024);
      uint32_t v_it = 0, u = 0, o_cnt = 0;
      StepCursor pc;
      pc.start(args, n_work);
      bool ok = true;
      if constexpr (C::MX) tmem_cp_atom_w(tbase + C::T_SFP, sdesc_rows16(smem_u32(sSFP)));  // P: scale 1 throughout
      while (pc.active && ok) {
        const int b = u & 1;
        ok = mbar_wait(&sm.p_full[b], (u >> 1) & 1, abort_flag);
        if (ok && pc.j == pc.it.lo) ok = mbar_wait(&sm.o_empty, (o_cnt++ & 1) ^ 1, abort_flag);
        const int vs = v_it % C::VST;
        if (ok) ok = mbar_wait(&sm.v_full[vs], (v_it / C::VST) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        const uint64_t b0 = sdesc_at(dv0, vs * C::V_BYTES);
        const bool acc = pc.j > pc.it.lo;
        const uint32_t sfv = tbase + C::T_SFV + vs * 4;
        if constexpr (C::MX) tmem_cp_atom_w(sfv, sdesc_rows16(smem_u32(sSFV + vs * C::SF_ATOM)));
#pragma unroll
        for (int k = 0; k < C::PV_MMAS; ++k) {
          const uint32_t a_t = tbase + C::T_P + b * 64 + k * (C::K_STEP * C::ESZ / 4);
          const uint64_t bd = sdesc_at(b0, k * C::K_STEP * 128);
          if constexpr (C::MX)  // K block k of 32 keys: byte k of the P and V atoms
            mma_mx_ts_w(tbase + C::T_O, a_t, bd, idesc_mx(128, C::DV, 0, 1, k, k), tbase + C::T_SFP, sfv,
                        (acc || k > 0) ? 1u : 0u);
          else if constexpr (C::DT == DT_E4M3)
            mma_f8_ts_w(tbase + C::T_O, a_t, bd, C::IDESC_PV, (acc || k > 0) ? 1u : 0u);
          else
            mma_f16_ts_w(tbase + C::T_O, a_t, bd, C::IDESC_PV, (acc || k > 0) ? 1u : 0u);
        }
        mma_commit_w(&sm.v_empty[vs]);
        mma_commit_w(&sm.pv_done[b]);
        ++v_it;
        if (pc.j == pc.it.hi) mma_commit_w(&sm.o_full);
        ++u;
        pc.advance(args, n_work);
      }
      if (*abort_flag) {  // every MMA this warp issued has completed before TMEM goes away
        mma_commit_w(&sm.drain[1]);
        if (!__all_sync(0xffffffffu, mbar_wait_timed(&sm.drain[1], 0, kDrainTimeoutNs)) && lane == 0)
          sm.drain_failed = 1;
      }
    }
  } else if (warp >= C::ACT_WARP0 && warp < C::ACT_WARP0 + 4 * C::NG) {
    // ------------------------------------------------ activation groups (and epilogue when folded)
    const int grp = (warp - C::ACT_WARP0) / 4;
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    const int col0 = C::GCOLS * grp;
    float qk_scale = args.scale;
    if (C::DT == DT_E4M3 && args.descale != nullptr) qk_scale *= args.descale[0] * args.descale[1];
    const ActConsts act_k = make_act_consts(qk_scale, C::DT == DT_BF16 ? kTruncBias : 1.0f);
    const float s_log2 = qk_scale * kLog2e;
    float v_scale = 1.0f;
    if (C::DT == DT_E4M3 && args.descale != nullptr) v_scale = args.descale[2];
    using OutT = typename std::conditional<C::DT == DT_FP16, __half, __nv_bfloat16>::type;
    OutT* out = reinterpret_cast<OutT*>(args.out);
    // 32-byte stores need a 32-byte aligned output (rows of dv = 128 are)
    const bool out_v8 = (reinterpret_cast<uintptr_t>(args.out) & 31) == 0;
    const bool gated = pv_gate_on_s(args.act);
    uint32_t u = 0, o_cnt = 0, stat_cnt = 0;

    // O of a finished item: this group's DV/4 columns of this thread's row.
    // Run after the next item's first step so that the item's last PV has
    // time to finish; the PV issuer waits o_empty before that item's first PV.
    auto epilogue = [&](const FwdItem& it, float l, float m) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.o_full, o_cnt++ & 1, abort_flag))) return false;
      tc_fence_after();
      // softmax runs with two groups and the separate epilogue warps, never here
      static_assert(!C::SOFTMAX || C::SEP_EPI, "the folded epilogue has no softmax statistics");
      (void)l;
      (void)m;
      const float f = v_scale;
      const int qrow = it.r0 + row;
      const bool row_valid = row < it.rows;
      OutT* orow = out + (static_cast<size_t>(it.q_start + qrow) * pb.h_q + it.h) * C::DV + grp * C::OCOLS;
      const uint32_t t_o = t_lane + C::T_O + grp * C::OCOLS;
      // every TMEM load first, so that O is released to the next item's PV
      // before the conversion and the global stores
      uint32_t o[C::OCOLS / C::OCH][C::OCH];
#pragma unroll
      for (int c = 0; c < C::OCOLS / C::OCH; ++c) tmem_ld_cols(t_o + c * C::OCH, o[c]);
#pragma unroll
      for (int c = 0; c < C::OCOLS / C::OCH; ++c) tmem_ld_wait(o[c]);
      tc_fence_before();
      mbar_arrive(&sm.o_empty);  // every TMEM read of O is done
      if constexpr (C::OCOLS == 32) {
        // 64 bytes of the row: paired 32-byte stores where the output allows
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float lo = __uint_as_float(o[e / 4][(2 * e) % 8]) * f;
          const float hi = __uint_as_float(o[e / 4][(2 * e) % 8 + 1]) * f;
          w[e] = C::DT == DT_FP16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
        }
        if (out_v8) {
          store_rows64_paired(reinterpret_cast<uint8_t*>(orow), static_cast<size_t>(pb.h_q) * C::DV * 2, lane, w,
                              row_valid);
        } else if (row_valid) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            *reinterpret_cast<uint4*>(orow + 8 * q4) = make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
        }
      } else if (row_valid) {
#pragma unroll
        for (int c = 0; c < C::OCOLS / C::OCH; ++c) {
#pragma unroll
          for (int q8 = 0; q8 < C::OCH / 8; ++q8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = __uint_as_float(o[c][8 * q8 + 2 * e]) * f;
              const float hi = __uint_as_float(o[c][8 * q8 + 2 * e + 1]) * f;
              w[e] = C::DT == DT_FP16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
            }
            *reinterpret_cast<uint4*>(orow + c * C::OCH + 8 * q8) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      return true;
    };

    // rescales this group's dv/NG columns of O by alpha (softmax)
    auto rescale_o = [&](float alpha) {
      const uint32_t t_o = t_lane + C::T_O + grp * C::OCOLS;
#pragma unroll
      for (int c = 0; c < C::OCOLS; c += C::OCH) {
        uint32_t o[C::OCH];
        tmem_ld_cols(t_o + c, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int e = 0; e < C::OCH; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st_cols(t_o + c, o);
      }
    };

    bool ok = true, pend = false;
    FwdItem pit{};
    float pl = 0.0f, pm = 0.0f;
    for (int round = 0; ok; ++round) {
      const int pos = zigzag_pos(round, blockIdx.x, gridDim.x);
      if (pos >= n_work) break;
      const FwdItem it = fwd_decode(args, pos);
      const int qrow = it.r0 + row;
      if (it.n == 0) {  // no allowed key for any row: exact zeros
        if (!C::SEP_EPI && row < it.rows) {
          OutT* orow = out + (static_cast<size_t>(it.q_start + qrow) * pb.h_q + it.h) * C::DV + grp * C::OCOLS;
          for (int q8 = 0; q8 < C::OCOLS / 8; ++q8) reinterpret_cast<uint4*>(orow)[q8] = make_uint4(0, 0, 0, 0);
          if (softmax && grp == 0 && args.lse != nullptr)
            args.lse[static_cast<size_t>(it.h) * pb.total_q + it.q_start + qrow] = -INFINITY;
        }
        continue;
      }
      int kmin = 1, kmax = 0;
      if (!(row < it.rows && key_range(qrow, qrow, it.lq, it.lk, pb.causal, pb.window, kmin, kmax))) {
        kmin = 1;
        kmax = 0;
      }
      float m = -INFINITY, l = 0.0f;
      for (int j = it.lo; j <= it.hi; ++j, ++u) {
        const int b = u & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.s_full[b], (u >> 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const int c_lo = kmin - j * kTileK, c_hi = kmax - j * kTileK;
        const uint32_t t_s = t_lane + C::T_S + b * 128 + col0;
        const uint32_t t_p = t_lane + C::T_P + b * 64 + grp * (C::GCOLS / 32) * C::P_COLS_PER_32;
        const StepSync sync{&sm.pv_done[b], u, abort_flag, gated};
        if constexpr (!softmax) {
          if (__all_sync(0xffffffffu, c_lo <= col0 && c_hi >= col0 + C::GCOLS - 1))
            ok = act_quarter_dispatch<C, false>(args.act, t_s, t_p, col0, act_k, c_lo, c_hi, sync);
          else
            ok = act_quarter_dispatch<C, true>(args.act, t_s, t_p, col0, act_k, c_lo, c_hi, sync);
          if (!ok) break;
        } else {
          // online softmax in the log2 domain; the groups agree on the row max
          uint32_t sa[C::GCOLS];
          tmem_ld32(t_s, *reinterpret_cast<uint32_t(*)[32]>(sa));
          if constexpr (C::GCOLS == 64) tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(sa + 32));
          tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(sa));
          if constexpr (C::GCOLS == 64) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(sa + 32));
          float mb = -INFINITY;
#pragma unroll
          for (int e = 0; e < C::GCOLS; ++e) {
            const int c0 = col0 + e;
            if (c0 >= c_lo && c0 <= c_hi) mb = fmaxf(mb, __uint_as_float(sa[e]) * s_log2);
          }
          // exchange through an mbarrier (bounded wait, unlike a named barrier,
          // so a warp whose wait gave up cannot strand the others here)
          ssm.red[u & 1][grp][row] = mb;
          mbar_arrive(&sm.red_full[u & 1]);
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.red_full[u & 1], (u >> 1) & 1, abort_flag));
          if (!ok) break;
#pragma unroll
          for (int g = 0; g < C::NG; ++g) mb = fmaxf(mb, ssm.red[u & 1][g][row]);
          // m is stale by at most 2^8: raise it (and rescale O) only past that
          const bool raise = mb > -INFINITY && (m == -INFINITY || mb > m + 8.0f);
          const float m_new = raise ? mb : m;
          const float alpha = raise && m != -INFINITY ? ex2_approx(m - m_new) : 1.0f;
          if (__any_sync(0xffffffffu, raise && m != -INFINITY) && j > it.lo) {
            // O holds the previous step's PV: wait for it, then rescale this group's columns of O
            ok = __all_sync(0xffffffffu, mbar_wait(&sm.pv_done[(u - 1) & 1], ((u - 1) >> 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            rescale_o(alpha);
          }
          l *= alpha;
          m = m_new;
          ok = sync.wait_p_buffer();
          if (!ok) break;
#pragma unroll
          for (int ch = 0; ch < C::GCOLS / 32; ++ch) {
            float p[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int cc = col0 + 32 * ch + e;
              const float v =
                  (cc >= c_lo && cc <= c_hi) ? ex2_approx(__uint_as_float(sa[32 * ch + e]) * s_log2 - m) : 0.0f;
              l += v;
              p[e] = v;
            }
            uint32_t pk[16];
            pack_p_chunk<C::DT>(p, pk);
            store_p_chunk<C::DT>(t_p + ch * C::P_COLS_PER_32, pk);
          }
        }
        tmem_st_wait();
        tc_fence_before();
#ifdef GDPA_TEST_HOOKS
        if (!(blockIdx.x == 0 && static_cast<int>(u) == args.test_skip_step))
#endif
        mbar_arrive(&sm.p_full[b]);
        if (!C::SEP_EPI && j == it.lo && pend) {
          ok = epilogue(pit, pl, pm);
          pend = false;
          if (!ok) break;
        }
      }
      if (!ok) break;
      if constexpr (C::SEP_EPI) {
        if (softmax) {  // hand the row statistics to the epilogue warps
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.stat_empty, (stat_cnt++ & 1) ^ 1, abort_flag));
          if (!ok) break;
          ssm.stat_l[grp][row] = l;
          if (grp == 0) ssm.stat_m[row] = m;
          mbar_arrive(&sm.stat_full);
        }
      } else {
        pend = true;
        pit = it;
        pl = l;
        pm = m;
      }
    }
    if constexpr (!C::SEP_EPI) {
      if (ok && pend) ok = epilogue(pit, pl, pm);
    }
  } else if (C::SEP_EPI && warp >= C::EPI_WARP0) {
    // ------------------------------------------------ epilogue warps (two activation groups)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t t_o = tbase + (static_cast<uint32_t>(quad * 32) << 16) + C::T_O;
    float v_scale = 1.0f;
    if (C::DT == DT_E4M3 && args.descale != nullptr) v_scale = args.descale[2];
    using OutT = typename std::conditional<C::DT == DT_FP16, __half, __nv_bfloat16>::type;
    OutT* out = reinterpret_cast<OutT*>(args.out);
    const bool out_v8 = (reinterpret_cast<uintptr_t>(args.out) & 31) == 0;
    uint32_t o_cnt = 0, stat_cnt = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int pos = zigzag_pos(round, blockIdx.x, gridDim.x);
      if (pos >= n_work) break;
      const FwdItem it = fwd_decode(args, pos);
      const int qrow = it.r0 + row;
      const bool row_valid = row < it.rows;
      OutT* orow = out + (static_cast<size_t>(it.q_start + qrow) * pb.h_q + it.h) * C::DV;
      float* lse_at = args.lse + static_cast<size_t>(it.h) * pb.total_q + it.q_start + qrow;
      if (it.n == 0) {  // no allowed key for any row: exact zeros
        if (row_valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
          for (int q4 = 0; q4 < C::DV * 2 / 16; ++q4) dst[q4] = make_uint4(0, 0, 0, 0);
          if (softmax && args.lse != nullptr) *lse_at = -INFINITY;
        }
        continue;
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&sm.o_full, o_cnt++ & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      float f = v_scale, lse = 0.0f;
      if (softmax) {
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.stat_full, stat_cnt++ & 1, abort_flag));
        if (!ok) break;
        float l = 0.0f;
#pragma unroll
        for (int g = 0; g < C::NG; ++g) l += ssm.stat_l[g][row];
        const float m = ssm.stat_m[row];
        mbar_arrive(&sm.stat_empty);
        f = l > 0.0f ? v_scale / l : 0.0f;
        lse = l > 0.0f ? m * 0.6931471805599453f + __logf(l) : -INFINITY;
      }
      // O from TMEM 32 columns at a time, packed to 16 bits; TMEM is released
      // as soon as the last columns are in registers
      constexpr int ECH = C::DV / 32;
      if constexpr (C::STAGE_BYTES > 0) {
        // through this warp's 32-row x 128-byte staging box (16-byte pieces
        // XOR-swizzled by row), 64 columns at a time, so that eight lanes
        // write one row's 128 contiguous bytes
        uint8_t* stg = sStage + quad * 4096;
        const size_t row_stride = static_cast<size_t>(pb.h_q) * C::DV;
        OutT* obase = out + (static_cast<size_t>(it.q_start + it.r0 + quad * 32) * pb.h_q + it.h) * C::DV;
#pragma unroll 1
        for (int ch = 0; ch < ECH; ++ch) {
          uint32_t o[32];
          tmem_ld32(t_o + ch * 32, o);
          tmem_ld_wait(o);
          if (ch == ECH - 1) {
            tc_fence_before();
            mbar_arrive(&sm.o_empty);  // every TMEM read of O is done
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = __uint_as_float(o[8 * q4 + 2 * e]) * f, hi = __uint_as_float(o[8 * q4 + 2 * e + 1]) * f;
              w[e] = C::DT == DT_FP16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
            }
            const int piece = 4 * (ch & 1) + q4;
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((piece ^ (lane & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if ((ch & 1) == 1 || ch == ECH - 1) {  // a 64-column half (or the last 32) is staged: write it out
            __syncwarp();
            const int piece = lane & 7, npieces = (ch & 1) ? 8 : 4;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = 4 * i + (lane >> 3);
              if (quad * 32 + r < it.rows && piece < npieces) {
                const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 128 + ((piece ^ (r & 7)) << 4));
                *reinterpret_cast<uint4*>(obase + r * row_stride + (ch >> 1) * 64 + piece * 8) = v;
              }
            }
            __syncwarp();
          }
        }
      } else {
#pragma unroll 1
        for (int ch = 0; ch < ECH; ++ch) {
          uint32_t o[32];
          tmem_ld32(t_o + ch * 32, o);
          tmem_ld_wait(o);
          if (ch == ECH - 1) {
            tc_fence_before();
            mbar_arrive(&sm.o_empty);
          }
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float lo = __uint_as_float(o[2 * e]) * f, hi = __uint_as_float(o[2 * e + 1]) * f;
            w[e] = C::DT == DT_FP16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
          }
          if (out_v8) {
            store_rows64_paired(reinterpret_cast<uint8_t*>(orow + ch * 32), static_cast<size_t>(pb.h_q) * C::DV * 2,
                                lane, w, row_valid);
          } else if (row_valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) dst[q4] = make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
          }
        }
      }
      if (softmax && row_valid && args.lse != nullptr) *lse_at = lse;
    }
  }

  // ------------------------------------------------ teardown
  // After an abort each role above has waited (time-bounded) for its own
  // TMA loads and MMAs in flight; only if one of those waits gave up does
  // the CTA also wait a fixed 1 ms before TMEM and shared memory go away.
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

// Whether e4m3 inputs run every elementwise activation with four groups.
constexpr bool kFp8FourGroups = false;

// Four activation groups where the activation's arithmetic, not the tensor
// core, sets the pace (16-bit GELU, tanh GELU, SiLU); two elsewhere, which
// leaves each thread more registers.
__host__ __device__ constexpr bool fwd_four_groups(int act, int dt) {
  return dt != DT_E4M3 ? (act == ACT_GELU || act == ACT_GELU_TANH || act == ACT_SILU) : kFp8FourGroups && act != ACT_SOFTMAX;
}

template <int DQK, int DV, int DT, int NG, bool SOFTMAX = false, bool MX = false>
cudaError_t launch_fwd_ng(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& a,
                          int grid, cudaStream_t stream) {
  using C = FwdCfg<DQK, DV, DT, NG, SOFTMAX, MX>;
  auto kern = gdpa_fwd_kernel<C>;
  const cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, stream, tq, tk, tv, a);
}

// MXFP8 (block-scaled e4m3): head dims with d_v = 128 only.
template <int DQK, int DV>
cudaError_t launch_fwd_mx(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& a,
                          int grid, cudaStream_t stream) {
  if constexpr (DV == 128 && DQK % 32 == 0) {
    if (a.act == ACT_SOFTMAX) return launch_fwd_ng<DQK, DV, DT_E4M3, 2, true, true>(tq, tk, tv, a, grid, stream);
    return launch_fwd_ng<DQK, DV, DT_E4M3, 2, false, true>(tq, tk, tv, a, grid, stream);
  } else {
    return cudaErrorNotSupported;
  }
}

template <int DQK, int DV, int DT>
cudaError_t launch_fwd_cfg(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& a,
                           int grid, cudaStream_t stream) {
  if constexpr (DT != DT_E4M3 || kFp8FourGroups) {
    if (fwd_four_groups(a.act, DT)) return launch_fwd_ng<DQK, DV, DT, 4>(tq, tk, tv, a, grid, stream);
  }
  if (a.act == ACT_SOFTMAX) return launch_fwd_ng<DQK, DV, DT, 2, true>(tq, tk, tv, a, grid, stream);
  return launch_fwd_ng<DQK, DV, DT, 2>(tq, tk, tv, a, grid, stream);
}

}  // namespace gdpa
