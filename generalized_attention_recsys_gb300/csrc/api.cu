// C ABI of libgdpa.so: argument checks, tensor maps, work lists, launches.
//
// The entry points follow the flash_attn_varlen_func statement of the
// problem on the gdpa/README.md page ("CUTE-DSL" API block): packed q/k/v with
// cumulative sequence offsets, max lengths, an activation, scale, causal flag
// and window. See include/gdpa.h for argument meaning and error behaviour.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "../../include/gdpa.h"
#include "act.cuh"
#include "args.h"
#include "common.cuh"

// The kernels' activation codes are the C ABI's, value for value.
static_assert(gdpa::ACT_IDENTITY == GDPA_ACT_IDENTITY && gdpa::ACT_GELU == GDPA_ACT_GELU &&
                  gdpa::ACT_GELU_TANH == GDPA_ACT_GELU_TANH && gdpa::ACT_FAST_GELU == GDPA_ACT_FAST_GELU &&
                  gdpa::ACT_RELU == GDPA_ACT_RELU && gdpa::ACT_RELU2 == GDPA_ACT_RELU2 &&
                  gdpa::ACT_LEAKY_RELU == GDPA_ACT_LEAKY_RELU && gdpa::ACT_SILU == GDPA_ACT_SILU &&
                  gdpa::ACT_HARDSWISH == GDPA_ACT_HARDSWISH && gdpa::ACT_SOFTMAX == GDPA_ACT_SOFTMAX &&
                  gdpa::ACT_FAST_GELU_BF16 == GDPA_ACT_FAST_GELU_BF16 && gdpa::ACT_FAST_SILU == GDPA_ACT_FAST_SILU &&
                  gdpa::ACT_COUNT == GDPA_ACT_FAST_SILU + 1,
              "activation codes differ between the kernels and gdpa.h");

namespace gdpa {

// Per-device status word written by kernels whose bounded waits gave up.
__device__ int g_status_word;

namespace {

constexpr int kMaxDevices = 64;

int* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  static int* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> g(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  static int counts[kMaxDevices] = {};
  if (counts[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    counts[dev] = n;
  }
  return counts[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [rows, heads, dim] row-major tensor as a 3-D map (dim, heads, rows) with
// a (128-byte, 1, 128-row) box and 128-byte swizzle. rows == 0 is encoded as
// one row over `fallback` (the kernels never read it then).
bool make_map(CUtensorMap* m, const void* ptr, int rows, int heads, int dim, int dtype, const void* fallback) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const int esz = dtype == DT_E4M3 ? 1 : 2;
  const CUtensorMapDataType dt = dtype == DT_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : dtype == DT_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  if (rows <= 0 || ptr == nullptr) {
    rows = 1;
    ptr = fallback;
  }
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(dim) * esz, static_cast<cuuint64_t>(heads) * dim * esz};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esz), 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [rows, heads, dim] accumulator as the target of TMA reduce-adds: boxes
// of 32 rows x 32 columns (128 bytes, the 128-byte swizzle span).
bool make_acc_map(CUtensorMap* m, float* ptr, int rows, int heads, int dim, const void* fallback) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  void* base = ptr;
  if (rows <= 0 || ptr == nullptr) {
    rows = 1;
    base = const_cast<void*>(fallback);
  }
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(dim) * 4, static_cast<cuuint64_t>(heads) * dim * 4};
  cuuint32_t box[3] = {32, 1, 32};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Upper bounds on work-list entries: sum over sequences of ceil(L / rows).
size_t fwd_list_cap(const gdpa_shape* s) {
  return static_cast<size_t>(s->total_q) / kFwdItemRows + static_cast<size_t>(s->batch) + 1;
}
size_t bwd_list_cap(const gdpa_shape* s) {
  return static_cast<size_t>(s->total_k) / kTileK + static_cast<size_t>(s->batch) + 1;
}
size_t list_bytes(size_t cap) { return round256(offsetof(WorkList, items) + sizeof(WorkEntry) * cap); }

// MXFP8 forward: the scale atoms (512 bytes each; see mx_stage_atoms), per work item and
// 4-block group of q, per 32-key group and kv head for k (4-block groups) and v.
constexpr size_t kAtom = 512;
size_t mx_nqb(const gdpa_shape* s) { return (static_cast<size_t>(s->d_qk) / 32 + 3) / 4; }
size_t mx_groups(const gdpa_shape* s) { return (static_cast<size_t>(s->total_k) + 31) / 32; }
size_t mx_q_atom_bytes(const gdpa_shape* s) { return round256(fwd_list_cap(s) * s->h_q * mx_nqb(s) * kAtom); }
size_t mx_k_atom_bytes(const gdpa_shape* s) { return round256(mx_groups(s) * s->h_kv * mx_nqb(s) * kAtom); }
size_t mx_v_atom_bytes(const gdpa_shape* s) { return round256(mx_groups(s) * s->h_kv * kAtom); }

// Deterministic backward: one fp32 dQ slice [total_q, h_q, d_qk] per key block.
size_t dq_part_bytes(const gdpa_shape* s, int max_k) {
  const size_t nkv = max_k > 0 ? (static_cast<size_t>(max_k) + kTileK - 1) / kTileK : 0;
  return nkv * static_cast<size_t>(s->total_q) * s->h_q * s->d_qk * sizeof(float);
}

// Sequences stay below 2^30 tokens, so that mask arithmetic (a position plus
// a window) cannot overflow an int; a longer window selects the same keys.
constexpr int kMaxSeqLen = 1 << 30;

int validate(const gdpa_shape* s, int max_q, int max_k, int act, int causal, int window) {
  (void)causal;
  (void)window;
  if (!s) return GDPA_ERR_INVALID;
  if (s->batch < 0 || s->total_q < 0 || s->total_k < 0 || max_q < 0 || max_k < 0) return GDPA_ERR_INVALID;
  if (s->h_q <= 0 || s->h_kv <= 0 || s->h_q % s->h_kv != 0) return GDPA_ERR_INVALID;
  if (s->dtype < GDPA_BF16 || s->dtype > GDPA_E4M3) return GDPA_ERR_INVALID;
  if (act < GDPA_ACT_IDENTITY || act > GDPA_ACT_FAST_SILU) return GDPA_ERR_INVALID;
  const bool ok_dims = (s->d_qk == 64 && s->d_v == 64) || (s->d_qk == 96 && s->d_v == 96) ||
                       (s->d_qk == 128 && s->d_v == 128) || (s->d_qk == 192 && s->d_v == 128);
  if (!ok_dims) return GDPA_ERR_UNSUPPORTED;
  if (static_cast<long long>(s->total_q) * s->h_q * (s->d_qk > s->d_v ? s->d_qk : s->d_v) >= (1ll << 40))
    return GDPA_ERR_UNSUPPORTED;
  if (max_q >= kMaxSeqLen || max_k >= kMaxSeqLen) return GDPA_ERR_UNSUPPORTED;
  return GDPA_OK;
}

// Work list: one decoded entry (WorkEntry) per block. mode 0: a 128-row
// query tile, cost = KV blocks it visits; mode 1: a 128-row key block, cost =
// query blocks that see it. Sequences are sorted by the cost of their
// heaviest block, heaviest first (counting sort over cost buckets), and each
// sequence's blocks stay together in the list, heaviest first (causal: the
// last query tile / the first key block). Zigzag dealing then gives every CTA
// a balanced mix, and the blocks that share a sequence's K and V (or, in the
// backward, its Q, dO and dQ rows) run at the same time on neighbouring
// CTAs, so those tiles are read from DRAM about once rather than once per
// block when the problem outgrows L2.
constexpr int kBuckets = 2048;

// The entry's block fields; w = its number of blocks to visit (the cost).
__device__ __forceinline__ int4 item_blocks(const Problem& pb, int mode, int blk, int lq, int lk) {
  int lo, hi;
  if (mode == 0) {
    const int r0 = blk * kFwdItemRows;
    const int rows = min(lq - r0, kFwdItemRows);
    if (rows <= 0 || !key_range(r0, r0 + rows - 1, lq, lk, pb.causal, pb.window, lo, hi))
      return make_int4(r0, rows > 0 ? rows : 0, 0, 0);
    return make_int4(r0, rows, lo / kTileK, hi / kTileK - lo / kTileK + 1);
  }
  const int k0 = blk * kTileK;
  const int krows = min(lk - k0, kTileK);
  if (krows <= 0 || !query_range(k0, k0 + krows - 1, lq, lk, pb.causal, pb.window, lo, hi))
    return make_int4(k0, krows > 0 ? krows : 0, 0, 0);
  return make_int4(k0, krows, lo / kTileQ, hi / kTileQ - lo / kTileQ + 1);
}

// Cost bucket of a sequence: its heaviest block's cost.
// Called by a whole warp for one sequence: its items are shared out over the lanes.
__device__ __forceinline__ int seq_bucket_warp(const Problem& pb, int mode, int nblk, int lq, int lk, int lane) {
  int c = 0;
  for (int blk = lane; blk < nblk; blk += 32) c = max(c, item_blocks(pb, mode, blk, lq, lk).w);
  return min(__reduce_max_sync(0xffffffffu, c), kBuckets - 1);
}

// Block 0 builds the list; any further blocks zero `clear` (n4 float4s, the
// backward's dQ accumulator) meanwhile, so that clear needs no launch of its own.
__global__ void __launch_bounds__(1024) build_worklist(Problem pb, int mode, WorkList* wl, int cap, float4* clear,
                                                       size_t n4) {
  pdl_wait();  // the workspace may still be in use by the previous kernel
  pdl_release();
  if (blockIdx.x > 0) {
    const size_t nthr = static_cast<size_t>(gridDim.x - 1) * blockDim.x;
    for (size_t i = (blockIdx.x - 1) * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4; i += nthr)
      clear[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  __shared__ int hist[kBuckets];
  for (int i = threadIdx.x; i < kBuckets; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int rows = mode == 0 ? kFwdItemRows : kTileK;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  // one warp per sequence (a sequence's items can number in the hundreds)
  for (int b = wid; b < pb.batch; b += nwarps) {
    int qs, lq, ks, lk;
    seq_bounds(pb.cu_q, b, pb.max_q, qs, lq);
    seq_bounds(pb.cu_k, b, pb.max_k, ks, lk);
    const int len = mode == 0 ? lq : lk;
    const int nblk = len > 0 ? (len + rows - 1) / rows : 0;
    if (nblk == 0) continue;
    const int c = seq_bucket_warp(pb, mode, nblk, lq, lk, lane);
    if (lane == 0) atomicAdd(&hist[c], nblk);
  }
  __syncthreads();
  // exclusive prefix over the buckets, heaviest first: each of the 1024
  // threads owns two consecutive positions of that order; a warp scan, then
  // a scan of the 32 warp totals
  static_assert(kBuckets == 2 * 1024, "two buckets a thread");
  __shared__ int warp_sum[32];
  const int c0 = kBuckets - 1 - 2 * static_cast<int>(threadIdx.x), c1 = c0 - 1;
  const int h0 = hist[c0], h1 = hist[c1];
  int incl = h0 + h1;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_sum[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int w = warp_sum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    warp_sum[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int excl = incl - (h0 + h1) + (wid > 0 ? warp_sum[wid - 1] : 0);
  hist[c0] = excl;
  hist[c1] = excl + h0;
  if (threadIdx.x == 0) {
    const int run = warp_sum[31];
    wl->count = run < cap ? run : cap;
  }
  __syncthreads();
  for (int b = wid; b < pb.batch; b += nwarps) {
    int qs, lq, ks, lk;
    seq_bounds(pb.cu_q, b, pb.max_q, qs, lq);
    seq_bounds(pb.cu_k, b, pb.max_k, ks, lk);
    const int len = mode == 0 ? lq : lk;
    const int nblk = len > 0 ? (len + rows - 1) / rows : 0;
    if (nblk == 0) continue;
    const int c = seq_bucket_warp(pb, mode, nblk, lq, lk, lane);
    int base = 0;
    if (lane == 0) base = atomicAdd(&hist[c], nblk);  // the sequence's slots
    base = __shfl_sync(0xffffffffu, base, 0);
    for (int i = lane; i < nblk; i += 32) {
      // causal costs grow with the query tile and shrink with the key block: heaviest first
      const int blk = mode == 0 ? nblk - 1 - i : i;
      const int p = base + i;
      if (p < cap) {
        wl->items[p].seq = make_int4(qs, lq, ks, lk);
        wl->items[p].blk = item_blocks(pb, mode, blk, lq, lk);
      }
    }
  }
}

// MXFP8: rearranges the caller's E8M0 scales into the atoms that tcgen05.cp
// copies to TMEM (row l, word j, byte b: tile row or value column l + 32 j,
// K block 4 g + b of atom g), so that the forward's producers load them with
// plain bulk copies.
//   q: per work item (entry e, head h: position e h_q + h) and atom g, rows
//      q_start + r0 + r of the item's tile (past its rows: 2^0);
//   k: per 32-key group G and kv head, and atom g: keys 32 G + r (the 128-key
//      tile that starts at G; past total_k: 2^0);
//   v: per 32-key group G and kv head: value column n, the four 32-key blocks
//      G..G+3 of the tile that starts at G.
// q and k go through shared memory a tile of rows at a time (a work entry's
// 128 rows, or the rows of up to 8 consecutive key groups), read in 16-byte
// chunks; one thread then writes one 16-byte atom row. The tile's row stride
// is an odd number of words, so the 32 rows a warp reads fall in 32 banks.
// Also checks that every key sequence starts on a 32-key block (V's blocks
// are counted from key 0): one that does not is reported as GDPA_ERR_INVALID.
constexpr int kStageSmem = 48 * 1024 - 16;        // tile bytes (mx_stage_atoms takes 48 KB: 16 for the read past the end)
constexpr int kStageRowWords = kStageSmem / 512;  // >= row stride (words) of a 128-row tile

// Odd number of words that holds a tile row of w bytes.
__device__ __forceinline__ int stage_stride(int w) { return ((w + 3) / 4) | 1; }

// Copies bytes [c0, c0 + w) of rows t0 .. t0 + n - 1 (n >= 1) of the row-major
// byte matrix src (rows of rl bytes, nbytes in all, 16-byte aligned) into
// tile rows 0 .. n - 1 (stride words apart), reading 16-byte chunks. With rl,
// c0 and w multiples of 4 it moves words, else bytes (E = 4 or 1 bytes).
template <typename E>
__device__ __forceinline__ void stage_rows_as(const uint8_t* src, size_t nbytes, int rl, int t0, int n, int c0, int w,
                                              uint32_t* tile, int stride) {
  constexpr int S = sizeof(E), PER = 16 / S;  // elements per chunk
  const E* se = reinterpret_cast<const E*>(src);
  E* te = reinterpret_cast<E*>(tile);
  const int rle = rl / S, c0e = c0 / S, we = w / S, se_stride = stride * 4 / S;
  const size_t ne = nbytes / S;  // whole elements in src (nbytes is a multiple of S)
  const size_t first = static_cast<size_t>(t0) * rle;
  const size_t lo = first + c0e, hi = first + static_cast<size_t>(n - 1) * rle + c0e + we;
  const size_t base = lo & ~static_cast<size_t>(PER - 1);
  const int nchunks = static_cast<int>((hi - base + PER - 1) / PER);
  const int rel0 = static_cast<int>(static_cast<long long>(base) - static_cast<long long>(first));  // >= -(PER - 1)
  constexpr int U = 4;
  for (int c = threadIdx.x; c < nchunks; c += U * blockDim.x) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int cu = c + u * blockDim.x;
      const size_t o = base + static_cast<size_t>(cu) * PER;
      v[u] = make_uint4(0, 0, 0, 0);
      if (cu < nchunks) {
        if (o + PER <= ne) {
          v[u] = __ldg(reinterpret_cast<const uint4*>(se + o));
        } else {
          E* ve = reinterpret_cast<E*>(&v[u]);
          for (int k = 0; k < PER && o + k < ne; ++k) ve[k] = se[o + k];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int cu = c + u * blockDim.x;
      if (cu >= nchunks) break;
      const E* ve = reinterpret_cast<const E*>(&v[u]);
      const int rel = rel0 + cu * PER;  // element offset from row t0's start
      int r = rel >= 0 ? rel / rle : -((-rel + rle - 1) / rle);
      int col = rel - r * rle;
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        if (r >= 0 && r < n && col >= c0e && col < c0e + we) te[r * se_stride + col - c0e] = ve[k];
        if (++col == rle) {
          col = 0;
          ++r;
        }
      }
    }
  }
}

__global__ void __launch_bounds__(256) mx_stage_atoms(Problem pb, const WorkList* wl, int nqb, int nkb, int dv,
                                                      const uint8_t* sf_q, const uint8_t* sf_k, const uint8_t* sf_v,
                                                      uint4* aq, uint4* ak, uint4* av, int* status) {
  extern __shared__ uint4 stage_smem[];  // kStageSmem bytes of tile, plus one word read past its end
  uint32_t* tile = reinterpret_cast<uint32_t*>(stage_smem);
  pdl_wait();  // the work list is the previous kernel's
  pdl_release();
  const int ngroups = (pb.total_k + 31) / 32;
  const int max_heads = (kStageRowWords - 1) * 4 / nkb;  // heads whose row fits an odd stride <= kStageRowWords
  const int hcq = min(pb.h_q, max_heads), hck = min(pb.h_kv, max_heads);
  const int cq = (pb.h_q + hcq - 1) / hcq, ck = (pb.h_kv + hck - 1) / hck;
  const int sk = stage_stride(hck * nkb);
  const int ngk = max(1, min(8, (kStageSmem / (4 * sk) - 96) / 32));  // key groups per k tile
  const int n_qu = wl->count * cq, n_ku = (ngroups + ngk - 1) / ngk * ck;
  for (int u = blockIdx.x; u < n_qu + n_ku; u += gridDim.x) {
    int h0, hc, heads, t0, nvalid, ng, atom0;  // atom0: the unit's first atom (for its first group and head h0)
    const uint8_t* src;
    size_t nbytes;
    uint4* dst;
    if (u < n_qu) {  // work entry e, heads h0 ..
      const int e = u / cq;
      h0 = (u - e * cq) * hcq;
      hc = min(hcq, pb.h_q - h0);
      heads = pb.h_q;
      t0 = wl->items[e].seq.x + wl->items[e].blk.x;
      nvalid = wl->items[e].blk.y;
      ng = 1;
      atom0 = (e * heads + h0) * nqb;
      src = sf_q;
      nbytes = static_cast<size_t>(pb.total_q) * pb.h_q * nkb;
      dst = aq;
    } else {  // key groups G0 .. G0 + ng - 1, kv heads h0 ..
      const int v = u - n_qu, gc = v / ck, g0 = gc * ngk;
      h0 = (v - gc * ck) * hck;
      hc = min(hck, pb.h_kv - h0);
      heads = pb.h_kv;
      t0 = 32 * g0;
      ng = min(ngk, ngroups - g0);
      nvalid = min(32 * ng + 96, pb.total_k - t0);
      atom0 = (g0 * heads + h0) * nqb;
      src = sf_k;
      nbytes = static_cast<size_t>(pb.total_k) * pb.h_kv * nkb;
      dst = ak;
    }
    const int w = hc * nkb, stride = stage_stride(w), rl = heads * nkb, c0 = h0 * nkb;
    __syncthreads();  // the previous tile's reads are done
    if (nvalid > 0) {
      if (((rl | c0 | w) & 3) == 0)
        stage_rows_as<uint32_t>(src, nbytes, rl, t0, nvalid, c0, w, tile, stride);
      else
        stage_rows_as<uint8_t>(src, nbytes, rl, t0, nvalid, c0, w, tile, stride);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < ng * hc * nqb * 32; i += blockDim.x) {  // one atom row each
      const int a = i >> 5, l = i & 31;
      const int gi = a / (hc * nqb), rem = a - gi * hc * nqb;
      const int hh = rem / nqb, g = rem - hh * nqb;
      const int ob = hh * nkb + 4 * g, ow = ob >> 2, sh = (ob & 3) * 8;  // the atom's bytes in a tile row
      const int nb = min(4, nkb - 4 * g);                                 // K blocks present (rest: 2^0)
      const uint32_t keep = nb == 4 ? 0xFFFFFFFFu : (1u << (8 * nb)) - 1;
      uint32_t wd[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = 32 * gi + l + 32 * j;
        wd[j] = 0x7F7F7F7Fu;
        if (r < nvalid) {
          const uint32_t* row = tile + r * stride + ow;
          const uint32_t x = sh ? __funnelshift_r(row[0], row[1], sh) : row[0];
          wd[j] = (x & keep) | (0x7F7F7F7Fu & ~keep);
        }
      }
      dst[(static_cast<size_t>(atom0) + static_cast<size_t>(gi) * heads * nqb + rem) * 32 + l] =
          make_uint4(wd[0], wd[1], wd[2], wd[3]);
    }
  }
  const int n_vr = ngroups * pb.h_kv * 32;  // v atom rows
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_vr; i += gridDim.x * blockDim.x) {
    const int a = i >> 5, l = i & 31;
    const int grp = a / pb.h_kv, head = a - grp * pb.h_kv;
    uint32_t wd[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      wd[j] = 0x7F7F7F7Fu;
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (grp + b < ngroups)
          wd[j] = (wd[j] & ~(0xFFu << (8 * b))) |
                  (static_cast<uint32_t>(sf_v[(static_cast<size_t>(grp + b) * pb.h_kv + head) * dv + l + 32 * j])
                   << (8 * b));
    }
    av[i] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
  }
  if (blockIdx.x == 0)
    for (int b = threadIdx.x; b < pb.batch; b += blockDim.x) {
      int ks, lk;
      seq_bounds(pb.cu_k, b, pb.max_k, ks, lk);
      if (ks % 32 != 0) atomicExch(status, 1);
    }
}

thread_local cudaEvent_t t_ev_before = nullptr, t_ev_after = nullptr;

#ifdef GDPA_TEST_HOOKS
// test-only builds: the step at which CTA 0 skips one arrive ([0] forward, [1] backward; -1 = none)
int g_test_skip[2] = {-1, -1};
#endif

void mark(cudaEvent_t ev, cudaStream_t stream) {
  if (ev) cudaEventRecord(ev, stream);
}

Problem make_problem(const gdpa_shape* s, const int32_t* cu_q, const int32_t* cu_k, int max_q, int max_k,
                     int causal, int window) {
  Problem pb;
  pb.batch = s->batch;
  pb.total_q = s->total_q;
  pb.total_k = s->total_k;
  pb.h_q = s->h_q;
  pb.h_kv = s->h_kv;
  pb.group = s->h_q / s->h_kv;
  pb.max_q = max_q;
  pb.max_k = max_k;
  pb.cu_q = cu_q;
  pb.cu_k = cu_k;
  pb.causal = causal ? 1 : 0;
  pb.window = window > 0 ? (window < kMaxSeqLen ? window : kMaxSeqLen) : 0;
  return pb;
}

}  // namespace
}  // namespace gdpa

using namespace gdpa;

extern "C" {

size_t gdpa_workspace_bytes(const gdpa_shape* s, int max_q, int max_k, int is_bwd) {
  if (validate(s, max_q, max_k, GDPA_ACT_IDENTITY, 0, 0) != GDPA_OK) return 0;
  if (!is_bwd) return list_bytes(fwd_list_cap(s));
  if (is_bwd == 3)  // gdpa_fwd_mxfp8: the forward's list and the scale atoms
    return list_bytes(fwd_list_cap(s)) + mx_q_atom_bytes(s) + mx_k_atom_bytes(s) + mx_v_atom_bytes(s);
  size_t b = list_bytes(bwd_list_cap(s));
  b += round256(static_cast<size_t>(s->total_q) * s->h_q * s->d_qk * sizeof(float));  // dQ accumulator
  b += round256(static_cast<size_t>(s->total_q) * s->h_q * sizeof(float));            // softmax rowsum(dO*O)
  if (is_bwd == 2) b += round256(dq_part_bytes(s, max_k));                          // deterministic dQ slices
  return b;
}

}  // extern "C"

namespace {

// The forward of gdpa_fwd (descale for e4m3) and gdpa_fwd_mxfp8 (sf_q/k/v).
int fwd_common(const gdpa_shape* s, const void* q, const void* k, const void* v, const int32_t* cu_q,
               const int32_t* cu_k, int max_q, int max_k, int act, float scale, int causal, int window,
               const float* descale, const uint8_t* sf_q, const uint8_t* sf_k, const uint8_t* sf_v, void* out,
               float* lse, void* workspace, size_t workspace_bytes, void* stream_) {
  int st = validate(s, max_q, max_k, act, causal, window);
  if (st != GDPA_OK) return st;
  const bool mx = sf_q != nullptr;
  if (mx) {
    if (s->dtype != GDPA_E4M3) return GDPA_ERR_INVALID;
    if (!((s->d_qk == 128 || s->d_qk == 192) && s->d_v == 128)) return GDPA_ERR_UNSUPPORTED;
    if (s->total_k > 0 && (!sf_k || !sf_v)) return GDPA_ERR_INVALID;
    if (!aligned16(sf_q) || (sf_k && !aligned16(sf_k)) || (sf_v && !aligned16(sf_v))) return GDPA_ERR_INVALID;
    if (!cu_k && max_k % 32 != 0) return GDPA_ERR_INVALID;  // fixed length: every key sequence starts on a block
  }
  if (s->total_q == 0 || s->batch == 0) return GDPA_OK;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return GDPA_ERR_INVALID;
  if (s->total_k > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return GDPA_ERR_INVALID;
  if ((cu_q == nullptr) != (cu_k == nullptr)) return GDPA_ERR_INVALID;
  if (!cu_q && (s->total_q != s->batch * max_q || s->total_k != s->batch * max_k)) return GDPA_ERR_INVALID;
  if (act == GDPA_ACT_SOFTMAX && !lse) return GDPA_ERR_INVALID;
  if (s->dtype == GDPA_E4M3 && !descale && !mx) return GDPA_ERR_INVALID;
  if (!workspace || !aligned16(workspace) || workspace_bytes < gdpa_workspace_bytes(s, max_q, max_k, mx ? 3 : 0))
    return GDPA_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const int nsm = sm_count();
  int* status = status_ptr();
  if (nsm <= 0 || !status) return GDPA_ERR_CUDA;

  const Problem pb = make_problem(s, cu_q, cu_k, max_q, max_k, causal, window);
  WorkList* wl = static_cast<WorkList*>(workspace);
  const int cap = static_cast<int>(fwd_list_cap(s));
  if (launch_pdl(build_worklist, dim3(1), dim3(1024), 0, stream, pb, 0, wl, cap, static_cast<float4*>(nullptr),
                 static_cast<size_t>(0)) != cudaSuccess)
    return GDPA_ERR_CUDA;
  uint8_t *atoms_q = nullptr, *atoms_k = nullptr, *atoms_v = nullptr;
  if (mx) {
    atoms_q = static_cast<uint8_t*>(workspace) + list_bytes(fwd_list_cap(s));
    atoms_k = atoms_q + mx_q_atom_bytes(s);
    atoms_v = atoms_k + mx_k_atom_bytes(s);
    if (launch_pdl(mx_stage_atoms, dim3(4 * nsm), dim3(256), kStageSmem + 16, stream, pb,
                   static_cast<const WorkList*>(wl), static_cast<int>(mx_nqb(s)), s->d_qk / 32, s->d_v, sf_q, sf_k,
                   sf_v, reinterpret_cast<uint4*>(atoms_q), reinterpret_cast<uint4*>(atoms_k),
                   reinterpret_cast<uint4*>(atoms_v), status) != cudaSuccess)
      return GDPA_ERR_CUDA;
  }

  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, s->total_q, s->h_q, s->d_qk, s->dtype, workspace) ||
      !make_map(&tk, k, s->total_k, s->h_kv, s->d_qk, s->dtype, workspace) ||
      !make_map(&tv, v, s->total_k, s->h_kv, s->d_v, s->dtype, workspace))
    return GDPA_ERR_CUDA;

  FwdArgs a;
  a.pb = pb;
  a.act = act;
  a.scale = scale;
  a.descale = mx ? nullptr : descale;
  a.sf_q = sf_q;
  a.sf_k = mx ? sf_k : nullptr;
  a.sf_v = mx ? sf_v : nullptr;
  a.atoms_q = atoms_q;
  a.atoms_k = atoms_k;
  a.atoms_v = atoms_v;
  a.out = out;
  a.lse = lse;
  a.work = wl;
  a.status = status;
#ifdef GDPA_TEST_HOOKS
  a.test_skip_step = g_test_skip[0];
#endif
  cudaError_t e;
  mark(t_ev_before, stream);
  switch (s->d_qk) {
    case 64: e = launch_fwd_d64(s->dtype, tq, tk, tv, a, nsm, stream); break;
    case 96: e = launch_fwd_d96(s->dtype, tq, tk, tv, a, nsm, stream); break;
    case 128: e = launch_fwd_d128(s->dtype, tq, tk, tv, a, nsm, stream); break;
    default: e = launch_fwd_d192(s->dtype, tq, tk, tv, a, nsm, stream); break;
  }
  mark(t_ev_after, stream);
  return e == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

}  // namespace

extern "C" {

int gdpa_fwd(const gdpa_shape* s, const void* q, const void* k, const void* v, const int32_t* cu_q,
             const int32_t* cu_k, int max_q, int max_k, int act, float scale, int causal, int window,
             const float* descale, void* out, float* lse, void* workspace, size_t workspace_bytes,
             void* stream_) {
  return fwd_common(s, q, k, v, cu_q, cu_k, max_q, max_k, act, scale, causal, window, descale, nullptr, nullptr,
                    nullptr, out, lse, workspace, workspace_bytes, stream_);
}

int gdpa_fwd_mxfp8(const gdpa_shape* s, const void* q, const void* k, const void* v, const uint8_t* q_scale,
                   const uint8_t* k_scale, const uint8_t* v_scale, const int32_t* cu_q, const int32_t* cu_k, int max_q,
                   int max_k, int act, float scale, int causal, int window, void* out, float* lse, void* workspace,
                   size_t workspace_bytes, void* stream_) {
  if (!q_scale) return GDPA_ERR_INVALID;
  return fwd_common(s, q, k, v, cu_q, cu_k, max_q, max_k, act, scale, causal, window, nullptr, q_scale, k_scale,
                    v_scale, out, lse, workspace, workspace_bytes, stream_);
}

int gdpa_bwd(const gdpa_shape* s, const void* q, const void* k, const void* v, const int32_t* cu_q,
             const int32_t* cu_k, int max_q, int max_k, int act, float scale, int causal, int window,
             const void* out, const float* lse, const void* dout, void* dq, void* dk, void* dv,
             int deterministic, void* workspace, size_t workspace_bytes, void* stream_) {
  int st = validate(s, max_q, max_k, act, causal, window);
  if (st != GDPA_OK) return st;
  if (s->dtype == GDPA_E4M3) return GDPA_ERR_UNSUPPORTED;
  if (s->batch == 0 || (s->total_q == 0 && s->total_k == 0)) return GDPA_OK;
  if ((cu_q == nullptr) != (cu_k == nullptr)) return GDPA_ERR_INVALID;
  if (!cu_q && (s->total_q != s->batch * max_q || s->total_k != s->batch * max_k)) return GDPA_ERR_INVALID;
  const void* need[] = {q, dout, dq};
  for (const void* p : need)
    if (s->total_q > 0 && (!p || !aligned16(p))) return GDPA_ERR_INVALID;
  const void* need_k[] = {k, v, dk, dv};
  for (const void* p : need_k)
    if (s->total_k > 0 && (!p || !aligned16(p))) return GDPA_ERR_INVALID;
  if (act == GDPA_ACT_SOFTMAX && (!out || !lse || !aligned16(out))) return GDPA_ERR_INVALID;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < gdpa_workspace_bytes(s, max_q, max_k, deterministic ? 2 : 1))
    return GDPA_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const int nsm = sm_count();
  int* status = status_ptr();
  if (nsm <= 0 || !status) return GDPA_ERR_CUDA;

  const Problem pb = make_problem(s, cu_q, cu_k, max_q, max_k, causal, window);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int cap = static_cast<int>(bwd_list_cap(s));
  WorkList* wl = reinterpret_cast<WorkList*>(ws);
  ws += list_bytes(cap);
  float* dq_acc = reinterpret_cast<float*>(ws);
  ws += round256(static_cast<size_t>(s->total_q) * s->h_q * s->d_qk * sizeof(float));
  float* drow = reinterpret_cast<float*>(ws);
  ws += round256(static_cast<size_t>(s->total_q) * s->h_q * sizeof(float));
  float* dq_part = deterministic ? reinterpret_cast<float*>(ws) : nullptr;

  // one key block per sequence (direct dQ) or deterministic slices: no accumulator to clear
  const bool accumulate = max_k > kTileK && !deterministic;
  const size_t n4 = accumulate ? static_cast<size_t>(s->total_q) * s->h_q * s->d_qk / 4 : 0;
  if (launch_pdl(build_worklist, dim3(n4 > 0 ? 1 + 2 * nsm : 1), dim3(1024), 0, stream, pb, 1, wl, cap,
                 reinterpret_cast<float4*>(dq_acc), n4) != cudaSuccess)
    return GDPA_ERR_CUDA;

  BwdArgs a;
  a.pb = pb;
  a.act = act;
  a.scale = scale;
  a.work = wl;
  a.status = status;
  a.out = out;
  a.lse = lse;
  a.dout = dout;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dq_acc = dq_acc;
  a.dq_part = dq_part;
  a.drow = drow;
#ifdef GDPA_TEST_HOOKS
  a.test_skip_step = g_test_skip[1];
#endif
  // one key block per sequence: each dQ row has a single producer, written in
  // place (deterministic by construction, so it serves both modes)
  a.dq_mode = max_k <= kTileK ? DQ_DIRECT : (deterministic ? DQ_SLICES : DQ_ACCUMULATE);
  a.n_kblocks = (max_k + kTileK - 1) / kTileK;
  a.d_qk = s->d_qk;
  a.d_v = s->d_v;
  a.dtype = s->dtype;
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!make_map(&tq, q, s->total_q, s->h_q, s->d_qk, s->dtype, workspace) ||
      !make_map(&tk, k, s->total_k, s->h_kv, s->d_qk, s->dtype, workspace) ||
      !make_map(&tv, v, s->total_k, s->h_kv, s->d_v, s->dtype, workspace) ||
      !make_map(&tdo, dout, s->total_q, s->h_q, s->d_v, s->dtype, workspace) ||
      !make_acc_map(&tdq, dq_acc, s->total_q, s->h_q, s->d_qk, workspace))
    return GDPA_ERR_CUDA;
  const cudaError_t e = launch_bwd(tq, tk, tv, tdo, tdq, a, nsm, stream, t_ev_before, t_ev_after);
  return e == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

int gdpa_get_status(void* stream_) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream_)) != cudaSuccess) return GDPA_ERR_CUDA;
  int* p = status_ptr();
  if (!p) return GDPA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GDPA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return GDPA_ERR_CUDA;
  }
  return v;
}

const char* gdpa_error_string(int s) {
  switch (s) {
    case GDPA_OK: return "ok";
    case GDPA_ERR_INVALID: return "invalid argument";
    case GDPA_ERR_UNSUPPORTED: return "unsupported configuration";
    case GDPA_ERR_CUDA: return "CUDA error";
    case GDPA_ERR_WORKSPACE: return "workspace missing or too small";
    case GDPA_ERR_TIMEOUT: return "device-side wait timed out";
    case GDPA_ERR_SCRATCH_LIMIT: return "problem exceeds the fixed scratch of the no-allocation forward";
    default: return "unknown status";
  }
}

int gdpa_num_sms(void) { return sm_count(); }

#ifdef GDPA_TEST_HOOKS
// Test-only builds: from the next call on, CTA 0 of the forward (kernel 0) or
// backward (kernel 1) skips one mbarrier arrive at `step` (-1: none), so that
// a bounded wait runs out and the call ends with GDPA_ERR_TIMEOUT.
int gdpa_test_set_skip(int kernel, int step) {
  if (kernel < 0 || kernel > 1) return GDPA_ERR_INVALID;
  g_test_skip[kernel] = step;
  return GDPA_OK;
}
#endif

int gdpa_set_profile_events(void* before_main, void* after_main) {
  t_ev_before = static_cast<cudaEvent_t>(before_main);
  t_ev_after = static_cast<cudaEvent_t>(after_main);
  return GDPA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- forward without allocation
//
// For callers that cannot allocate device memory (see gdpa_fwd_noalloc in
// gdpa.h): the forward's only scratch, the work list, lives in this fixed
// array instead of a caller workspace. Host code must not pass the symbol
// itself to a kernel (on the host it names a stand-in, not device memory);
// it passes the address cudaGetSymbolAddress returns for the current device.

namespace {

static __device__ __align__(256) unsigned char g_fwd_noalloc_scratch[GDPA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached; NULL on failure.
void* noalloc_scratch_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  static void* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> g(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace

extern "C" int gdpa_fwd_noalloc(const gdpa_shape* s, const void* q, const void* k, const void* v,
                                const int32_t* cu_q, const int32_t* cu_k, int max_q, int max_k, int act,
                                float scale, int causal, int window, const float* descale, void* out, float* lse,
                                void* stream) {
  const int st = validate(s, max_q, max_k, act, causal, window);
  if (st != GDPA_OK) return st;
  const size_t need = gdpa_workspace_bytes(s, max_q, max_k, 0);
  if (need > GDPA_NOALLOC_SCRATCH_BYTES) return GDPA_ERR_SCRATCH_LIMIT;
  if (s->total_q == 0 || s->batch == 0) return GDPA_OK;
  void* scratch = noalloc_scratch_ptr();
  if (!scratch) return GDPA_ERR_CUDA;
  return gdpa_fwd(s, q, k, v, cu_q, cu_k, max_q, max_k, act, scale, causal, window, descale, out, lse, scratch,
                  GDPA_NOALLOC_SCRATCH_BYTES, stream);
}
