// Problem description shared by the schedule builder and the GDPA kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace gdpa {

constexpr int kTileQ = 128;   // query rows per Q tile (TMEM lanes)
constexpr int kTileK = 128;   // key rows per KV block
constexpr int kFwdItemRows = kTileQ;  // a forward work item is one Q tile of one (sequence, head)

enum DType : int { DT_BF16 = 0, DT_FP16 = 1, DT_E4M3 = 2 };

// Programmatic dependent launch. Every kernel of the library is launched so
// that it may start while the previous kernel on the stream finishes; it
// calls pdl_wait() before it reads or writes memory that an earlier kernel
// may still use (the wait returns once that kernel has completed and its
// writes are visible; without a programmatic predecessor it returns at
// once), and pdl_release() to let the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

struct Problem {
  int batch, total_q, total_k;
  int h_q, h_kv, group;  // group = h_q / h_kv
  int max_q, max_k;
  const int* cu_q;  // NULL = fixed length max_q
  const int* cu_k;  // NULL = fixed length max_k
  int causal, window;
};

__device__ __forceinline__ void seq_bounds(const int* cu, int b, int fixed_len, int& start, int& len) {
  if (cu) {
    start = cu[b];
    len = cu[b + 1] - start;
  } else {
    start = b * fixed_len;
    len = fixed_len;
  }
}

// Keys allowed for any query row in [r_first, r_last] (rows within the
// sequence) as an inclusive range [kmin, kmax] of key indices; returns false
// when no row of the range sees any key. Query row i sits at key position
// i + Lk - Lq. causal: keys <= that position (and > position - window when
// window > 0); non-causal window: |position - key| < window.
__host__ __device__ __forceinline__ bool key_range(int r_first, int r_last, int lq, int lk, int causal,
                                                   int window, int& kmin, int& kmax) {
  if (lk <= 0 || r_last < r_first) return false;
  const int off = lk - lq;
  if (causal) {
    kmax = r_last + off;
    kmin = window > 0 ? r_first + off - window + 1 : 0;
  } else if (window > 0) {
    kmax = r_last + off + window - 1;
    kmin = r_first + off - window + 1;
  } else {
    kmax = lk - 1;
    kmin = 0;
  }
  if (kmin < 0) kmin = 0;
  if (kmax > lk - 1) kmax = lk - 1;
  return kmax >= kmin;
}

// Same for query rows: the rows that see any key in [k_first, k_last].
__host__ __device__ __forceinline__ bool query_range(int k_first, int k_last, int lq, int lk, int causal,
                                                     int window, int& rmin, int& rmax) {
  if (lq <= 0 || k_last < k_first) return false;
  const int off = lk - lq;
  if (causal) {
    rmin = k_first - off;                                    // position >= key
    rmax = window > 0 ? k_last - off + window - 1 : lq - 1;  // position - key < window
  } else if (window > 0) {
    rmin = k_first - off - window + 1;
    rmax = k_last - off + window - 1;
  } else {
    rmin = 0;
    rmax = lq - 1;
  }
  if (rmin < 0) rmin = 0;
  if (rmax > lq - 1) rmax = lq - 1;
  return rmax >= rmin;
}

// One work-list entry, decoded when the list is built, so that a kernel role
// needs one 32-byte load per item instead of a work-list load followed by
// dependent cu_seqlens loads:
//   seq = (q_start, lq, k_start, lk) of the item's sequence;
//   blk = forward:  (r0, rows, lo, n): the Q tile's first row and row count,
//                   its first KV block and number of KV blocks (0: no key
//                   is visible to any of its rows);
//         backward: (k0, krows, qlo, nq): the key block's first row and row
//                   count, its first query block and number of query blocks.
struct WorkEntry {
  int4 seq;
  int4 blk;
};

// Work list written by the schedule kernel: count, then entries sorted by
// cost, heaviest first. The kernels visit list position p as
// (entry p / heads, head p % heads).
struct WorkList {
  int count;
  int pad[7];
  WorkEntry items[1];
};

// Snake ("zigzag") order over the sorted list: round r visits positions
// r*G + c for even r and (r+1)*G - 1 - c for odd r, so each CTA c receives
// a balanced mix of heavy and light items.
__device__ __forceinline__ int zigzag_pos(int round, int cta, int grid) {
  return (round & 1) ? (round + 1) * grid - 1 - cta : round * grid + cta;
}

}  // namespace gdpa
