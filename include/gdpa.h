/*
 * gdpa.h -- C ABI of libgdpa.so: Generalized Dot Product Attention (GDPA)
 * forward and backward on one NVIDIA GB300 (sm_103a).
 *
 * What is computed (gdpa/README.md of facebookresearch/ads_model_kernel_library,
 * intro paragraph and "Features"): for every sequence b and query head h, with
 * kv head g = h / (h_q / h_kv),
 *
 *     Z = scale * Q_bh K_bg^T,   P = where(M, act(Z), 0),   O = P V_bg
 *
 * M is the causal / sliding-window / length mask; masked and out-of-length
 * positions contribute exactly zero and there is no row normalisation. The
 * backward (same page, "Features": forward and backward kernels) returns
 *
 *     dV_bg += P^T dO,  dS = scale * where(M, (dO V_bg^T) * act'(Z), 0),
 *     dQ_bh = dS K_bg,  dK_bg += dS^T Q_bh.
 *
 * GDPA_ACT_SOFTMAX selects ordinary softmax attention (online softmax with a
 * log-sum-exp per row, as in the Dao-AILab/flash-attention overview) for
 * cross-checking.
 *
 * The argument list follows the page's "CUTE-DSL" API block,
 * flash_attn_varlen_func(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
 * max_seqlen_k, activation=...): packed (jagged) tensors plus cumulative
 * sequence offsets.
 *
 * Layouts. q [total_q, h_q, d_qk], k [total_k, h_kv, d_qk],
 * v [total_k, h_kv, d_v], out/dout [total_q, h_q, d_v], all row-major with the
 * head dimension contiguous (element strides h*d, d, 1). cu_seqlens_q/k are
 * int32 [batch+1] device arrays, non-decreasing, cu[0] = 0, cu[batch] = total;
 * NULL means every sequence has max_seqlen tokens (the fixed-length
 * [batch, seq, heads, dim] layout of flash_attn_func, the same memory).
 * lse is float [h_q, total_q].
 *
 * Ownership. The caller allocates every buffer, including the workspace, whose
 * size gdpa_workspace_bytes() returns. The library allocates no device memory
 * and keeps no per-call state. Calls are asynchronous on `stream` (a
 * cudaStream_t passed as void*; NULL is the legacy default stream).
 *
 * Errors. Problems visible on the host are returned before any launch:
 * GDPA_ERR_INVALID (null or misaligned pointer, negative size, h_q % h_kv,
 * bad enum), GDPA_ERR_UNSUPPORTED (head dims other than (64,64), (96,96),
 * (128,128), (192,128); FP8 backward; max_seqlen of 2^30 or more),
 * GDPA_ERR_WORKSPACE (too small),
 * GDPA_ERR_CUDA (a launch or tensor-map encode failed). A window of 2^30 or
 * more is the same as none. Every device-side wait
 * is bounded; a wait that gives up records GDPA_ERR_TIMEOUT in a per-device
 * status word that gdpa_get_status() returns. cu_seqlens consistency
 * (monotone, lengths <= max_seqlen, cu[batch] = total) is a caller
 * precondition. The backward checks the one part of it that sizes its
 * writes: a key block beyond max_seqlen_k records GDPA_ERR_INVALID in the
 * status word and that block writes no dq (the rest of the call still
 * runs, so dq is then incomplete).
 */
#ifndef GDPA_H_
#define GDPA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdpa_status {
  GDPA_OK = 0,
  GDPA_ERR_INVALID = 1,
  GDPA_ERR_UNSUPPORTED = 2,
  GDPA_ERR_CUDA = 3,
  GDPA_ERR_WORKSPACE = 4,
  GDPA_ERR_TIMEOUT = 5,
  GDPA_ERR_SCRATCH_LIMIT = 6 /* problem too large for gdpa_fwd_noalloc's fixed scratch */
} gdpa_status;

/* Storage type of q, k, v. out/dout/dq/dk/dv use the same type, except that
 * the FP8 forward writes bf16 out. */
typedef enum gdpa_dtype { GDPA_BF16 = 0, GDPA_FP16 = 1, GDPA_E4M3 = 2 } gdpa_dtype;

/* Activations ("Features" on the gdpa/README.md page). GELU_TANH is
 * GELUApprox; FAST_GELU evaluates the same tanh-form GELU; LEAKY_RELU uses
 * slope 0.01; derivatives at kinks follow PyTorch. FAST_GELU_BF16 and
 * FAST_SILU are cheaper forward evaluations of GELU_TANH and SILU (results
 * within about 6e-3 * max(1, |z|) beyond one bf16 ulp, and 6e-4 * max(1, |z|),
 * of the exact functions); their backward uses the GELU_TANH and SILU
 * derivatives. */
typedef enum gdpa_act {
  GDPA_ACT_IDENTITY = 0,
  GDPA_ACT_GELU = 1,
  GDPA_ACT_GELU_TANH = 2,
  GDPA_ACT_FAST_GELU = 3,
  GDPA_ACT_RELU = 4,
  GDPA_ACT_RELU2 = 5,
  GDPA_ACT_LEAKY_RELU = 6,
  GDPA_ACT_SILU = 7,
  GDPA_ACT_HARDSWISH = 8,
  GDPA_ACT_SOFTMAX = 9,
  GDPA_ACT_FAST_GELU_BF16 = 10, /* FastGELU (BF16): the tanh form evaluated in packed bf16 */
  GDPA_ACT_FAST_SILU = 11       /* FastSiLU: z (1 + tanh(z / 2)) / 2 with the hardware tanh */
} gdpa_act;

typedef struct gdpa_shape {
  int batch;   /* number of sequences B (>= 0) */
  int total_q; /* rows of q and out: sum of query lengths (B*max_seqlen_q when cu_seqlens_q is NULL) */
  int total_k; /* rows of k and v */
  int h_q;     /* query heads */
  int h_kv;    /* key/value heads; h_q % h_kv == 0 (MHA, GQA, MQA) */
  int d_qk;    /* head dim of q and k */
  int d_v;     /* head dim of v and out */
  int dtype;   /* gdpa_dtype */
} gdpa_shape;

/* Bytes of device workspace that gdpa_fwd (is_bwd = 0), gdpa_bwd
 * (is_bwd = 1), gdpa_bwd with deterministic != 0 (is_bwd = 2) or
 * gdpa_fwd_mxfp8 (is_bwd = 3) needs for this problem; 0 for an invalid
 * shape. The size depends only on the arguments given here. The
 * deterministic backward adds one fp32 dQ slice [total_q, h_q, d_qk] per
 * 128-key block of the longest key sequence; gdpa_fwd_mxfp8 adds its scales
 * rearranged into 512-byte tensor-memory copy atoms (about 4 d_qk / 32 + 1
 * bytes per query or key row and head, rounded up to 128-row tiles). */
size_t gdpa_workspace_bytes(const gdpa_shape* shape, int max_seqlen_q, int max_seqlen_k, int is_bwd);

/* Forward. scale multiplies Q K^T before the activation (1/sqrt(d_qk) is the
 * usual choice). causal != 0 aligns query i of a length-Lq sequence with key
 * i + Lk - Lq and allows keys at or before it. window > 0 limits each query
 * to keys at distance < window from that position (with causal: the window
 * keys ending at it); window <= 0 disables it. descale_qkv: FP8 only, device
 * float[3] of per-tensor scales (q, k, v) so that value = code * scale; NULL
 * otherwise. lse: required (device float [h_q, total_q]) for
 * GDPA_ACT_SOFTMAX, ignored (may be NULL) otherwise. All device pointers
 * must be 16-byte aligned. */
int gdpa_fwd(const gdpa_shape* shape, const void* q, const void* k, const void* v,
             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int max_seqlen_q,
             int max_seqlen_k, int act, float scale, int causal, int window,
             const float* descale_qkv, void* out, float* lse, void* workspace,
             size_t workspace_bytes, void* stream);

/* MXFP8 forward ("MXFP8 forward" is listed as coming soon on the gdpa/README.md
 * page, "Features", Datatypes; the block-scale layout is not on the page and
 * follows the OCP Microscaling (MX) v1.0 format: blocks of 32 elements share
 * one E8M0 scale byte s, element value = e4m3 code * 2^(s - 127), s = 255
 * being NaN). q, k, v hold e4m3 codes (shape->dtype = GDPA_E4M3) in the
 * layouts above; out is bf16. The blocks run along the contraction of each
 * GEMM:
 *   q_scale [total_q, h_q, d_qk / 32]: block i of q[t, h, :] is elements 32i..32i+31;
 *   k_scale [total_k, h_kv, d_qk / 32]: likewise for k;
 *   v_scale [ceil(total_k / 32), h_kv, d_v]: block j of column v[:, g, n] is
 *     packed key tokens 32j..32j+31, so every key sequence must start at a
 *     multiple of 32 (cu_seqlens_k[b] % 32 == 0; without cu_seqlens,
 *     max_seqlen_k % 32 == 0, checked on the host). A sequence that does not
 *     records GDPA_ERR_INVALID in the status word (its rows are then wrong).
 *     Keys past a sequence's end inside its last block are ignored.
 * The MMAs apply the scales (tcgen05 kind::mxf8f6f4); P is quantised to e4m3
 * with scale 2^0. Head dims (128, 128) and (192, 128); every activation,
 * softmax included. The scale pointers must be 16-byte aligned. The
 * workspace is gdpa_workspace_bytes(shape, ..., 3) bytes: a first kernel
 * rearranges the scales there into the atoms that the MMAs' scale copies
 * read. Other arguments and errors as for gdpa_fwd (descale is not used). */
int gdpa_fwd_mxfp8(const gdpa_shape* shape, const void* q, const void* k, const void* v,
                   const uint8_t* q_scale, const uint8_t* k_scale, const uint8_t* v_scale,
                   const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int max_seqlen_q,
                   int max_seqlen_k, int act, float scale, int causal, int window, void* out,
                   float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* Backward (bf16/fp16 only). Arguments as for gdpa_fwd; out and lse are read
 * only for GDPA_ACT_SOFTMAX (they must be the forward's results) and may be
 * NULL otherwise. dout has out's layout; dq, dk, dv have q's, k's and v's.
 * dk/dv of a kv head sum the contributions of its query-head group in a
 * fixed order, so they are the same bits on every call. dq sums the
 * contributions of all key blocks: with deterministic = 0 they are added
 * into an fp32 accumulator in the workspace in whatever order the key
 * blocks finish (results may differ in the last bits between calls); with
 * deterministic != 0 each key block writes its own fp32 slice and a final
 * kernel adds the slices in key-block order, so dq is bitwise reproducible
 * (at the cost of the slices' memory, see gdpa_workspace_bytes, and their
 * HBM traffic). FA's flash_attn_varlen_func(deterministic=...) is the model.
 * When max_seqlen_k <= 128 every sequence has one key block, so each dq row
 * has a single producer: the kernel then writes dq directly in the output
 * type (no accumulator, reproducible in either mode). */
int gdpa_bwd(const gdpa_shape* shape, const void* q, const void* k, const void* v,
             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int max_seqlen_q,
             int max_seqlen_k, int act, float scale, int causal, int window, const void* out,
             const float* lse, const void* dout, void* dq, void* dk, void* dv, int deterministic,
             void* workspace, size_t workspace_bytes, void* stream);

/* Synchronises `stream`, then returns and clears the device-side status of
 * the current device (GDPA_OK, GDPA_ERR_TIMEOUT, or GDPA_ERR_INVALID for a
 * key block beyond max_seqlen_k in the backward), or GDPA_ERR_CUDA if the
 * synchronisation itself failed. */
int gdpa_get_status(void* stream);

/* Static, human-readable text for a status code. */
const char* gdpa_error_string(int status);

/* Timing hook. When set, every later gdpa_fwd / gdpa_bwd call made by this
 * host thread records `before_main` (a cudaEvent_t passed as void*) on its
 * stream right before the main GDPA kernel launch and `after_main` right
 * after it, so the pair brackets that kernel alone (not the work-list,
 * dQ-clear or dQ-convert kernels). Pass NULL, NULL to stop. The events are
 * owned by the caller and must stay valid while set. Returns GDPA_OK. */
int gdpa_set_profile_events(void* before_main, void* after_main);

/* Forward without any allocation. No counterpart on the pages: this is an
 * addition of this library for callers that cannot call cudaMalloc -- for
 * example a plugin running inside a host framework whose device memory is
 * owned entirely by that framework's allocator, or a deployment that forbids
 * allocations after start-up to keep a fixed, pre-planned memory footprint.
 *
 * Same arguments and results as gdpa_fwd, minus the workspace: the scratch
 * that gdpa_fwd takes from `workspace` (the cost-sorted work list) lives
 * instead in a fixed device array of GDPA_NOALLOC_SCRATCH_BYTES inside the
 * library, which every GPU that loads the library holds until the process
 * exits. The caller still allocates q, k, v, out, lse and the cu_seqlens.
 *
 * - Problems whose work list needs more than GDPA_NOALLOC_SCRATCH_BYTES
 *   (gdpa_workspace_bytes(shape, ..., 0) above it) return
 *   GDPA_ERR_SCRATCH_LIMIT before anything is launched.
 * - The first call on each device looks up that device's address of the
 *   array (cudaGetSymbolAddress, with the device current); make that first
 *   call before any stream capture.
 * - The call allocates nothing: no cudaMalloc, cudaFree or allocating
 *   library routine.
 * - All calls on a device share the one array and each call rewrites it
 *   completely before reading it (nothing in it has to start at zero), so
 *   calls that overlap on the GPU -- on different streams or from
 *   different host threads -- race and must be serialised by the caller. */
#define GDPA_NOALLOC_SCRATCH_BYTES (512u * 1024u)
int gdpa_fwd_noalloc(const gdpa_shape* shape, const void* q, const void* k, const void* v,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int max_seqlen_q,
                     int max_seqlen_k, int act, float scale, int causal, int window,
                     const float* descale_qkv, void* out, float* lse, void* stream);

/* Number of multiprocessors the persistent kernels are sized for on the
 * current device (the grid of every main kernel), or -1 on error. */
int gdpa_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* GDPA_H_ */
