/*
 * sdpa.h — C ABI of libsdpa.so: scaled dot-product attention forward for NVIDIA GB300 (sm_103a).
 *
 * The operation (onnx-light "include_nn_kernels.h", class Attention, baseline formula):
 *
 *     Y = Softmax( Q K^T * scale + bias ) V
 *
 * with the variants spelled out by three operator contracts:
 *   - ai.onnx::Attention v23/v24 (same page, class Attention, "Supported features"):
 *     rank-3 / rank-4 layouts, default scale 1/sqrt(head_size), is_causal aligned to the
 *     upper-left corner, softcap c*tanh(s/c), grouped query heads, FLOAT (added) or BOOL
 *     (true = attend) attn_mask broadcast over (batch, heads, q, kv) and padded with
 *     -inf/false when shorter than the key axis, past_key/past_value concatenated into
 *     present_key/present_value, nonpad_kv_seqlen masking keys j >= n[b];
 *   - com.microsoft::MultiHeadAttention (onnx-light-cpu "Custom operators", Python API,
 *     section Microsoft MultiHeadAttention): projection-bias segments, int32 key-padding
 *     lengths or binary masks offset by mask_filter_value (default -10000), additive
 *     attention bias, past/present with P+L positions, unidirectional masking;
 *   - com.microsoft::GroupQueryAttention (same page, section Microsoft GroupQueryAttention):
 *     causal attention at absolute positions, local_window_size counting the current token,
 *     head_sink as a per-head virtual logit that joins the softmax denominator and adds no
 *     value; seqlens_k = key length - 1 ("Custom operators", C++ API,
 *     GroupQueryAttentionFusionPattern).
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a DEVICE pointer on the current CUDA device, except the
 *     sdpa_params struct itself, which is read on the host during the call and may be
 *     freed when the call returns.
 *   - The caller owns every buffer.  The library keeps no pointer past the asynchronous
 *     completion of the work it enqueues on `stream` and allocates no device memory:
 *     scratch goes through the caller's workspace (size from sdpa_workspace_size).
 *   - Outputs never alias inputs (class Attention: CanRunInPlace() is false); overlapping
 *     byte ranges are rejected with SDPA_ERR_ALIAS.
 *   - Every argument is validated on the host before anything is enqueued; on an error
 *     nothing is launched, the return value names the class of error and sdpa_last_error()
 *     holds a one-line message (thread-local).  Functions never throw.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream); the
 *     call returns without synchronising.  Device-side failures of bounded waits are
 *     reported later through sdpa_query_status().
 */
#ifndef SDPA_GB300_H
#define SDPA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sdpa_stream_t;   /* same type as cudaStream_t */

#if defined(__GNUC__)
#define SDPA_API __attribute__((visibility("default")))
#else
#define SDPA_API
#endif

/* ---- status codes ---- */
#define SDPA_OK               0
#define SDPA_ERR_INVALID      1   /* attribute value outside its contract (e.g. window 0)   */
#define SDPA_ERR_SHAPE        2   /* inconsistent sizes / head counts                        */
#define SDPA_ERR_UNSUPPORTED  3   /* valid request this library does not implement           */
#define SDPA_ERR_ALIGNMENT    4   /* pointer or stride not aligned as documented             */
#define SDPA_ERR_ALIAS        5   /* an output overlaps an input or another output           */
#define SDPA_ERR_OVERFLOW     6   /* a size or index does not fit the kernels' index types   */
#define SDPA_ERR_WORKSPACE    7   /* workspace missing or smaller than sdpa_workspace_size() */
#define SDPA_ERR_CUDA         8   /* a CUDA runtime/driver call failed                       */
#define SDPA_ERR_TIMEOUT      9   /* a bounded device-side wait expired (via query_status)   */
#define SDPA_ERR_NULL        10   /* a required pointer is NULL                              */
#define SDPA_ERR_BOUNDS      11   /* bounds-checking build only: an index check failed and   */
                                  /* the access was skipped (via sdpa_query_status)          */

typedef enum { SDPA_F32 = 0, SDPA_F16 = 1, SDPA_BF16 = 2 } sdpa_dtype;

/* A logical (batch, head, seq, dim) view of device memory.  Strides are in ELEMENTS of
 * the view's type; the last (dim) axis has stride 1.  A stride of 0 broadcasts that axis
 * (masks only).  data == NULL means "absent".
 * Rank-3 packed tensors (B, S, N*D) are views with stride_b = S*N*D, stride_n = D,
 * stride_s = N*D; rank-4 (B, N, S, D) tensors have stride_b = N*S*D, stride_n = S*D,
 * stride_s = D. */
typedef struct {
  void* data;
  int64_t stride_b, stride_n, stride_s;
} sdpa_view;

/* Where query row i sits on the key axis for the causal and window rules. */
typedef enum {
  SDPA_CAUSAL_NONE = 0,
  SDPA_CAUSAL_UPPER_LEFT = 1,   /* pos(i) = i  (ai.onnx::Attention is_causal)                */
  SDPA_CAUSAL_LOWER_RIGHT = 2   /* pos(i) = Tv(b) - S + i, Tv(b) = seqlens_k[b] + 1 under
                                   SDPA_LEN_SEQLENS_K_I32, else T = P + L (GQA causal,
                                   MHA unidirectional: absolute positions)                   */
} sdpa_causal;

/* Second mask slot (beside the additive one). */
typedef enum {
  SDPA_KEEP_NONE = 0,
  SDPA_KEEP_BOOL_U8 = 1,        /* uint8: 0 excludes the key (ai.onnx BOOL attn_mask)       */
  SDPA_KEEP_FILTER_I32 = 2      /* int32: 0 adds mask_filter_value (MHA binary key mask)    */
} sdpa_keep_kind;

/* Per-batch key-length vector, `lens` of B elements (device). */
typedef enum {
  SDPA_LEN_NONE = 0,
  SDPA_LEN_NONPAD_I64 = 1,      /* int64: keys j >= lens[b] excluded (nonpad_kv_seqlen)     */
  SDPA_LEN_KEYLEN_I32 = 2,      /* int32: keys j >= lens[b] get mask_filter_value (MHA)     */
  SDPA_LEN_SEQLENS_K_I32 = 3    /* int32: keys j > lens[b] excluded (GQA seqlens_k)         */
} sdpa_len_kind;

/* One attention problem.  T = P + L keys: the P past rows followed by the L new rows.
 *
 * Per score s_ij = scale * <q_i, k_j> the stages are, in order (class Attention,
 * qk_matmul_output_mode list): + additive mask, softcap, then the keep mask, the
 * filter/length rules and the structural rules.  A key that any rule excludes stays
 * excluded through softcap.  With softcap_before_bias = 1 the additive mask is added
 * after softcap instead.  The sink logit enters the denominator as given.  A row with
 * no admitted key and no sink is written as zeros. */
typedef struct {
  int32_t struct_size;          /* must be sizeof(sdpa_params) */
  int32_t B, Nq, Nkv;           /* batch, query heads, kv heads (Nq % Nkv == 0)            */
  int32_t S, L, P;              /* query rows, new kv rows, past kv rows                     */
  int32_t H, Hv;                /* q/k head size, v head size                                */
  sdpa_dtype dtype;             /* element type of q, k, v, past, present, y, the projection
                                   biases and head_sink                                      */
  sdpa_view q;                  /* (B, Nq, S, H)                                             */
  sdpa_view k, v;               /* (B, Nkv, L, H) / (B, Nkv, L, Hv)                          */
  sdpa_view past_k, past_v;     /* (B, Nkv, P, H) / (B, Nkv, P, Hv); required iff P > 0      */
  sdpa_view present_k, present_v; /* outputs (B, Nkv, P+L, H/Hv) or both absent             */
  sdpa_view y;                  /* output (B, Nq, S, Hv)                                     */
  const void* q_bias;           /* (Nq*H) added to q, or NULL                                */
  const void* k_bias;           /* (Nkv*H) added to the new k rows (and to present), or NULL */
  const void* v_bias;           /* (Nkv*Hv) added to the new v rows (and to present), or NULL*/
  const void* head_sink;        /* (Nq) sink logits, or NULL                                 */
  int32_t has_scale;            /* 0: scale = 1/sqrt(H)                                      */
  float scale;
  float softcap;                /* <= 0: off; must be finite                                 */
  int32_t causal;               /* sdpa_causal                                               */
  int64_t window;               /* -1: unlimited; > 0: keys pos-window+1 .. pos (needs causal)*/
  sdpa_view add_mask;           /* additive mask / attention bias, (b, h, i, j < add_mask_T) */
  sdpa_dtype add_mask_dtype;
  int64_t add_mask_T;           /* keys j >= add_mask_T are excluded                         */
  sdpa_view keep_mask;          /* (b, h, i, j < keep_mask_T), kind below                    */
  int32_t keep_kind;            /* sdpa_keep_kind; keys j >= keep_mask_T count as 0          */
  int64_t keep_mask_T;
  int32_t len_kind;             /* sdpa_len_kind                                             */
  const void* lens;             /* (B) device vector                                         */
  float mask_filter_value;      /* MHA: -10000                                               */
  int32_t softcap_before_bias;  /* 0: pages' stage order; 1: softcap, then the additive mask */
  /* Rotary embedding of Q and of the new K rows before attention (GroupQueryAttention's
   * rotary, class RotaryEmbedding's rotation): rank-2 caches (rotary_max_pos, R/2) in
   * dtype, R = rotary_dim (0: H).  Absolute positions: query row i at Tv(b) - S + i and new
   * key row j at Tv(b) - L + j, Tv(b) = seqlens_k[b] + 1 under SDPA_LEN_SEQLENS_K_I32, else
   * T = P + L.  present holds the rotated keys.  A position outside the cache is reported
   * by sdpa_query_status as SDPA_ERR_INVALID.  rotary_cos == NULL: no rotation. */
  const void* rotary_cos;
  const void* rotary_sin;
  int64_t rotary_max_pos;
  int32_t rotary_dim;
  int32_t rotary_interleaved;
  /* Auxiliary qk output of class Attention (qk_matmul_output_mode), written by
   * sdpa_attn_fwd when qk_out.data != NULL: a (B, Nq, S, P+L) FLOAT view (last dimension
   * contiguous) of the scores at stage qk_mode: 0 = scale * Q K^T; 1 = with the additive
   * bias and every mask (an excluded key is -inf); 2 = after softcap (the softmax's
   * logits); 3 = the softmax probabilities, the sink in the denominator (an excluded key is
   * 0).  The decode entry points reject it (SDPA_ERR_UNSUPPORTED). */
  sdpa_view qk_out;
  int32_t qk_mode;
} sdpa_params;

/* Which entry point a workspace query is for. */
#define SDPA_OP_FWD    0
#define SDPA_OP_DECODE 1
#define SDPA_OP_BWD    2

/* Prefill / general forward.  Writes y (and present_k/present_v when given).
 * workspace: device scratch of at least sdpa_workspace_size(p, SDPA_OP_FWD) bytes
 * (NULL allowed when that size is 0), 256-byte aligned.
 * Alignment: data pointers 16-byte aligned; H and Hv multiples of 8 (16-bit types) or 4
 * (f32), at most 256; strides of q/k/v/past/present/y multiples of 8 (16-bit) or 4 (f32).
 * Returns SDPA_OK or an SDPA_ERR_* code. */
SDPA_API int sdpa_attn_fwd(const sdpa_params* p, void* workspace, size_t workspace_bytes,
                  sdpa_stream_t stream);

/* Decode forward for few query rows per head (S <= 16): the keys of each (batch, kv head)
 * are split into chunks processed in parallel and merged by a second kernel; past K/V are
 * read once and, when present outputs are given, copied into them in the same pass.
 * Same semantics, arguments and rules as sdpa_attn_fwd; workspace from
 * sdpa_workspace_size(p, SDPA_OP_DECODE). */
SDPA_API int sdpa_attn_decode(const sdpa_params* p, void* workspace, size_t workspace_bytes,
                     sdpa_stream_t stream);

/* Decode without a workspace, for callers that cannot allocate device memory: a host
 * or plugin framework that owns the whole device memory budget and gives its extensions
 * no allocator, or a latency-critical serving loop that cannot afford cudaMalloc's
 * implicit device-wide synchronisation or its failure under memory pressure.  (The
 * documentation pages have no counterpart: this is a deployment variant of
 * sdpa_attn_decode, not part of the operator contracts.)
 * Same semantics, arguments and rules as sdpa_attn_decode; the split partials go to a
 * fixed 8 MiB device array inside the library instead of a caller workspace.  That array
 * is reserved on every GPU that loads the library until the process exits.
 *  - Limit: the partials, B*Nq*S rows x nsplit chunks x (Hv + 2) floats (each part
 *    rounded up to 256 bytes; sdpa_workspace_size(p, SDPA_OP_DECODE) reports the figure),
 *    must fit in 8 MiB, else SDPA_ERR_WORKSPACE is returned and nothing is launched.
 *    E.g. 2048 rows, T = 4096, Hv = 128 need about 4.3 MiB.
 *  - The first call on each device looks up the array's device address with that device
 *    current, and so does the first call after the device's context has changed (e.g.
 *    after cudaDeviceReset, which may load the library's device code elsewhere); make
 *    those calls before any stream capture on the device.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 *  - Every call on a device shares the one array, which keeps the last call's contents
 *    (nothing in it needs to start at zero: each call writes every slot it reads).  Calls
 *    that overlap on the GPU race on it and corrupt each other's results: issue them in
 *    order on one stream. */
SDPA_API int sdpa_attn_decode_static(const sdpa_params* p, sdpa_stream_t stream);

/* Backward of the attention: the gradient graph of onnx-light-cpu "Custom operators" (C++
 * API, RegisterCustomOperatorGradients, GroupQueryAttention gradient).  With P the stage-3
 * probabilities of the forward (class Attention, qk_matmul_output_mode 3, sink in the
 * denominator):
 *     dP = dY V^T,  dS = P (dP - rowsum(P dP)) scale,  dQ = dS K,  dK = dS^T Q,  dV = P^T dY,
 * the query heads of a group summed onto their kv head, every output rounded once to dtype.
 * p describes the forward problem exactly as for sdpa_attn_fwd (p->y may be absent and is not
 * written).  dy: (B, Nq, S, Hv) upstream gradient; outputs dq (B, Nq, S, H), dk (B, Nkv, P+L, H),
 * dv (B, Nkv, P+L, Hv): gradients with respect to the rows the scores see (Q plus its projection
 * bias; the P past rows followed by the L new rows plus their biases), all views of dtype
 * elements, written in full (zeros where no score depends on them).  workspace:
 * sdpa_workspace_size(p, SDPA_OP_BWD) bytes (two fp32 values per query row, plus copies of
 * the biased Q and of the T key / value rows when there are biases or past rows), 256-byte
 * aligned.
 * Subset: float16 / bfloat16, H == Hv in {64, 128}, no rotary, no qk output, no present
 * outputs; every mask and length rule of sdpa_attn_fwd and head_sink.  softcap > 0 returns
 * SDPA_ERR_UNSUPPORTED (the gradient graph has no softcap).
 * Alignment and aliasing rules as for sdpa_attn_fwd; outputs overlap no input. */
SDPA_API int sdpa_attn_bwd(const sdpa_params* p, sdpa_view dy, sdpa_view dq, sdpa_view dk, sdpa_view dv,
                           void* workspace, size_t workspace_bytes, sdpa_stream_t stream);

/* Bytes of device workspace the entry point `op` (SDPA_OP_FWD / SDPA_OP_DECODE / SDPA_OP_BWD) needs for
 * these parameters; 0 when none.  Pure host function (no CUDA call); returns 0 and sets
 * sdpa_last_error() when the parameters are invalid. */
SDPA_API size_t sdpa_workspace_size(const sdpa_params* p, int op);

/* Host-only validation of p for `op` (SDPA_OP_FWD / SDPA_OP_DECODE / SDPA_OP_BWD), exactly as
 * the entry points perform it before any launch (for SDPA_OP_BWD: the problem's parameters and
 * the backward's subset; the gradient views are checked by sdpa_attn_bwd itself).  No CUDA
 * call.  Returns SDPA_OK or the error code the entry point would return. */
SDPA_API int sdpa_validate(const sdpa_params* p, int op);

/* RotaryEmbedding (onnx-light "include_nn_kernels.h", class RotaryEmbedding): y = x with
 * the first R channels of every head rotated in pairs (d, d + R/2), or (2d, 2d + 1) when
 * interleaved, by the angle of cache row `pos`: (x1, x2) -> (x1 cos - x2 sin, x2 cos + x1 sin);
 * channels >= R are copied.  x, y: (B, N, S, D) views (rank-3 or rank-4 via strides), dtype
 * elements, may not overlap.  Caches: R/2 contiguous entries per row in dtype; with
 * position_ids (B, S) int64 (device) they are rank-2 (max_pos rows) and row = position_ids[b,
 * s]; with position_ids NULL they are rank-3 (B, S, R/2) and max_pos must be B*S.
 * R = rotary_dim (0: D), even.  Positions outside [0, max_pos) are reported by
 * sdpa_query_status as SDPA_ERR_INVALID. */
SDPA_API int sdpa_rotary(sdpa_dtype dtype, int32_t B, int32_t N, int32_t S, int32_t D, sdpa_view x, sdpa_view y,
                         const void* cos_cache, const void* sin_cache, int64_t max_pos,
                         const int64_t* position_ids, int32_t rotary_dim, int32_t interleaved,
                         sdpa_stream_t stream);

/* present[b, n, 0:P] = past[b, n, :]; present[b, n, P:P+L] = cur[b, n, :] (+ bias[n*D:(n+1)*D]
 * rounded once to dtype when bias is non-NULL).  (class Attention, past_key/past_value
 * and Result.present_key; MHA: present holds P+L positions; GQA: present holds the whole
 * past followed by the current step.)  Without bias the copy is bit-exact.
 * past may be absent (data NULL) only when P == 0.  present must not overlap past/cur.
 * Alignment: pointers and strides as for sdpa_attn_fwd with D in place of H. */
SDPA_API int sdpa_kv_concat(sdpa_dtype dtype, int32_t B, int32_t N, int32_t P, int32_t L, int32_t D,
                   sdpa_view past, sdpa_view cur, const void* bias, sdpa_view present,
                   sdpa_stream_t stream);

/* Synchronises `stream`, then reads and clears the current device's status words: set when
 * a bounded wait of a kernel expires (SDPA_ERR_TIMEOUT) or a rotary position falls outside
 * its cache (SDPA_ERR_INVALID).  Returns SDPA_OK, one of those codes, or SDPA_ERR_CUDA when
 * the synchronisation itself failed. */
SDPA_API int sdpa_query_status(sdpa_stream_t stream);

/* Message for the last error on the calling thread ("" when none).  Valid until the next
 * call on this thread. */
SDPA_API const char* sdpa_last_error(void);

/* Name of the last kernel path the calling thread launched (e.g. "prefill_tc_bf16_h128"),
 * for tests and profiling. */
SDPA_API const char* sdpa_last_kernel_name(void);

/* Number of kernels this library has launched in this process (all threads), for
 * benchmarks that count their device work. */
SDPA_API int64_t sdpa_launch_count(void);

/* Library version string. */
SDPA_API const char* sdpa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SDPA_GB300_H */
