/*
 * Double-precision CPU oracle for the scaled dot-product attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or call
 * this code: only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no header, helper or constant with the CUDA library.
 *
 * What it computes (the plain definition, written out with no blocking or fusion):
 *   onnx-light "include_nn_kernels.h", class Attention: Y = Softmax(Q K^T * scale + bias) V,
 *   extended by the contracts of com.microsoft::MultiHeadAttention and
 *   com.microsoft::GroupQueryAttention ("Custom operators" page, sections
 *   "Microsoft MultiHeadAttention" and "Microsoft GroupQueryAttention").
 *
 * Every tensor is a strided view of a host buffer holding the element type named by
 * ORC_* codes below; the last (head) dimension is contiguous.  Elements are widened to
 * double exactly before any arithmetic.
 */
#ifndef SDPA_ORACLE_H
#define SDPA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_U8 = 3, ORC_I32 = 4, ORC_I64 = 5, ORC_F64 = 6 };

/* causal alignment of query row i */
enum {
  ORC_CAUSAL_NONE = 0,
  ORC_CAUSAL_UPPER_LEFT = 1,   /* query i sits at key position i                              */
  ORC_CAUSAL_LOWER_RIGHT = 2   /* query i sits at key position (valid_total - S + i)          */
};
/* the second mask slot */
enum {
  ORC_KEEP_NONE = 0,
  ORC_KEEP_BOOL = 1,           /* u8: 0 excludes the key (ai.onnx BOOL attn_mask)             */
  ORC_KEEP_FILTER = 2          /* i32: 0 adds mask_filter_value (MHA binary key mask)         */
};
/* per-batch key-length vector */
enum {
  ORC_LEN_NONE = 0,
  ORC_LEN_NONPAD_I64 = 1,      /* keys j >= len[b] excluded (ai.onnx nonpad_kv_seqlen)         */
  ORC_LEN_KEYLEN_I32 = 2,      /* keys j >= len[b] get mask_filter_value (MHA key padding)    */
  ORC_LEN_SEQLENS_K_I32 = 3    /* keys j > len[b] excluded (GQA seqlens_k = total - 1)        */
};

typedef struct {
  const void* data;            /* NULL = absent */
  int32_t dtype;               /* ORC_* */
  int64_t sb, sh, ss;          /* element strides of (batch, head, seq); last dim stride 1 */
} orc_tensor;

typedef struct {
  int32_t B, Nq, Nkv, S, L, P, H, Hv;   /* total keys T = P + L */
  orc_tensor q;                /* (B, Nq, S, H)   */
  orc_tensor k, v;             /* (B, Nkv, L, H) / (B, Nkv, L, Hv) */
  orc_tensor past_k, past_v;   /* (B, Nkv, P, H) / (B, Nkv, P, Hv), data NULL when P == 0 */
  const void* q_bias;          /* (Nq*H) projection-bias segments, dtype of q, or NULL */
  const void* k_bias;          /* (Nkv*H)  */
  const void* v_bias;          /* (Nkv*Hv) */
  int32_t bias_dtype;          /* dtype of q_bias / k_bias / v_bias / head_sink */
  double scale;                /* multiplier of Q K^T */
  double softcap;              /* <= 0: off */
  int32_t causal;              /* ORC_CAUSAL_* */
  int64_t window;              /* -1: unlimited; > 0: keys pos-window+1 .. pos */
  const void* head_sink;       /* (Nq) or NULL */
  orc_tensor add_mask;         /* additive (b, h, i, j), j < add_mask_T; data NULL = absent */
  int64_t add_mask_T;          /* keys j >= add_mask_T are excluded                */
  orc_tensor keep_mask;        /* (b, h, i, j) u8 or i32 */
  int32_t keep_kind;           /* ORC_KEEP_* */
  int64_t keep_mask_T;
  int32_t len_kind;            /* ORC_LEN_* */
  const void* lens;            /* (B) int64 or int32 */
  double mask_filter_value;
  int32_t softcap_before_bias; /* 0: bias then softcap (the ai.onnx stage order); 1: softcap then bias */
} orc_params;

/* Attention output for selected query rows.  rows holds nrows triples (b, h, i);
 * out receives nrows * Hv doubles.  nthreads <= 0 uses every online core.
 * Returns the number of threads used, or a negative value on a bad argument. */
int oracle_attention_rows(const orc_params* p, const int64_t* rows, int64_t nrows, double* out,
                          int nthreads);

/* The auxiliary qk output of class Attention (qk_matmul_output_mode) for selected query
 * rows: out receives nrows * (P+L) doubles, the scores of each row at stage `mode`:
 * 0 = scale * Q K^T; 1 = with the additive bias and masks (an excluded key is -inf);
 * 2 = after softcap (the logits of the softmax); 3 = softmax probabilities, the sink in the
 * denominator (an excluded key is 0; a row with nothing admitted is all 0).
 * Returns the number of threads used, or a negative value on a bad argument. */
int oracle_qk_rows(const orc_params* p, int32_t mode, const int64_t* rows, int64_t nrows, double* out,
                   int nthreads);

/* Backward of the attention (the GroupQueryAttention gradient graph): given dY (B, Nq, S,
 * Hv), writes dQ (B, Nq, S, H), dK (B, Nkv, P+L, H) and dV (B, Nkv, P+L, Hv) as contiguous
 * doubles (gradients with respect to the rows the scores see: past rows first).
 * P = the stage-3 probabilities; dS = P (dY V^T - rowsum(P dY V^T)) * scale; dQ = dS K;
 * dK = dS^T Q and dV = P^T dY summed over the query heads of each kv head.  Softcap > 0 is
 * rejected.  Returns the number of threads used, or a negative value on a bad argument. */
int oracle_attention_backward(const orc_params* p, const orc_tensor* dy, double* dq, double* dk, double* dv,
                              int nthreads);

/* Present tensor (B, N, P+L, D), contiguous, in dtype: past positions followed by the new
 * ones (new + bias, rounded once to dtype, when bias is given). */
int oracle_present(int32_t dtype, int32_t B, int32_t N, int32_t P, int32_t L, int32_t D,
                   const orc_tensor* past, const orc_tensor* cur, const void* bias, void* out);

/* Rotary positional embedding (onnx-light "include_nn_kernels.h", class RotaryEmbedding):
 * x is a (B, N, S, D) view; out is a contiguous (B, N, S, D) double array.  Channel pairs
 * are (d, d + R/2) for d < R/2, or (2d, 2d + 1) when interleaved; R = rotary_dim (0 means
 * D).  Each pair (x1, x2) becomes (x1 cos - x2 sin, x2 cos + x1 sin) with cos = cos[pos, d]
 * and sin = sin[pos, d]; channels >= R pass through.  The angle row comes from
 * positions[b * pos_sb + s] (int64) indexing a rank-2 cache (row stride cache_ld), or,
 * when positions is NULL, from the rank-3 cache row (b * S + s). */
int oracle_rotary(int32_t B, int32_t N, int32_t S, int32_t D, const orc_tensor* x, int32_t rotary_dim,
                  int32_t interleaved, const void* cos_cache, const void* sin_cache, int32_t cache_dtype,
                  int64_t cache_ld, const int64_t* positions, int64_t pos_sb, double* out);

/* Element conversions, exposed so they can be pinned against library conversions. */
double oracle_to_double(int32_t dtype, const void* base, int64_t index);
uint16_t oracle_round_f16(double x);
uint16_t oracle_round_bf16(double x);
/* n doubles rounded once to dtype (F32 / F16 / BF16), written contiguously to out. */
int oracle_round_array(int32_t dtype, const double* in, int64_t n, void* out);

#ifdef __cplusplus
}
#endif
#endif
