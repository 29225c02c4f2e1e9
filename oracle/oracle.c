/*
 * Double-precision CPU oracle for the scaled dot-product attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY: used by the test suite, the smoke check and the benchmark's
 * CPU-baseline leg, never by the product path.  Plain loops, no blocking, no SIMD, no
 * reordering beyond what the definition states.  Sources (onnx-light documentation):
 *
 *  - "include_nn_kernels.h", class Attention (ai.onnx::Attention v23/v24): the baseline
 *    formula Y = Softmax(Q K^T * scale + attn_bias) V; default scale 1/sqrt(head_size);
 *    is_causal aligned to the upper-left corner; softcap c*tanh(s/c) on pre-softmax scores;
 *    the stage order raw -> +bias -> softcap -> softmax of qk_matmul_output_mode 0..3;
 *    grouped heads (q_num_heads a multiple of kv_num_heads); float masks added, bool
 *    masks with true = attend, a mask shorter than the key axis padded with -inf/false;
 *    past K/V concatenated in front of K/V; nonpad_kv_seqlen masking j >= n[b].
 *  - "Custom operators" (Python API), section Microsoft MultiHeadAttention: projection
 *    bias split (q | k | v), query segment only for rank-4 key/value; int32 key-padding
 *    lengths or binary masks; additive attention bias; mask_filter_value default -10000;
 *    past/present with P+L positions; unidirectional.
 *  - same page, section Microsoft GroupQueryAttention: causal attention with absolute
 *    positions, local_window_size counting the current token, head_sink as a virtual
 *    logit in the denominator that adds no value; present holds the whole past then the
 *    current step.
 *  - "Custom operators" (C++ API), GroupQueryAttentionFusionPattern: seqlens_k is the key
 *    sequence length minus one.
 *
 * Readings taken where the pages leave a step open (each is listed in the design notes):
 *  - an excluded key (bool false, causal, window, nonpad, seqlens_k, mask padding, or a
 *    -inf float-mask entry) stays excluded through softcap (a literal softcap of -inf
 *    would give -c and re-admit it);
 *  - MHA key-padding lengths and binary masks add mask_filter_value after softcap;
 *  - the sink logit is used as given (not scaled, not capped);
 *  - a row with no admitted key and no sink outputs zeros;
 *  - GQA head mapping is contiguous: kv head = q head / (Nq / Nkv);
 *  - projection bias is added to the new key/value rows only, never to the past cache.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---- element conversions (exact widening, round-to-nearest-even narrowing) ---- */

static double f16_bits_to_double(uint16_t h) {
  int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = ldexp((double)m, -24);                /* zero and subnormals */
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m + 1024), e - 25);           /* 1.m * 2^(e-15) */
  return sign ? -v : v;
}

static double bf16_bits_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;                       /* bf16 is the top half of a binary32 */
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

double oracle_to_double(int32_t dtype, const void* base, int64_t index) {
  switch (dtype) {
    case ORC_F32: return (double)((const float*)base)[index];
    case ORC_F16: return f16_bits_to_double(((const uint16_t*)base)[index]);
    case ORC_BF16: return bf16_bits_to_double(((const uint16_t*)base)[index]);
    case ORC_U8: return (double)((const uint8_t*)base)[index];
    case ORC_I32: return (double)((const int32_t*)base)[index];
    case ORC_I64: return (double)((const int64_t*)base)[index];
    case ORC_F64: return ((const double*)base)[index];
    default: return NAN;
  }
}

/* Round x to a binary format with `prec` significant bits, smallest normal exponent emin,
 * largest exponent emax; returns (biased exponent, stored mantissa) packed with sign. */
static uint16_t round_to_format(double x, int prec, int emin, int emax, int ebits) {
  const int stored = prec - 1;
  const uint16_t sign = signbit(x) ? (uint16_t)(1u << (stored + ebits)) : 0;
  const uint16_t inf = (uint16_t)(((1u << ebits) - 1) << stored);
  if (isnan(x)) return (uint16_t)(inf | (1u << (stored - 1)));
  double a = fabs(x);
  if (isinf(a)) return sign | inf;
  if (a < ldexp(1.0, emin)) {
    /* subnormal range: an integer count of 2^(emin - stored) units; a count of
       2^stored is exactly the smallest normal and encodes as such */
    double units = nearbyint(ldexp(a, stored - emin));
    return sign | (uint16_t)units;
  }
  int E;
  frexp(a, &E);                                          /* a = f * 2^E, f in [0.5, 1) */
  int e = E - 1;                                         /* a in [2^e, 2^(e+1)) */
  double mant = nearbyint(ldexp(a, stored - e));         /* in [2^stored, 2^prec] */
  if (mant == ldexp(1.0, prec)) { mant = ldexp(1.0, stored); e += 1; }
  if (e > emax) return sign | inf;
  const int bias = emax;
  return sign | (uint16_t)((uint32_t)(e + bias) << stored) | (uint16_t)(mant - ldexp(1.0, stored));
}

uint16_t oracle_round_f16(double x) { return round_to_format(x, 11, -14, 15, 5); }
uint16_t oracle_round_bf16(double x) { return round_to_format(x, 8, -126, 127, 8); }

/* ---- attention, one query row at a time ---- */

static int64_t offset4(const orc_tensor* t, int64_t b, int64_t h, int64_t s) {
  return b * t->sb + h * t->sh + s * t->ss;
}

static int64_t len_of(const orc_params* p, int64_t b) {
  if (p->len_kind == ORC_LEN_NONPAD_I64) return ((const int64_t*)p->lens)[b];
  return (int64_t)((const int32_t*)p->lens)[b];
}

/* key (or value) row j of kv head kh, after concatenating the past in front of the new
   rows and adding the projection-bias segment to new rows */
static void kv_row(const orc_params* p, int is_value, int64_t b, int64_t kh, int64_t j,
                   double* row) {
  const int64_t D = is_value ? p->Hv : p->H;
  const orc_tensor* past = is_value ? &p->past_v : &p->past_k;
  const orc_tensor* cur = is_value ? &p->v : &p->k;
  const void* bias = is_value ? p->v_bias : p->k_bias;
  if (j < p->P) {
    const int64_t o = offset4(past, b, kh, j);
    for (int64_t d = 0; d < D; ++d) row[d] = oracle_to_double(past->dtype, past->data, o + d);
  } else {
    const int64_t o = offset4(cur, b, kh, j - p->P);
    for (int64_t d = 0; d < D; ++d) {
      row[d] = oracle_to_double(cur->dtype, cur->data, o + d);
      if (bias) row[d] += oracle_to_double(p->bias_dtype, bias, kh * D + d);
    }
  }
}

typedef struct {
  double* q;      /* H  */
  double* krow;   /* H  */
  double* vrow;   /* Hv */
  double* raw;    /* T: scale * <q, k_j>                                    */
  double* nocap;  /* T: raw with every bias and mask term, before softcap   */
  double* s;      /* T: the logit that enters the softmax                   */
  char* alive;    /* T  */
} row_scratch;

/* kv head of query head h: query heads form contiguous groups of Nq / Nkv */
static int64_t kv_head(const orc_params* p, int64_t h) {
  const int64_t group = p->Nq / p->Nkv;
  return h / group;
}

/* softcap c * tanh(x / c); a -inf logit stays -inf */
static double capped(const orc_params* p, double x) {
  if (p->softcap <= 0.0 || (isinf(x) && x < 0)) return x;
  return p->softcap * tanh(x / p->softcap);
}

/* Scores of query row (b, h, i) against every key j < T, through every stage: the scaled
 * product, the additive mask (ai.onnx order: before softcap; softcap_before_bias: after),
 * softcap, the mask_filter_value terms of the MultiHeadAttention masks (after softcap), and
 * the exclusions (boolean mask, causal, window, lengths, a mask shorter than T). */
static void score_row(const orc_params* p, int64_t b, int64_t h, int64_t i, row_scratch* w) {
  const int64_t T = (int64_t)p->P + p->L;
  const int64_t kh = kv_head(p, h);

  /* query row, with the query segment of the projection bias */
  const int64_t qo = offset4(&p->q, b, h, i);
  for (int64_t d = 0; d < p->H; ++d) {
    w->q[d] = oracle_to_double(p->q.dtype, p->q.data, qo + d);
    if (p->q_bias) w->q[d] += oracle_to_double(p->bias_dtype, p->q_bias, h * p->H + d);
  }

  /* key position of this query row for the causal and window rules */
  int64_t pos = 0;
  if (p->causal == ORC_CAUSAL_UPPER_LEFT) {
    pos = i;
  } else if (p->causal == ORC_CAUSAL_LOWER_RIGHT) {
    const int64_t valid_total = (p->len_kind == ORC_LEN_SEQLENS_K_I32) ? len_of(p, b) + 1 : T;
    pos = valid_total - p->S + i;
  }

  for (int64_t j = 0; j < T; ++j) {
    kv_row(p, 0, b, kh, j, w->krow);
    double dot = 0.0;
    for (int64_t d = 0; d < p->H; ++d) dot += w->q[d] * w->krow[d];
    const double raw = p->scale * dot;
    int excluded = 0;

    /* additive mask / attention bias */
    double addv = 0.0;
    if (p->add_mask.data) {
      if (j < p->add_mask_T)
        addv = oracle_to_double(p->add_mask.dtype, p->add_mask.data,
                                offset4(&p->add_mask, b, h, i) + j);
      else
        excluded = 1;                        /* a mask shorter than T is padded with -inf */
    }

    /* second mask slot */
    double filt = 0.0;                       /* mask_filter_value terms */
    if (p->keep_kind != ORC_KEEP_NONE) {
      double keep = 0.0;
      if (j < p->keep_mask_T)
        keep = oracle_to_double(p->keep_mask.dtype, p->keep_mask.data,
                                offset4(&p->keep_mask, b, h, i) + j);
      if (keep == 0.0) {
        if (p->keep_kind == ORC_KEEP_BOOL) excluded = 1;
        else filt += p->mask_filter_value;
      }
    }

    /* structural rules */
    if (p->causal != ORC_CAUSAL_NONE && j > pos) excluded = 1;
    if (p->window > 0 && j < pos - p->window + 1) excluded = 1;
    if (p->len_kind == ORC_LEN_NONPAD_I64 && j >= len_of(p, b)) excluded = 1;
    if (p->len_kind == ORC_LEN_KEYLEN_I32 && j >= len_of(p, b)) filt += p->mask_filter_value;
    if (p->len_kind == ORC_LEN_SEQLENS_K_I32 && j > len_of(p, b)) excluded = 1;

    const double s = p->softcap_before_bias ? capped(p, raw) + addv + filt
                                            : capped(p, raw + addv) + filt;
    const double nocap = raw + addv + filt;
    if (isinf(s) && s < 0) excluded = 1;
    w->raw[j] = raw;
    w->nocap[j] = excluded ? -INFINITY : nocap;
    w->s[j] = excluded ? -INFINITY : s;
    w->alive[j] = (char)!excluded;
  }
}

/* Softmax statistics of a scored row with the optional sink logit in the denominator:
 * m = max(max_j s_j, sink), l = sum_j exp(s_j - m) + exp(sink - m).  Returns 0 when no
 * key is admitted and there is no finite sink (the row's output is then all zeros). */
static int softmax_stats(const orc_params* p, int64_t h, const row_scratch* w, double* mp, double* lp) {
  const int64_t T = (int64_t)p->P + p->L;
  const int has_sink = p->head_sink != NULL;
  const double sink = has_sink ? oracle_to_double(p->bias_dtype, p->head_sink, h) : -INFINITY;
  double m = sink;
  int64_t n_alive = 0;
  for (int64_t j = 0; j < T; ++j)
    if (w->alive[j]) { ++n_alive; if (w->s[j] > m) m = w->s[j]; }
  if (n_alive == 0 && !(has_sink && isfinite(sink))) return 0;   /* nothing admitted */
  double l = has_sink ? exp(sink - m) : 0.0;
  for (int64_t j = 0; j < T; ++j)
    if (w->alive[j]) l += exp(w->s[j] - m);
  *mp = m;
  *lp = l;
  return 1;
}

static void attention_row(const orc_params* p, int64_t b, int64_t h, int64_t i, double* y,
                          row_scratch* w) {
  const int64_t T = (int64_t)p->P + p->L;
  const int64_t kh = kv_head(p, h);
  score_row(p, b, h, i, w);
  for (int64_t d = 0; d < p->Hv; ++d) y[d] = 0.0;
  double m, l;
  if (!softmax_stats(p, h, w, &m, &l)) return;                  /* zeros */
  for (int64_t j = 0; j < T; ++j) {
    if (!w->alive[j]) continue;
    const double e = exp(w->s[j] - m);
    kv_row(p, 1, b, kh, j, w->vrow);
    for (int64_t d = 0; d < p->Hv; ++d) y[d] += e * w->vrow[d];
  }
  for (int64_t d = 0; d < p->Hv; ++d) y[d] /= l;
}

/* The auxiliary qk output of class Attention (qk_matmul_output_mode): the T scores of
 * row (b, h, i) at stage 0 (scale * Q K^T), 1 (with the bias and masks; an excluded key is
 * -inf), 2 (after softcap) or 3 (softmax probabilities; an excluded key is 0). */
static void qk_row(const orc_params* p, int32_t mode, int64_t b, int64_t h, int64_t i, double* out,
                   row_scratch* w) {
  const int64_t T = (int64_t)p->P + p->L;
  score_row(p, b, h, i, w);
  if (mode == 0) { for (int64_t j = 0; j < T; ++j) out[j] = w->raw[j]; return; }
  if (mode == 1) { for (int64_t j = 0; j < T; ++j) out[j] = w->nocap[j]; return; }
  if (mode == 2) { for (int64_t j = 0; j < T; ++j) out[j] = w->s[j]; return; }
  double m, l;
  const int any = softmax_stats(p, h, w, &m, &l);
  for (int64_t j = 0; j < T; ++j) out[j] = (any && w->alive[j]) ? exp(w->s[j] - m) / l : 0.0;
}

typedef struct {
  const orc_params* p;
  const int64_t* rows;
  int64_t nrows;
  double* out;
  int tid, nthreads;
  int status;
  int32_t qk_mode;    /* -1: attention output rows; 0..3: qk output rows */
} worker_arg;

static void* worker(void* argp) {
  worker_arg* a = (worker_arg*)argp;
  const orc_params* p = a->p;
  const int64_t T = (int64_t)p->P + p->L;
  row_scratch w;
  w.q = (double*)malloc(sizeof(double) * (size_t)(p->H + 1));
  w.krow = (double*)malloc(sizeof(double) * (size_t)(p->H + 1));
  w.vrow = (double*)malloc(sizeof(double) * (size_t)(p->Hv + 1));
  w.raw = (double*)malloc(sizeof(double) * (size_t)(T + 1));
  w.nocap = (double*)malloc(sizeof(double) * (size_t)(T + 1));
  w.s = (double*)malloc(sizeof(double) * (size_t)(T + 1));
  w.alive = (char*)malloc((size_t)(T + 1));
  if (!w.q || !w.krow || !w.vrow || !w.raw || !w.nocap || !w.s || !w.alive) {
    a->status = -2;
  } else {
    for (int64_t r = a->tid; r < a->nrows; r += a->nthreads) {
      if (a->qk_mode < 0)
        attention_row(p, a->rows[3 * r], a->rows[3 * r + 1], a->rows[3 * r + 2],
                      a->out + r * p->Hv, &w);
      else
        qk_row(p, a->qk_mode, a->rows[3 * r], a->rows[3 * r + 1], a->rows[3 * r + 2],
               a->out + r * T, &w);
    }
  }
  free(w.q); free(w.krow); free(w.vrow); free(w.raw); free(w.nocap); free(w.s); free(w.alive);
  return NULL;
}

static int run_rows(const orc_params* p, int32_t qk_mode, const int64_t* rows, int64_t nrows, double* out,
                    int nthreads) {
  if (!p || !rows || !out || nrows < 0) return -1;
  if (p->Nkv <= 0 || p->Nq % p->Nkv != 0) return -1;
  if (p->window > 0 && p->causal == ORC_CAUSAL_NONE) return -1;
  if (p->len_kind != ORC_LEN_NONE && !p->lens) return -1;
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
    if (b < 0 || b >= p->B || h < 0 || h >= p->Nq || i < 0 || i >= p->S) return -1;
  }
  if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (nthreads < 1) nthreads = 1;
  if ((int64_t)nthreads > nrows) nthreads = nrows > 0 ? (int)nrows : 1;

  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  worker_arg* args = (worker_arg*)malloc(sizeof(worker_arg) * (size_t)nthreads);
  if (!th || !args) { free(th); free(args); return -2; }
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    args[t] = (worker_arg){p, rows, nrows, out, t, nthreads, 0, qk_mode};
    if (pthread_create(&th[t], NULL, worker, &args[t]) != 0) break;
    ++started;
  }
  int status = 0;
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  for (int t = 0; t < started; ++t) if (args[t].status) status = args[t].status;
  if (started < nthreads) {
    /* finish the rows of threads that could not be started on this thread */
    for (int t = started; t < nthreads; ++t) {
      worker_arg a = {p, rows, nrows, out, t, nthreads, 0, qk_mode};
      worker(&a);
      if (a.status) status = a.status;
    }
  }
  free(th);
  free(args);
  return status ? status : nthreads;
}

int oracle_attention_rows(const orc_params* p, const int64_t* rows, int64_t nrows, double* out,
                          int nthreads) {
  return run_rows(p, -1, rows, nrows, out, nthreads);
}

int oracle_qk_rows(const orc_params* p, int32_t mode, const int64_t* rows, int64_t nrows, double* out,
                   int nthreads) {
  if (mode < 0 || mode > 3) return -1;
  return run_rows(p, mode, rows, nrows, out, nthreads);
}

/* ---- backward: the GroupQueryAttention gradient graph ("Custom operators", C++ API,
 * RegisterCustomOperatorGradients).  Probabilities P from the forward's stage 3 (class
 * Attention, mode 3); softmax backward dS = P * (dP - rowsum(P * dP)) with dP = dY V^T; the
 * score scale replayed on dS; dQ = dS K, dK = dS^T Q and dV = P^T dY, the grouped query
 * heads summed back onto their kv head.  Softcap has no place in that graph: rejected. ---- */

typedef struct {
  const orc_params* p;
  const orc_tensor* dy;
  double *dq, *dk, *dv;
  int tid, nthreads;
  int status;
} bwd_arg;

static void* bwd_worker(void* argp) {
  bwd_arg* a = (bwd_arg*)argp;
  const orc_params* p = a->p;
  const int64_t T = (int64_t)p->P + p->L;
  const int64_t group = p->Nq / p->Nkv;
  row_scratch w;
  w.q = (double*)malloc(sizeof(double) * (size_t)(p->H + 1));
  w.krow = (double*)malloc(sizeof(double) * (size_t)(p->H + 1));
  w.vrow = (double*)malloc(sizeof(double) * (size_t)(p->Hv + 1));
  w.raw = (double*)malloc(sizeof(double) * (size_t)(T + 1));
  w.nocap = (double*)malloc(sizeof(double) * (size_t)(T + 1));
  w.s = (double*)malloc(sizeof(double) * (size_t)(T + 1));
  w.alive = (char*)malloc((size_t)(T + 1));
  double* prob = (double*)malloc(sizeof(double) * (size_t)(T + 1));
  double* dp = (double*)malloc(sizeof(double) * (size_t)(T + 1));
  double* dyrow = (double*)malloc(sizeof(double) * (size_t)(p->Hv + 1));
  if (!w.q || !w.krow || !w.vrow || !w.raw || !w.nocap || !w.s || !w.alive || !prob || !dp || !dyrow) {
    a->status = -2;
  } else {
    /* one (batch, kv head) per unit: every write of the unit lands in its own rows */
    for (int64_t unit = a->tid; unit < (int64_t)p->B * p->Nkv; unit += a->nthreads) {
      const int64_t b = unit / p->Nkv, kh = unit % p->Nkv;
      for (int64_t h = kh * group; h < (kh + 1) * group; ++h)
        for (int64_t i = 0; i < p->S; ++i) {
          qk_row(p, 3, b, h, i, prob, &w);             /* P of the row; w->q holds q_i */
          const int64_t yo = offset4(a->dy, b, h, i);
          for (int64_t d = 0; d < p->Hv; ++d) dyrow[d] = oracle_to_double(a->dy->dtype, a->dy->data, yo + d);
          double delta = 0.0;                           /* rowsum(P * dP) */
          for (int64_t j = 0; j < T; ++j) {
            dp[j] = 0.0;
            if (prob[j] == 0.0) continue;
            kv_row(p, 1, b, kh, j, w.vrow);
            double acc = 0.0;
            for (int64_t d = 0; d < p->Hv; ++d) acc += dyrow[d] * w.vrow[d];
            dp[j] = acc;
            delta += prob[j] * acc;
          }
          double* dqr = a->dq + ((b * p->Nq + h) * p->S + i) * p->H;
          for (int64_t j = 0; j < T; ++j) {
            if (prob[j] == 0.0) continue;
            const double ds = prob[j] * (dp[j] - delta) * p->scale;
            kv_row(p, 0, b, kh, j, w.krow);
            double* dkr = a->dk + ((b * p->Nkv + kh) * T + j) * p->H;
            double* dvr = a->dv + ((b * p->Nkv + kh) * T + j) * p->Hv;
            for (int64_t d = 0; d < p->H; ++d) {
              dqr[d] += ds * w.krow[d];
              dkr[d] += ds * w.q[d];
            }
            for (int64_t d = 0; d < p->Hv; ++d) dvr[d] += prob[j] * dyrow[d];
          }
        }
    }
  }
  free(w.q); free(w.krow); free(w.vrow); free(w.raw); free(w.nocap); free(w.s); free(w.alive);
  free(prob); free(dp); free(dyrow);
  return NULL;
}

int oracle_attention_backward(const orc_params* p, const orc_tensor* dy, double* dq, double* dk, double* dv,
                              int nthreads) {
  if (!p || !dy || !dy->data || !dq || !dk || !dv) return -1;
  if (p->Nkv <= 0 || p->Nq % p->Nkv != 0) return -1;
  if (p->window > 0 && p->causal == ORC_CAUSAL_NONE) return -1;
  if (p->len_kind != ORC_LEN_NONE && !p->lens) return -1;
  if (p->softcap > 0.0) return -1;
  const int64_t T = (int64_t)p->P + p->L;
  memset(dq, 0, sizeof(double) * (size_t)((int64_t)p->B * p->Nq * p->S * p->H));
  memset(dk, 0, sizeof(double) * (size_t)((int64_t)p->B * p->Nkv * T * p->H));
  memset(dv, 0, sizeof(double) * (size_t)((int64_t)p->B * p->Nkv * T * p->Hv));
  if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  const int64_t units = (int64_t)p->B * p->Nkv;
  if (nthreads < 1) nthreads = 1;
  if ((int64_t)nthreads > units) nthreads = units > 0 ? (int)units : 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  bwd_arg* args = (bwd_arg*)malloc(sizeof(bwd_arg) * (size_t)nthreads);
  if (!th || !args) { free(th); free(args); return -2; }
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    args[t] = (bwd_arg){p, dy, dq, dk, dv, t, nthreads, 0};
    if (pthread_create(&th[t], NULL, bwd_worker, &args[t]) != 0) break;
    ++started;
  }
  int status = 0;
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  for (int t = 0; t < started; ++t) if (args[t].status) status = args[t].status;
  for (int t = started; t < nthreads; ++t) {
    bwd_arg a1 = {p, dy, dq, dk, dv, t, nthreads, 0};
    bwd_worker(&a1);
    if (a1.status) status = a1.status;
  }
  free(th);
  free(args);
  return status ? status : nthreads;
}

/* ---- rounding of a double array to an element type (once, to nearest even) ---- */

int oracle_round_array(int32_t dtype, const double* in, int64_t n, void* out) {
  if (dtype != ORC_F32 && dtype != ORC_F16 && dtype != ORC_BF16) return -1;
  for (int64_t i = 0; i < n; ++i) {
    if (dtype == ORC_F32) ((float*)out)[i] = (float)in[i];
    else if (dtype == ORC_F16) ((uint16_t*)out)[i] = oracle_round_f16(in[i]);
    else ((uint16_t*)out)[i] = oracle_round_bf16(in[i]);
  }
  return 0;
}

/* ---- present = concat(past, new) along the sequence axis ---- */

int oracle_present(int32_t dtype, int32_t B, int32_t N, int32_t P, int32_t L, int32_t D,
                   const orc_tensor* past, const orc_tensor* cur, const void* bias, void* out) {
  if (dtype != ORC_F32 && dtype != ORC_F16 && dtype != ORC_BF16) return -1;
  const size_t esz = dtype == ORC_F32 ? 4 : 2;
  const int64_t T = (int64_t)P + L;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t t = 0; t < T; ++t) {
        char* dst = (char*)out + (((b * N + n) * T + t) * D) * (int64_t)esz;
        if (t < P) {
          const char* src = (const char*)past->data + offset4(past, b, n, t) * (int64_t)esz;
          memcpy(dst, src, (size_t)D * esz);                      /* bit copy */
        } else if (!bias) {
          const char* src = (const char*)cur->data + offset4(cur, b, n, t - P) * (int64_t)esz;
          memcpy(dst, src, (size_t)D * esz);
        } else {
          const int64_t o = offset4(cur, b, n, t - P);
          for (int64_t d = 0; d < D; ++d) {
            const double x = oracle_to_double(dtype, cur->data, o + d) +
                             oracle_to_double(dtype, bias, n * D + d);
            if (dtype == ORC_F32) ((float*)dst)[d] = (float)x;   /* one rounding */
            else if (dtype == ORC_F16) ((uint16_t*)dst)[d] = oracle_round_f16(x);
            else ((uint16_t*)dst)[d] = oracle_round_bf16(x);
          }
        }
      }
  return 0;
}

/* ---- rotary positional embedding (class RotaryEmbedding; RoFormer's rotation of channel
 * pairs by position-dependent angles given through the cos / sin caches) ---- */

int oracle_rotary(int32_t B, int32_t N, int32_t S, int32_t D, const orc_tensor* x, int32_t rotary_dim,
                  int32_t interleaved, const void* cos_cache, const void* sin_cache, int32_t cache_dtype,
                  int64_t cache_ld, const int64_t* positions, int64_t pos_sb, double* out) {
  const int32_t R = rotary_dim > 0 ? rotary_dim : D;
  if (R > D || R % 2 != 0 || !x || !cos_cache || !sin_cache) return -1;
  const int32_t half = R / 2;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t s = 0; s < S; ++s) {
        const int64_t xo = offset4(x, b, n, s);
        double* o = out + ((b * N + n) * S + s) * D;
        for (int64_t d = 0; d < D; ++d) o[d] = oracle_to_double(x->dtype, x->data, xo + d);
        const int64_t row = positions ? positions[b * pos_sb + s] : b * S + s;
        for (int64_t d = 0; d < half; ++d) {
          const double c = oracle_to_double(cache_dtype, cos_cache, row * cache_ld + d);
          const double sn = oracle_to_double(cache_dtype, sin_cache, row * cache_ld + d);
          const int64_t i1 = interleaved ? 2 * d : d;
          const int64_t i2 = interleaved ? 2 * d + 1 : d + half;
          const double x1 = oracle_to_double(x->dtype, x->data, xo + i1);
          const double x2 = oracle_to_double(x->dtype, x->data, xo + i2);
          o[i1] = x1 * c - x2 * sn;
          o[i2] = x2 * c + x1 * sn;
        }
      }
  return 0;
}
