// Internal definitions shared by the CUDA kernels of libsdpa (not part of the C ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sdpa.h"

namespace sdpa {

// ---------------------------------------------------------------------------------------
// Element types
// ---------------------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float to_f32(float x) { return x; }
  static __device__ __forceinline__ float from_f32(float x) { return x; }
  static __device__ __forceinline__ float from_f64(double x) { return (float)x; }
  static __device__ __forceinline__ double to_f64(float x) { return (double)x; }
  static constexpr int kVec = 4;   // elements per 16-byte vector
};
template <> struct Elem<__half> {
  static __device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f32(float x) { return __float2half_rn(x); }
  static __device__ __forceinline__ __half from_f64(double x) { return __double2half(x); }
  static __device__ __forceinline__ double to_f64(__half x) { return (double)__half2float(x); }
  static constexpr int kVec = 8;
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f64(double x) { return __double2bfloat16(x); }
  static __device__ __forceinline__ double to_f64(__nv_bfloat16 x) { return (double)__bfloat162float(x); }
  static constexpr int kVec = 8;
};

// Unpack a 16-byte vector of T into floats.
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& u, float* f) {
  if constexpr (sizeof(T) == 4) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  } else {
    const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = Elem<T>::to_f32(e[i]);
  }
}

__device__ __forceinline__ float load_scalar(const void* base, int dtype, int64_t idx) {
  switch (dtype) {
    case SDPA_F32: return reinterpret_cast<const float*>(base)[idx];
    case SDPA_F16: return __half2float(reinterpret_cast<const __half*>(base)[idx]);
    default: return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  }
}

// ---------------------------------------------------------------------------------------
// Resolved problem description passed to kernels by value
// ---------------------------------------------------------------------------------------
struct View {
  const void* p;
  int64_t sb, sh, ss;
  __host__ __device__ int64_t off(int64_t b, int64_t h, int64_t s) const { return b * sb + h * sh + s * ss; }
};

struct Rules {
  const void* add; int add_dtype; int64_t add_sb, add_sh, add_ss, add_T;
  const void* keep; int keep_kind; int64_t keep_sb, keep_sh, keep_ss, keep_T;
  int len_kind; const void* lens;
  int causal; int64_t window;
  float softcap; int softcap_before_bias; float filter;
};

struct Problem {
  int B, Nq, Nkv, S, L, P, H, Hv;
  int64_t T;
  int group;                 // Nq / Nkv
  View q, k, v, past_k, past_v, present_k, present_v, y;
  const void* q_bias; const void* k_bias; const void* v_bias; const void* head_sink;
  float scale;
  Rules r;
};

// Per-row constants for the score rules.
struct RowCtx {
  int64_t pos;       // key position of the query row (causal / window)
  int64_t len;       // per-batch length (len_kind != NONE)
};

__device__ __forceinline__ int64_t batch_len(const Rules& r, int b) {
  if (r.len_kind == SDPA_LEN_NONPAD_I64) return reinterpret_cast<const int64_t*>(r.lens)[b];
  if (r.len_kind == SDPA_LEN_NONE) return 0;
  return (int64_t)reinterpret_cast<const int32_t*>(r.lens)[b];
}

__device__ __forceinline__ RowCtx row_ctx(const Rules& r, int S, int64_t T, int b, int i) {
  RowCtx c;
  c.len = batch_len(r, b);
  if (r.causal == SDPA_CAUSAL_UPPER_LEFT) c.pos = i;
  else if (r.causal == SDPA_CAUSAL_LOWER_RIGHT)
    c.pos = ((r.len_kind == SDPA_LEN_SEQLENS_K_I32) ? c.len + 1 : T) - S + i;
  else c.pos = 0;
  return c;
}

__device__ __forceinline__ float softcap_f(float s, float c) { return c * tanhf(s / c); }

// Applies every stage after the scaled dot product to score s of key j in row (b, h, i).
// Returns -inf for an excluded key.
__device__ __forceinline__ float apply_rules(const Rules& r, const RowCtx& c, float s, int b, int h,
                                             int i, int64_t j) {
  bool excl = false;
  float addv = 0.f;
  if (r.add) {
    if (j < r.add_T) addv = load_scalar(r.add, r.add_dtype, b * r.add_sb + h * r.add_sh + i * r.add_ss + j);
    else excl = true;
  }
  if (!r.softcap_before_bias) s += addv;
  if (r.softcap > 0.f && !excl && s != -INFINITY) s = softcap_f(s, r.softcap);
  if (r.softcap_before_bias) s += addv;
  if (r.keep_kind != SDPA_KEEP_NONE) {
    bool keep = false;
    if (j < r.keep_T) {
      const int64_t o = b * r.keep_sb + h * r.keep_sh + i * r.keep_ss + j;
      keep = (r.keep_kind == SDPA_KEEP_BOOL_U8) ? (reinterpret_cast<const uint8_t*>(r.keep)[o] != 0)
                                                : (reinterpret_cast<const int32_t*>(r.keep)[o] != 0);
    }
    if (!keep) {
      if (r.keep_kind == SDPA_KEEP_BOOL_U8) excl = true;
      else s += r.filter;
    }
  }
  if (r.causal != SDPA_CAUSAL_NONE && j > c.pos) excl = true;
  if (r.window > 0 && j < c.pos - r.window + 1) excl = true;
  if (r.len_kind == SDPA_LEN_NONPAD_I64 && j >= c.len) excl = true;
  if (r.len_kind == SDPA_LEN_KEYLEN_I32 && j >= c.len) s += r.filter;
  if (r.len_kind == SDPA_LEN_SEQLENS_K_I32 && j > c.len) excl = true;
  return excl ? -INFINITY : s;
}

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------------------
// Bounds-checking debug build (compiled with -DSDPA_BOUNDS_CHECK)
// ---------------------------------------------------------------------------------------
// SDPA_IN_BOUNDS(cond, site) guards an index before the access it feeds: in the debug build a
// false condition records `site` (the first failing check wins) in the translation unit's
// status word and yields false, so the caller skips the access instead of faulting; in the
// normal build it is `true` and costs nothing.  Each kernel translation unit defines its
// reader with SDPA_DEFINE_BOUNDS_TAKE(name); sdpa_query_status reports a recorded site as
// SDPA_ERR_BOUNDS.
#ifdef SDPA_BOUNDS_CHECK
static __device__ int g_bounds_site;   // one per translation unit
__device__ __forceinline__ bool bounds_ok(bool cond, int site) {
  if (!cond) atomicCAS(&g_bounds_site, 0, site);
  return cond;
}
#define SDPA_IN_BOUNDS(cond, site) (::sdpa::bounds_ok((cond), (site)))
#define SDPA_DEFINE_BOUNDS_TAKE(name)                                          \
  cudaError_t name(int* site) {                                                \
    int v = 0;                                                                 \
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_bounds_site, sizeof v);         \
    if (e != cudaSuccess) return e;                                            \
    *site = v;                                                                 \
    if (v) {                                                                   \
      const int zero = 0;                                                      \
      e = cudaMemcpyToSymbol(g_bounds_site, &zero, sizeof zero);               \
    }                                                                          \
    return e;                                                                  \
  }
#else
#define SDPA_IN_BOUNDS(cond, site) true
#define SDPA_DEFINE_BOUNDS_TAKE(name) \
  cudaError_t name(int* site) {       \
    *site = 0;                        \
    return cudaSuccess;               \
  }
#endif

}  // namespace sdpa
