// C ABI of libsdpa: argument validation, planning and launch (see include/sdpa.h).
//
// Every check runs on the host before anything is enqueued, following the contracts'
// rejection rules (onnx-light-cpu "Custom operators": GroupQueryAttention rejects a
// local_window_size of 0, below -1, above INT32_MAX, or with causal off; MultiHeadAttention
// rejects shared past/present buffers; class Attention never runs in place).
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "internal.h"
#include "prefill_tc.h"

namespace sdpa {

static std::atomic<long long> g_launches{0};
void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

namespace {

thread_local std::string g_error;
thread_local const char* g_kernel = "";

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_error = buf;
  return code;
}

int esize(int dt) { return dt == SDPA_F32 ? 4 : 2; }
int vec_elems(int dt) { return 16 / esize(dt); }

struct Extent {
  uintptr_t lo = 0, hi = 0;   // [lo, hi) bytes; hi == lo when empty/absent
  const char* name = "";
};

// Validates a (B, N, S, D) view; records its byte extent.
int check_view(const sdpa_view& v, const char* name, int dt, int64_t B, int64_t N, int64_t S,
               int64_t D, bool required, bool allow_broadcast, Extent* ext) {
  ext->name = name;
  ext->lo = ext->hi = 0;
  const bool empty = B == 0 || N == 0 || S == 0 || D == 0;
  if (!v.data) {
    if (required && !empty) return fail(SDPA_ERR_NULL, "%s: data pointer is NULL", name);
    return SDPA_OK;
  }
  if (v.stride_b < 0 || v.stride_n < 0 || v.stride_s < 0)
    return fail(SDPA_ERR_INVALID, "%s: negative stride", name);
  if (!allow_broadcast && !empty && ((B > 1 && v.stride_b == 0) || (N > 1 && v.stride_n == 0) ||
                                     (S > 1 && v.stride_s == 0)))
    return fail(SDPA_ERR_INVALID, "%s: zero stride on a non-broadcast view", name);
  if (empty) return SDPA_OK;
  const int64_t lim = (int64_t)1 << 40;
  if (v.stride_b > lim || v.stride_n > lim || v.stride_s > lim || B > lim || S > lim)
    return fail(SDPA_ERR_OVERFLOW, "%s: stride or extent beyond 2^40 elements", name);
  const double last = (double)(B - 1) * v.stride_b + (double)(N - 1) * v.stride_n +
                      (double)(S - 1) * v.stride_s + (double)D;
  if (last * esize(dt) > 9.0e18) return fail(SDPA_ERR_OVERFLOW, "%s: byte extent overflows", name);
  const int64_t last_i = (B - 1) * v.stride_b + (N - 1) * v.stride_n + (S - 1) * v.stride_s + D;
  ext->lo = (uintptr_t)v.data;
  ext->hi = ext->lo + (uintptr_t)(last_i * esize(dt));
  return SDPA_OK;
}

int check_aligned_view(const sdpa_view& v, const char* name, int dt) {
  if (!v.data) return SDPA_OK;
  const int ve = vec_elems(dt);
  if (((uintptr_t)v.data & 15u) != 0) return fail(SDPA_ERR_ALIGNMENT, "%s: pointer not 16-byte aligned", name);
  if (v.stride_b % ve || v.stride_n % ve || v.stride_s % ve)
    return fail(SDPA_ERR_ALIGNMENT, "%s: strides must be multiples of %d elements", name, ve);
  return SDPA_OK;
}

bool overlap(const Extent& a, const Extent& b) {
  if (a.hi == a.lo || b.hi == b.lo) return false;
  return a.lo < b.hi && b.lo < a.hi;
}

Extent flat(const void* p, size_t bytes, const char* name) {
  Extent e;
  e.name = name;
  if (p && bytes) { e.lo = (uintptr_t)p; e.hi = e.lo + bytes; }
  return e;
}

// Rotary embedding of Q and the new K rows requested through sdpa_params.
struct Rot {
  bool on = false;
  const void* cos = nullptr;
  const void* sin = nullptr;
  int64_t max_pos = 0;
  int R = 0, interleaved = 0;
};

// Validation shared by every attention entry point.  Fills `pr` (and `rot`) on success.
int validate(const sdpa_params* p, int op, Problem* pr, Rot* rot = nullptr) {
  if (!p) return fail(SDPA_ERR_NULL, "params is NULL");
  if (p->struct_size != (int32_t)sizeof(sdpa_params))
    return fail(SDPA_ERR_INVALID, "struct_size %d != sizeof(sdpa_params) %d", p->struct_size,
                (int)sizeof(sdpa_params));
  if (op != SDPA_OP_FWD && op != SDPA_OP_DECODE && op != SDPA_OP_BWD) return fail(SDPA_ERR_INVALID, "unknown op %d", op);
  const int dt = p->dtype;
  if (dt != SDPA_F32 && dt != SDPA_F16 && dt != SDPA_BF16) return fail(SDPA_ERR_INVALID, "dtype %d", dt);
  if (p->B < 0 || p->S < 0 || p->L < 0 || p->P < 0)
    return fail(SDPA_ERR_SHAPE, "negative size (B=%d S=%d L=%d P=%d)", p->B, p->S, p->L, p->P);
  if (p->Nq < 1 || p->Nkv < 1 || p->H < 1 || p->Hv < 1)
    return fail(SDPA_ERR_SHAPE, "Nq, Nkv, H and Hv must be >= 1");
  if (p->Nq % p->Nkv != 0)
    return fail(SDPA_ERR_SHAPE, "q heads (%d) must be a multiple of kv heads (%d)", p->Nq, p->Nkv);
  const int ve = vec_elems(dt);
  if (p->H > 256 || p->Hv > 256 || p->H % ve || p->Hv % ve)
    return fail(SDPA_ERR_UNSUPPORTED, "head sizes must be multiples of %d and at most 256 (H=%d Hv=%d)",
                ve, p->H, p->Hv);
  if (p->causal < SDPA_CAUSAL_NONE || p->causal > SDPA_CAUSAL_LOWER_RIGHT)
    return fail(SDPA_ERR_INVALID, "causal mode %d", p->causal);
  if (p->window == 0 || p->window < -1 || p->window > 2147483647LL)
    return fail(SDPA_ERR_INVALID, "window %lld: must be -1 or in [1, INT32_MAX]", (long long)p->window);
  if (p->window > 0 && p->causal == SDPA_CAUSAL_NONE)
    return fail(SDPA_ERR_INVALID, "a local window needs causal masking");
  if (!std::isfinite(p->softcap)) return fail(SDPA_ERR_INVALID, "softcap must be finite");
  if (p->has_scale && !std::isfinite(p->scale)) return fail(SDPA_ERR_INVALID, "scale must be finite");
  if (!std::isfinite(p->mask_filter_value)) return fail(SDPA_ERR_INVALID, "mask_filter_value must be finite");
  if (p->keep_kind < SDPA_KEEP_NONE || p->keep_kind > SDPA_KEEP_FILTER_I32)
    return fail(SDPA_ERR_INVALID, "keep_kind %d", p->keep_kind);
  if (p->len_kind < SDPA_LEN_NONE || p->len_kind > SDPA_LEN_SEQLENS_K_I32)
    return fail(SDPA_ERR_INVALID, "len_kind %d", p->len_kind);
  if (p->len_kind != SDPA_LEN_NONE && !p->lens && p->B > 0) return fail(SDPA_ERR_NULL, "lens is NULL");
  if (p->keep_kind != SDPA_KEEP_NONE && !p->keep_mask.data) return fail(SDPA_ERR_NULL, "keep_mask is NULL");
  if (p->add_mask.data && p->add_mask_dtype != SDPA_F32 && p->add_mask_dtype != SDPA_F16 &&
      p->add_mask_dtype != SDPA_BF16)
    return fail(SDPA_ERR_INVALID, "add_mask_dtype %d", p->add_mask_dtype);
  if (p->add_mask_T < 0 || p->keep_mask_T < 0) return fail(SDPA_ERR_SHAPE, "negative mask width");
  if ((p->present_k.data == nullptr) != (p->present_v.data == nullptr))
    return fail(SDPA_ERR_INVALID, "present_k and present_v must be given together");
  if (p->P > 0 && (!p->past_k.data || !p->past_v.data))
    return fail(SDPA_ERR_SHAPE, "P=%d past rows but past_k/past_v absent", p->P);
  if (p->P == 0 && (p->past_k.data || p->past_v.data))
    return fail(SDPA_ERR_SHAPE, "past_k/past_v given with P=0");
  if (p->qk_out.data) {
    if (op == SDPA_OP_DECODE)
      return fail(SDPA_ERR_UNSUPPORTED, "the qk output is written by sdpa_attn_fwd only");
    if (p->qk_mode < 0 || p->qk_mode > 3) return fail(SDPA_ERR_INVALID, "qk_mode %d: must be 0..3", p->qk_mode);
  }
  if ((p->rotary_cos == nullptr) != (p->rotary_sin == nullptr))
    return fail(SDPA_ERR_INVALID, "rotary_cos and rotary_sin must be given together");
  const bool rot_on = p->rotary_cos != nullptr;
  const int rot_R = rot_on ? (p->rotary_dim ? p->rotary_dim : p->H) : 0;
  if (rot_on) {
    if (rot_R < 2 || rot_R > p->H || rot_R % 2)
      return fail(SDPA_ERR_INVALID, "rotary_dim %d: must be even and in [2, H=%d] (0 means H)", p->rotary_dim, p->H);
    if (p->rotary_interleaved != 0 && p->rotary_interleaved != 1)
      return fail(SDPA_ERR_INVALID, "rotary_interleaved must be 0 or 1");
    if (p->rotary_max_pos < 1 || p->rotary_max_pos > ((int64_t)1 << 40))
      return fail(SDPA_ERR_SHAPE, "rotary_max_pos %lld out of range", (long long)p->rotary_max_pos);
    if (p->q_bias || p->k_bias)
      return fail(SDPA_ERR_UNSUPPORTED, "rotary embedding together with q/k projection biases");
    if (((uintptr_t)p->rotary_cos | (uintptr_t)p->rotary_sin) % esize(dt))
      return fail(SDPA_ERR_ALIGNMENT, "rotary caches not aligned to the element size");
  }
  if (op == SDPA_OP_DECODE) {
    if (p->S > 16) return fail(SDPA_ERR_UNSUPPORTED, "decode handles S <= 16 (S=%d); use sdpa_attn_fwd", p->S);
    if (!decode_supported((sdpa_dtype)dt, p->H, p->Hv))
      return fail(SDPA_ERR_UNSUPPORTED, "decode needs H == Hv with H*elem_size in {128, 256, 512} bytes");
  }
  const int64_t T = (int64_t)p->P + p->L;
  if ((int64_t)p->B * p->Nq * (int64_t)p->S > ((int64_t)1 << 31) - 1 || T > ((int64_t)1 << 31) - 1)
    return fail(SDPA_ERR_OVERFLOW, "B*Nq*S or P+L exceeds 2^31-1");

  // views
  Extent eq, ek, ev, epk, epv, eprk, eprv, ey, eam, ekm;
  int rc;
  if ((rc = check_view(p->q, "q", dt, p->B, p->Nq, p->S, p->H, true, false, &eq))) return rc;
  if ((rc = check_view(p->k, "k", dt, p->B, p->Nkv, p->L, p->H, true, false, &ek))) return rc;
  if ((rc = check_view(p->v, "v", dt, p->B, p->Nkv, p->L, p->Hv, true, false, &ev))) return rc;
  if ((rc = check_view(p->past_k, "past_k", dt, p->B, p->Nkv, p->P, p->H, p->P > 0, false, &epk))) return rc;
  if ((rc = check_view(p->past_v, "past_v", dt, p->B, p->Nkv, p->P, p->Hv, p->P > 0, false, &epv))) return rc;
  if ((rc = check_view(p->present_k, "present_k", dt, p->B, p->Nkv, T, p->H, false, false, &eprk))) return rc;
  if ((rc = check_view(p->present_v, "present_v", dt, p->B, p->Nkv, T, p->Hv, false, false, &eprv))) return rc;
  if ((rc = check_view(p->y, "y", dt, p->B, p->Nq, p->S, p->Hv, op != SDPA_OP_BWD, false, &ey))) return rc;
  Extent eqk;
  if ((rc = check_view(p->qk_out, "qk_out", SDPA_F32, p->B, p->Nq, p->S, T, false, false, &eqk))) return rc;
  const int mdt = p->add_mask.data ? p->add_mask_dtype : SDPA_F32;
  if ((rc = check_view(p->add_mask, "add_mask", mdt, p->B, p->Nq, p->S, p->add_mask_T, false, true, &eam))) return rc;
  // keep masks are u8 or i32: reuse the f32/f16 element sizes for the extent
  const int kdt = (p->keep_kind == SDPA_KEEP_FILTER_I32) ? SDPA_F32 : SDPA_F16;
  if (p->keep_kind != SDPA_KEEP_NONE) {
    if ((rc = check_view(p->keep_mask, "keep_mask", kdt, p->B, p->Nq, p->S, p->keep_mask_T, true, true, &ekm))) return rc;
    if (p->keep_kind == SDPA_KEEP_BOOL_U8 && ekm.hi > ekm.lo) {   // u8: half the f16 extent
      ekm.hi = ekm.lo + (ekm.hi - ekm.lo) / 2;
    }
  }
  for (const sdpa_view* v : {&p->q, &p->k, &p->v, &p->past_k, &p->past_v, &p->present_k, &p->present_v, &p->y}) {
    const char* nm = v == &p->q ? "q" : v == &p->k ? "k" : v == &p->v ? "v" : v == &p->past_k ? "past_k"
                   : v == &p->past_v ? "past_v" : v == &p->present_k ? "present_k" : v == &p->present_v ? "present_v" : "y";
    if ((rc = check_aligned_view(*v, nm, dt))) return rc;
  }
  for (const void* ptr : {p->q_bias, p->k_bias, p->v_bias})
    if (ptr && ((uintptr_t)ptr & 15u)) return fail(SDPA_ERR_ALIGNMENT, "projection bias not 16-byte aligned");

  // aliasing: outputs against every input and against each other
  const Extent inputs[] = {eq, ek, ev, epk, epv, eam, ekm,
                           flat(p->q_bias, (size_t)p->Nq * p->H * esize(dt), "q_bias"),
                           flat(p->k_bias, (size_t)p->Nkv * p->H * esize(dt), "k_bias"),
                           flat(p->v_bias, (size_t)p->Nkv * p->Hv * esize(dt), "v_bias"),
                           flat(p->head_sink, (size_t)p->Nq * esize(dt), "head_sink"),
                           flat(p->lens, (size_t)p->B * (p->len_kind == SDPA_LEN_NONPAD_I64 ? 8 : 4), "lens"),
                           flat(p->rotary_cos, (size_t)p->rotary_max_pos * (rot_R / 2) * esize(dt), "rotary_cos"),
                           flat(p->rotary_sin, (size_t)p->rotary_max_pos * (rot_R / 2) * esize(dt), "rotary_sin")};
  for (const Extent& o : {ey, eprk, eprv, eqk}) {
    for (const Extent& in : inputs)
      if (overlap(o, in)) return fail(SDPA_ERR_ALIAS, "output %s overlaps input %s", o.name, in.name);
  }
  if (overlap(ey, eprk) || overlap(ey, eprv) || overlap(eprk, eprv) || overlap(eqk, ey) || overlap(eqk, eprk) ||
      overlap(eqk, eprv))
    return fail(SDPA_ERR_ALIAS, "outputs y / present_k / present_v / qk_out overlap");

  // resolved problem
  Problem& r = *pr;
  std::memset(&r, 0, sizeof r);
  r.B = p->B; r.Nq = p->Nq; r.Nkv = p->Nkv; r.S = p->S; r.L = p->L; r.P = p->P; r.H = p->H; r.Hv = p->Hv;
  r.T = T;
  r.group = p->Nq / p->Nkv;
  auto cv = [](const sdpa_view& v) { return View{v.data, v.stride_b, v.stride_n, v.stride_s}; };
  r.q = cv(p->q); r.k = cv(p->k); r.v = cv(p->v); r.past_k = cv(p->past_k); r.past_v = cv(p->past_v);
  r.present_k = cv(p->present_k); r.present_v = cv(p->present_v); r.y = cv(p->y);
  r.q_bias = p->q_bias; r.k_bias = p->k_bias; r.v_bias = p->v_bias; r.head_sink = p->head_sink;
  r.scale = p->has_scale ? p->scale : (float)(1.0 / std::sqrt((double)p->H));
  Rules& ru = r.r;
  ru.add = p->add_mask.data; ru.add_dtype = p->add_mask_dtype;
  ru.add_sb = p->add_mask.stride_b; ru.add_sh = p->add_mask.stride_n; ru.add_ss = p->add_mask.stride_s;
  ru.add_T = p->add_mask_T;
  ru.keep = p->keep_kind != SDPA_KEEP_NONE ? p->keep_mask.data : nullptr;
  ru.keep_kind = p->keep_kind;
  ru.keep_sb = p->keep_mask.stride_b; ru.keep_sh = p->keep_mask.stride_n; ru.keep_ss = p->keep_mask.stride_s;
  ru.keep_T = p->keep_mask_T;
  ru.len_kind = p->len_kind; ru.lens = p->lens;
  ru.causal = p->causal; ru.window = p->window;
  ru.softcap = p->softcap > 0.f ? p->softcap : 0.f;
  ru.softcap_before_bias = p->softcap_before_bias ? 1 : 0;
  ru.filter = p->mask_filter_value;
  if (rot) {
    *rot = Rot{};
    if (rot_on) {
      rot->on = true; rot->cos = p->rotary_cos; rot->sin = p->rotary_sin;
      rot->max_pos = p->rotary_max_pos; rot->R = rot_R; rot->interleaved = p->rotary_interleaved;
    }
  }
  return SDPA_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(SDPA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Bytes of workspace sdpa_attn_fwd needs: K/V materialised for the tensor-core path when
// past rows or projection biases are present and no present output can hold them.
// The tensor-core path takes the problem when the kernel fits it and the K and V views it
// will read (the inputs, present, or the materialised copies) walk their axes alike.
bool tc_usable(const Problem& r, sdpa_dtype dt) {
  if (!tc_eligible(r, dt)) return false;
  const bool needs_total = r.P > 0 || r.k_bias || r.v_bias;
  if (needs_total && !r.present_k.p) return true;            // contiguous copies, same order
  const View& k = needs_total ? r.present_k : r.k;
  const View& v = needs_total ? r.present_v : r.v;
  return tc_same_axis_order(k, v, r.B, r.Nkv, needs_total ? r.T : r.L);
}

size_t fwd_workspace(const Problem& r, sdpa_dtype dt) {
  if (!tc_usable(r, dt)) return 0;
  const bool needs_total = r.P > 0 || r.k_bias || r.v_bias;
  if (!needs_total || r.present_k.p) return 0;
  const size_t bytes = (size_t)r.B * r.Nkv * (size_t)r.T * (r.H + r.Hv) * esize(dt);
  return (bytes + 255) & ~(size_t)255;
}

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

// Past rows or k / v projection biases: the backward works on contiguous copies of the T key
// and value rows the scores see (past rows first, biases added), as the forward does.
bool bwd_materialise_kv(const Problem& r) { return r.P > 0 || r.k_bias || r.v_bias; }

// The backward's subset: the GroupQueryAttention gradient graph has no softcap, and this
// library's kernels take 16-bit types, H == Hv in {64, 128} and no rotary step.
int bwd_check(const sdpa_params* p, const Problem& r, const Rot& rot) {
  const sdpa_dtype dt = (sdpa_dtype)p->dtype;
  if (p->softcap > 0.f) return fail(SDPA_ERR_UNSUPPORTED, "the backward has no softcap derivative");
  if (dt == SDPA_F32) return fail(SDPA_ERR_UNSUPPORTED, "backward: float16 / bfloat16 only");
  if (!bwd_tc_supported(r, dt)) return fail(SDPA_ERR_UNSUPPORTED, "backward: H == Hv in {64, 128} only");
  if (rot.on) return fail(SDPA_ERR_UNSUPPORTED, "backward: no rotary step");
  if (p->qk_out.data) return fail(SDPA_ERR_UNSUPPORTED, "backward: no qk output");
  if (p->present_k.data) return fail(SDPA_ERR_INVALID, "backward: present outputs are not written");
  if (!bwd_materialise_kv(r) && !tc_same_axis_order(r.k, r.v, r.B, r.Nkv, r.T))
    return fail(SDPA_ERR_UNSUPPORTED, "backward: k and v views must walk their axes in the same order");
  return SDPA_OK;
}

// Backward workspace: log2-sum-exp and delta per query row, then Q + q_bias when there is a
// q bias, then the key and value rows the scores see when they must be materialised.
struct BwdWs {
  size_t lse2 = 0, delta = 0, q = 0, k = 0, v = 0, total = 0;
};
BwdWs bwd_layout(const Problem& r, sdpa_dtype dt) {
  BwdWs w;
  const size_t stat = align256((size_t)r.B * r.Nq * (size_t)r.S * sizeof(float));
  w.lse2 = 0;
  w.delta = stat;
  w.total = 2 * stat;
  if (r.q_bias) { w.q = w.total; w.total += align256((size_t)r.B * r.Nq * (size_t)r.S * r.H * esize(dt)); }
  if (bwd_materialise_kv(r)) {
    w.k = w.total; w.total += align256((size_t)r.B * r.Nkv * (size_t)r.T * r.H * esize(dt));
    w.v = w.total; w.total += align256((size_t)r.B * r.Nkv * (size_t)r.T * r.Hv * esize(dt));
  }
  return w;
}
size_t bwd_workspace(const Problem& r, sdpa_dtype dt) { return bwd_layout(r, dt).total; }

// Bytes of workspace for the rotated copies of Q and of the new K rows; 0 without rotary.
size_t rot_workspace(const Problem& r, const Rot& rot, sdpa_dtype dt) {
  if (!rot.on) return 0;
  return align256((size_t)r.B * r.Nq * r.S * r.H * esize(dt)) +
         align256((size_t)r.B * r.Nkv * r.L * r.H * esize(dt));
}

// The problem as the attention kernels see it after the rotary step: r.q and r.k point at
// contiguous copies at the start of `ws` (a stand-in 256-byte aligned address when ws is
// NULL, for sizing), so every later step (present included) reads rotated Q and K.
Problem after_rotary(const Problem& r, const Rot& rot, sdpa_dtype dt, void* ws) {
  Problem a = r;
  if (!rot.on) return a;
  char* base = ws ? reinterpret_cast<char*>(ws) : reinterpret_cast<char*>((uintptr_t)256);
  const size_t qbytes = align256((size_t)r.B * r.Nq * r.S * r.H * esize(dt));
  a.q = View{base, (int64_t)r.Nq * r.S * r.H, (int64_t)r.S * r.H, r.H};
  // the K copy walks its axes in V's order, so the tensor-core path can read both
  int order[3];
  tc_axis_order(r.v, r.B, r.Nkv, r.L, order);
  const int64_t ext[3] = {r.L, r.Nkv, r.B};
  int64_t str[3], cur = r.H;
  for (int i = 0; i < 3; ++i) { str[order[i]] = cur; cur *= ext[order[i]]; }
  a.k = View{base + qbytes, str[2], str[1], str[0]};
  return a;
}

// GroupQueryAttention's rotary step at absolute positions: query row i of batch b sits at
// Tv(b) - S + i and new key row j at Tv(b) - L + j, where Tv(b) = seqlens_k[b] + 1 under
// SDPA_LEN_SEQLENS_K_I32 and T = P + L otherwise (the causal alignment's positions).
// Writes the rotated rows to the views of after_rotary(r, rot, dt, ws).
int run_rotary(const Problem& r, const Rot& rot, sdpa_dtype dt, void* ws, cudaStream_t st) {
  const Problem a = after_rotary(r, rot, dt, ws);
  RotaryPos rp{};
  rp.mode = kRotaryAbsolute;
  rp.cache_ld = rot.R / 2;
  rp.max_pos = rot.max_pos;
  rp.lens = r.r.len_kind == SDPA_LEN_SEQLENS_K_I32 ? reinterpret_cast<const int32_t*>(r.r.lens) : nullptr;
  RotaryJob jobs[2];
  jobs[0] = RotaryJob{r.q, a.q, r.B, r.Nq, r.S, rp};
  jobs[0].rp.new_rows = r.S;
  jobs[0].rp.base = r.T - r.S;
  jobs[1] = RotaryJob{r.k, a.k, r.B, r.Nkv, r.L, rp};
  jobs[1].rp.new_rows = r.L;
  jobs[1].rp.base = r.T - r.L;
  const cudaError_t e = launch_rotary(dt, jobs, 2, r.H, rot.cos, rot.sin, rot.R, rot.interleaved, st);
  return e == cudaSuccess ? SDPA_OK : cuda_fail(e, "rotary launch");
}

// The qk output (class Attention's qk_matmul_output) after the attention launch.
thread_local std::string g_kernel_pair;
int run_qk(const Problem& r, const View* k_total, const sdpa_params* p, sdpa_dtype dt, cudaStream_t st) {
  const View out{p->qk_out.data, p->qk_out.stride_b, p->qk_out.stride_n, p->qk_out.stride_s};
  const char* name = "";
  const cudaError_t e = launch_qk(r, k_total, out, p->qk_mode, dt, st, &name);
  if (e != cudaSuccess) return cuda_fail(e, "qk output launch");
  g_kernel_pair = std::string(g_kernel) + "+" + name;
  g_kernel = g_kernel_pair.c_str();
  return SDPA_OK;
}

int run_concat_present(const Problem& r, sdpa_dtype dt, cudaStream_t st) {
  cudaError_t e = launch_kv_concat(dt, r.B, r.Nkv, r.P, r.L, r.H, r.past_k, r.k, r.k_bias, r.present_k, st);
  if (e == cudaSuccess)
    e = launch_kv_concat(dt, r.B, r.Nkv, r.P, r.L, r.Hv, r.past_v, r.v, r.v_bias, r.present_v, st);
  return e == cudaSuccess ? SDPA_OK : cuda_fail(e, "kv_concat launch");
}

}  // namespace
}  // namespace sdpa

using namespace sdpa;

extern "C" {

int sdpa_validate(const sdpa_params* p, int op) {
  Problem r;
  Rot rot;
  const int rc = validate(p, op, &r, &rot);
  if (rc || op != SDPA_OP_BWD) return rc;
  return bwd_check(p, r, rot);
}

size_t sdpa_workspace_size(const sdpa_params* p, int op) {
  Problem r;
  Rot rot;
  if (validate(p, op, &r, &rot) != SDPA_OK) return 0;
  const sdpa_dtype dt = (sdpa_dtype)p->dtype;
  const size_t pre = rot_workspace(r, rot, dt);
  if (op == SDPA_OP_DECODE) return pre + plan_decode(r.B, r.Nq, r.Nkv, r.S, r.T, r.Hv).ws_bytes;
  if (op == SDPA_OP_BWD) return bwd_check(p, r, rot) == SDPA_OK ? bwd_workspace(r, (sdpa_dtype)p->dtype) : 0;
  return pre + fwd_workspace(after_rotary(r, rot, dt, nullptr), dt);
}

int sdpa_attn_fwd(const sdpa_params* p, void* workspace, size_t workspace_bytes, sdpa_stream_t stream) {
  Problem r;
  Rot rot;
  int rc = validate(p, SDPA_OP_FWD, &r, &rot);
  if (rc) return rc;
  const sdpa_dtype dt = (sdpa_dtype)p->dtype;
  const size_t pre = rot_workspace(r, rot, dt);
  const size_t need = pre + fwd_workspace(after_rotary(r, rot, dt, nullptr), dt);
  if (need && (!workspace || workspace_bytes < need))
    return fail(SDPA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if (need && ((uintptr_t)workspace & 255u)) return fail(SDPA_ERR_ALIGNMENT, "workspace not 256-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  g_error.clear();
  if (rot.on) {
    if ((rc = run_rotary(r, rot, dt, workspace, st))) return rc;
    r = after_rotary(r, rot, dt, workspace);
    workspace = reinterpret_cast<char*>(workspace) + pre;
  }

  const int64_t rows = (int64_t)r.B * r.Nq * r.S;
  if (tc_usable(r, dt) && rows > 0) {
    // the tensor-core kernel reads one K and one V view of T rows
    Problem a = r;
    const bool needs_total = r.P > 0 || r.k_bias || r.v_bias;
    if (r.present_k.p) {
      if ((rc = run_concat_present(r, dt, st))) return rc;
    }
    if (needs_total) {
      View tk, tv;
      if (r.present_k.p) {
        tk = r.present_k; tv = r.present_v;
      } else {
        char* base = reinterpret_cast<char*>(workspace);
        const int64_t es = esize(dt);
        tk = View{base, (int64_t)r.Nkv * r.T * r.H, r.T * r.H, r.H};
        tv = View{base + (size_t)r.B * r.Nkv * r.T * r.H * es, (int64_t)r.Nkv * r.T * r.Hv, r.T * r.Hv, r.Hv};
        cudaError_t e = launch_kv_concat(dt, r.B, r.Nkv, r.P, r.L, r.H, r.past_k, r.k, r.k_bias, tk, st);
        if (e == cudaSuccess) e = launch_kv_concat(dt, r.B, r.Nkv, r.P, r.L, r.Hv, r.past_v, r.v, r.v_bias, tv, st);
        if (e != cudaSuccess) return cuda_fail(e, "kv materialisation");
      }
      a.k = tk; a.v = tv; a.P = 0; a.L = (int)r.T; a.k_bias = nullptr; a.v_bias = nullptr;
      a.past_k = View{}; a.past_v = View{};
    }
    a.present_k = View{}; a.present_v = View{};
    const char* name = "";
    cudaError_t e = launch_prefill_tc(a, dt, st, &name);
    if (e != cudaSuccess) return cuda_fail(e, "prefill_tc launch");
    g_kernel = name;
    if (p->qk_out.data && (rc = run_qk(r, &a.k, p, dt, st))) return rc;
    return SDPA_OK;
  }

  if (r.present_k.p) {
    if ((rc = run_concat_present(r, dt, st))) return rc;
  }
  if (rows > 0) {
    Problem a = r;
    a.present_k = View{}; a.present_v = View{};
    cudaError_t e = launch_simt_fwd(a, dt, st);
    if (e != cudaSuccess) return cuda_fail(e, "simt_fwd launch");
    g_kernel = dt == SDPA_F32 ? "simt_fwd_f32" : dt == SDPA_F16 ? "simt_fwd_f16" : "simt_fwd_bf16";
    if (p->qk_out.data) {
      // one view of all T key rows, where the inputs already hold one
      const View* kt = (r.P == 0 && !r.k_bias) ? &r.k : (r.present_k.p ? &r.present_k : nullptr);
      if ((rc = run_qk(r, kt, p, dt, st))) return rc;
    }
  }
  return SDPA_OK;
}

int sdpa_attn_decode(const sdpa_params* p, void* workspace, size_t workspace_bytes, sdpa_stream_t stream) {
  Problem r;
  Rot rot;
  int rc = validate(p, SDPA_OP_DECODE, &r, &rot);
  if (rc) return rc;
  const sdpa_dtype dt = (sdpa_dtype)p->dtype;
  const DecodePlan plan = plan_decode(r.B, r.Nq, r.Nkv, r.S, r.T, r.Hv);
  const size_t pre = rot_workspace(r, rot, dt);
  const size_t need = pre + plan.ws_bytes;
  if (need && (!workspace || workspace_bytes < need))
    return fail(SDPA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if (need && ((uintptr_t)workspace & 255u)) return fail(SDPA_ERR_ALIGNMENT, "workspace not 256-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  g_error.clear();
  if (rot.on) {
    if ((rc = run_rotary(r, rot, dt, workspace, st))) return rc;
    r = after_rotary(r, rot, dt, workspace);
    workspace = reinterpret_cast<char*>(workspace) + pre;
  }
  const int64_t rows = (int64_t)r.B * r.Nq * r.S;
  if (rows == 0) {
    if (r.present_k.p) return run_concat_present(r, dt, st);
    return SDPA_OK;
  }
  cudaError_t e = launch_decode(r, dt, plan, workspace, st);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  g_kernel = dt == SDPA_F32 ? "decode_splitkv_f32" : dt == SDPA_F16 ? "decode_splitkv_f16" : "decode_splitkv_bf16";
  return SDPA_OK;
}

int sdpa_attn_decode_static(const sdpa_params* p, sdpa_stream_t stream) {
  Problem r;
  Rot rot;
  int rc = validate(p, SDPA_OP_DECODE, &r, &rot);
  if (rc) return rc;
  if (rot.on)
    return fail(SDPA_ERR_UNSUPPORTED, "rotary embedding needs a workspace for the rotated rows; "
                "call sdpa_attn_decode");
  const sdpa_dtype dt = (sdpa_dtype)p->dtype;
  const DecodePlan plan = plan_decode(r.B, r.Nq, r.Nkv, r.S, r.T, r.Hv);
  if (plan.ws_bytes > decode_static_scratch_bytes())
    return fail(SDPA_ERR_WORKSPACE,
                "decode partials need %zu bytes but the built-in scratch holds %zu; "
                "call sdpa_attn_decode with a workspace instead", plan.ws_bytes,
                decode_static_scratch_bytes());
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  g_error.clear();
  const int64_t rows = (int64_t)r.B * r.Nq * r.S;
  if (rows == 0) {
    if (r.present_k.p) return run_concat_present(r, dt, st);
    return SDPA_OK;
  }
  cudaError_t e = launch_decode_static(r, dt, plan, st);
  if (e != cudaSuccess) return cuda_fail(e, "decode (built-in scratch) launch");
  g_kernel = dt == SDPA_F32 ? "decode_splitkv_f32" : dt == SDPA_F16 ? "decode_splitkv_f16" : "decode_splitkv_bf16";
  return SDPA_OK;
}

int sdpa_kv_concat(sdpa_dtype dtype, int32_t B, int32_t N, int32_t P, int32_t L, int32_t D,
                   sdpa_view past, sdpa_view cur, const void* bias, sdpa_view present, sdpa_stream_t stream) {
  if (dtype != SDPA_F32 && dtype != SDPA_F16 && dtype != SDPA_BF16) return fail(SDPA_ERR_INVALID, "dtype %d", dtype);
  if (B < 0 || N < 1 || P < 0 || L < 0 || D < 1) return fail(SDPA_ERR_SHAPE, "bad sizes");
  if (D % vec_elems(dtype) || D > 4096) return fail(SDPA_ERR_UNSUPPORTED, "D must be a multiple of %d, at most 4096", vec_elems(dtype));
  if ((int64_t)P + L > ((int64_t)1 << 31) - 1) return fail(SDPA_ERR_OVERFLOW, "P+L too large");
  if (P > 0 && !past.data) return fail(SDPA_ERR_SHAPE, "P=%d but past is absent", P);
  Extent ep, ec, eo;
  int rc;
  if ((rc = check_view(past, "past", dtype, B, N, P, D, P > 0, false, &ep))) return rc;
  if ((rc = check_view(cur, "cur", dtype, B, N, L, D, true, false, &ec))) return rc;
  if ((rc = check_view(present, "present", dtype, B, N, (int64_t)P + L, D, true, false, &eo))) return rc;
  for (const sdpa_view* v : {&past, &cur, &present})
    if ((rc = check_aligned_view(*v, v == &past ? "past" : v == &cur ? "cur" : "present", dtype))) return rc;
  if (bias && ((uintptr_t)bias & 15u)) return fail(SDPA_ERR_ALIGNMENT, "bias not 16-byte aligned");
  const Extent eb = flat(bias, (size_t)N * D * esize(dtype), "bias");
  if (overlap(eo, ep) || overlap(eo, ec) || overlap(eo, eb))
    return fail(SDPA_ERR_ALIAS, "present overlaps an input");
  g_error.clear();
  auto cv = [](const sdpa_view& v) { return View{v.data, v.stride_b, v.stride_n, v.stride_s}; };
  cudaError_t e = launch_kv_concat(dtype, B, N, P, L, D, cv(past), cv(cur), bias, cv(present),
                                   reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_concat launch");
  g_kernel = "kv_concat";
  return SDPA_OK;
}

int sdpa_rotary(sdpa_dtype dtype, int32_t B, int32_t N, int32_t S, int32_t D, sdpa_view x, sdpa_view y,
                const void* cos_cache, const void* sin_cache, int64_t max_pos, const int64_t* position_ids,
                int32_t rotary_dim, int32_t interleaved, sdpa_stream_t stream) {
  if (dtype != SDPA_F32 && dtype != SDPA_F16 && dtype != SDPA_BF16) return fail(SDPA_ERR_INVALID, "dtype %d", dtype);
  if (B < 0 || S < 0 || N < 1 || D < 2) return fail(SDPA_ERR_SHAPE, "bad sizes (B=%d N=%d S=%d D=%d)", B, N, S, D);
  const int R = rotary_dim ? rotary_dim : D;
  if (R < 2 || R > D || R % 2)
    return fail(SDPA_ERR_INVALID, "rotary_dim %d: must be even and in [2, D=%d] (0 means D)", rotary_dim, D);
  if (interleaved != 0 && interleaved != 1) return fail(SDPA_ERR_INVALID, "interleaved must be 0 or 1");
  if (!cos_cache || !sin_cache) return fail(SDPA_ERR_NULL, "cos_cache / sin_cache is NULL");
  if ((int64_t)B * S == 0) { g_error.clear(); return SDPA_OK; }      // nothing to rotate
  if (((uintptr_t)cos_cache | (uintptr_t)sin_cache) % esize(dtype))
    return fail(SDPA_ERR_ALIGNMENT, "caches not aligned to the element size");
  if ((int64_t)B * N * (int64_t)S > ((int64_t)1 << 40)) return fail(SDPA_ERR_OVERFLOW, "B*N*S too large");
  if (position_ids) {
    if (max_pos < 1 || max_pos > ((int64_t)1 << 40)) return fail(SDPA_ERR_SHAPE, "max_pos %lld", (long long)max_pos);
    if ((uintptr_t)position_ids & 7u) return fail(SDPA_ERR_ALIGNMENT, "position_ids not 8-byte aligned");
  } else if (max_pos != (int64_t)B * S) {
    return fail(SDPA_ERR_SHAPE, "without position_ids the caches are (B, S, R/2): max_pos must be B*S=%lld",
                (long long)B * S);
  }
  Extent ex, ey;
  int rc;
  if ((rc = check_view(x, "x", dtype, B, N, S, D, true, false, &ex))) return rc;
  if ((rc = check_view(y, "y", dtype, B, N, S, D, true, false, &ey))) return rc;
  const bool same = x.data == y.data && x.stride_b == y.stride_b && x.stride_n == y.stride_n &&
                    x.stride_s == y.stride_s;
  const size_t cache_bytes = (size_t)max_pos * (R / 2) * esize(dtype);
  if (!same && overlap(ex, ey)) return fail(SDPA_ERR_ALIAS, "y partially overlaps x");
  if (overlap(ey, flat(cos_cache, cache_bytes, "cos_cache")) || overlap(ey, flat(sin_cache, cache_bytes, "sin_cache")) ||
      overlap(ey, flat(position_ids, (size_t)B * S * 8, "position_ids")))
    return fail(SDPA_ERR_ALIAS, "y overlaps a cache or position_ids");
  g_error.clear();
  auto cv = [](const sdpa_view& v) { return View{v.data, v.stride_b, v.stride_n, v.stride_s}; };
  RotaryPos rp{};
  rp.mode = position_ids ? kRotaryPositionIds : kRotaryPerToken;
  rp.positions = position_ids;
  rp.pos_sb = S;
  rp.max_pos = max_pos;
  rp.cache_ld = R / 2;
  const RotaryJob job{cv(x), cv(y), B, N, S, rp};
  cudaError_t e = launch_rotary(dtype, &job, 1, D, cos_cache, sin_cache, R, interleaved,
                                reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rotary launch");
  g_kernel = "rotary";
  return SDPA_OK;
}

int sdpa_attn_bwd(const sdpa_params* p, sdpa_view dy, sdpa_view dq, sdpa_view dk, sdpa_view dv, void* workspace,
                  size_t workspace_bytes, sdpa_stream_t stream) {
  Problem r;
  Rot rot;
  int rc = validate(p, SDPA_OP_BWD, &r, &rot);
  if (rc) return rc;
  if ((rc = bwd_check(p, r, rot))) return rc;
  const int dt = p->dtype;
  Extent edy, edq, edk, edv;
  if ((rc = check_view(dy, "dy", dt, r.B, r.Nq, r.S, r.Hv, true, false, &edy))) return rc;
  if ((rc = check_view(dq, "dq", dt, r.B, r.Nq, r.S, r.H, true, false, &edq))) return rc;
  if ((rc = check_view(dk, "dk", dt, r.B, r.Nkv, r.T, r.H, true, false, &edk))) return rc;
  if ((rc = check_view(dv, "dv", dt, r.B, r.Nkv, r.T, r.Hv, true, false, &edv))) return rc;
  for (const sdpa_view* v : {&dy, &dq, &dk, &dv})
    if ((rc = check_aligned_view(*v, v == &dy ? "dy" : v == &dq ? "dq" : v == &dk ? "dk" : "dv", dt))) return rc;
  Extent eq, ek, ev, epk, epv;
  check_view(p->q, "q", dt, r.B, r.Nq, r.S, r.H, true, false, &eq);
  check_view(p->k, "k", dt, r.B, r.Nkv, r.L, r.H, true, false, &ek);
  check_view(p->v, "v", dt, r.B, r.Nkv, r.L, r.Hv, true, false, &ev);
  check_view(p->past_k, "past_k", dt, r.B, r.Nkv, r.P, r.H, r.P > 0, false, &epk);
  check_view(p->past_v, "past_v", dt, r.B, r.Nkv, r.P, r.Hv, r.P > 0, false, &epv);
  const Extent ins[] = {eq, ek, ev, epk, epv, edy, flat(p->head_sink, (size_t)r.Nq * esize(dt), "head_sink"),
                        flat(p->lens, (size_t)r.B * (p->len_kind == SDPA_LEN_NONPAD_I64 ? 8 : 4), "lens"),
                        flat(p->q_bias, (size_t)r.Nq * r.H * esize(dt), "q_bias"),
                        flat(p->k_bias, (size_t)r.Nkv * r.H * esize(dt), "k_bias"),
                        flat(p->v_bias, (size_t)r.Nkv * r.Hv * esize(dt), "v_bias")};
  for (const Extent& o : {edq, edk, edv})
    for (const Extent& in : ins)
      if (overlap(o, in)) return fail(SDPA_ERR_ALIAS, "output %s overlaps input %s", o.name, in.name);
  if (overlap(edq, edk) || overlap(edq, edv) || overlap(edk, edv))
    return fail(SDPA_ERR_ALIAS, "outputs dq / dk / dv overlap");
  const BwdWs wl = bwd_layout(r, (sdpa_dtype)dt);
  const size_t need = wl.total;
  if (need && (!workspace || workspace_bytes < need))
    return fail(SDPA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if (need && ((uintptr_t)workspace & 255u)) return fail(SDPA_ERR_ALIGNMENT, "workspace not 256-byte aligned");
  for (const Extent& o : {edq, edk, edv})
    if (need && overlap(flat(workspace, need, "workspace"), o)) return fail(SDPA_ERR_ALIAS, "workspace overlaps an output");
  g_error.clear();
  if ((int64_t)r.B * r.Nq * r.S == 0 && (int64_t)r.B * r.Nkv * r.T == 0) return SDPA_OK;
  auto cv = [](const sdpa_view& v) { return View{v.data, v.stride_b, v.stride_n, v.stride_s}; };
  char* ws = reinterpret_cast<char*>(workspace);
  float* lse2 = reinterpret_cast<float*>(ws + wl.lse2);
  float* delta = reinterpret_cast<float*>(ws + wl.delta);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the rows the scores see: Q + q_bias, and concat(past, new + bias) for K and V
  Problem b = r;
  cudaError_t e = cudaSuccess;
  if (r.q_bias) {
    const View qm{ws + wl.q, (int64_t)r.Nq * r.S * r.H, (int64_t)r.S * r.H, r.H};
    e = launch_kv_concat((sdpa_dtype)dt, r.B, r.Nq, 0, r.S, r.H, View{}, r.q, r.q_bias, qm, st);
    b.q = qm;
    b.q_bias = nullptr;
  }
  if (e == cudaSuccess && bwd_materialise_kv(r)) {
    const View km{ws + wl.k, (int64_t)r.Nkv * r.T * r.H, r.T * r.H, r.H};
    const View vm{ws + wl.v, (int64_t)r.Nkv * r.T * r.Hv, r.T * r.Hv, r.Hv};
    e = launch_kv_concat((sdpa_dtype)dt, r.B, r.Nkv, r.P, r.L, r.H, r.past_k, r.k, r.k_bias, km, st);
    if (e == cudaSuccess) e = launch_kv_concat((sdpa_dtype)dt, r.B, r.Nkv, r.P, r.L, r.Hv, r.past_v, r.v, r.v_bias, vm, st);
    b.k = km; b.v = vm; b.P = 0; b.L = (int)r.T; b.k_bias = nullptr; b.v_bias = nullptr;
    b.past_k = View{}; b.past_v = View{};
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward: materialising the scored rows");
  const char* name = "";
  e = launch_bwd_tc(b, (sdpa_dtype)dt, cv(dy), cv(dq), cv(dk), cv(dv), lse2, delta, st, &name);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  g_kernel = name;
  return SDPA_OK;
}

int sdpa_query_status(sdpa_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int status = 0, rot_status = 0, qk_status = 0, bwd_status = 0;
  e = take_prefill_status(&status);
  if (e == cudaSuccess) e = take_rotary_status(&rot_status);
  if (e == cudaSuccess) e = take_qk_status(&qk_status);
  if (e == cudaSuccess) e = take_bwd_status(&bwd_status);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (!status) status = qk_status;
  if (!status) status = bwd_status;
  // the bounds-checking build: the first failing index check of each kernel family
  int site = 0;
  for (auto take : {take_bounds_prefill, take_bounds_decode, take_bounds_concat, take_bounds_simt}) {
    int v = 0;
    if ((e = take(&v)) != cudaSuccess) return cuda_fail(e, "bounds status read");
    if (!site) site = v;
  }
  if (site) return fail(SDPA_ERR_BOUNDS, "an index check failed at site %d; the access was skipped", site);
  if (status) return fail(SDPA_ERR_TIMEOUT, "a bounded device wait expired (code %d)", status);
  if (rot_status) return fail(SDPA_ERR_INVALID, "a rotary position fell outside its cos/sin cache");
  return SDPA_OK;
}

const char* sdpa_last_error(void) { return g_error.c_str(); }
const char* sdpa_last_kernel_name(void) { return g_kernel; }
int64_t sdpa_launch_count(void) { return (int64_t)g_launches.load(std::memory_order_relaxed); }
const char* sdpa_version(void) { return "sdpa-gb300 0.1 (sm_103a)"; }

}  // extern "C"
