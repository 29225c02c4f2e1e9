// Split-KV decode: few query rows per head (S small) against a long key axis.
//
// Semantics are those of onnx-light class Attention / MultiHeadAttention /
// GroupQueryAttention (see sdpa.h); the split itself is this library's design: the key
// axis of each (batch, kv head) is cut into chunks, one CTA per (chunk, kv head, batch,
// row group) scores its chunk for every query row of the group (the grouped query heads
// share one read of K/V), and a merge kernel combines the chunk partials (m, l, o) by
// log-sum-exp together with the head sink.
//
// Memory path: each key row is read as LPK 16-byte vectors by LPK consecutive lanes
// (coalesced, read-only path), two keys per lane group in flight per iteration, and,
// when present outputs are requested, written straight back out with streaming stores,
// so past K/V cross HBM exactly once in each direction.
#include "internal.h"

#include <algorithm>

namespace sdpa {
namespace {

constexpr int kThreads = 128;
constexpr int kUnroll = 2;
constexpr int kTargetCtas = 16 * 152;   // enough CTAs to fill the GPU several times

template <typename T>
__device__ __forceinline__ const uint4* row_vec(const Problem& p, bool value, int b, int kh, int64_t j) {
  const View& v = (j < p.P) ? (value ? p.past_v : p.past_k) : (value ? p.v : p.k);
  const int64_t jj = (j < p.P) ? j : j - p.P;
  return reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(v.p) + v.off(b, kh, jj));
}

template <typename T>
__device__ __forceinline__ void add_bias_round(uint4& u, float* f, const T* bias) {
  // f += bias (float, used for the scores); u = round(f64 sum) (stored to present)
  T* e = reinterpret_cast<T*>(&u);
  constexpr int V = Elem<T>::kVec;
#pragma unroll
  for (int x = 0; x < V; ++x) {
    const double s = Elem<T>::to_f64(e[x]) + Elem<T>::to_f64(bias[x]);
    f[x] = (float)s;
    e[x] = Elem<T>::from_f64(s);
  }
}

template <typename T, int LPK, int R>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const Problem p, const int nsplit,
                                                                const int64_t chunk, const int row_groups,
                                                                float* __restrict__ ws_ml,
                                                                float* __restrict__ ws_o) {
  constexpr int V = Elem<T>::kVec;
  constexpr int KPI = kThreads / LPK;   // keys per CTA per step (one per lane group)
  constexpr int H = LPK * V;            // head size handled (checked by the host)
  extern __shared__ float smem[];       // [KPI][R][H] partial accumulators
  __shared__ float sm_m[KPI][R], sm_l[KPI][R];

  const int split = blockIdx.x;
  const int kh = blockIdx.y / row_groups, rg = blockIdx.y % row_groups;
  const int b = blockIdx.z;
  const int grp = threadIdx.x / LPK, t = threadIdx.x % LPK;
  const int rows_total = p.group * p.S;
  const int r0 = rg * R;
  const int nr = min(R, rows_total - r0);

  float q[R][V];
  int qh[R], qi[R];
  RowCtx ctx[R];
  const T* qb = reinterpret_cast<const T*>(p.q_bias);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int rr = r0 + min(r, nr - 1);
    qh[r] = kh * p.group + rr / p.S;
    qi[r] = rr % p.S;
    ctx[r] = row_ctx(p.r, p.S, p.T, b, qi[r]);
    uint4 u = *(reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.q.p) + p.q.off(b, qh[r], qi[r])) + t);
    unpack16<T>(u, q[r]);
    if (qb) {
#pragma unroll
      for (int e = 0; e < V; ++e) q[r][e] += Elem<T>::to_f32(qb[qh[r] * H + t * V + e]);
    }
  }

  float m[R], l[R], acc[R][V];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -INFINITY; l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < V; ++e) acc[r][e] = 0.f;
  }

  const int64_t j_begin = (int64_t)split * chunk;
  const int64_t j_end = min(p.T, j_begin + chunk);
  const bool write_present = p.present_k.p != nullptr && rg == 0;
  const T* kb = reinterpret_cast<const T*>(p.k_bias);
  const T* vb = reinterpret_cast<const T*>(p.v_bias);

  // every thread runs the same number of steps (the shuffles below need whole warps)
  for (int64_t base = j_begin; base < j_end; base += (int64_t)KPI * kUnroll) {
    uint4 kvec[kUnroll], vvec[kUnroll];
    int64_t jj[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      jj[u] = base + grp + (int64_t)u * KPI;
      kvec[u] = make_uint4(0u, 0u, 0u, 0u);
      vvec[u] = make_uint4(0u, 0u, 0u, 0u);
      if (jj[u] < j_end && SDPA_IN_BOUNDS(jj[u] >= 0 && jj[u] < p.T && t * V < H, 201)) {
        kvec[u] = __ldg(row_vec<T>(p, false, b, kh, jj[u]) + t);
        vvec[u] = __ldg(row_vec<T>(p, true, b, kh, jj[u]) + t);
      }
    }
    float vf[kUnroll][V];
    float s[R][kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const bool valid = jj[u] < j_end;
      float kf[V];
      unpack16<T>(kvec[u], kf);
      unpack16<T>(vvec[u], vf[u]);
      if (valid && jj[u] >= p.P) {
        if (kb) add_bias_round<T>(kvec[u], kf, kb + kh * H + t * V);
        if (vb) add_bias_round<T>(vvec[u], vf[u], vb + kh * H + t * V);
      }
      if (valid && write_present && SDPA_IN_BOUNDS(jj[u] < p.T && kh < p.Nkv, 202)) {
        T* pk = reinterpret_cast<T*>(const_cast<void*>(p.present_k.p)) + p.present_k.off(b, kh, jj[u]);
        T* pv = reinterpret_cast<T*>(const_cast<void*>(p.present_v.p)) + p.present_v.off(b, kh, jj[u]);
        __stcs(reinterpret_cast<uint4*>(pk) + t, kvec[u]);
        __stcs(reinterpret_cast<uint4*>(pv) + t, vvec[u]);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < V; ++e) dot = fmaf(q[r][e], kf[e], dot);
#pragma unroll
        for (int o = LPK / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        s[r][u] = valid ? apply_rules(p.r, ctx[r], dot * p.scale, b, qh[r], qi[r], jj[u]) : -INFINITY;
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float mx = m[r];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) mx = fmaxf(mx, s[r][u]);
      if (mx == -INFINITY) continue;
      const float corr = exp2f((m[r] - mx) * kLog2e);
      l[r] *= corr;
#pragma unroll
      for (int e = 0; e < V; ++e) acc[r][e] *= corr;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const float w = (s[r][u] == -INFINITY) ? 0.f : exp2f((s[r][u] - mx) * kLog2e);
        l[r] += w;
#pragma unroll
        for (int e = 0; e < V; ++e) acc[r][e] = fmaf(w, vf[u][e], acc[r][e]);
      }
      m[r] = mx;
    }
  }

  // merge the lane groups of this CTA
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (t == 0) { sm_m[grp][r] = m[r]; sm_l[grp][r] = l[r]; }
#pragma unroll
    for (int e = 0; e < V; ++e) smem[(grp * R + r) * H + t * V + e] = acc[r][e];
  }
  __syncthreads();
  for (int x = threadIdx.x; x < nr * H; x += kThreads) {
    const int r = x / H, d = x % H;
    float M = -INFINITY;
    for (int g = 0; g < KPI; ++g) M = fmaxf(M, sm_m[g][r]);
    float O = 0.f, Ls = 0.f;
    if (M != -INFINITY) {
      for (int g = 0; g < KPI; ++g) {
        const float mg = sm_m[g][r];
        if (mg == -INFINITY) continue;
        const float w = exp2f((mg - M) * kLog2e);
        O = fmaf(w, smem[(g * R + r) * H + d], O);
        Ls = fmaf(w, sm_l[g][r], Ls);
      }
    }
    const int rr = r0 + r;
    const int h = kh * p.group + rr / p.S, i = rr % p.S;
    const int64_t slot = (((int64_t)b * p.Nq + h) * p.S + i) * nsplit + split;
    if (!SDPA_IN_BOUNDS(h < p.Nq && i < p.S && split < nsplit, 203)) continue;
    ws_o[slot * H + d] = O;
    if (d == 0) { ws_ml[slot * 2] = M; ws_ml[slot * 2 + 1] = Ls; }
  }
}

template <typename T>
__global__ void __launch_bounds__(128) decode_merge_kernel(const Problem p, const int nsplit,
                                                           const float* __restrict__ ws_ml,
                                                           const float* __restrict__ ws_o) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 4 + warp;
  const int64_t nrows = (int64_t)p.B * p.Nq * p.S;
  if (row >= nrows) return;
  const int i = (int)(row % p.S);
  const int h = (int)((row / p.S) % p.Nq);
  const int b = (int)(row / ((int64_t)p.S * p.Nq));
  const float* ml = ws_ml + row * nsplit * 2;
  const float* o = ws_o + row * nsplit * p.Hv;

  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ml[2 * s]);
  float sk = -INFINITY;
  if (p.head_sink) {
    sk = Elem<T>::to_f32(reinterpret_cast<const T*>(p.head_sink)[h]);
    M = fmaxf(M, sk);
  }
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float Ls = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const float ms = ml[2 * s];
      if (ms == -INFINITY) continue;
      const float w = exp2f((ms - M) * kLog2e);
      Ls = fmaf(w, ml[2 * s + 1], Ls);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int d = lane + 32 * e;
        if (d < p.Hv) acc[e] = fmaf(w, o[(int64_t)s * p.Hv + d], acc[e]);
      }
    }
    if (sk != -INFINITY) Ls += exp2f((sk - M) * kLog2e);
  }
  const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
  T* y = reinterpret_cast<T*>(const_cast<void*>(p.y.p)) + p.y.off(b, h, i);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int d = lane + 32 * e;
    if (d < p.Hv) y[d] = Elem<T>::from_f32(acc[e] * inv);
  }
}

template <typename T, int LPK, int R>
cudaError_t launch_split(const Problem& p, const DecodePlan& plan, float* ml, float* o, cudaStream_t st) {
  constexpr int KPI = kThreads / LPK;
  constexpr int H = LPK * Elem<T>::kVec;
  const size_t smem = sizeof(float) * KPI * R * H;
  const dim3 grid(plan.nsplit, p.Nkv * plan.row_groups, p.B);
  decode_split_kernel<T, LPK, R><<<grid, kThreads, smem, st>>>(p, plan.nsplit, plan.chunk, plan.row_groups, ml, o);
  count_launch();
  return cudaGetLastError();
}

template <typename T, int R>
cudaError_t launch_lpk(const Problem& p, const DecodePlan& plan, float* ml, float* o, cudaStream_t st) {
  const int lpk = p.H / Elem<T>::kVec;
  switch (lpk) {
    case 8: return launch_split<T, 8, R>(p, plan, ml, o, st);
    case 16: return launch_split<T, 16, R>(p, plan, ml, o, st);
    default: return launch_split<T, 32, R>(p, plan, ml, o, st);
  }
}

template <typename T>
cudaError_t launch_t(const Problem& p, const DecodePlan& plan, void* ws, cudaStream_t st) {
  const int64_t rows = (int64_t)p.B * p.Nq * p.S;
  float* ml = reinterpret_cast<float*>(ws);
  const size_t ml_bytes = (((size_t)rows * plan.nsplit * 2 * sizeof(float)) + 255) & ~(size_t)255;
  float* o = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + ml_bytes);
  cudaError_t e = (plan.rows_per_cta == 1) ? launch_lpk<T, 1>(p, plan, ml, o, st)
                                           : launch_lpk<T, 4>(p, plan, ml, o, st);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((rows + 3) / 4);
  decode_merge_kernel<T><<<grid, 128, 0, st>>>(p, plan.nsplit, ml, o);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

bool decode_supported(sdpa_dtype dt, int H, int Hv) {
  if (H != Hv) return false;
  const int vec = (dt == SDPA_F32) ? 4 : 8;
  const int lpk = H / vec;
  return H % vec == 0 && (lpk == 8 || lpk == 16 || lpk == 32);
}

DecodePlan plan_decode(int B, int Nq, int Nkv, int S, int64_t T, int Hv) {
  DecodePlan pl{};
  const int group = Nq / Nkv;
  const int rows_total = group * S;
  pl.rows_per_cta = rows_total <= 1 ? 1 : 4;
  pl.row_groups = (rows_total + pl.rows_per_cta - 1) / pl.rows_per_cta;
  const int64_t units = std::max<int64_t>(1, (int64_t)B * Nkv * pl.row_groups);
  const int64_t Tc = std::max<int64_t>(T, 1);
  int64_t nsplit = std::max<int64_t>((Tc + 1023) / 1024,
                                     std::min<int64_t>((Tc + 63) / 64, (kTargetCtas + units - 1) / units));
  nsplit = std::max<int64_t>(1, std::min<int64_t>(nsplit, 65535));
  pl.chunk = (Tc + nsplit - 1) / nsplit;
  pl.nsplit = (int)((Tc + pl.chunk - 1) / pl.chunk);
  const size_t rows = (size_t)B * Nq * S;
  const size_t ml = ((rows * pl.nsplit * 2 * sizeof(float)) + 255) & ~(size_t)255;
  const size_t o = ((rows * pl.nsplit * (size_t)Hv * sizeof(float)) + 255) & ~(size_t)255;
  pl.ws_bytes = rows ? ml + o : 0;
  return pl;
}

cudaError_t launch_decode(const Problem& p, sdpa_dtype dt, const DecodePlan& plan, void* ws, cudaStream_t st) {
  switch (dt) {
    case SDPA_F32: return launch_t<float>(p, plan, ws, st);
    case SDPA_F16: return launch_t<__half>(p, plan, ws, st);
    default: return launch_t<__nv_bfloat16>(p, plan, ws, st);
  }
}

SDPA_DEFINE_BOUNDS_TAKE(take_bounds_decode)

}  // namespace sdpa
