// General-purpose forward kernel: one warp per query row, fp32 arithmetic throughout.
//
// It evaluates the definition of onnx-light "include_nn_kernels.h", class Attention
// (Y = Softmax(Q K^T * scale + bias) V) with every rule of the MultiHeadAttention and
// GroupQueryAttention contracts, as an online softmax over tiles of 32 keys: lane l scores
// key j0 + l, the warp takes the tile maximum, rescales its running sum and accumulator,
// then accumulates the tile's weighted value rows with each lane owning Hv/32 output
// columns.  It serves fp32 problems (where tensor-core tf32 would miss a 1e-4 bound) and
// shapes the tensor-core path does not tile.
#include "internal.h"

namespace sdpa {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxAccPerLane = 8;   // Hv <= 256

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename T>
__device__ __forceinline__ const T* kv_row(const Problem& p, bool value, int b, int kh, int64_t j) {
  if (j < p.P) {
    const View& v = value ? p.past_v : p.past_k;
    return reinterpret_cast<const T*>(v.p) + v.off(b, kh, j);
  }
  const View& v = value ? p.v : p.k;
  return reinterpret_cast<const T*>(v.p) + v.off(b, kh, j - p.P);
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) simt_fwd_kernel(const Problem p) {
  extern __shared__ float q_smem[];  // kWarps x H
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t nrows = (int64_t)p.B * p.Nq * p.S;
  if (row >= nrows) return;            // warp-uniform; no block-wide barrier follows
  const int i = (int)(row % p.S);
  const int h = (int)((row / p.S) % p.Nq);
  const int b = (int)(row / ((int64_t)p.S * p.Nq));
  const int kh = h / p.group;
  constexpr int V = Elem<T>::kVec;

  float* qs = q_smem + warp * p.H;
  const T* qrow = reinterpret_cast<const T*>(p.q.p) + p.q.off(b, h, i);
  const T* qb = reinterpret_cast<const T*>(p.q_bias);
  for (int d = lane; d < p.H; d += 32)
    qs[d] = Elem<T>::to_f32(qrow[d]) + (qb ? Elem<T>::to_f32(qb[h * p.H + d]) : 0.f);
  __syncwarp();

  const RowCtx ctx = row_ctx(p.r, p.S, p.T, b, i);
  const T* kb = reinterpret_cast<const T*>(p.k_bias);
  const T* vb = reinterpret_cast<const T*>(p.v_bias);

  float m = -INFINITY, l = 0.f;
  float acc[kMaxAccPerLane];
#pragma unroll
  for (int e = 0; e < kMaxAccPerLane; ++e) acc[e] = 0.f;

  for (int64_t j0 = 0; j0 < p.T; j0 += 32) {
    const int64_t j = j0 + lane;
    float s = -INFINITY;
    if (j < p.T && SDPA_IN_BOUNDS(j >= 0 && kh < p.Nkv && i < p.S, 401)) {
      const T* krow = kv_row<T>(p, false, b, kh, j);
      const bool add_bias = kb && j >= p.P;
      float dot = 0.f;
      for (int d = 0; d < p.H; d += V) {
        float f[V];
        unpack16<T>(*reinterpret_cast<const uint4*>(krow + d), f);
#pragma unroll
        for (int e = 0; e < V; ++e) {
          const float kv = add_bias ? f[e] + Elem<T>::to_f32(kb[kh * p.H + d + e]) : f[e];
          dot = fmaf(qs[d + e], kv, dot);
        }
      }
      s = apply_rules(p.r, ctx, dot * p.scale, b, h, i, j);
    }
    const float m_new = fmaxf(m, warp_max(s));
    if (m_new == -INFINITY) continue;                   // nothing admitted so far (uniform)
    const float corr = exp2f((m - m_new) * kLog2e);     // 0 when m is still -inf
    const float pj = (s == -INFINITY) ? 0.f : exp2f((s - m_new) * kLog2e);
    l = l * corr + warp_sum(pj);
#pragma unroll
    for (int e = 0; e < kMaxAccPerLane; ++e) acc[e] *= corr;
    const int nk = (int)(p.T - j0 < 32 ? p.T - j0 : 32);
    for (int jj = 0; jj < nk; ++jj) {
      const float w = __shfl_sync(0xffffffffu, pj, jj);
      if (w == 0.f) continue;                           // uniform across the warp
      const int64_t jv = j0 + jj;
      if (!SDPA_IN_BOUNDS(jv < p.T, 402)) continue;
      const T* vrow = kv_row<T>(p, true, b, kh, jv);
      const bool add_bias = vb && jv >= p.P;
#pragma unroll
      for (int e = 0; e < kMaxAccPerLane; ++e) {
        const int d = lane + 32 * e;
        if (d < p.Hv) {
          float x = Elem<T>::to_f32(vrow[d]);
          if (add_bias) x += Elem<T>::to_f32(vb[kh * p.Hv + d]);
          acc[e] = fmaf(w, x, acc[e]);
        }
      }
    }
    m = m_new;
  }

  if (p.head_sink) {
    const float sk = Elem<T>::to_f32(reinterpret_cast<const T*>(p.head_sink)[h]);
    const float m_new = fmaxf(m, sk);
    if (m_new != -INFINITY) {
      const float corr = exp2f((m - m_new) * kLog2e);
      l = l * corr + exp2f((sk - m_new) * kLog2e);
#pragma unroll
      for (int e = 0; e < kMaxAccPerLane; ++e) acc[e] *= corr;
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  T* yrow = reinterpret_cast<T*>(const_cast<void*>(p.y.p)) + p.y.off(b, h, i);
#pragma unroll
  for (int e = 0; e < kMaxAccPerLane; ++e) {
    const int d = lane + 32 * e;
    if (d < p.Hv) yrow[d] = Elem<T>::from_f32(acc[e] * inv);
  }
}

}  // namespace

cudaError_t launch_simt_fwd(const Problem& p, sdpa_dtype dt, cudaStream_t st) {
  const int64_t nrows = (int64_t)p.B * p.Nq * p.S;
  if (nrows == 0) return cudaSuccess;
  const dim3 grid((unsigned)((nrows + kWarps - 1) / kWarps));
  const size_t smem = sizeof(float) * kWarps * p.H;
  switch (dt) {
    case SDPA_F32: simt_fwd_kernel<float><<<grid, kWarps * 32, smem, st>>>(p); break;
    case SDPA_F16: simt_fwd_kernel<__half><<<grid, kWarps * 32, smem, st>>>(p); break;
    default: simt_fwd_kernel<__nv_bfloat16><<<grid, kWarps * 32, smem, st>>>(p); break;
  }
  count_launch();
  return cudaGetLastError();
}

SDPA_DEFINE_BOUNDS_TAKE(take_bounds_simt)

}  // namespace sdpa
