// Rotary positional embedding (onnx-light "include_nn_kernels.h", class RotaryEmbedding):
// channel pairs (d, d + R/2) — or (2d, 2d + 1) when interleaved — of the first R channels of
// every head are rotated by the angle whose cosine and sine sit in row `pos` of the caches;
// the other channels are copied.  Used standalone (sdpa_rotary) and, with absolute
// positions, on Q and the new K rows before attention (GroupQueryAttention's rotary).
//
// Memory bound: every element is read and written once, the cache rows come from L2.
// The main kernel moves 16-byte vectors: one thread rotates V = 16 / sizeof(T) pairs (the
// split layout: a vector of the first half and its partner vector R/2 further on; the
// interleaved layout: one vector holding V/2 adjacent pairs) or copies one pass-through
// vector.  Up to two jobs (Q and the new K rows) share one launch.  Shapes or pointers that
// do not allow 16-byte vectors take the scalar kernel (one thread per pair).  Both compute
// x1 c - x2 s and x2 c + x1 s in fp32 with the same operation order, so they agree bit for
// bit, and round once to the element type.
#include "internal.h"

#include <algorithm>

namespace sdpa {

static __device__ int g_rotary_status;

namespace {

// Cache row of (b, s) for a job; rows outside [0, max_pos) are recorded and clamped, so the
// cache reads stay in bounds.
__device__ __forceinline__ int64_t cache_row(const RotaryPos& rp, int b, int s, int S) {
  int64_t row;
  if (rp.mode == kRotaryPositionIds) {
    row = rp.positions[(int64_t)b * rp.pos_sb + s];
  } else if (rp.mode == kRotaryPerToken) {
    row = (int64_t)b * S + s;
  } else {                                  // absolute: base(b) + s
    const int64_t base = rp.lens ? (int64_t)rp.lens[b] + 1 - rp.new_rows : rp.base;
    row = base + s;
  }
  if (row < 0 || row >= rp.max_pos) {
    atomicExch(&g_rotary_status, 1);
    row = row < 0 ? 0 : rp.max_pos - 1;
  }
  return row;
}

__device__ __forceinline__ void rot2(float x1, float x2, float c, float s, float& o1, float& o2) {
  o1 = fmaf(x1, c, -x2 * s);
  o2 = fmaf(x2, c, x1 * s);
}

// ---------------------------------------------------------------- scalar kernel

template <typename T>
__global__ void __launch_bounds__(256) rotary_scalar_kernel(const RotaryJob j, const T* __restrict__ cos_c,
                                                            const T* __restrict__ sin_c, int D, int R,
                                                            int interleaved) {
  const int half = R / 2;
  const int per_row = half + (D - R);       // rotated pairs + copied channels
  const int64_t total = (int64_t)j.B * j.N * j.S * per_row;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % per_row);
    const int64_t rowi = idx / per_row;
    const int s = (int)(rowi % j.S);
    const int64_t bn = rowi / j.S;
    const int n = (int)(bn % j.N);
    const int b = (int)(bn / j.N);
    const T* xr = reinterpret_cast<const T*>(j.x.p) + j.x.off(b, n, s);
    T* yr = reinterpret_cast<T*>(const_cast<void*>(j.y.p)) + j.y.off(b, n, s);
    if (c >= half) {                        // pass-through channel
      const int d = R + (c - half);
      yr[d] = xr[d];
      continue;
    }
    const int64_t row = cache_row(j.rp, b, s, j.S);
    const float cs = Elem<T>::to_f32(cos_c[row * j.rp.cache_ld + c]);
    const float sn = Elem<T>::to_f32(sin_c[row * j.rp.cache_ld + c]);
    const int i1 = interleaved ? 2 * c : c;
    const int i2 = interleaved ? 2 * c + 1 : c + half;
    float o1, o2;
    rot2(Elem<T>::to_f32(xr[i1]), Elem<T>::to_f32(xr[i2]), cs, sn, o1, o2);
    yr[i1] = Elem<T>::from_f32(o1);
    yr[i2] = Elem<T>::from_f32(o2);
  }
}

// ---------------------------------------------------------------- 16-byte vector kernel

template <typename T, int N>
struct alignas(N * sizeof(T)) Pack { T v[N]; };

// One unit of a job: unit -> (row, u); u < urot rotates, the rest copy one vector.
template <typename T, bool kInter>
__device__ __forceinline__ void rotary_unit(const RotaryJob& j, int64_t unit, int urot, int units_per_row,
                                            const T* __restrict__ cos_c, const T* __restrict__ sin_c, int R,
                                            bool small) {
  constexpr int V = 16 / (int)sizeof(T);
  int64_t row;
  int u, s, n, b;
  if (small) {                              // 32-bit index arithmetic
    const uint32_t un = (uint32_t)unit, upr = (uint32_t)units_per_row;
    const uint32_t r32 = un / upr;
    u = (int)(un - r32 * upr);
    const uint32_t bn = r32 / (uint32_t)j.S;
    s = (int)(r32 - bn * (uint32_t)j.S);
    b = (int)(bn / (uint32_t)j.N);
    n = (int)(bn - (uint32_t)b * (uint32_t)j.N);
    row = r32;
  } else {
    row = unit / units_per_row;
    u = (int)(unit - row * units_per_row);
    const int64_t bn = row / j.S;
    s = (int)(row - bn * j.S);
    b = (int)(bn / j.N);
    n = (int)(bn - (int64_t)b * j.N);
  }
  const T* xr = reinterpret_cast<const T*>(j.x.p) + j.x.off(b, n, s);
  T* yr = reinterpret_cast<T*>(const_cast<void*>(j.y.p)) + j.y.off(b, n, s);
  if (u >= urot) {                          // pass-through vector
    const int c = R + (u - urot) * V;
    *reinterpret_cast<uint4*>(yr + c) = *reinterpret_cast<const uint4*>(xr + c);
    return;
  }
  const int64_t crow = cache_row(j.rp, b, s, j.S) * j.rp.cache_ld;
  if (!kInter) {
    const int c0 = u * V, c1 = c0 + R / 2;
    const Pack<T, V> a = *reinterpret_cast<const Pack<T, V>*>(xr + c0);
    const Pack<T, V> p = *reinterpret_cast<const Pack<T, V>*>(xr + c1);
    const Pack<T, V> cs = *reinterpret_cast<const Pack<T, V>*>(cos_c + crow + c0);
    const Pack<T, V> sn = *reinterpret_cast<const Pack<T, V>*>(sin_c + crow + c0);
    Pack<T, V> o1, o2;
#pragma unroll
    for (int e = 0; e < V; ++e) {
      float r1, r2;
      rot2(Elem<T>::to_f32(a.v[e]), Elem<T>::to_f32(p.v[e]), Elem<T>::to_f32(cs.v[e]), Elem<T>::to_f32(sn.v[e]),
           r1, r2);
      o1.v[e] = Elem<T>::from_f32(r1);
      o2.v[e] = Elem<T>::from_f32(r2);
    }
    *reinterpret_cast<Pack<T, V>*>(yr + c0) = o1;
    *reinterpret_cast<Pack<T, V>*>(yr + c1) = o2;
  } else {
    const int c0 = u * V;
    const Pack<T, V> a = *reinterpret_cast<const Pack<T, V>*>(xr + c0);
    const Pack<T, V / 2> cs = *reinterpret_cast<const Pack<T, V / 2>*>(cos_c + crow + c0 / 2);
    const Pack<T, V / 2> sn = *reinterpret_cast<const Pack<T, V / 2>*>(sin_c + crow + c0 / 2);
    Pack<T, V> o;
#pragma unroll
    for (int e = 0; e < V / 2; ++e) {
      float r1, r2;
      rot2(Elem<T>::to_f32(a.v[2 * e]), Elem<T>::to_f32(a.v[2 * e + 1]), Elem<T>::to_f32(cs.v[e]),
           Elem<T>::to_f32(sn.v[e]), r1, r2);
      o.v[2 * e] = Elem<T>::from_f32(r1);
      o.v[2 * e + 1] = Elem<T>::from_f32(r2);
    }
    *reinterpret_cast<Pack<T, V>*>(yr + c0) = o;
  }
}

template <typename T, bool kInter>
__global__ void __launch_bounds__(256) rotary_vec_kernel(const RotaryJob j0, const RotaryJob j1, int64_t units0,
                                                         int64_t units1, int urot, int units_per_row,
                                                         const T* __restrict__ cos_c, const T* __restrict__ sin_c,
                                                         int R) {
  const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (unit < units0) {
    rotary_unit<T, kInter>(j0, unit, urot, units_per_row, cos_c, sin_c, R, units0 < ((int64_t)1 << 31));
  } else if (unit - units0 < units1) {
    rotary_unit<T, kInter>(j1, unit - units0, urot, units_per_row, cos_c, sin_c, R, units1 < ((int64_t)1 << 31));
  }
}

bool view_vec_ok(const View& v, int V) {
  return ((uintptr_t)v.p & 15u) == 0 && v.sb % V == 0 && v.sh % V == 0 && v.ss % V == 0;
}

template <typename T>
cudaError_t launch_t(const RotaryJob* jobs, int njobs, int D, const void* cos_c, const void* sin_c, int R,
                     int interleaved, cudaStream_t st) {
  constexpr int V = 16 / (int)sizeof(T);
  const int64_t ld = jobs[0].rp.cache_ld;
  bool vec = D % V == 0 && (interleaved ? R % V == 0 : (R / 2) % V == 0);
  const unsigned cache_align = interleaved ? 8u : 16u;
  vec = vec && (((uintptr_t)cos_c | (uintptr_t)sin_c) & (cache_align - 1)) == 0 &&
        ld % (interleaved ? V / 2 : V) == 0;
  for (int i = 0; i < njobs; ++i) vec = vec && view_vec_ok(jobs[i].x, V) && view_vec_ok(jobs[i].y, V);
  const T* cp = reinterpret_cast<const T*>(cos_c);
  const T* sp = reinterpret_cast<const T*>(sin_c);
  const int urot = interleaved ? R / V : R / (2 * V);
  const int upr = urot + (D - R) / V;
  int64_t units[2] = {0, 0};
  for (int i = 0; i < njobs; ++i) units[i] = (int64_t)jobs[i].B * jobs[i].N * jobs[i].S * upr;
  const int64_t total = units[0] + units[1];
  vec = vec && (total + 255) / 256 <= 0x7fffffffLL;            // one unit per thread
  if (vec) {
    if (total == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((total + 255) / 256);
    const RotaryJob& j1 = njobs > 1 ? jobs[1] : jobs[0];
    if (interleaved)
      rotary_vec_kernel<T, true><<<grid, 256, 0, st>>>(jobs[0], j1, units[0], units[1], urot, upr, cp, sp, R);
    else
      rotary_vec_kernel<T, false><<<grid, 256, 0, st>>>(jobs[0], j1, units[0], units[1], urot, upr, cp, sp, R);
    count_launch(1);
    return cudaGetLastError();
  }
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  for (int i = 0; i < njobs; ++i) {
    const RotaryJob& j = jobs[i];
    const int64_t total = (int64_t)j.B * j.N * j.S * (R / 2 + (D - R));
    if (total == 0) continue;
    const unsigned grid = (unsigned)std::min<int64_t>((total + 255) / 256, (int64_t)sms * 16);
    rotary_scalar_kernel<T><<<grid, 256, 0, st>>>(j, cp, sp, D, R, interleaved);
    count_launch(1);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_rotary(sdpa_dtype dt, const RotaryJob* jobs, int njobs, int D, const void* cos_c,
                          const void* sin_c, int R, int interleaved, cudaStream_t st) {
  switch (dt) {
    case SDPA_F32: return launch_t<float>(jobs, njobs, D, cos_c, sin_c, R, interleaved, st);
    case SDPA_F16: return launch_t<__half>(jobs, njobs, D, cos_c, sin_c, R, interleaved, st);
    default: return launch_t<__nv_bfloat16>(jobs, njobs, D, cos_c, sin_c, R, interleaved, st);
  }
}

cudaError_t take_rotary_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_rotary_status, sizeof v);
  if (e != cudaSuccess) return e;
  *status = v;
  if (v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_rotary_status, &zero, sizeof zero);
  }
  return e;
}

}  // namespace sdpa
