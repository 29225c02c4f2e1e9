// Rotary positional embedding (onnx-light "include_nn_kernels.h", class RotaryEmbedding):
// channel pairs (d, d + R/2) — or (2d, 2d + 1) when interleaved — of the first R channels of
// every head are rotated by the angle whose cosine and sine sit in row `pos` of the caches;
// the other channels are copied.  Used standalone (sdpa_rotary) and, with absolute
// positions, on Q and the new K rows before attention (GroupQueryAttention's rotary).
//
// One thread per rotated pair (plus copy threads for pass-through channels), fp32
// arithmetic, one rounding to the element type.  Memory bound.
#include "internal.h"

#include <algorithm>

namespace sdpa {

static __device__ int g_rotary_status;

namespace {

template <typename T>
__global__ void __launch_bounds__(256) rotary_kernel(const View x, const View y, const T* __restrict__ cos_c,
                                                     const T* __restrict__ sin_c, RotaryPos rp, int B, int N,
                                                     int S, int D, int R, int interleaved) {
  const int half = R / 2;
  const int per_row = half + (D - R);       // rotated pairs + copied channels
  const int64_t total = (int64_t)B * N * S * per_row;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % per_row);
    const int64_t rowi = idx / per_row;
    const int s = (int)(rowi % S);
    const int64_t bn = rowi / S;
    const int n = (int)(bn % N);
    const int b = (int)(bn / N);
    const T* xr = reinterpret_cast<const T*>(x.p) + x.off(b, n, s);
    T* yr = reinterpret_cast<T*>(const_cast<void*>(y.p)) + y.off(b, n, s);
    if (c >= half) {                        // pass-through channel
      const int d = R + (c - half);
      yr[d] = xr[d];
      continue;
    }
    int64_t row;
    if (rp.mode == kRotaryPositionIds) {
      row = rp.positions[(int64_t)b * rp.pos_sb + s];
    } else if (rp.mode == kRotaryPerToken) {
      row = (int64_t)b * S + s;
    } else {                                // absolute: base(b) + s
      int64_t base = rp.base;
      if (rp.lens) base = (int64_t)rp.lens[b] + 1 - rp.new_rows;
      row = base + s;
    }
    if (row < 0 || row >= rp.max_pos) {     // outside the cache: record it, leave a copy
      atomicExch(&g_rotary_status, 1);
      row = row < 0 ? 0 : rp.max_pos - 1;
    }
    const float cs = Elem<T>::to_f32(cos_c[row * rp.cache_ld + c]);
    const float sn = Elem<T>::to_f32(sin_c[row * rp.cache_ld + c]);
    const int i1 = interleaved ? 2 * c : c;
    const int i2 = interleaved ? 2 * c + 1 : c + half;
    const float x1 = Elem<T>::to_f32(xr[i1]), x2 = Elem<T>::to_f32(xr[i2]);
    yr[i1] = Elem<T>::from_f32(fmaf(x1, cs, -x2 * sn));
    yr[i2] = Elem<T>::from_f32(fmaf(x2, cs, x1 * sn));
  }
}

template <typename T>
cudaError_t launch_t(int B, int N, int S, int D, const View& x, const View& y, const void* cos_c, const void* sin_c,
                     const RotaryPos& rp, int R, int interleaved, cudaStream_t st) {
  const int64_t total = (int64_t)B * N * S * (R / 2 + (D - R));
  if (total == 0) return cudaSuccess;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const unsigned grid = (unsigned)std::min<int64_t>((total + 255) / 256, (int64_t)sms * 16);
  rotary_kernel<T><<<grid, 256, 0, st>>>(x, y, reinterpret_cast<const T*>(cos_c), reinterpret_cast<const T*>(sin_c),
                                         rp, B, N, S, D, R, interleaved);
  count_launch(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rotary(sdpa_dtype dt, int B, int N, int S, int D, const View& x, const View& y, const void* cos_c,
                          const void* sin_c, const RotaryPos& rp, int R, int interleaved, cudaStream_t st) {
  switch (dt) {
    case SDPA_F32: return launch_t<float>(B, N, S, D, x, y, cos_c, sin_c, rp, R, interleaved, st);
    case SDPA_F16: return launch_t<__half>(B, N, S, D, x, y, cos_c, sin_c, rp, R, interleaved, st);
    default: return launch_t<__nv_bfloat16>(B, N, S, D, x, y, cos_c, sin_c, rp, R, interleaved, st);
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
