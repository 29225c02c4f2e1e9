// present = concat(past, cur) along the sequence axis (onnx-light class Attention:
// past_key/past_value concatenated with K/V into present_key/present_value; MHA: present
// holds P+L positions; GQA: the whole past followed by the current step).
//
// One thread per 16-byte chunk of the output, grid-stride, read-only loads and
// streaming stores.  Without bias the copy is bit-exact; with the MHA projection-bias
// segment the sum is formed in double and rounded once to the element type.
#include "internal.h"

#include <algorithm>

namespace sdpa {
namespace {

template <typename T, bool kBias>
__global__ void __launch_bounds__(256) kv_concat_kernel(View past, View cur, const T* __restrict__ bias,
                                                        View present, int B, int N, int P, int L,
                                                        int D) {
  constexpr int V = Elem<T>::kVec;
  const int chunks_per_row = D / V;
  const int64_t T_total = (int64_t)P + L;
  const int64_t total = (int64_t)B * N * T_total * chunks_per_row;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % chunks_per_row);
    const int64_t row = idx / chunks_per_row;
    const int64_t t = row % T_total;
    const int64_t bn = row / T_total;
    const int n = (int)(bn % N);
    const int b = (int)(bn / N);
    const T* src;
    bool add = false;
    if (t < P) {
      src = reinterpret_cast<const T*>(past.p) + past.off(b, n, t);
    } else {
      src = reinterpret_cast<const T*>(cur.p) + cur.off(b, n, t - P);
      add = kBias;
    }
    if (!SDPA_IN_BOUNDS(t < T_total && b < B && c < chunks_per_row, 301)) continue;
    uint4 u = __ldg(reinterpret_cast<const uint4*>(src) + c);
    if (kBias && add) {
      T* e = reinterpret_cast<T*>(&u);
#pragma unroll
      for (int x = 0; x < V; ++x)
        e[x] = Elem<T>::from_f64(Elem<T>::to_f64(e[x]) + Elem<T>::to_f64(bias[(int64_t)n * D + c * V + x]));
    }
    T* dst = reinterpret_cast<T*>(const_cast<void*>(present.p)) + present.off(b, n, t);
    __stcs(reinterpret_cast<uint4*>(dst) + c, u);
  }
}

template <typename T>
cudaError_t launch_t(int B, int N, int P, int L, int D, const View& past, const View& cur,
                     const void* bias, const View& present, cudaStream_t st) {
  const int64_t total = (int64_t)B * N * ((int64_t)P + L) * (D / Elem<T>::kVec);
  if (total == 0) return cudaSuccess;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (total + 255) / 256;
  const unsigned grid = (unsigned)std::min<int64_t>(want, (int64_t)sms * 16);
  if (bias)
    kv_concat_kernel<T, true><<<grid, 256, 0, st>>>(past, cur, reinterpret_cast<const T*>(bias), present,
                                                    B, N, P, L, D);
  else
    kv_concat_kernel<T, false><<<grid, 256, 0, st>>>(past, cur, nullptr, present, B, N, P, L, D);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kv_concat(sdpa_dtype dt, int B, int N, int P, int L, int D, const View& past,
                             const View& cur, const void* bias, const View& present, cudaStream_t st) {
  switch (dt) {
    case SDPA_F32: return launch_t<float>(B, N, P, L, D, past, cur, bias, present, st);
    case SDPA_F16: return launch_t<__half>(B, N, P, L, D, past, cur, bias, present, st);
    default: return launch_t<__nv_bfloat16>(B, N, P, L, D, past, cur, bias, present, st);
  }
}

SDPA_DEFINE_BOUNDS_TAKE(take_bounds_concat)

}  // namespace sdpa
