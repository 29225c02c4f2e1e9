// Tensor-core prefill path (placeholder until the tcgen05 kernel lands).
#include "prefill_tc.h"

namespace sdpa {

static __device__ int g_prefill_status;

bool tc_eligible(const Problem&, sdpa_dtype) { return false; }

cudaError_t launch_prefill_tc(const Problem&, sdpa_dtype, cudaStream_t, const char** name) {
  *name = "";
  return cudaErrorNotSupported;
}

cudaError_t take_prefill_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_prefill_status, sizeof v);
  if (e != cudaSuccess) return e;
  *status = v;
  if (v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_prefill_status, &zero, sizeof zero);
  }
  return e;
}

}  // namespace sdpa
