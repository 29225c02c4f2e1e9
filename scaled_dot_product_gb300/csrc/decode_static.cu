// Allocation-free variant of the split-KV decode entry point.
//
// Some callers cannot call cudaMalloc, or any allocating routine, on the path that runs
// attention: a host application or plugin framework that owns the whole device memory
// budget and hands its extensions no allocator, or a latency-critical serving loop where
// cudaMalloc's implicit device-wide synchronisation and its chance of failing under memory
// pressure are not acceptable.  sdpa_attn_decode asks such callers for a workspace;
// this variant needs none: the decode partials live in a fixed device array that is part
// of the library image, reserved on every GPU that loads the library until the process
// exits.
#include <mutex>

#include "internal.h"

namespace sdpa {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;   // 8 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device, looked up once per device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

size_t decode_static_scratch_bytes() { return kStaticScratchBytes; }

cudaError_t launch_decode_static(const Problem& p, sdpa_dtype dt, const DecodePlan& plan, cudaStream_t st) {
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return e;
  // Every (row, chunk) slot the merge kernel reads is written by the split kernel of the
  // same call, so nothing in the array has to start at zero.
  return launch_decode(p, dt, plan, scratch, st);
}

}  // namespace sdpa
