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
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace sdpa {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;   // 8 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_setup_mutex;
struct ScratchSlot {
  CUcontext ctx;   // the context the address belongs to
  void* ptr;
};
ScratchSlot g_scratch[kMaxDevices] = {};

// The driver's cuCtxGetCurrent, reached through the runtime (the library links no driver
// library); nullptr when unavailable.
PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  return fn;
}

// Device address of g_decode_scratch on the current device, looked up the first time the
// device is used and again whenever its context has changed since (after cudaDeviceReset
// the module is loaded anew and the array may sit elsewhere).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  ScratchSlot& slot = g_scratch[dev];
  CUcontext ctx = nullptr;
  auto get_ctx = ctx_get_current();
  if (slot.ptr && get_ctx && get_ctx(&ctx) == CUDA_SUCCESS && ctx == slot.ctx) {
    *out = slot.ptr;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_decode_scratch);   // also makes the device's context current
  if (e != cudaSuccess) return e;
  ctx = nullptr;
  if (get_ctx && get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  slot.ctx = ctx;
  slot.ptr = ctx ? p : nullptr;   // without a context handle, look the address up every call
  *out = p;
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
