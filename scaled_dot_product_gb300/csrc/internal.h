// Launch functions implemented by the kernel translation units and called by api.cu.
// Each returns cudaSuccess or the launch error; none allocates memory.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "common.cuh"

namespace sdpa {

// Counts one kernel launch (reported by sdpa_launch_count()).
void count_launch(int n = 1);

// General forward (any S): one warp per query row, fp32 arithmetic, reads past and new
// K/V rows in place (projection bias added on the fly).
cudaError_t launch_simt_fwd(const Problem& p, sdpa_dtype dt, cudaStream_t st);

// present = concat(past, cur (+bias)); bit-exact without bias.
cudaError_t launch_kv_concat(sdpa_dtype dt, int B, int N, int P, int L, int D, const View& past,
                             const View& cur, const void* bias, const View& present, cudaStream_t st);

// Rotary embedding: where the cache row of (batch b, row s) comes from.
enum { kRotaryPositionIds = 0, kRotaryPerToken = 1, kRotaryAbsolute = 2 };
struct RotaryPos {
  int mode;
  const int64_t* positions;  // kRotaryPositionIds: positions[b * pos_sb + s]
  int64_t pos_sb;
  int64_t base;              // kRotaryAbsolute: base + s, or lens[b] + 1 - new_rows + s with lens
  const int32_t* lens;
  int new_rows;
  int64_t max_pos;           // rows in the caches
  int64_t cache_ld;          // cache row length (R / 2)
};
// One rotation: (B, N, S, D) view x into y, cache rows chosen by rp.
struct RotaryJob {
  View x, y;
  int B, N, S;
  RotaryPos rp;
};
// njobs (1 or 2) jobs sharing D, the caches, R and the pair layout.
cudaError_t launch_rotary(sdpa_dtype dt, const RotaryJob* jobs, int njobs, int D, const void* cos_c,
                          const void* sin_c, int R, int interleaved, cudaStream_t st);
cudaError_t take_rotary_status(int* status);

// Auxiliary qk output (B, Nq, S, T) fp32 at stage `mode` (0..3).  k_total: one view of all
// T key rows when one exists (enables the tensor-core kernel), else nullptr.
cudaError_t launch_qk(const Problem& p, const View* k_total, const View& out, int mode, sdpa_dtype dt,
                      cudaStream_t st, const char** name);
cudaError_t take_qk_status(int* status);

// Split-KV decode: partials into the workspace, then the merge kernel writes y.
struct DecodePlan {
  int rows_per_cta;     // query rows (group heads x S) handled by one CTA
  int row_groups;       // ceil(group * S / rows_per_cta)
  int nsplit;           // key chunks per (batch, kv head)
  int64_t chunk;        // keys per chunk
  size_t ws_bytes;      // partials: m, l and unnormalised outputs
};
DecodePlan plan_decode(int B, int Nq, int Nkv, int S, int64_t T, int Hv);
cudaError_t launch_decode(const Problem& p, sdpa_dtype dt, const DecodePlan& plan, void* workspace,
                          cudaStream_t st);
bool decode_supported(sdpa_dtype dt, int H, int Hv);

// Backward (tensor cores): statistics pass, then dK/dV and dQ.  lse2 / delta: B*Nq*S floats.
bool bwd_tc_supported(const Problem& p, sdpa_dtype dt);
cudaError_t launch_bwd_tc(const Problem& p, sdpa_dtype dt, const View& dy, const View& dq, const View& dk,
                          const View& dv, float* lse2, float* delta, cudaStream_t st, const char** name);
cudaError_t take_bwd_status(int* status);

// Bounds-checking debug build: the first failing index check of each translation unit
// (its site code; 0 when none), read and cleared.  Always 0 in the normal build.
cudaError_t take_bounds_prefill(int* site);
cudaError_t take_bounds_decode(int* site);
cudaError_t take_bounds_concat(int* site);
cudaError_t take_bounds_simt(int* site);

// Decode with the partials in the library's own device array (no workspace).
size_t decode_static_scratch_bytes();
cudaError_t launch_decode_static(const Problem& p, sdpa_dtype dt, const DecodePlan& plan, cudaStream_t st);

}  // namespace sdpa
