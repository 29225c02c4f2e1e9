// Tensor-core (tcgen05 / TMEM / TMA) prefill path.
#pragma once

#include "common.cuh"

namespace sdpa {

void count_launch(int n);

// True when the problem fits the tensor-core kernel (16-bit types, supported head sizes,
// TMA-compatible alignment).  Pure host function.
bool tc_eligible(const Problem& p, sdpa_dtype dt);

// Order in which the kernel's tensor maps walk the (seq, head, batch) axes of a view
// (ids 0, 1, 2): increasing stride, size-1 axes last.  The K and V views one launch reads
// must share it (tc_same_axis_order).
void tc_axis_order(const View& v, int64_t B, int64_t N, int64_t S, int order[3]);
bool tc_same_axis_order(const View& k, const View& v, int64_t B, int64_t N, int64_t T);

// Launches the fused kernel; p.k / p.v must hold all T key rows (P == 0, no kv bias).
cudaError_t launch_prefill_tc(const Problem& p, sdpa_dtype dt, cudaStream_t st, const char** name);

// Reads and clears the device status word the kernel sets when a bounded wait expires.
cudaError_t take_prefill_status(int* status);

}  // namespace sdpa
