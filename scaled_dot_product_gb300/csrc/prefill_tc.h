// Tensor-core (tcgen05 / TMEM / TMA) prefill path.
#pragma once

#include <cudaTypedefs.h>

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

// Driver entry point of cuTensorMapEncodeTiled (nullptr when unavailable), and the 4-D
// 16-bit map over a (B, N, Seq, D) view the kernels use (box 64 x box_rows rows, 128-byte
// swizzle); ds / dn / db receive the map dimension of seq / head / batch.
PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn();
bool tc_make_map(CUtensorMap* map, const View& v, sdpa_dtype dt, int64_t B, int64_t N, int64_t Sq, int D, int* ds,
                 int* dn, int* db, int box_rows = 128);

// Launches the fused kernel; p.k / p.v must hold all T key rows (P == 0, no kv bias).
cudaError_t launch_prefill_tc(const Problem& p, sdpa_dtype dt, cudaStream_t st, const char** name);

// The same kernel as the statistics pass of the backward: per query row (index
// (b * Nq + h) * S + i) the log2-sum-exp of the scores in units of q.k * scale * log2(e)
// (+inf for a row with nothing admitted) and delta = dY . O, O the normalised output in fp32.
// y is written only when p.y.p is set.  Any rule set but softcap.
cudaError_t launch_prefill_tc_stats(const Problem& p, sdpa_dtype dt, float* lse2, float* delta, const View* dy,
                                    cudaStream_t st, const char** name);

// Reads and clears the device status word the kernel sets when a bounded wait expires.
cudaError_t take_prefill_status(int* status);

}  // namespace sdpa
