// Auxiliary qk output of onnx-light "include_nn_kernels.h", class Attention (attribute
// qk_matmul_output_mode): the FLOAT tensor (B, Nq, S, T) of one stage of the scores --
//   0  scale * Q K^T
//   1  with the additive bias and the masks (an excluded key reads -inf)
//   2  after softcap: the logits the softmax sees
//   3  the softmax probabilities, the sink in the denominator (an excluded key reads 0)
//
// Tensor-core kernel (16-bit inputs, H = 64 or 128, one K view of all T rows): one CTA per
// 128-row query tile of one (batch, head), streaming every key tile of its kv head.
//   warp 0     TMA producer: Q once, then K_0, K_1, ... through a shared-memory ring
//   warp 1     MMA issuer: S_j = Q K_j^T into one of two tensor-memory buffers
//   warps 2-17 epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. (its 32 query
//              rows) and owns one 32-key column chunk (w - 2) / 4 of every tile; each
//              thread turns its row's 32 products into the requested stage, writes them to
//              a shared-memory slot in the 128-byte swizzle, and lane 0 stores the 32 x 32
//              block with a TMA store (clipped at S and T by the tensor map)
// Stage 3 runs the key tiles twice: the first pass gathers each row's maximum and sum
// (per chunk, combined through shared memory), the second writes the probabilities.
// The output write bounds the kernel (HBM).  Rules that are key intervals (causal,
// window, lengths) plus an additive mask take a per-row fast path; boolean / filter masks
// and key-padding filter values go through the general rule function.
//
// General kernel (every other case): one warp per query row, lane l on key j0 + l.
//
// Every barrier wait is bounded; on expiry the tensor-core kernel drains what it issued,
// frees its tensor memory and records SDPA_ERR_TIMEOUT for sdpa_query_status.
#include <algorithm>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "prefill_tc.h"
#include "tc_ptx.cuh"

namespace sdpa {

static __device__ int g_qk_status;

namespace {

using namespace ptx;

constexpr int kRows = 128;          // query rows per CTA (tensor-memory lanes)
constexpr int kKeys = 128;          // keys per tile
constexpr int kEpiWarps = 16;       // 4 lane quarters x 4 column chunks
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kOutBufs = 2;         // staging slots per epilogue warp
constexpr int kOutSlot = 32 * 32 * 4;   // 32 rows x 32 fp32 (128-byte swizzle)
constexpr uint64_t kDrainNs = 2000000000ull;

template <int H>
struct QkCfg {
  static constexpr int kRegions = H / 64;
  static constexpr int kRegionBytes = 128 * 128;
  static constexpr int kTile = 128 * H * 2;
  static constexpr int kStages = (H == 128) ? 2 : 4;
  static constexpr int kKOff = kTile;
  static constexpr int kOutOff = kKOff + kStages * kTile;
  static constexpr int kSmem = kOutOff + kEpiWarps * kOutBufs * kOutSlot + 1024;   // + alignment slack
  static_assert(kSmem + 512 <= 227 * 1024, "shared memory (dynamic + static)");
  static constexpr uint32_t kTmemCols = 256;
};

struct QkArgs {
  int B, Nq, Nkv, S, T, group, mode, q_tiles;
  float scale;
  Rules r;          // every rule, softcap included (stages 2 and 3)
  Rules r1;         // the same rules without softcap (stage 1)
  int q_ds, q_dn, q_db, k_ds, k_dn, k_db, o_ds, o_dn, o_db;
  const void* head_sink;
  int fast;         // rules are key intervals plus at most an additive mask
  uint64_t wait_ns;
};

__device__ __forceinline__ void perm3(int ds, int dn, int db, int s, int n, int b, int& c1, int& c2, int& c3) {
  c1 = ds == 1 ? s : (dn == 1 ? n : b);
  c2 = ds == 2 ? s : (dn == 2 ? n : b);
  c3 = ds == 3 ? s : (dn == 3 ? n : b);
}

// Stage value of one product; -inf marks an excluded key from stage 1 on.
__device__ __forceinline__ float stage_value(int mode, const Rules& r, const Rules& r1, const RowCtx& ctx,
                                             float raw, int b, int h, int i, int64_t j) {
  if (mode == 0) return raw;
  return apply_rules(mode == 1 ? r1 : r, ctx, raw, b, h, i, j);
}

__device__ __noinline__ float generic_stage(const Rules& r, const RowCtx& ctx, float raw, int b, int h, int i,
                                            int64_t j) {
  return apply_rules(r, ctx, raw, b, h, i, j);
}

// tanh(x) = sign(x) (1 - 2 / (e^{2|x|} + 1)): absolute error a few 1e-7 (the exponential's
// relative error and the final subtraction), far inside the qk output's bound even after
// the softcap amplitude multiplies it.
__device__ __forceinline__ float tanh_exp(float x) {
  const float e = ex2_approx(fabsf(x) * (2.f * kLog2e));
  return copysignf(1.f - __fdividef(2.f, e + 1.f), x);
}

template <typename T>
__device__ __forceinline__ float sink_of(const void* sink, int h) {
  return Elem<T>::to_f32(reinterpret_cast<const T*>(sink)[h]);
}

template <int H, bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
    qk_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap to, const QkArgs a) {
  using C = QkCfg<H>;
  using T = typename std::conditional<kBF16, __nv_bfloat16, __half>::type;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_q, bar_drain;
  __shared__ __align__(8) uint64_t bar_full[C::kStages], bar_empty[C::kStages];
  __shared__ __align__(8) uint64_t bar_sfull[2], bar_sfree[2], bar_red[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int t = blockIdx.x;
  const int qt = t % a.q_tiles; t /= a.q_tiles;
  const int h = t % a.Nq; t /= a.Nq;
  const int b = t;
  const int kvh = h / a.group;
  const int m0 = qt * kRows;
  const int nT = (a.T + kKeys - 1) / kKeys;
  const int nit = (a.mode == 3 ? 2 : 1) * nT;      // MMA tiles issued

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase, sK = sbase + C::kKOff, sOut = sbase + C::kOutOff;
  const uint32_t b_q = smem_u32(&bar_q), b_drain = smem_u32(&bar_drain);
  auto b_full = [&](int s) { return smem_u32(&bar_full[s]); };
  auto b_empty = [&](int s) { return smem_u32(&bar_empty[s]); };
  auto b_sfull = [&](int x) { return smem_u32(&bar_sfull[x]); };
  auto b_sfree = [&](int x) { return smem_u32(&bar_sfree[x]); };
  volatile int* abortp = &abort_flag;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(b_q, 1);
    mbar_init(b_drain, 1);
    for (int s = 0; s < C::kStages; ++s) { mbar_init(b_full(s), 1); mbar_init(b_empty(s), 1); }
    for (int x = 0; x < 2; ++x) {
      mbar_init(b_sfull(x), 1);
      mbar_init(b_sfree(x), 32 * kEpiWarps);
      mbar_init(smem_u32(&bar_red[x]), 32 * kEpiWarps);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ================================================================ TMA producer
    if (nit > 0) {
      const uint32_t leader = elect_one();   // issues every copy, MMA and commit of the warp
      if (leader) prefetch_tmap(&tq);
      if (leader) prefetch_tmap(&tk);
      int c1, c2, c3;
      if (leader) mbar_arrive_expect_tx(b_q, C::kTile);
      perm3(a.q_ds, a.q_dn, a.q_db, m0, h, b, c1, c2, c3);
      for (int r = 0; r < C::kRegions; ++r) if (leader) tma_load_4d(sQ + r * C::kRegionBytes, &tq, b_q, 64 * r, c1, c2, c3);
      int issued = 0;
      bool ok = true;
      for (int it = 0; it < nit && ok; ++it) {
        const int st = it % C::kStages;
        if (it >= C::kStages &&
            !(ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_empty(st), ((it / C::kStages) - 1) & 1, abortp, a.wait_ns))))
          break;
        if (leader) mbar_arrive_expect_tx(b_full(st), C::kTile);
        perm3(a.k_ds, a.k_dn, a.k_db, (it % nT) * kKeys, kvh, b, c1, c2, c3);
        for (int r = 0; r < C::kRegions; ++r)
          if (leader) tma_load_4d(sK + st * C::kTile + r * C::kRegionBytes, &tk, b_full(st), 64 * r, c1, c2, c3);
        ++issued;
      }
      if (__any_sync(0xffffffffu, !ok || *abortp)) {
        // some role gave up: let every copy already issued land before the CTA can exit
        mbar_wait_bounded(b_q, 0, nullptr, kDrainNs);
        for (int s = 0; s < C::kStages && s < issued; ++s) {
          const int last = s + ((issued - 1 - s) / C::kStages) * C::kStages;
          mbar_wait_bounded(b_full(s), (last / C::kStages) & 1, nullptr, kDrainNs);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (nit > 0) {
      const uint32_t leader = elect_one();   // issues every copy, MMA and commit of the warp
      constexpr uint32_t kId = idesc_f16(kBF16, kRows, kKeys, false);
      const uint64_t dQ = desc_sw128(sQ, 16, 1024);
      const uint64_t dK0 = desc_sw128(sK, 16, 1024);
      bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_q, 0, abortp, a.wait_ns));
      tc_fence_after();
      for (int it = 0; it < nit && ok; ++it) {
        const int buf = it & 1, st = it % C::kStages;
        if (it >= 2) {
          if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_sfree(buf), ((it >> 1) - 1) & 1, abortp, a.wait_ns)))) break;
          tc_fence_after();
        }
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_full(st), (it / C::kStages) & 1, abortp, a.wait_ns)))) break;
        tc_fence_after();
        const uint64_t dk = dK0 + (uint64_t)((st * C::kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < H / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk / 4) * C::kRegionBytes + (kk % 4) * 32) >> 4);
          if (leader) mma_f16_ss(tmem + buf * kKeys, dQ + off, dk + off, kId, kk > 0);
        }
        if (leader) mma_commit(b_sfull(buf));
        if (leader) mma_commit(b_empty(st));
      }
      // every MMA this thread issued completes before the CTA frees its tensor memory
      if (leader) mma_commit(b_drain);
      mbar_wait_bounded(b_drain, 0, nullptr, kDrainNs);
    }
    __syncwarp();
  } else {
    // ================================================================ epilogue warps
    const int quarter = warp & 3;                    // tensor-memory lanes 32*quarter ..
    const int chunk = (warp - 2) >> 2;               // key columns 32*chunk .. of each tile
    const int row = quarter * 32 + lane;
    const int i = m0 + row;
    const bool valid = i < a.S;
    const RowCtx ctx = row_ctx(a.r, a.S, a.T, b, valid ? i : 0);
    // admitted key interval of the row under the interval rules
    int64_t lo = 0, hi = (int64_t)a.T - 1;
    if (a.r.causal != SDPA_CAUSAL_NONE) hi = min(hi, ctx.pos);
    if (a.r.window > 0) lo = max(lo, ctx.pos - a.r.window + 1);
    if (a.r.len_kind == SDPA_LEN_NONPAD_I64) hi = min(hi, ctx.len - 1);
    if (a.r.len_kind == SDPA_LEN_SEQLENS_K_I32) hi = min(hi, ctx.len);
    const void* mrow = nullptr;
    if (a.r.add && valid) {
      const int esz = a.r.add_dtype == SDPA_F32 ? 4 : 2;
      mrow = reinterpret_cast<const char*>(a.r.add) +
             ((int64_t)b * a.r.add_sb + (int64_t)h * a.r.add_sh + (int64_t)i * a.r.add_ss) * esz;
    }
    const float cap = a.r.softcap, cap_inv = cap > 0.f ? 1.f / cap : 0.f;
    const uint32_t tcol = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)chunk * 32;
    const uint32_t slots = sOut + (uint32_t)(warp - 2) * kOutBufs * kOutSlot;
    const bool warp_rows = m0 + quarter * 32 < a.S;  // some row of this warp is in the output
    int os1, os2, os3;
    perm3(a.o_ds, a.o_dn, a.o_db, m0 + quarter * 32, h, b, os1, os2, os3);
    float m_run = -INFINITY, l_run = 0.f;            // stage 3, first pass (log2 domain)
    float m_fin = -INFINITY, inv_l = 0.f;            // stage 3, second pass
    int nstore = 0;
    bool ok = true;
    for (int it = 0; it < nit && ok; ++it) {
      const int buf = it & 1;
      const int j = it % nT;
      const bool gather = a.mode == 3 && it < nT;    // stage 3, first pass: statistics only
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_sfull(buf), (it >> 1) & 1, abortp, a.wait_ns))))
        break;
      tc_fence_after();
      uint32_t u[32];
      tmem_ld32(tcol + buf * kKeys, u);
      tmem_ld_wait();
      // the chunk is in registers: once every warp has its chunk the MMA warp may reuse it
      tc_fence_before();
      mbar_arrive(b_sfree(buf));
      const int key0 = j * kKeys + chunk * 32;
      float v[32];
      if (a.mode == 0) {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(u[e]) * a.scale;
      } else if (a.fast) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int64_t key = (int64_t)key0 + e;
          const float raw = __uint_as_float(u[e]) * a.scale;
          float addv = 0.f;
          bool excl = !valid || key < lo || key > hi;
          if (mrow) {
            if (key < a.r.add_T) addv = load_scalar(mrow, a.r.add_dtype, key);
            else excl = true;
          }
          float x;
          if (a.mode == 1 || cap == 0.f) x = raw + addv;
          else if (!a.r.softcap_before_bias) {
            x = raw + addv;
            x = (x == -INFINITY) ? x : cap * tanh_exp(x * cap_inv);
          } else {
            x = cap * tanh_exp(raw * cap_inv) + addv;
          }
          v[e] = (excl || x == -INFINITY) ? -INFINITY : x;
        }
      } else {
        const Rules& rr = a.mode == 1 ? a.r1 : a.r;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int64_t key = (int64_t)key0 + e;
          v[e] = (valid && key < a.T) ? generic_stage(rr, ctx, __uint_as_float(u[e]) * a.scale, b, h, i, key)
                                      : -INFINITY;
        }
      }
      if (gather) {
        float mt = -INFINITY;
#pragma unroll
        for (int e = 0; e < 32; ++e) mt = fmaxf(mt, v[e]);
        if (mt != -INFINITY) {
          const float m_new = fmaxf(m_run, mt * kLog2e);
          l_run *= ex2_approx(m_run - m_new);           // 0 while m_run is -inf (l_run is 0 then)
          m_run = m_new;
#pragma unroll
          for (int e = 0; e < 32; ++e) l_run += ex2_approx(fmaf(v[e], kLog2e, -m_run));   // exp(-inf) = 0
        }
        if (it == nT - 1) {
          // end of the first pass: combine the four chunks of each row, fold in the sink.
          // The staging slots are idle in this pass: the statistics borrow their space.
          float (*red_m)[kRows] = reinterpret_cast<float (*)[kRows]>(smem + C::kOutOff);
          float (*red_l)[kRows] = reinterpret_cast<float (*)[kRows]>(smem + C::kOutOff + 4 * kRows * 4);
          red_m[chunk][row] = m_run;
          red_l[chunk][row] = l_run;
          mbar_arrive(smem_u32(&bar_red[0]));
          if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bar_red[0]), 0, abortp, a.wait_ns))))
            break;
          float m = fmaxf(fmaxf(red_m[0][row], red_m[1][row]), fmaxf(red_m[2][row], red_m[3][row]));
          if (a.head_sink) m = fmaxf(m, sink_of<T>(a.head_sink, h) * kLog2e);
          float l = 0.f;
          if (m != -INFINITY) {
#pragma unroll
            for (int c = 0; c < 4; ++c) l += red_l[c][row] * ex2_approx(red_m[c][row] - m);
            if (a.head_sink) l += ex2_approx(fmaf(sink_of<T>(a.head_sink, h), kLog2e, -m));
          }
          m_fin = m;
          inv_l = (m != -INFINITY && l > 0.f) ? 1.f / l : 0.f;
          // every row read before the slots are reused
          mbar_arrive(smem_u32(&bar_red[1]));
          if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bar_red[1]), 0, abortp, a.wait_ns))))
            break;
        }
        continue;
      }
      if (a.mode == 3) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          v[e] = (m_fin == -INFINITY) ? 0.f : ex2_approx(fmaf(v[e], kLog2e, -m_fin)) * inv_l;
      }
      if (!warp_rows || key0 >= a.T) continue;        // the block lies outside the output
      // stage the 32 x 32 block in shared memory (128-byte swizzle) and store it
      const int slot = nstore % kOutBufs;
      if (nstore >= kOutBufs) {
        if (lane == 0) bulk_wait_read<kOutBufs - 1>();   // the slot's previous store has read it
        __syncwarp();
      }
      const uint32_t sl = slots + (uint32_t)slot * kOutSlot;
      const uint32_t rowaddr = sl + (uint32_t)lane * 128;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_shared_v4(rowaddr + (uint32_t)((q ^ (lane & 7)) << 4), __float_as_uint(v[4 * q]),
                     __float_as_uint(v[4 * q + 1]), __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3]));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_4d(&to, sl, key0, os1, os2, os3);
        bulk_commit();
      }
      ++nstore;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && abort_flag) atomicExch(&g_qk_status, (int)SDPA_ERR_TIMEOUT);
}

// ---------------------------------------------------------------------- general kernel

constexpr int kSimtWarps = 4;

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
__global__ void __launch_bounds__(kSimtWarps * 32) qk_simt_kernel(const Problem p, const View out, int mode) {
  extern __shared__ float q_smem[];  // kSimtWarps x H
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kSimtWarps + warp;
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
  Rules r1 = p.r;
  r1.softcap = 0.f;
  const T* kb = reinterpret_cast<const T*>(p.k_bias);
  float* orow = reinterpret_cast<float*>(const_cast<void*>(out.p)) + out.off(b, h, i);
  float m = -INFINITY, l = 0.f, inv = 0.f;

  for (int pass = 0; pass < (mode == 3 ? 2 : 1); ++pass) {
    const bool gather = mode == 3 && pass == 0;
    for (int64_t j0 = 0; j0 < p.T; j0 += 32) {
      const int64_t j = j0 + lane;
      float v = -INFINITY;
      if (j < p.T) {
        const T* krow = j < p.P ? reinterpret_cast<const T*>(p.past_k.p) + p.past_k.off(b, kh, j)
                                : reinterpret_cast<const T*>(p.k.p) + p.k.off(b, kh, j - p.P);
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
        v = stage_value(mode, p.r, r1, ctx, dot * p.scale, b, h, i, j);
      }
      if (gather) {
        const float mt = warp_max(v);
        if (mt == -INFINITY) continue;                  // uniform across the warp
        const float m_new = fmaxf(m, mt);
        l = l * exp2f((m - m_new) * kLog2e) + warp_sum(v == -INFINITY ? 0.f : exp2f((v - m_new) * kLog2e));
        m = m_new;
        continue;
      }
      if (mode == 3) v = (v == -INFINITY || m == -INFINITY) ? 0.f : exp2f((v - m) * kLog2e) * inv;
      if (j < p.T) orow[j] = v;
    }
    if (gather) {
      if (p.head_sink) {
        const float sk = sink_of<T>(p.head_sink, h);
        const float m_new = fmaxf(m, sk);
        if (m_new != -INFINITY) {
          l = l * exp2f((m - m_new) * kLog2e) + exp2f((sk - m_new) * kLog2e);
          m = m_new;
        }
      }
      inv = (m != -INFINITY && l > 0.f) ? 1.f / l : 0.f;
    }
  }
}

// 4-D fp32 map over the (B, Nq, S, T) output: dim 0 = T, dims 1..3 = seq / head / batch by
// increasing stride.  Box: 32 keys x 32 rows, 128-byte swizzle.
bool make_out_map(CUtensorMap* map, const View& o, int64_t B, int64_t N, int64_t S, int64_t T, int* ds, int* dn,
                  int* db) {
  auto enc = tc_encode_fn();
  if (!enc) return false;
  int order[3];
  tc_axis_order(o, B, N, S, order);
  const int64_t ext[3] = {S, N, B};
  const int64_t str[3] = {o.ss, o.sh, o.sb};
  cuuint64_t dims[4] = {(cuuint64_t)T, 0, 0, 0};
  cuuint64_t strides[3];
  cuuint32_t box[4] = {32, 1, 1, 1};
  int64_t prev_end = T * 4;
  for (int k = 0; k < 3; ++k) {
    const int id = order[k];
    dims[k + 1] = (cuuint64_t)ext[id];
    int64_t sb = str[id] * 4;
    if (ext[id] == 1) sb = ((prev_end + 15) / 16) * 16;   // never stepped: any legal stride
    strides[k] = (cuuint64_t)sb;
    prev_end = std::max<int64_t>(prev_end, sb * ext[id]);
    if (id == 0) { box[k + 1] = 32; *ds = k + 1; }
    if (id == 1) *dn = k + 1;
    if (id == 2) *db = k + 1;
  }
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(o.p), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

uint64_t qk_wait_limit_ns() {
  static uint64_t v = [] {
    const char* e = std::getenv("SDPA_WAIT_LIMIT_NS");
    return e ? std::strtoull(e, nullptr, 10) : 4000000000ull;
  }();
  return v;
}

template <int H, bool kBF16>
cudaError_t launch_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& to, const QkArgs& a,
                      cudaStream_t st) {
  using C = QkCfg<H>;
  auto kern = qk_tc_kernel<H, kBF16>;
  static cudaError_t attr_err = cudaSuccess;
  static std::once_flag once;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t grid = (int64_t)a.B * a.Nq * a.q_tiles;
  kern<<<(unsigned)grid, kThreads, C::kSmem, st>>>(tq, tk, to, a);
  count_launch(1);
  return cudaGetLastError();
}

bool out_view_tma_ok(const View& o) {
  return ((uintptr_t)o.p & 15u) == 0 && o.sb % 4 == 0 && o.sh % 4 == 0 && o.ss % 4 == 0 &&
         o.sb <= ((int64_t)1 << 37) && o.sh <= ((int64_t)1 << 37) && o.ss <= ((int64_t)1 << 37);
}

}  // namespace

cudaError_t launch_qk(const Problem& p, const View* k_total, const View& out, int mode, sdpa_dtype dt,
                      cudaStream_t st, const char** name) {
  const int64_t rows = (int64_t)p.B * p.Nq * p.S;
  if (rows == 0 || p.T == 0) return cudaSuccess;
  const bool tc = (dt == SDPA_F16 || dt == SDPA_BF16) && (p.H == 64 || p.H == 128) && k_total != nullptr &&
                  p.q_bias == nullptr && p.T <= ((int64_t)1 << 30) && out_view_tma_ok(out) &&
                  tc_encode_fn() != nullptr;
  if (tc) {
    QkArgs a{};
    a.B = p.B; a.Nq = p.Nq; a.Nkv = p.Nkv; a.S = p.S; a.T = (int)p.T; a.group = p.group; a.mode = mode;
    a.q_tiles = (p.S + kRows - 1) / kRows;
    a.scale = p.scale;
    a.r = p.r;
    a.r1 = p.r;
    a.r1.softcap = 0.f;
    a.head_sink = p.head_sink;
    a.fast = p.r.keep_kind == SDPA_KEEP_NONE && p.r.len_kind != SDPA_LEN_KEYLEN_I32;
    a.wait_ns = qk_wait_limit_ns();
    CUtensorMap tq, tk, to;
    bool ok = tc_make_map(&tq, p.q, dt, p.B, p.Nq, p.S, p.H, &a.q_ds, &a.q_dn, &a.q_db) &&
              tc_make_map(&tk, *k_total, dt, p.B, p.Nkv, p.T, p.H, &a.k_ds, &a.k_dn, &a.k_db) &&
              make_out_map(&to, out, p.B, p.Nq, p.S, p.T, &a.o_ds, &a.o_dn, &a.o_db);
    if (ok) {
      const bool bf = dt == SDPA_BF16;
      if (p.H == 128) {
        *name = bf ? "qk_tc_bf16_h128" : "qk_tc_f16_h128";
        return bf ? launch_tc<128, true>(tq, tk, to, a, st) : launch_tc<128, false>(tq, tk, to, a, st);
      }
      *name = bf ? "qk_tc_bf16_h64" : "qk_tc_f16_h64";
      return bf ? launch_tc<64, true>(tq, tk, to, a, st) : launch_tc<64, false>(tq, tk, to, a, st);
    }
  }
  const dim3 grid((unsigned)((rows + kSimtWarps - 1) / kSimtWarps));
  const size_t smem = sizeof(float) * kSimtWarps * p.H;
  switch (dt) {
    case SDPA_F32: qk_simt_kernel<float><<<grid, kSimtWarps * 32, smem, st>>>(p, out, mode); break;
    case SDPA_F16: qk_simt_kernel<__half><<<grid, kSimtWarps * 32, smem, st>>>(p, out, mode); break;
    default: qk_simt_kernel<__nv_bfloat16><<<grid, kSimtWarps * 32, smem, st>>>(p, out, mode); break;
  }
  count_launch(1);
  *name = dt == SDPA_F32 ? "qk_simt_f32" : dt == SDPA_F16 ? "qk_simt_f16" : "qk_simt_bf16";
  return cudaGetLastError();
}

cudaError_t take_qk_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_qk_status, sizeof v);
  if (e != cudaSuccess) return e;
  *status = v;
  if (v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_qk_status, &zero, sizeof zero);
  }
  return e;
}

}  // namespace sdpa
