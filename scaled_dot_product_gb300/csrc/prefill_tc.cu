// Fused tensor-core prefill for GB300 (sm_103a): TMA-staged Q/K/V tiles, tcgen05.mma with
// accumulators in tensor memory, an online softmax with fp32 statistics in registers,
// and the masking rules of onnx-light class Attention / MultiHeadAttention /
// GroupQueryAttention applied per element in registers.
//
// One CTA owns two 128-row query tiles (A, B) of one (batch, query head) and streams the
// key/value tiles of its kv head through a shared-memory ring:
//
//   warp 0      TMA producer: Q tiles once, then K_0, V_0, K_1, V_1, ... into the ring
//   warp 1      MMA issuer (one thread): S_X = Q_X K_j^T into TMEM, O_X += P_X V_j
//   warps 4-7   softmax for tile A: each thread owns one query row (TMEM lane = row)
//   warps 8-11  softmax for tile B
//
// The two softmax warpgroups alternate with the tensor core: while one works on its
// scores the MMA warp computes the other's products.  Running maxima are kept in the
// base-2 domain and only moved (with a rescale of the TMEM accumulator) when they grow
// by more than 2^8, so most tiles skip the rescale.  P is written to shared memory in
// the K-major 128-byte-swizzled layout the second MMA reads.
//
// Every barrier wait is bounded: on expiry the kernel raises an abort flag, drains the
// copies and MMAs it issued, frees its tensor memory and records SDPA_ERR_TIMEOUT in a
// device status word (read by sdpa_query_status).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "prefill_tc.h"
#include "tc_ptx.cuh"

namespace sdpa {

static __device__ int g_prefill_status;

namespace {

using namespace ptx;

constexpr int kBM = 128;        // query rows per tile (TMEM lanes)
constexpr int kBN = 128;        // keys per tile
constexpr int kThreads = 384;   // 12 warps
constexpr float kRescaleThreshold = 8.f;   // log2 units

template <int H>
struct Cfg {
  static constexpr int kRegions = H / 64;              // 128-byte swizzle regions per row
  static constexpr int kRegionBytes = 128 * 128;       // 128 rows x 128 bytes
  static constexpr int kQTile = kBM * H * 2;
  static constexpr int kKVTile = kBN * H * 2;
  static constexpr int kStages = (H == 128) ? 3 : 6;
  static constexpr int kPTile = kBM * kBN * 2;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = 2 * kQTile;
  static constexpr int kPOff = kKVOff + kStages * kKVTile;
  static constexpr int kSmem = kPOff + 2 * kPTile + 1024;   // + alignment slack
  static constexpr int kTmemS0 = 0, kTmemS1 = 128, kTmemO0 = 256, kTmemO1 = 256 + H;
  static constexpr uint32_t kTmemCols = 512;
};

struct TcArgs {
  int B, Nq, Nkv, S, T, group, npairs;
  float scale, scale_log2, cap_in, cap_out_log2;   // cap_* used when softcap > 0
  int has_softcap;
  int causal, window, len_kind;
  const void* lens;
  int generic;                                      // per-element rules beyond the structural ones
  Rules r;
  int q_ds, q_dn, q_db, kv_ds, kv_dn, kv_db;        // tensor-map dimension of seq / head / batch
  void* y;
  int64_t y_sb, y_sh, y_ss;
  const void* q_bias;
  const void* head_sink;
  uint64_t wait_ns;
};

__device__ __forceinline__ int64_t min64(int64_t x, int64_t y) { return x < y ? x : y; }
__device__ __forceinline__ int64_t max64(int64_t x, int64_t y) { return x > y ? x : y; }

__device__ __forceinline__ void perm_coords(int ds, int dn, int db, int s, int n, int b, int& c1, int& c2, int& c3) {
  c1 = ds == 1 ? s : (dn == 1 ? n : b);
  c2 = ds == 2 ? s : (dn == 2 ? n : b);
  c3 = ds == 3 ? s : (dn == 3 ? n : b);
}

__device__ __forceinline__ int64_t lens_of(const TcArgs& a, int b) {
  if (a.len_kind == SDPA_LEN_NONE) return 0;
  if (a.len_kind == SDPA_LEN_NONPAD_I64) return reinterpret_cast<const int64_t*>(a.lens)[b];
  return reinterpret_cast<const int32_t*>(a.lens)[b];
}

// Key position of query row i for the causal / window rules.
__device__ __forceinline__ int64_t pos_of(const TcArgs& a, int64_t len_b, int64_t i) {
  if (a.causal == SDPA_CAUSAL_UPPER_LEFT) return i;
  if (a.causal == SDPA_CAUSAL_LOWER_RIGHT)
    return ((a.len_kind == SDPA_LEN_SEQLENS_K_I32) ? len_b + 1 : (int64_t)a.T) - a.S + i;
  return (int64_t)a.T - 1;
}

// Admitted key interval [lo, hi] of query row i under the structural rules.
__device__ __forceinline__ void key_bounds(const TcArgs& a, int64_t len_b, int64_t i, int64_t& lo, int64_t& hi) {
  hi = (int64_t)a.T - 1;
  lo = 0;
  const int64_t pos = pos_of(a, len_b, i);
  if (a.causal != SDPA_CAUSAL_NONE) hi = min64(hi, pos);
  if (a.window > 0) lo = max64(lo, pos - a.window + 1);
  if (a.len_kind == SDPA_LEN_NONPAD_I64) hi = min64(hi, len_b - 1);
  if (a.len_kind == SDPA_LEN_SEQLENS_K_I32) hi = min64(hi, len_b);
}

__device__ __noinline__ float generic_score(const Rules& r, const RowCtx& ctx, float s_nat, int b, int h, int i,
                                            int64_t j) {
  return apply_rules(r, ctx, s_nat, b, h, i, j);
}

template <int H, bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const TcArgs a) {
  using C = Cfg<H>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_q, bar_qready, bar_drain;
  __shared__ __align__(8) uint64_t bar_full[C::kStages], bar_empty[C::kStages];
  __shared__ __align__(8) uint64_t bar_s[2], bar_p[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work unit: (query-tile pair, batch, kv head, head within the group), heavy first
  int t = blockIdx.x;
  const int g_idx = t % a.group; t /= a.group;
  const int kvh = t % a.Nkv; t /= a.Nkv;
  const int b = t % a.B; t /= a.B;
  const int pair = a.npairs - 1 - t;
  const int qh = kvh * a.group + g_idx;
  const int m0 = pair * 2 * kBM;
  const int m1 = min(a.S, m0 + 2 * kBM);
  const int64_t len_b = lens_of(a, b);

  // key tiles any row of this CTA can admit
  int64_t lo_first, hi_first, lo_last, hi_last;
  key_bounds(a, len_b, m0, lo_first, hi_first);
  key_bounds(a, len_b, m1 - 1, lo_last, hi_last);
  const int64_t lo_key = max64(0, min64(lo_first, lo_last));
  const int64_t hi_key = min64((int64_t)a.T - 1, max64(hi_first, hi_last));
  const int kv_t0 = (int)(lo_key / kBN);
  const int n_tiles = (hi_key >= lo_key) ? (int)(hi_key / kBN) - kv_t0 + 1 : 0;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::kQOff, sKV = sbase + C::kKVOff, sP = sbase + C::kPOff;
  const uint32_t b_q = smem_u32(&bar_q), b_qready = smem_u32(&bar_qready), b_drain = smem_u32(&bar_drain);
  auto b_full = [&](int s) { return smem_u32(&bar_full[s]); };
  auto b_empty = [&](int s) { return smem_u32(&bar_empty[s]); };
  auto b_s = [&](int x) { return smem_u32(&bar_s[x]); };
  auto b_p = [&](int x) { return smem_u32(&bar_p[x]); };
  volatile int* abortp = &abort_flag;
  constexpr uint64_t kDrainNs = 2000000000ull;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(b_q, 1);
    mbar_init(b_qready, 2 * kBM);
    mbar_init(b_drain, 1);
    for (int s = 0; s < C::kStages; ++s) { mbar_init(b_full(s), 1); mbar_init(b_empty(s), 1); }
    for (int x = 0; x < 2; ++x) { mbar_init(b_s(x), 1); mbar_init(b_p(x), kBM); }
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
    if (lane == 0 && n_tiles > 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      int c1, c2, c3;
      mbar_arrive_expect_tx(b_q, 2 * C::kQTile);
      for (int x = 0; x < 2; ++x) {
        perm_coords(a.q_ds, a.q_dn, a.q_db, m0 + x * kBM, qh, b, c1, c2, c3);
        for (int r = 0; r < C::kRegions; ++r)
          tma_load_4d(sQ + x * C::kQTile + r * C::kRegionBytes, &tq, b_q, 64 * r, c1, c2, c3);
      }
      int seq = 0;
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        for (int kind = 0; kind < 2 && ok; ++kind, ++seq) {
          const int st = seq % C::kStages;
          if (seq >= C::kStages) {
            ok = mbar_wait_bounded(b_empty(st), ((seq / C::kStages) - 1) & 1, abortp, a.wait_ns);
            if (!ok) break;
          }
          mbar_arrive_expect_tx(b_full(st), C::kKVTile);
          perm_coords(a.kv_ds, a.kv_dn, a.kv_db, (kv_t0 + j) * kBN, kvh, b, c1, c2, c3);
          for (int r = 0; r < C::kRegions; ++r)
            tma_load_4d(sKV + st * C::kKVTile + r * C::kRegionBytes, kind == 0 ? &tk : &tv, b_full(st), 64 * r,
                        c1, c2, c3);
        }
      }
      if (!ok) {
        // let every copy already issued land before the CTA can exit
        mbar_wait_bounded(b_q, 0, nullptr, kDrainNs);
        const int issued = seq;
        for (int s = 0; s < C::kStages && s < issued; ++s) {
          const int last = s + ((issued - 1 - s) / C::kStages) * C::kStages;
          mbar_wait_bounded(b_full(s), (last / C::kStages) & 1, nullptr, kDrainNs);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kIdQK = idesc_f16(kBF16, kBM, kBN, false);
      constexpr uint32_t kIdPV = idesc_f16(kBF16, kBM, H, true);
      const uint32_t tS[2] = {tmem + C::kTmemS0, tmem + C::kTmemS1};
      const uint32_t tO[2] = {tmem + C::kTmemO0, tmem + C::kTmemO1};
      auto wait_full = [&](int seq) -> bool {
        const bool ok = mbar_wait_bounded(b_full(seq % C::kStages), (seq / C::kStages) & 1, abortp, a.wait_ns);
        tc_fence_after();
        return ok;
      };
      auto issue_S = [&](int x, int st) {
        const uint32_t q0 = sQ + x * C::kQTile, k0 = sKV + st * C::kKVTile;
#pragma unroll
        for (int kk = 0; kk < H / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::kRegionBytes + (kk % 4) * 32;
          mma_f16_ss(tS[x], desc_sw128(q0 + off, 16, 1024), desc_sw128(k0 + off, 16, 1024), kIdQK, kk > 0);
        }
      };
      auto issue_PV = [&](int x, int st, bool acc) {
        const uint32_t p0 = sP + x * C::kPTile, v0 = sKV + st * C::kKVTile;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t aoff = (kk / 4) * C::kRegionBytes + (kk % 4) * 32;
          mma_f16_ss(tO[x], desc_sw128(p0 + aoff, 16, 1024), desc_sw128(v0 + kk * 2048, C::kRegionBytes, 1024),
                     kIdPV, (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait_bounded(a.q_bias ? b_qready : b_q, 0, abortp, a.wait_ns);
      tc_fence_after();
      if (ok) ok = wait_full(0);
      if (ok) {
        const int st0 = 0;
        issue_S(0, st0);
        mma_commit(b_s(0));
        issue_S(1, st0);
        mma_commit(b_s(1));
        mma_commit(b_empty(st0));
      }
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int vseq = 2 * j + 1, kseq = 2 * j + 2;
        const int vst = vseq % C::kStages, kst = kseq % C::kStages;
        const bool more = j + 1 < n_tiles;
        if (!(ok = wait_full(vseq))) break;
        // tile A
        if (!(ok = mbar_wait_bounded(b_p(0), j & 1, abortp, a.wait_ns))) break;
        tc_fence_after();
        issue_PV(0, vst, j > 0);
        if (more) {
          if (!(ok = wait_full(kseq))) break;
          issue_S(0, kst);
        }
        mma_commit(b_s(0));
        // tile B
        if (!(ok = mbar_wait_bounded(b_p(1), j & 1, abortp, a.wait_ns))) break;
        tc_fence_after();
        issue_PV(1, vst, j > 0);
        mma_commit(b_empty(vst));
        if (more) {
          issue_S(1, kst);
          mma_commit(b_empty(kst));
        }
        mma_commit(b_s(1));
      }
      // every MMA this thread issued completes before the CTA frees its tensor memory
      mma_commit(b_drain);
      mbar_wait_bounded(b_drain, 0, nullptr, kDrainNs);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ================================================================ softmax warpgroups
    const int x = (warp - 4) >> 2;                  // query tile A or B
    const int sub = warp & 3;                       // TMEM sub-partition of this warp
    const int row = sub * 32 + lane;                // row in the tile == TMEM lane
    const int64_t i = (int64_t)m0 + x * kBM + row;  // query row
    const bool valid = i < a.S;
    int64_t lo = 1, hi = 0;
    if (valid) key_bounds(a, len_b, i, lo, hi);
    // T <= 2^30, so the bounds fit 32 bits once clamped to [-1, T]
    const int lo32 = (int)max64(-1, min64(lo, a.T));
    const int hi32 = (int)max64(-1, min64(hi, a.T));
    RowCtx ctx;
    ctx.len = len_b;
    ctx.pos = pos_of(a, len_b, i);
    const uint32_t trow = tmem + ((uint32_t)(sub * 32) << 16);
    const uint32_t tS = trow + (x == 0 ? C::kTmemS0 : C::kTmemS1);
    const uint32_t tO = trow + (x == 0 ? C::kTmemO0 : C::kTmemO1);
    const uint32_t pRow = sP + x * C::kPTile + row * 128;
    const int swz = row & 7;
    bool ok = true;

    if (n_tiles > 0 && a.q_bias) {
      // add the query segment of the projection bias to this row of Q in shared memory
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_q, 0, abortp, a.wait_ns));
      if (ok) {
        const uint32_t qRow = sQ + x * C::kQTile + row * 128;
        const auto* qb = reinterpret_cast<const typename std::conditional<kBF16, __nv_bfloat16, __half>::type*>(a.q_bias) +
                         (int64_t)qh * H;
#pragma unroll
        for (int r = 0; r < C::kRegions; ++r)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t addr = qRow + r * C::kRegionBytes + ((c ^ swz) << 4);
            uint32_t w[4];
            ld_shared_v4(addr, w[0], w[1], w[2], w[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float lo_f, hi_f;
              const int col = r * 64 + c * 8 + 2 * e;
              if constexpr (kBF16) {
                __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w[e]);
                lo_f = __bfloat162float(v.x) + __bfloat162float(qb[col]);
                hi_f = __bfloat162float(v.y) + __bfloat162float(qb[col + 1]);
                w[e] = pack_bf16x2(lo_f, hi_f);
              } else {
                __half2 v = *reinterpret_cast<__half2*>(&w[e]);
                lo_f = __half2float(v.x) + __half2float(qb[col]);
                hi_f = __half2float(v.y) + __half2float(qb[col + 1]);
                w[e] = pack_f16x2(lo_f, hi_f);
              }
            }
            st_shared_v4(addr, w[0], w[1], w[2], w[3]);
          }
        fence_proxy_async_smem();
      }
      mbar_arrive(b_qready);
    }

    float m_use = -INFINITY, l = 0.f;
    for (int j = 0; j < n_tiles && ok; ++j) {
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_s(x), j & 1, abortp, a.wait_ns)))) break;
      tc_fence_after();
      uint32_t u[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) tmem_ld32(tS + c * 32, u + c * 32);
      tmem_ld_wait();
      float s[kBN];
#pragma unroll
      for (int e = 0; e < kBN; ++e) s[e] = __uint_as_float(u[e]);
      const int key0 = (kv_t0 + j) * kBN;
      float mx = -INFINITY;
      if (!a.generic) {
        const bool full = (lo32 <= key0) && (key0 + kBN - 1 <= hi32);
        if (a.has_softcap) {
#pragma unroll
          for (int e = 0; e < kBN; ++e) s[e] = tanh_approx(s[e] * a.cap_in) * a.cap_out_log2;
        } else {
#pragma unroll
          for (int e = 0; e < kBN; ++e) s[e] *= a.scale_log2;
        }
        if (!full) {
#pragma unroll
          for (int e = 0; e < kBN; ++e) {
            const int key = key0 + e;
            s[e] = (key >= lo32 && key <= hi32) ? s[e] : -INFINITY;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < kBN; ++e) {
          const int key = key0 + e;
          float v = -INFINITY;
          if (key >= lo32 && key <= hi32)
            v = generic_score(a.r, ctx, s[e] * a.scale, b, qh, (int)i, key) * kLog2e;
          s[e] = v;
        }
      }
#pragma unroll
      for (int e = 0; e < kBN; ++e) mx = fmaxf(mx, s[e]);

      // move the running maximum only when it grows by more than 2^8
      const float m_new = fmaxf(m_use, mx);
      const bool need = m_new > m_use + kRescaleThreshold;
      float corr = 1.f;
      if (need) {
        corr = ex2_approx(m_use - m_new);
        m_use = m_new;
      }
      const bool dead = (m_use == -INFINITY);
      float rowsum = 0.f;
#pragma unroll
      for (int c = 0; c < kBN / 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = dead ? 0.f : ex2_approx(s[c * 8 + 2 * e] - m_use);
          const float p1 = dead ? 0.f : ex2_approx(s[c * 8 + 2 * e + 1] - m_use);
          rowsum += p0 + p1;
          w[e] = kBF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
        }
        st_shared_v4(pRow + (c >> 3) * C::kRegionBytes + (((c & 7) ^ swz) << 4), w[0], w[1], w[2], w[3]);
      }
      l = l * corr + rowsum;
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // rescale this warp's rows of the accumulator (factor 1 for rows that kept their max)
#pragma unroll
        for (int c = 0; c < H / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
          tmem_st32(tO + c * 32, o);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(b_p(x));
    }

    // ---- epilogue: O / (l + sink term), rounded once to the output type
    if (ok && n_tiles > 0) ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_s(x), n_tiles & 1, abortp, a.wait_ns));
    if (ok) {
      tc_fence_after();
      float denom = l;
      if (a.head_sink && m_use != -INFINITY) {
        float sk;
        if constexpr (kBF16) sk = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.head_sink)[qh]);
        else sk = __half2float(reinterpret_cast<const __half*>(a.head_sink)[qh]);
        denom += ex2_approx(sk * kLog2e - m_use);
      }
      const float inv = (denom > 0.f && m_use != -INFINITY) ? 1.f / denom : 0.f;
      using T = typename std::conditional<kBF16, __nv_bfloat16, __half>::type;
      T* yrow = reinterpret_cast<T*>(a.y) + (int64_t)b * a.y_sb + (int64_t)qh * a.y_sh + i * a.y_ss;
#pragma unroll
      for (int c = 0; c < H / 32; ++c) {
        uint32_t o[32];
        if (n_tiles > 0) {
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float v0 = __uint_as_float(o[q * 8 + 2 * e]) * inv;
              const float v1 = __uint_as_float(o[q * 8 + 2 * e + 1]) * inv;
              w[e] = kBF16 ? pack_bf16x2(v0, v1) : pack_f16x2(v0, v1);
            }
            *reinterpret_cast<uint4*>(yrow + c * 32 + q * 8) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && abort_flag) atomicExch(&g_prefill_status, (int)SDPA_ERR_TIMEOUT);
}

// ---------------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 4-D map over a (B, N, Seq, D) view: dim 0 = D (contiguous); dims 1..3 = seq / head /
// batch ordered by increasing stride (size-1 axes last).  Box: 64 x 128 rows.
bool make_map(CUtensorMap* map, const View& v, sdpa_dtype dt, int64_t B, int64_t N, int64_t Sq, int D, int* ds,
              int* dn, int* db) {
  auto enc = encode_fn();
  if (!enc) return false;
  struct Ax { int64_t ext, stride; int id; };
  Ax ax[3] = {{Sq, v.ss, 0}, {N, v.sh, 1}, {B, v.sb, 2}};
  std::stable_sort(ax, ax + 3, [](const Ax& l, const Ax& r) {
    const bool l1 = l.ext == 1, r1 = r.ext == 1;
    if (l1 != r1) return r1;             // size-1 axes go last
    return l.stride < r.stride;
  });
  const int64_t es = 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, 0, 0, 0};
  cuuint64_t strides[3];
  cuuint32_t box[4] = {64, 1, 1, 1};
  int64_t prev_end = (int64_t)D * es;  // bytes spanned so far
  for (int k = 0; k < 3; ++k) {
    dims[k + 1] = (cuuint64_t)ax[k].ext;
    int64_t sb = ax[k].stride * es;
    if (ax[k].ext == 1) sb = ((prev_end + 15) / 16) * 16;   // never stepped: any legal stride
    strides[k] = (cuuint64_t)sb;
    prev_end = std::max<int64_t>(prev_end, sb * ax[k].ext);
    if (ax[k].id == 0) { box[k + 1] = kBN; *ds = k + 1; }
    if (ax[k].id == 1) *dn = k + 1;
    if (ax[k].id == 2) *db = k + 1;
  }
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, dt == SDPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                   const_cast<void*>(v.p), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

uint64_t wait_limit_ns() {
  static uint64_t v = [] {
    const char* e = std::getenv("SDPA_WAIT_LIMIT_NS");
    return e ? std::strtoull(e, nullptr, 10) : 4000000000ull;
  }();
  return v;
}

template <int H, bool kBF16>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const TcArgs& a,
                     int64_t units, cudaStream_t st) {
  using C = Cfg<H>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(prefill_tc_kernel<H, kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  prefill_tc_kernel<H, kBF16><<<(unsigned)units, kThreads, C::kSmem, st>>>(tq, tk, tv, a);
  count_launch(1);
  return cudaGetLastError();
}

}  // namespace

bool tc_eligible(const Problem& p, sdpa_dtype dt) {
  if (dt != SDPA_F16 && dt != SDPA_BF16) return false;
  if (p.H != p.Hv || (p.H != 64 && p.H != 128)) return false;
  if (p.T < 1 || p.S < 16) return false;
  if (p.T > (int64_t)1 << 30 || p.r.window > (int64_t)1 << 30) return false;
  for (const View* v : {&p.q, &p.k, &p.v})
    if (v->sb > ((int64_t)1 << 38) || v->sh > ((int64_t)1 << 38) || v->ss > ((int64_t)1 << 38)) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const Problem& p, sdpa_dtype dt, cudaStream_t st, const char** name) {
  TcArgs a{};
  a.B = p.B; a.Nq = p.Nq; a.Nkv = p.Nkv; a.S = p.S; a.T = (int)p.T; a.group = p.group;
  a.npairs = (p.S + 2 * kBM - 1) / (2 * kBM);
  a.scale = p.scale;
  a.scale_log2 = p.scale * kLog2e;
  a.has_softcap = p.r.softcap > 0.f;
  a.cap_in = a.has_softcap ? p.scale / p.r.softcap : 0.f;
  a.cap_out_log2 = a.has_softcap ? p.r.softcap * kLog2e : 0.f;
  a.causal = p.r.causal;
  a.window = (int)p.r.window;
  a.len_kind = p.r.len_kind;
  a.lens = p.r.lens;
  a.generic = (p.r.add != nullptr) || (p.r.keep_kind != SDPA_KEEP_NONE) || (p.r.len_kind == SDPA_LEN_KEYLEN_I32);
  a.r = p.r;
  a.y = const_cast<void*>(p.y.p);
  a.y_sb = p.y.sb; a.y_sh = p.y.sh; a.y_ss = p.y.ss;
  a.q_bias = p.q_bias;
  a.head_sink = p.head_sink;
  a.wait_ns = wait_limit_ns();
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, p.q, dt, p.B, p.Nq, p.S, p.H, &a.q_ds, &a.q_dn, &a.q_db) ||
      !make_map(&tk, p.k, dt, p.B, p.Nkv, p.T, p.H, &a.kv_ds, &a.kv_dn, &a.kv_db))
    return cudaErrorInvalidValue;
  int vds, vdn, vdb;
  if (!make_map(&tv, p.v, dt, p.B, p.Nkv, p.T, p.Hv, &vds, &vdn, &vdb)) return cudaErrorInvalidValue;
  if (vds != a.kv_ds || vdn != a.kv_dn || vdb != a.kv_db) return cudaErrorInvalidValue;   // k and v views differ in order
  const int64_t units = (int64_t)p.B * p.Nkv * a.npairs * p.group;
  if (units > 0x7fffffff) return cudaErrorInvalidValue;
  const bool bf = dt == SDPA_BF16;
  if (p.H == 128) {
    *name = bf ? "prefill_tc_bf16_h128" : "prefill_tc_f16_h128";
    return bf ? launch_t<128, true>(tq, tk, tv, a, units, st) : launch_t<128, false>(tq, tk, tv, a, units, st);
  }
  *name = bf ? "prefill_tc_bf16_h64" : "prefill_tc_f16_h64";
  return bf ? launch_t<64, true>(tq, tk, tv, a, units, st) : launch_t<64, false>(tq, tk, tv, a, units, st);
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
