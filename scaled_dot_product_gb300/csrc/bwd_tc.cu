// Tensor-core backward of the attention for GB300 (sm_103a): the gradient graph of
// onnx-light-cpu "Custom operators" (C++ API, RegisterCustomOperatorGradients,
// GroupQueryAttention gradient).  From the stage-3 probabilities P of the forward (class
// Attention, qk_matmul_output_mode 3):
//
//   dP = dY V^T,   dS = P (dP - rowsum(P dP)) scale,   dQ = dS K,   dK = dS^T Q,   dV = P^T dY,
//
// with the query heads of a group summed onto their kv head ("reduce groups").
//
// Three launches.  The statistics pass is the forward kernel (prefill_tc.cu) writing, per
// query row, the log2-sum-exp L_i of its scores and delta_i = dY_i . O_i (= rowsum(P dP)).
// Then two kernels recompute the scores tile by tile, so no S x T matrix is stored:
//
// The score scale of dS is applied once, to the accumulated dQ and dK when they are stored.
//
//   bwd_dkdv_kernel   one CTA per (128-key tile, kv head, batch); loops over the query
//                     tiles and the grouped query heads that see the key tile:
//                       S^T = K Q^T, dP^T = V dY^T            (tcgen05, both operands in smem)
//                       P^T = 2^(S^T scale log2e - L), dS^T   (one thread per key, in registers)
//                       dV += P^T dY, dK += dS^T Q            (tcgen05, P^T / dS^T in TMEM)
//   bwd_dq_kernel     one CTA per (128-row query tile, query head, batch); loops over key tiles:
//                       S = Q K^T, dP = dY V^T;  dS;  dQ += dS K
//
// Roles per CTA: warp 0 TMA producer, warp 1 MMA issuer (one thread), warps 4-7 one thread
// per TMEM lane (the key row in dK/dV, the query row in dQ).  P^T and dS^T overwrite the
// tensor-memory columns of S^T and dP^T they came from; the MMA warp issues the next tile's
// products only after the accumulating MMAs that read them.  Every barrier wait is bounded:
// on expiry the kernel raises an abort flag, drains what it issued, frees its tensor memory
// and records SDPA_ERR_TIMEOUT.
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "internal.h"
#include "prefill_tc.h"
#include "tc_ptx.cuh"

namespace sdpa {

static __device__ int g_bwd_status;

namespace {

using namespace ptx;

constexpr int kBM = 128;   // rows per tile (TMEM lanes)

struct BwdArgs {
  int B, Nq, Nkv, S, T, group;
  float scale, scale_log2;
  int causal, window, len_kind;
  const void* lens;
  const float* lse2;        // (B, Nq, S) log2-sum-exp in units of q.k scale log2e
  const float* delta;       // (B, Nq, S) rowsum(P dP)
  int q_ds, q_dn, q_db;     // map dimension of seq / head / batch (Q map)
  int g_ds, g_dn, g_db;     // dY map
  int kv_ds, kv_dn, kv_db;  // K and V maps
  void* out0;               // dK (dK/dV kernel) or dQ (dQ kernel)
  int64_t o0_sb, o0_sh, o0_ss;
  void* out1;               // dV (dK/dV kernel)
  int64_t o1_sb, o1_sh, o1_ss;
  int nq_tiles, nk_tiles;
  uint64_t wait_ns;
  Rules r;                  // masks: additive, keep (bool / binary), key-padding lengths
  int has_extra;            // any of them present
};

// H: head size; STEP: rows of the streamed tiles (the queries of one dK/dV step, the keys of
// one dQ step).  With STEP = 64 and H = 64 a CTA needs 256 TMEM columns and 96 KB of shared
// memory, so two CTAs share an SM and one's score pass runs under the other's products.
template <int H, int STEP>
struct BCfg {
  static constexpr int kRegions = H / 64;              // 128-byte swizzle regions per row
  static constexpr int kRegionBytes = 128 * 128;       // resident tile: 128 rows x 128 bytes
  static constexpr int kSRegionBytes = STEP * 128;     // streamed tile: STEP rows x 128 bytes
  static constexpr int kTile = kBM * H * 2;            // resident 128-row tile
  static constexpr int kSTile = STEP * H * 2;          // streamed STEP-row tile
  static constexpr int kStages = (H == 128) ? 2 : 4;
  // two resident tiles, then kStages stages of two streamed tiles each
  static constexpr int kSmem = 2 * kTile + 2 * kStages * kSTile + 1024;
  static constexpr int kTmemS = 0, kTmemP = STEP, kTmemA0 = 2 * STEP, kTmemA1 = 2 * STEP + H;
  static constexpr uint32_t kTmemCols = (2 * STEP + 2 * H <= 256) ? 256 : 512;
  static constexpr int kThreads = 256;                 // 4 control warps + one warpgroup
  static constexpr int kMinBlocks = (kTmemCols == 256) ? 2 : 1;
};

__device__ __forceinline__ void perm_coords(int ds, int dn, int db, int s, int n, int b, int& c1, int& c2, int& c3) {
  c1 = ds == 1 ? s : (dn == 1 ? n : b);
  c2 = ds == 2 ? s : (dn == 2 ? n : b);
  c3 = ds == 3 ? s : (dn == 3 ? n : b);
}

__device__ __forceinline__ int64_t bmin(int64_t x, int64_t y) { return x < y ? x : y; }
__device__ __forceinline__ int64_t bmax(int64_t x, int64_t y) { return x > y ? x : y; }

__device__ __forceinline__ int64_t len_of(const BwdArgs& a, int b) {
  if (a.len_kind == SDPA_LEN_NONPAD_I64) return reinterpret_cast<const int64_t*>(a.lens)[b];
  if (a.len_kind == SDPA_LEN_SEQLENS_K_I32 || a.len_kind == SDPA_LEN_KEYLEN_I32)
    return reinterpret_cast<const int32_t*>(a.lens)[b];
  return 0;
}

// Offset of the causal alignment: query row i sits at key position i + off.
__device__ __forceinline__ int64_t pos_off(const BwdArgs& a, int64_t len_b) {
  if (a.causal == SDPA_CAUSAL_LOWER_RIGHT)
    return ((a.len_kind == SDPA_LEN_SEQLENS_K_I32) ? len_b + 1 : (int64_t)a.T) - a.S;
  return 0;
}

// Last admitted key of the whole row set (length rules only).
__device__ __forceinline__ int64_t key_limit(const BwdArgs& a, int64_t len_b) {
  int64_t hi = (int64_t)a.T - 1;
  if (a.len_kind == SDPA_LEN_NONPAD_I64) hi = bmin(hi, len_b - 1);
  if (a.len_kind == SDPA_LEN_SEQLENS_K_I32) hi = bmin(hi, len_b);
  return hi;
}

// Admitted key interval [lo, hi] of query row i (causal, window, lengths).
__device__ __forceinline__ void key_range(const BwdArgs& a, int64_t len_b, int64_t i, int64_t& lo, int64_t& hi) {
  hi = key_limit(a, len_b);
  lo = 0;
  if (a.causal != SDPA_CAUSAL_NONE) {
    const int64_t pos = i + pos_off(a, len_b);
    hi = bmin(hi, pos);
    if (a.window > 0) lo = bmax(lo, pos - a.window + 1);
  }
}

// Admitted query interval [lo, hi] of key j (the same rules seen from the key side).
__device__ __forceinline__ void query_range(const BwdArgs& a, int64_t len_b, int64_t j, int64_t& lo, int64_t& hi) {
  lo = 0;
  hi = (int64_t)a.S - 1;
  if (j > key_limit(a, len_b)) { lo = 1; hi = 0; return; }
  if (a.causal != SDPA_CAUSAL_NONE) {
    const int64_t off = pos_off(a, len_b);
    lo = bmax(lo, j - off);                              // pos(i) >= j
    if (a.window > 0) hi = bmin(hi, j + a.window - 1 - off);   // pos(i) - W + 1 <= j
  }
}

// Additive term of score (i, j) in natural units from the masks: the float mask (-inf past
// its end), a keep mask (bool: -inf for a dropped key; binary: + mask_filter_value) and
// MultiHeadAttention key-padding lengths (+ mask_filter_value from the length on).
__device__ __forceinline__ float extra_term(const Rules& r, int64_t len_b, int b, int h, int64_t i, int64_t j) {
  float e = 0.f;
  if (r.add) {
    if (j >= r.add_T) return -INFINITY;
    e += load_scalar(r.add, r.add_dtype, b * r.add_sb + h * r.add_sh + i * r.add_ss + j);
  }
  if (r.keep_kind != SDPA_KEEP_NONE) {
    bool keep = false;
    if (j < r.keep_T) {
      const int64_t o = b * r.keep_sb + h * r.keep_sh + i * r.keep_ss + j;
      keep = (r.keep_kind == SDPA_KEEP_BOOL_U8) ? (reinterpret_cast<const uint8_t*>(r.keep)[o] != 0)
                                                : (reinterpret_cast<const int32_t*>(r.keep)[o] != 0);
    }
    if (!keep) {
      if (r.keep_kind == SDPA_KEEP_BOOL_U8) return -INFINITY;
      e += r.filter;
    }
  }
  if (r.len_kind == SDPA_LEN_KEYLEN_I32 && j >= len_b) e += r.filter;
  return e;
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return kBF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}

// One 128 x (32 NCH) tile of scores and score gradients in TMEM (this thread's lane = one row):
// P = 2^(s scale log2e - L) on admitted entries and dS' = P (dP - delta) (the score scale is
// applied once to the accumulated dQ / dK instead); P goes over the first 64 columns of S and
// dS' over the first 64 columns of dP (or of S when P is not wanted), as packed 16-bit pairs.
// Entry e of the row is admitted when e_lo <= e <= e_hi (full: every entry); -L and -delta
// come per entry from shared memory (kPerCol) or are the row's own.
template <bool kBF16, bool kWantP, bool kPerCol, int NCH, bool kMask = false, typename F = int>
__device__ __forceinline__ void grad_tile(uint32_t tS, uint32_t tdP, float scale_log2, int e_lo, int e_hi,
                                          bool full, float nL_row, float nd_row, const float* nL_col,
                                          const float* nd_col, F extra = 0) {
  const f2_t sl2 = f2_pack(scale_log2, scale_log2);
  const f2_t nL_r = f2_pack(nL_row, nL_row), nd_r = f2_pack(nd_row, nd_row);
#pragma unroll 1
  for (int c = 0; c < NCH; ++c) {
    uint32_t us[32], ud[32];
    tmem_ld32(tS + c * 32, us);
    tmem_ld32(tdP + c * 32, ud);
    tmem_ld_wait();
    uint32_t pw[16], dw[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const int col = c * 32 + e;
      f2_t nL = nL_r, nd = nd_r;
      if constexpr (kPerCol) {
        const float2 Lv = *reinterpret_cast<const float2*>(nL_col + col);
        const float2 dv = *reinterpret_cast<const float2*>(nd_col + col);
        nL = f2_pack(Lv.x, Lv.y);
        nd = f2_pack(dv.x, dv.y);
      }
      if constexpr (kMask) {
        // the masks' additive terms (natural units) join the exponent's offset
        float a0, a1;
        f2_unpack(nL, a0, a1);
        nL = f2_pack(fmaf(extra(col), kLog2e, a0), fmaf(extra(col + 1), kLog2e, a1));
      }
      float p0, p1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(us[e]), __uint_as_float(us[e + 1])), sl2, nL), p0, p1);
      p0 = ex2_approx(p0);
      p1 = ex2_approx(p1);
      if (!full) {
        if (col < e_lo || col > e_hi) p0 = 0.f;
        if (col + 1 < e_lo || col + 1 > e_hi) p1 = 0.f;
      }
      const f2_t pp = f2_pack(p0, p1);
      const f2_t g = f2_mul(pp, f2_add(f2_pack(__uint_as_float(ud[e]), __uint_as_float(ud[e + 1])), nd));
      float g0, g1;
      f2_unpack(g, g0, g1);
      if constexpr (kWantP) pw[e >> 1] = pack2<kBF16>(p0, p1);
      dw[e >> 1] = pack2<kBF16>(g0, g1);
    }
    // chunk c's 16 packed columns land in columns already read (16c..16c+15 < 32(c+1))
    if constexpr (kWantP) tmem_st16(tS + c * 16, pw);
    tmem_st16(kWantP ? tdP + c * 16 : tS + c * 16, dw);
  }
  tmem_st_wait();
}

// Writes a 128-lane accumulator row (D columns, fp32 in TMEM) times mul as 16-bit values,
// or zeros.
template <int D, bool kBF16>
__device__ __forceinline__ void store_row(uint32_t tAcc, bool have, bool valid, float mul, void* dst) {
  using T = typename std::conditional<kBF16, __nv_bfloat16, __half>::type;
  T* out = reinterpret_cast<T*>(dst);
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    if (have) {
      tmem_ld32(tAcc + c * 32, o);
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
        for (int e = 0; e < 4; ++e)
          w[e] = pack2<kBF16>(__uint_as_float(o[q * 8 + 2 * e]) * mul, __uint_as_float(o[q * 8 + 2 * e + 1]) * mul);
        *reinterpret_cast<uint4*>(out + c * 32 + q * 8) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

constexpr uint64_t kDrainNs = 2000000000ull;

// ------------------------------------------------------------------------- dK, dV
template <int H, int STEP, bool kBF16>
__global__ void __launch_bounds__(BCfg<H, STEP>::kThreads, BCfg<H, STEP>::kMinBlocks)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tg,
                    const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, const BwdArgs a) {
  using C = BCfg<H, STEP>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_kv, bar_sready, bar_pready, bar_acc, bar_stat[2];
  __shared__ __align__(8) uint64_t bar_full[C::kStages], bar_empty[C::kStages];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ __align__(16) float sh_L[2][kBM], sh_d[2][kBM];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // work unit: key tile (heavy first under causal rules), then (batch, kv head)
  const int kt = blockIdx.x / (a.B * a.Nkv);
  const int bh = blockIdx.x % (a.B * a.Nkv);
  const int b = bh / a.Nkv, kvh = bh % a.Nkv;
  const int64_t len_b = len_of(a, b);
  const int64_t k0 = (int64_t)kt * kBM, k1 = bmin((int64_t)a.T, k0 + kBM) - 1;

  // query steps that admit some key of this tile: a contiguous range (the bounds grow with i)
  const int nqs = (a.S + STEP - 1) / STEP;
  int qt_lo = nqs, qt_hi = -1;
  for (int qt = 0; qt < nqs; ++qt) {
    int64_t lo0, hi0, lo1, hi1;
    key_range(a, len_b, (int64_t)qt * STEP, lo0, hi0);
    key_range(a, len_b, bmin((int64_t)a.S, (int64_t)qt * STEP + STEP) - 1, lo1, hi1);
    const int64_t lo = bmin(lo0, lo1), hi = bmax(hi0, hi1);
    if (hi >= lo && lo <= k1 && hi >= k0) {
      if (qt < qt_lo) qt_lo = qt;
      qt_hi = qt;
    }
  }
  const int nqt = qt_hi >= qt_lo ? qt_hi - qt_lo + 1 : 0;
  const int n_steps = nqt * a.group;   // step n: query step qt_lo + n / group, head n % group

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase, sV = sbase + C::kTile, sRing = sbase + 2 * C::kTile;
  const uint32_t b_kv = smem_u32(&bar_kv), b_sready = smem_u32(&bar_sready), b_pready = smem_u32(&bar_pready);
  const uint32_t b_acc = smem_u32(&bar_acc);
  auto b_full = [&](int s) { return smem_u32(&bar_full[s]); };
  auto b_empty = [&](int s) { return smem_u32(&bar_empty[s]); };
  volatile int* abortp = &abort_flag;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(b_kv, 1);
    mbar_init(smem_u32(&bar_stat[0]), kBM);
    mbar_init(smem_u32(&bar_stat[1]), kBM);
    mbar_init(b_sready, 1);
    mbar_init(b_pready, kBM);
    mbar_init(b_acc, 1);
    for (int s = 0; s < C::kStages; ++s) { mbar_init(b_full(s), 1); mbar_init(b_empty(s), 1); }
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
    // ======================================================== TMA producer
    if (n_steps > 0) {
      const uint32_t leader = elect_one();   // issues every copy, MMA and commit of the warp
      if (leader) {
        prefetch_tmap(&tq); prefetch_tmap(&tg); prefetch_tmap(&tk); prefetch_tmap(&tv);
      }
      int c1, c2, c3;
      if (leader) mbar_arrive_expect_tx(b_kv, 2 * C::kTile);
      perm_coords(a.kv_ds, a.kv_dn, a.kv_db, (int)k0, kvh, b, c1, c2, c3);
      for (int r = 0; r < C::kRegions; ++r) {
        if (leader) tma_load_4d(sK + r * C::kRegionBytes, &tk, b_kv, 64 * r, c1, c2, c3);
        if (leader) tma_load_4d(sV + r * C::kRegionBytes, &tv, b_kv, 64 * r, c1, c2, c3);
      }
      int n = 0;
      for (; n < n_steps; ++n) {
        const int st = n % C::kStages;
        if (n >= C::kStages &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(b_empty(st), ((n / C::kStages) - 1) & 1, abortp, a.wait_ns)))
          break;
        const int qt = qt_lo + n / a.group, h = kvh * a.group + n % a.group;
        const uint32_t sQ = sRing + st * 2 * C::kSTile, sG = sQ + C::kSTile;
        if (leader) mbar_arrive_expect_tx(b_full(st), 2 * C::kSTile);
        perm_coords(a.q_ds, a.q_dn, a.q_db, qt * STEP, h, b, c1, c2, c3);
        for (int r = 0; r < C::kRegions; ++r) if (leader) tma_load_4d(sQ + r * C::kSRegionBytes, &tq, b_full(st), 64 * r, c1, c2, c3);
        perm_coords(a.g_ds, a.g_dn, a.g_db, qt * STEP, h, b, c1, c2, c3);
        for (int r = 0; r < C::kRegions; ++r) if (leader) tma_load_4d(sG + r * C::kSRegionBytes, &tg, b_full(st), 64 * r, c1, c2, c3);
      }
      if (__any_sync(0xffffffffu, n < n_steps || *abortp)) {
        // some role gave up: let every copy already issued land before the CTA can exit
        mbar_wait_bounded(b_kv, 0, nullptr, kDrainNs);
        for (int s = 0; s < C::kStages && s < n; ++s) {
          const int last = s + ((n - 1 - s) / C::kStages) * C::kStages;
          mbar_wait_bounded(b_full(s), (last / C::kStages) & 1, nullptr, kDrainNs);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================================================== MMA issuer
    if (n_steps > 0) {
      const uint32_t leader = elect_one();   // issues every copy, MMA and commit of the warp
      constexpr uint32_t kIdS = idesc_f16(kBF16, kBM, STEP, false);  // M keys, N queries
      constexpr uint32_t kIdA = idesc_f16(kBF16, kBM, H, true);      // M keys, N head dims
      const uint32_t tS = tmem + C::kTmemS, tP = tmem + C::kTmemP;
      const uint32_t tdK = tmem + C::kTmemA0, tdV = tmem + C::kTmemA1;
      const uint64_t dK = desc_sw128(sK, 16, 1024), dV = desc_sw128(sV, 16, 1024);
      bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_kv, 0, abortp, a.wait_ns));
      tc_fence_after();
      for (int n = 0; n < n_steps && ok; ++n) {
        const int st = n % C::kStages;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_full(st), (n / C::kStages) & 1, abortp, a.wait_ns)))) break;
        tc_fence_after();
        const uint32_t sQ = sRing + st * 2 * C::kSTile, sG = sQ + C::kSTile;
        const uint64_t dQk = desc_sw128(sQ, 16, 1024), dGk = desc_sw128(sG, 16, 1024);
        const uint64_t dQm = desc_sw128(sQ, C::kSRegionBytes, 1024), dGm = desc_sw128(sG, C::kSRegionBytes, 1024);
        // S^T = K Q^T and dP^T = V dY^T (after the accumulations of step n-1 read P^T / dS^T)
#pragma unroll
        for (int kk = 0; kk < H / 16; ++kk) {
          const uint64_t offa = (uint64_t)(((kk / 4) * C::kRegionBytes + (kk % 4) * 32) >> 4);
          const uint64_t offb = (uint64_t)(((kk / 4) * C::kSRegionBytes + (kk % 4) * 32) >> 4);
          if (leader) mma_f16_ss(tS, dK + offa, dQk + offb, kIdS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < H / 16; ++kk) {
          const uint64_t offa = (uint64_t)(((kk / 4) * C::kRegionBytes + (kk % 4) * 32) >> 4);
          const uint64_t offb = (uint64_t)(((kk / 4) * C::kSRegionBytes + (kk % 4) * 32) >> 4);
          if (leader) mma_f16_ss(tP, dV + offa, dGk + offb, kIdS, kk > 0);
        }
        if (leader) mma_commit(b_sready);
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_pready, n & 1, abortp, a.wait_ns)))) break;
        tc_fence_after();
        // dV += P^T dY and dK += dS^T Q: A from TMEM (16 queries = 8 columns per K step)
#pragma unroll
        for (int kk = 0; kk < STEP / 16; ++kk)
          if (leader) mma_f16_ts(tdV, tS + kk * 8, dGm + (uint64_t)((kk * 2048) >> 4), kIdA, (n > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < STEP / 16; ++kk)
          if (leader) mma_f16_ts(tdK, tP + kk * 8, dQm + (uint64_t)((kk * 2048) >> 4), kIdA, (n > 0 || kk > 0) ? 1u : 0u);
        if (leader) mma_commit(b_empty(st));
      }
      // the accumulators are final (or the CTA gave up) once every MMA completes
      if (leader) mma_commit(b_acc);
      mbar_wait_bounded(b_acc, 0, nullptr, kDrainNs);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ======================================================== one thread per key row
    const int sub = warp & 3;
    const int row = sub * 32 + lane;
    const int64_t j = k0 + row;                       // key of this thread
    const uint32_t trow = tmem + ((uint32_t)(sub * 32) << 16);
    const uint32_t tS = trow + C::kTmemS, tP = trow + C::kTmemP;
    int64_t qlo = 1, qhi = 0;
    if (j < a.T) query_range(a, len_b, j, qlo, qhi);
    bool ok = true;
    for (int n = 0; n < n_steps && ok; ++n) {
      const int qt = qt_lo + n / a.group, h = kvh * a.group + n % a.group;
      const int64_t q0 = (int64_t)qt * STEP;
      // statistics of the step's STEP query rows into shared memory (row q0 + row), double
      // buffered: a thread rewrites buffer n & 1 only after every thread arrived for step n-1,
      // that is after every thread finished reading it in step n-2
      {
        const int64_t i = q0 + row;
        float L = INFINITY, d = 0.f;
        if (row < STEP && i < a.S) {
          const int64_t idx = ((int64_t)b * a.Nq + h) * a.S + i;
          L = a.lse2[idx];
          d = a.delta[idx];
        }
        sh_L[n & 1][row] = -L;
        sh_d[n & 1][row] = -d;
        const uint32_t bst = smem_u32(&bar_stat[n & 1]);
        mbar_arrive(bst);
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(bst, (n >> 1) & 1, abortp, a.wait_ns)))) break;
      }
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_sready, n & 1, abortp, a.wait_ns)))) break;
      tc_fence_after();
      const int e_lo = (int)bmax(-1, bmin((int64_t)STEP, qlo - q0));
      const int e_hi = (int)bmax(-1, bmin((int64_t)STEP, qhi - q0));
      const bool full = __all_sync(0xffffffffu, e_lo <= 0 && e_hi >= STEP - 1);
      if (a.has_extra) {
        // rows past S (a ragged last step) have L = +inf; their masks are not read
        auto extra = [&](int col) { return q0 + col < a.S ? extra_term(a.r, len_b, b, h, q0 + col, j) : 0.f; };
        grad_tile<kBF16, true, true, STEP / 32, true>(tS, tP, a.scale_log2, e_lo, e_hi, full, 0.f, 0.f,
                                                      sh_L[n & 1], sh_d[n & 1], extra);
      } else {
        grad_tile<kBF16, true, true, STEP / 32>(tS, tP, a.scale_log2, e_lo, e_hi, full, 0.f, 0.f, sh_L[n & 1],
                                                 sh_d[n & 1]);
      }
      tc_fence_before();
      mbar_arrive(b_pready);
    }
    if (ok && n_steps > 0) ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_acc, 0, abortp, a.wait_ns));
    if (ok) {
      tc_fence_after();
      const bool valid = j < a.T;
      char* dk = reinterpret_cast<char*>(a.out0) + (b * a.o0_sb + (int64_t)kvh * a.o0_sh + j * a.o0_ss) * 2;
      char* dv = reinterpret_cast<char*>(a.out1) + (b * a.o1_sb + (int64_t)kvh * a.o1_sh + j * a.o1_ss) * 2;
      store_row<H, kBF16>(trow + C::kTmemA0, n_steps > 0, valid, a.scale, dk);
      store_row<H, kBF16>(trow + C::kTmemA1, n_steps > 0, valid, 1.f, dv);
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && abort_flag) atomicExch(&g_bwd_status, (int)SDPA_ERR_TIMEOUT);
}

// ------------------------------------------------------------------------- dQ
template <int H, int STEP, bool kBF16>
__global__ void __launch_bounds__(BCfg<H, STEP>::kThreads, BCfg<H, STEP>::kMinBlocks)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tg,
                  const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, const BwdArgs a) {
  using C = BCfg<H, STEP>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_q, bar_sready, bar_pready, bar_acc;
  __shared__ __align__(8) uint64_t bar_full[C::kStages], bar_empty[C::kStages];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // work unit: query tile (heavy first), then (batch, query head)
  int t = blockIdx.x;
  const int bh = t % (a.B * a.Nq);
  const int qt = a.nq_tiles - 1 - t / (a.B * a.Nq);
  const int b = bh / a.Nq, qh = bh % a.Nq, kvh = qh / a.group;
  const int64_t len_b = len_of(a, b);
  const int64_t m0 = (int64_t)qt * kBM, m1 = bmin((int64_t)a.S, m0 + kBM);
  int64_t lo0, hi0, lo1, hi1;
  key_range(a, len_b, m0, lo0, hi0);
  key_range(a, len_b, m1 - 1, lo1, hi1);
  const int64_t klo = bmax(0, bmin(lo0, lo1)), khi = bmin((int64_t)a.T - 1, bmax(hi0, hi1));
  const int kt0 = (int)(klo / STEP);
  const int n_steps = khi >= klo ? (int)(khi / STEP) - kt0 + 1 : 0;   // STEP keys per step

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase, sG = sbase + C::kTile, sRing = sbase + 2 * C::kTile;
  const uint32_t b_q = smem_u32(&bar_q), b_sready = smem_u32(&bar_sready), b_pready = smem_u32(&bar_pready);
  const uint32_t b_acc = smem_u32(&bar_acc);
  auto b_full = [&](int s) { return smem_u32(&bar_full[s]); };
  auto b_empty = [&](int s) { return smem_u32(&bar_empty[s]); };
  volatile int* abortp = &abort_flag;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(b_q, 1);
    mbar_init(b_sready, 1);
    mbar_init(b_pready, kBM);
    mbar_init(b_acc, 1);
    for (int s = 0; s < C::kStages; ++s) { mbar_init(b_full(s), 1); mbar_init(b_empty(s), 1); }
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
    // ======================================================== TMA producer
    if (n_steps > 0) {
      const uint32_t leader = elect_one();   // issues every copy, MMA and commit of the warp
      if (leader) {
        prefetch_tmap(&tq); prefetch_tmap(&tg); prefetch_tmap(&tk); prefetch_tmap(&tv);
      }
      int c1, c2, c3;
      if (leader) mbar_arrive_expect_tx(b_q, 2 * C::kTile);
      perm_coords(a.q_ds, a.q_dn, a.q_db, (int)m0, qh, b, c1, c2, c3);
      for (int r = 0; r < C::kRegions; ++r) if (leader) tma_load_4d(sQ + r * C::kRegionBytes, &tq, b_q, 64 * r, c1, c2, c3);
      perm_coords(a.g_ds, a.g_dn, a.g_db, (int)m0, qh, b, c1, c2, c3);
      for (int r = 0; r < C::kRegions; ++r) if (leader) tma_load_4d(sG + r * C::kRegionBytes, &tg, b_q, 64 * r, c1, c2, c3);
      int n = 0;
      for (; n < n_steps; ++n) {
        const int st = n % C::kStages;
        if (n >= C::kStages &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(b_empty(st), ((n / C::kStages) - 1) & 1, abortp, a.wait_ns)))
          break;
        const uint32_t sK = sRing + st * 2 * C::kSTile, sV = sK + C::kSTile;
        if (leader) mbar_arrive_expect_tx(b_full(st), 2 * C::kSTile);
        perm_coords(a.kv_ds, a.kv_dn, a.kv_db, (kt0 + n) * STEP, kvh, b, c1, c2, c3);
        for (int r = 0; r < C::kRegions; ++r) {
          if (leader) tma_load_4d(sK + r * C::kSRegionBytes, &tk, b_full(st), 64 * r, c1, c2, c3);
          if (leader) tma_load_4d(sV + r * C::kSRegionBytes, &tv, b_full(st), 64 * r, c1, c2, c3);
        }
      }
      if (__any_sync(0xffffffffu, n < n_steps || *abortp)) {
        mbar_wait_bounded(b_q, 0, nullptr, kDrainNs);
        for (int s = 0; s < C::kStages && s < n; ++s) {
          const int last = s + ((n - 1 - s) / C::kStages) * C::kStages;
          mbar_wait_bounded(b_full(s), (last / C::kStages) & 1, nullptr, kDrainNs);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================================================== MMA issuer
    if (n_steps > 0) {
      const uint32_t leader = elect_one();   // issues every copy, MMA and commit of the warp
      constexpr uint32_t kIdS = idesc_f16(kBF16, kBM, STEP, false);  // M queries, N keys
      constexpr uint32_t kIdA = idesc_f16(kBF16, kBM, H, true);      // M queries, N head dims
      const uint32_t tS = tmem + C::kTmemS, tP = tmem + C::kTmemP, tdQ = tmem + C::kTmemA0;
      const uint64_t dQ = desc_sw128(sQ, 16, 1024), dG = desc_sw128(sG, 16, 1024);
      bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_q, 0, abortp, a.wait_ns));
      tc_fence_after();
      for (int n = 0; n < n_steps && ok; ++n) {
        const int st = n % C::kStages;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_full(st), (n / C::kStages) & 1, abortp, a.wait_ns)))) break;
        tc_fence_after();
        const uint32_t sK = sRing + st * 2 * C::kSTile, sV = sK + C::kSTile;
        const uint64_t dKk = desc_sw128(sK, 16, 1024), dVk = desc_sw128(sV, 16, 1024);
        const uint64_t dKm = desc_sw128(sK, C::kSRegionBytes, 1024);
        // S = Q K^T and dP = dY V^T (after dQ of step n-1 read dS)
#pragma unroll
        for (int kk = 0; kk < H / 16; ++kk) {
          const uint64_t offa = (uint64_t)(((kk / 4) * C::kRegionBytes + (kk % 4) * 32) >> 4);
          const uint64_t offb = (uint64_t)(((kk / 4) * C::kSRegionBytes + (kk % 4) * 32) >> 4);
          if (leader) mma_f16_ss(tS, dQ + offa, dKk + offb, kIdS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < H / 16; ++kk) {
          const uint64_t offa = (uint64_t)(((kk / 4) * C::kRegionBytes + (kk % 4) * 32) >> 4);
          const uint64_t offb = (uint64_t)(((kk / 4) * C::kSRegionBytes + (kk % 4) * 32) >> 4);
          if (leader) mma_f16_ss(tP, dG + offa, dVk + offb, kIdS, kk > 0);
        }
        if (leader) mma_commit(b_sready);
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_pready, n & 1, abortp, a.wait_ns)))) break;
        tc_fence_after();
        // dQ += dS K: dS from TMEM (16 keys = 8 columns per K step), K MN-major
#pragma unroll
        for (int kk = 0; kk < STEP / 16; ++kk)
          if (leader) mma_f16_ts(tdQ, tS + kk * 8, dKm + (uint64_t)((kk * 2048) >> 4), kIdA, (n > 0 || kk > 0) ? 1u : 0u);
        if (leader) mma_commit(b_empty(st));
      }
      if (leader) mma_commit(b_acc);
      mbar_wait_bounded(b_acc, 0, nullptr, kDrainNs);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ======================================================== one thread per query row
    const int sub = warp & 3;
    const int row = sub * 32 + lane;
    const int64_t i = m0 + row;
    const uint32_t trow = tmem + ((uint32_t)(sub * 32) << 16);
    const uint32_t tS = trow + C::kTmemS, tP = trow + C::kTmemP;
    const bool valid = i < a.S;
    int64_t lo = 1, hi = 0;
    float L = INFINITY, d = 0.f;
    if (valid) {
      key_range(a, len_b, i, lo, hi);
      const int64_t idx = ((int64_t)b * a.Nq + qh) * a.S + i;
      L = a.lse2[idx];
      d = a.delta[idx];
    }
    bool ok = true;
    for (int n = 0; n < n_steps && ok; ++n) {
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_sready, n & 1, abortp, a.wait_ns)))) break;
      tc_fence_after();
      const int64_t key0 = (int64_t)(kt0 + n) * STEP;
      const int e_lo = (int)bmax(-1, bmin((int64_t)STEP, lo - key0));
      const int e_hi = (int)bmax(-1, bmin((int64_t)STEP, hi - key0));
      const bool full = __all_sync(0xffffffffu, e_lo <= 0 && e_hi >= STEP - 1);
      if (a.has_extra) {
        auto extra = [&](int col) { return valid ? extra_term(a.r, len_b, b, qh, i, key0 + col) : 0.f; };
        grad_tile<kBF16, false, false, STEP / 32, true>(tS, tP, a.scale_log2, e_lo, e_hi, full, -L, -d, nullptr,
                                                        nullptr, extra);
      } else {
        grad_tile<kBF16, false, false, STEP / 32>(tS, tP, a.scale_log2, e_lo, e_hi, full, -L, -d, nullptr, nullptr);
      }
      tc_fence_before();
      mbar_arrive(b_pready);
    }
    if (ok && n_steps > 0) ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_acc, 0, abortp, a.wait_ns));
    if (ok) {
      tc_fence_after();
      char* dq = reinterpret_cast<char*>(a.out0) + (b * a.o0_sb + (int64_t)qh * a.o0_sh + i * a.o0_ss) * 2;
      store_row<H, kBF16>(trow + C::kTmemA0, n_steps > 0, valid, a.scale, dq);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && abort_flag) atomicExch(&g_bwd_status, (int)SDPA_ERR_TIMEOUT);
}

uint64_t bwd_wait_ns() {
  static uint64_t v = [] {
    const char* e = std::getenv("SDPA_WAIT_LIMIT_NS");
    return e ? std::strtoull(e, nullptr, 10) : 4000000000ull;
  }();
  return v;
}

// Maps: tq / tg cover Q and dY, tk / tv K and V; the "s" maps have STEP-row boxes (the
// streamed tiles), the others 128-row boxes (the resident ones).
template <int H, int STEP, bool kBF16>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tg, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tqs, const CUtensorMap& tgs, const CUtensorMap& tks,
                         const CUtensorMap& tvs, const BwdArgs& a_kv, const BwdArgs& a_q, cudaStream_t st) {
  using C = BCfg<H, STEP>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(bwd_dkdv_kernel<H, STEP, kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(bwd_dq_kernel<H, STEP, kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t g1 = (int64_t)a_kv.nk_tiles * a_kv.B * a_kv.Nkv;
  const int64_t g2 = (int64_t)a_q.nq_tiles * a_q.B * a_q.Nq;
  if (g1 > 0x7fffffff || g2 > 0x7fffffff) return cudaErrorInvalidValue;
  if (g1 > 0) {
    bwd_dkdv_kernel<H, STEP, kBF16><<<(unsigned)g1, C::kThreads, C::kSmem, st>>>(tqs, tgs, tk, tv, a_kv);
    count_launch(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (g2 > 0) {
    bwd_dq_kernel<H, STEP, kBF16><<<(unsigned)g2, C::kThreads, C::kSmem, st>>>(tq, tg, tks, tvs, a_q);
    count_launch(1);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

bool bwd_tc_supported(const Problem& p, sdpa_dtype dt) {
  if (dt != SDPA_F16 && dt != SDPA_BF16) return false;
  if (p.H != p.Hv || (p.H != 64 && p.H != 128)) return false;
  return p.T <= (int64_t)1 << 30 && p.S <= (1 << 30) && p.r.window <= (int64_t)1 << 30;
}

cudaError_t launch_bwd_tc(const Problem& p, sdpa_dtype dt, const View& dy, const View& dq, const View& dk,
                          const View& dv, float* lse2, float* delta, cudaStream_t st, const char** name) {
  // statistics pass: the forward kernel writes L and delta, no y
  Problem fp = p;
  fp.y = View{};
  const char* fname = "";
  cudaError_t e = launch_prefill_tc_stats(fp, dt, lse2, delta, &dy, st, &fname);
  if (e != cudaSuccess) return e;

  BwdArgs a{};
  a.B = p.B; a.Nq = p.Nq; a.Nkv = p.Nkv; a.S = p.S; a.T = (int)p.T; a.group = p.group;
  a.scale = p.scale;
  a.scale_log2 = p.scale * kLog2e;
  a.causal = p.r.causal;
  a.window = (int)p.r.window;
  a.len_kind = p.r.len_kind;
  a.lens = p.r.lens;
  a.lse2 = lse2;
  a.delta = delta;
  a.r = p.r;
  a.has_extra = p.r.add != nullptr || p.r.keep_kind != SDPA_KEEP_NONE || p.r.len_kind == SDPA_LEN_KEYLEN_I32;
  a.nq_tiles = (p.S + kBM - 1) / kBM;
  a.nk_tiles = (int)((p.T + kBM - 1) / kBM);
  a.wait_ns = bwd_wait_ns();
  if (!tc_encode_fn()) return cudaErrorNotSupported;
  // 64-row streamed tiles for H = 64 (two CTAs per SM), 128 rows for H = 128
  const int step = p.H == 64 ? 64 : 128;
  CUtensorMap tq, tg, tk, tv, tqs, tgs, tks, tvs;
  int vds, vdn, vdb, x1, x2, x3;
  if (!tc_make_map(&tq, p.q, dt, p.B, p.Nq, p.S, p.H, &a.q_ds, &a.q_dn, &a.q_db) ||
      !tc_make_map(&tg, dy, dt, p.B, p.Nq, p.S, p.Hv, &a.g_ds, &a.g_dn, &a.g_db) ||
      !tc_make_map(&tk, p.k, dt, p.B, p.Nkv, p.T, p.H, &a.kv_ds, &a.kv_dn, &a.kv_db) ||
      !tc_make_map(&tv, p.v, dt, p.B, p.Nkv, p.T, p.Hv, &vds, &vdn, &vdb) ||
      !tc_make_map(&tqs, p.q, dt, p.B, p.Nq, p.S, p.H, &x1, &x2, &x3, step) ||
      !tc_make_map(&tgs, dy, dt, p.B, p.Nq, p.S, p.Hv, &x1, &x2, &x3, step) ||
      !tc_make_map(&tks, p.k, dt, p.B, p.Nkv, p.T, p.H, &x1, &x2, &x3, step) ||
      !tc_make_map(&tvs, p.v, dt, p.B, p.Nkv, p.T, p.Hv, &x1, &x2, &x3, step))
    return cudaErrorInvalidValue;
  if (vds != a.kv_ds || vdn != a.kv_dn || vdb != a.kv_db) return cudaErrorInvalidValue;
  BwdArgs akv = a, aq = a;
  akv.out0 = const_cast<void*>(dk.p); akv.o0_sb = dk.sb; akv.o0_sh = dk.sh; akv.o0_ss = dk.ss;
  akv.out1 = const_cast<void*>(dv.p); akv.o1_sb = dv.sb; akv.o1_sh = dv.sh; akv.o1_ss = dv.ss;
  aq.out0 = const_cast<void*>(dq.p); aq.o0_sb = dq.sb; aq.o0_sh = dq.sh; aq.o0_ss = dq.ss;
  const bool bf = dt == SDPA_BF16;
  if (p.H == 128) {
    *name = bf ? "bwd_tc_bf16_h128" : "bwd_tc_f16_h128";
    return bf ? launch_bwd_t<128, 128, true>(tq, tg, tk, tv, tqs, tgs, tks, tvs, akv, aq, st)
              : launch_bwd_t<128, 128, false>(tq, tg, tk, tv, tqs, tgs, tks, tvs, akv, aq, st);
  }
  *name = bf ? "bwd_tc_bf16_h64" : "bwd_tc_f16_h64";
  return bf ? launch_bwd_t<64, 64, true>(tq, tg, tk, tv, tqs, tgs, tks, tvs, akv, aq, st)
            : launch_bwd_t<64, 64, false>(tq, tg, tk, tv, tqs, tgs, tks, tvs, akv, aq, st);
}

cudaError_t take_bwd_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_bwd_status, sizeof v);
  if (e != cudaSuccess) return e;
  *status = v;
  if (v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof zero);
  }
  return e;
}

}  // namespace sdpa
