// Fused tensor-core prefill for GB300 (sm_103a): TMA-staged Q/K/V tiles, tcgen05.mma with
// accumulators in tensor memory, an online softmax with fp32 statistics in registers,
// and the masking rules of onnx-light class Attention / MultiHeadAttention /
// GroupQueryAttention applied per element in registers.
//
// Persistent: one CTA per SM walks a share of the work units (heavy first).  A unit is two
// 128-row query tiles that stream the same key/value tiles: two query heads of one GQA group
// over one row block, or two consecutive row blocks of one head.
//
//   warp 0      TMA producer: the unit's first K tile, its Q tiles (once the previous unit's
//               last S MMAs have read the buffer), then V_0, K_1, V_1, ... into the ring
//   warp 1      MMA issuer (the whole warp runs the loop, one elected lane issues):
//               S_X = Q_X K_j^T into TMEM, O_X += P_X V_j with P read from TMEM
//   warps 4-7   softmax of tile 0: each thread owns one query row (TMEM lane = row)
//   warps 8-11  softmax of tile 1
//
// The two softmax warpgroups alternate with the tensor core: while one works on its
// scores the MMA warp computes the other's products.  Running maxima are kept in the
// base-2 domain and only moved (with a rescale of the TMEM accumulator) when they grow
// by more than 2^8, so most tiles skip the rescale.  A unit's epilogue (each softmax warp
// stages its rows of y in shared memory and writes them with TMA stores) runs at the top of
// the warp's next pass over the unit list; before the first unit the same code runs once dry.
//
// Every barrier wait is bounded: on expiry the kernel raises an abort flag, drains the
// copies and MMAs it issued, frees its tensor memory and records SDPA_ERR_TIMEOUT in a
// device status word (read by sdpa_query_status).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
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
// CTA shape for QT 128-row query tiles per CTA and SPLIT softmax threads per query row (each
// owns 128 / SPLIT score columns of a key tile).  The kernel instantiates QT = 2 (one CTA per
// SM) and SPLIT = 1.
template <int QT, int SPLIT>
struct Layout {
  static constexpr int kSmxThreads = 128 * QT * SPLIT;    // softmax warpgroups
  static constexpr int kThreads = 128 + kSmxThreads;      // + 4 control warps
  static constexpr int kMinBlocks = (QT == 1) ? 2 : 1;
  // Register split (setmaxnreg): the control warpgroup shrinks to kCtlRegs, the softmax
  // warpgroups grow to kSmxRegs.  The sum must not exceed what the block was launched with
  // (kThreads x the kernel's register count), which the host checks before every launch.
  static constexpr int kLaunchRegs = (65536 / (kThreads * kMinBlocks)) & ~7;
#ifndef SDPA_CTL_REGS_SMALL
#define SDPA_CTL_REGS_SMALL 56
#endif
  // (88 with two tiles: the MMA warp's descriptors and counters fit without spilling, and the
  // softmax warpgroups keep 208)
  static constexpr int kCtlRegs = (kLaunchRegs <= 96) ? SDPA_CTL_REGS_SMALL : ((QT == 1) ? 64 : 88);
  static constexpr int kSmxRegs = ((kLaunchRegs * kThreads - kCtlRegs * 128) / kSmxThreads) & ~7;
  static_assert(kSmxRegs <= 256 && kSmxRegs >= kLaunchRegs, "register split");
  static_assert(kCtlRegs * 128 + kSmxRegs * kSmxThreads <= kLaunchRegs * kThreads, "register split");
};
constexpr float kRescaleThreshold = 8.f;   // log2 units
// Softcap tanh(u) on |u| <= kTanhPolyLimit uses u - u^3/3 + 2u^5/15 on the FMA pipe: the
// alternating Taylor series' error is below its next term, 17/315 u^7 <= 3.3e-6.
constexpr float kTanhPolyLimit = 0.25f;
constexpr float kTanhA1 = -1.f / 3.f, kTanhA2 = 2.f / 15.f;

// Softcap with a fixed maximum (bf16 only): tanh(u) on |u| <= kTanhPolyLimit by the odd cubic
// minimax fit a1 u + a3 u^3 (Remez exchange on [0, 0.25]; maximum error 7.8e-6).
constexpr float kTanhMM1 = 0.99984343f, kTanhMM3 = -0.32319898f;

__device__ __forceinline__ float tanh_poly(float u) {
  const float z = u * u;
  const float q = fmaf(z, kTanhA2, kTanhA1);
  const float w = u * z;
  return fmaf(w, q, u);
}

// Keys outside the admitted interval [elo, ehi] of a row's tile segment (element indices) take
// the value fill.  Per 32-column chunk the admitted keys are formed once as a bit set, so each
// key then costs one bit test and one select, with no branches (branches that overwrite parts
// of the score array cost registers in the softmax warps).
template <int N>
__device__ __forceinline__ void clip_interval(float (&s)[N], int elo, int ehi, float fill) {
#pragma unroll
  for (int c0 = 0; c0 < N; c0 += 32) {
    const int lo = max(elo - c0, 0), hi = min(ehi - c0, 31);
    const uint32_t up = 0xffffffffu >> (31 - max(hi, 0));   // bits 0 .. hi
    const uint32_t m = (lo <= hi) ? (up & (0xffffffffu << min(lo, 31))) : 0u;
#pragma unroll
    for (int e = 0; e < 32; ++e) s[c0 + e] = ((m >> e) & 1u) ? s[c0 + e] : fill;
  }
}

// Shapes of one kernel variant: H = head size of Q and K, HV = head size of V (64 or 128 each).
template <int H, int HV, int kQT, bool kMaskStage = false>
struct Cfg {
  static_assert(kQT == 2, "two query tiles per CTA");
  static_assert((H == 64 || H == 128) && (HV == 64 || HV == 128), "head sizes");
  static constexpr int kRegions = H / 64;              // 128-byte swizzle regions per Q / K row
  static constexpr int kVRegions = HV / 64;            // ... per V row
  static constexpr int kRegionBytes = 128 * 128;       // 128 rows x 128 bytes
  static constexpr int kQTile = kBM * H * 2;
  static constexpr int kKTile = kBN * H * 2;
  static constexpr int kVTile = kBN * HV * 2;
  static constexpr int kKVTile = kKTile > kVTile ? kKTile : kVTile;   // one ring slot
  // Q holds the unit's two tiles; the next unit's tiles load once the current unit's last S
  // MMAs have read them
  static constexpr int kQBuf = kQT * kQTile;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQBuf;
  // additive-mask staging: per softmax warp its 32 rows x 128 16-bit columns, 16-byte chunks
  // of row r swizzled by r mod 16
  static constexpr int kMaskWarpBytes = 32 * kBN * 2;
  static constexpr int kMaskBytes = kMaskStage ? 4 * kQT * kMaskWarpBytes : 0;
  // output staging for the TMA stores of y: per softmax warp 32 rows x 64 columns (4 KB,
  // 128-byte swizzle); the additive-mask mode reuses the warp's mask region
  static constexpr int kYWarpBytes = 32 * 128;
  static constexpr int kYBytes = kMaskStage ? 0 : 4 * kQT * kYWarpBytes;
  // K/V ring depth: what is left of the shared memory, at most 10 slots, and 6 with a staged
  // mask, whose ragged last tile is read through L1 (measured: 8 slots left it too little
  // L1 and were slower)
  static constexpr int kSmemMax = 232448;
  static constexpr int kStagesFit = (kSmemMax - 1024 - kQBuf - kMaskBytes - kYBytes) / kKVTile;
  static constexpr int kStagesCap = kMaskStage ? 6 : 10;
  static constexpr int kStages = kStagesFit < kStagesCap ? kStagesFit : kStagesCap;
  static constexpr int kMaskOff = kKVOff + kStages * kKVTile;
  static constexpr int kYOff = kMaskOff + kMaskBytes;
  static constexpr int kSmem = kYOff + kYBytes + 1024;   // + alignment slack
  static_assert(kSmem <= kSmemMax && kStages >= 3, "shared memory");
  // Tensor memory: S_X (128 columns each), O_X (HV columns each) and P_X (16-bit, two per
  // column: 64 columns).  With HV = 128 there is no room for P: P_X overwrites the first 64
  // columns of S_X once S_X is in registers.
  static constexpr bool kAlias = (HV == 128);
  static constexpr int kTmemS0 = 0, kTmemS1 = 128;
  static constexpr int kTmemO0 = 128 * kQT, kTmemO1 = kTmemO0 + HV;
  static constexpr int kTmemP0 = kAlias ? kTmemS0 : kTmemO0 + kQT * HV;
  static constexpr int kTmemP1 = kAlias ? kTmemS1 : kTmemP0 + 64;
  static constexpr uint32_t kTmemCols = 256 * kQT;
};

struct TcArgs {
  int B, Nq, Nkv, S, T, group;
  int nunits;                                       // work units (two query tiles each)
  int nrow;                                         // row blocks per (batch, head or head pair)
  int pairs;                                        // units per (batch, kv head, row block)
  int head_pairs;                                   // 1: the tiles of a unit are two heads of a group
  float scale, scale_log2, cap_in, cap_out_log2;   // cap_* used when softcap > 0
  int has_softcap;
  int cap_fixed;                                    // bf16 softcap: fixed row maximum (below)
  float fx_a, fx_b, fx_lim;                         // cubic coefficients on raw q.k, its range
  int causal, window, len_kind;
  const void* lens;
  int generic;                                      // per-element rules beyond the structural ones
  int add_fast;                                     // additive mask only: vectorised path
  int add_vec;                                      // bytes per mask load (2, 4, 8 or 16)
  int add_stage;                                    // mask tiles staged through shared memory
  int keep_fast;                                    // keep mask / key-length filter, no float mask
  int keep_vec;                                     // keep-mask rows allow 16-byte loads
  float filter_raw;                                 // mask_filter_value in units of raw q.k
  Rules r;
  int q_ds, q_dn, q_db, kv_ds, kv_dn, kv_db;        // tensor-map dimension of seq / head / batch
  void* y;                                          // NULL: y is not written (statistics only)
  int64_t y_sb, y_sh, y_ss;
  int y_ds, y_dn, y_db;                             // tensor-map dimension of seq / head / batch of y
  // Row statistics for the backward pass (one thread per row only): the log2-sum-exp of the
  // row in units of q.k scale log2(e), and delta = dY . O (O normalised, fp32), indexed
  // (b * Nq + h) * S + i.  NULL: not written.
  float* lse2_out;
  float* delta_out;
  const void* dy;
  int64_t dy_sb, dy_sh, dy_ss;
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

// Mask values of columns c0 .. c0+7 of one 16-bit mask row into w[4] (elements 2v, 2v+1 in
// w[v]): the widest loads the row alignment vec allows, -inf past the mask's T_mask columns.
template <typename M>
__device__ __forceinline__ void load_mask_chunk(const M* row, int c0, int64_t T_mask, int vec, uint32_t* w) {
  static_assert(sizeof(M) == 2, "16-bit masks");
  const unsigned short* h = reinterpret_cast<const unsigned short*>(row);
  if ((int64_t)c0 + 8 <= T_mask) {
    if (vec >= 16) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(h + c0));
      w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
    } else if (vec >= 8) {
      const uint2 u0 = __ldg(reinterpret_cast<const uint2*>(h + c0)), u1 = __ldg(reinterpret_cast<const uint2*>(h + c0 + 4));
      w[0] = u0.x; w[1] = u0.y; w[2] = u1.x; w[3] = u1.y;
    } else if (vec >= 4) {
#pragma unroll
      for (int v = 0; v < 4; ++v) w[v] = __ldg(reinterpret_cast<const uint32_t*>(h + c0) + v);
    } else {
#pragma unroll
      for (int v = 0; v < 4; ++v) w[v] = (uint32_t)__ldg(h + c0 + 2 * v) | ((uint32_t)__ldg(h + c0 + 2 * v + 1) << 16);
    }
  } else {
    const unsigned short ninf = std::is_same<M, __half>::value ? 0xFC00u : 0xFF80u;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int64_t e0 = (int64_t)c0 + 2 * v, e1 = e0 + 1;
      const uint32_t lo = e0 < T_mask ? __ldg(h + e0) : ninf;
      const uint32_t hi = e1 < T_mask ? __ldg(h + e1) : ninf;
      w[v] = lo | (hi << 16);
    }
  }
}

// Additive-mask staging.  One warp copies the 128-column tile of its 32 mask rows into its
// shared-memory region with coalesced cp.async (row-contiguous; 16-byte chunk c of row r at
// r * 256 + (c ^ (r & 15)) * 16), so that each thread can then read its own row without bank
// conflicts.  row0 is the warp's first mask row, row_bytes the row stride, rows the rows that
// exist (the rest are not read), vec the alignment of every row start (4, 8 or 16 bytes).
__device__ __forceinline__ void stage_mask_tile(uint32_t dst, const char* row0, int64_t row_bytes, int rows,
                                                int vec, int lane) {
  if (vec >= 16) {
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const int r = 2 * n + (lane >> 4), c = lane & 15;
      if (r < rows) ptx::cp_async16(dst + r * 256 + ((c ^ (r & 15)) << 4), row0 + r * row_bytes + c * 16);
    }
  } else if (vec >= 8) {
#pragma unroll 8
    for (int r = 0; r < 32; ++r)
      if (r < rows)
        ptx::cp_async8(dst + r * 256 + (((lane >> 1) ^ (r & 15)) << 4) + ((lane & 1) << 3), row0 + r * row_bytes + lane * 8);
  } else {
#pragma unroll 4
    for (int r = 0; r < 32; ++r)
      if (r < rows) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int q = h * 32 + lane;
          ptx::cp_async4(dst + r * 256 + (((q >> 2) ^ (r & 15)) << 4) + ((q & 3) << 2), row0 + r * row_bytes + q * 4);
        }
      }
  }
  ptx::cp_async_commit();
}

template <typename M>
__device__ __forceinline__ float mask_elem(const uint32_t* raw, int e) {
  const unsigned short bits = (unsigned short)((e & 1) ? (raw[e >> 1] >> 16) : (raw[e >> 1] & 0xFFFFu));
  if constexpr (std::is_same<M, __half>::value) return __half2float(__ushort_as_half(bits));
  else return __bfloat162float(__ushort_as_bfloat16(bits));
}

__device__ __noinline__ float generic_score(const Rules& r, const RowCtx& ctx, float s_nat, int b, int h, int i,
                                            int64_t j) {
  return apply_rules(r, ctx, s_nat, b, h, i, j);
}

// Score-rule paths, fixed per launch.  kCapFixed: interval rules with softcap on bf16.  The
// capped logits lie in [-c, c], so the softmax uses the fixed maximum c (log2 domain: c log2 e)
// instead of a running one: no row maximum, no rescale of the accumulator.  Every weight is
// then at least 2^(-2 c log2 e), a normal number in fp32 and bf16 for c <= 40.
// kKeep: interval rules plus a keep mask (ai.onnx BOOL attn_mask, MultiHeadAttention binary
// key mask) and MultiHeadAttention key-padding lengths, neither softcap nor a float mask.
enum RuleMode { kPlain = 0, kAddMask = 1, kGeneric = 2, kCapFixed = 3, kKeep = 4 };

// Keep bits of keys [k0, k0 + 128) of one keep-mask row (bit e of word e / 32 set = keep);
// keys >= T_keep count as not kept.  u8 rows (bool) or int32 rows (binary), any non-zero
// value keeps.
__device__ __forceinline__ void keep_bits128(const void* row, bool is_u8, int k0, int64_t T_keep, bool vec,
                                             uint32_t* kb) {
  if (vec && (int64_t)k0 + 128 <= T_keep) {
    if (is_u8) {
      const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(row) + k0);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint4 lo = __ldg(p + 2 * w), hi = __ldg(p + 2 * w + 1);
        const uint32_t words[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        uint32_t bits = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t m = __vcmpne4(words[q], 0u);   // 0xff per non-zero byte
          const uint32_t nib = ((m >> 7) & 1u) | ((m >> 14) & 2u) | ((m >> 21) & 4u) | ((m >> 28) & 8u);
          bits |= nib << (4 * q);
        }
        kb[w] = bits;
      }
    } else {
      const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const int32_t*>(row) + k0);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t bits = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 u = __ldg(p + 8 * w + q);
          bits |= ((u.x != 0u) ? 1u : 0u) << (4 * q);
          bits |= ((u.y != 0u) ? 2u : 0u) << (4 * q);
          bits |= ((u.z != 0u) ? 4u : 0u) << (4 * q);
          bits |= ((u.w != 0u) ? 8u : 0u) << (4 * q);
        }
        kb[w] = bits;
      }
    }
  } else {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t bits = 0;
      for (int q = 0; q < 32; ++q) {
        const int64_t key = (int64_t)k0 + 32 * w + q;
        bool keep = false;
        if (key < T_keep)
          keep = is_u8 ? (reinterpret_cast<const uint8_t*>(row)[key] != 0)
                       : (reinterpret_cast<const int32_t*>(row)[key] != 0);
        bits |= (keep ? 1u : 0u) << q;
      }
      kb[w] = bits;
    }
  }
}

// Work unit: two 128-row query tiles (0, 1) that stream the same key/value tiles of one kv
// head.  With an even group they are two query heads of the group over the same rows (same
// key range, same structural rules); otherwise two consecutive row blocks of one head.
struct Unit {
  int b, kvh;
  int qh[2];          // query head of each tile
  int m[2];           // first query row of each tile
  int kv_t0, n_tiles; // key tiles some row of the unit admits
  int64_t len_b;
};

// k-th unit of CTA c among G: units are numbered heavy first and dealt round by round, the
// direction alternating (0..G-1, then G-1..0, ...), which balances the causal rows' costs.
__device__ __forceinline__ int unit_at(int k, int c, int G) { return k * G + ((k & 1) ? (G - 1 - c) : c); }

__device__ __forceinline__ void decode_unit(const TcArgs& a, int u, Unit& w) {
  int t = u;
  const int g = t % a.pairs; t /= a.pairs;
  w.kvh = t % a.Nkv; t /= a.Nkv;
  w.b = t % a.B; t /= a.B;
  const int ru = a.nrow - 1 - t;   // unit 0 takes the last (heaviest) row block
  if (a.head_pairs) {
    w.qh[0] = w.kvh * a.group + 2 * g;
    w.qh[1] = w.qh[0] + 1;
    w.m[0] = w.m[1] = ru * kBM;
  } else {
    w.qh[0] = w.qh[1] = w.kvh * a.group + g;
    w.m[0] = ru * 2 * kBM;
    w.m[1] = w.m[0] + kBM;
  }
  w.len_b = lens_of(a, w.b);
  const int last = min(a.S, w.m[1] + kBM) - 1;
  int64_t lo_f, hi_f, lo_l, hi_l;
  key_bounds(a, w.len_b, w.m[0], lo_f, hi_f);
  key_bounds(a, w.len_b, last, lo_l, hi_l);
  const int64_t lo_key = max64(0, min64(lo_f, lo_l));
  const int64_t hi_key = min64((int64_t)a.T - 1, max64(hi_f, hi_l));
  w.kv_t0 = (int)(lo_key / kBN);
  w.n_tiles = (hi_key >= lo_key) ? (int)(hi_key / kBN) - w.kv_t0 + 1 : 0;
}

template <int H, int HV, bool kBF16, int kMode, int SPLIT, bool kStats>
__global__ void __launch_bounds__(Layout<2, SPLIT>::kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap ty,
                      const TcArgs a) {
  // additive mask through shared memory (H = 64; H = 128 reads it per thread)
  constexpr bool kStage = (kMode == kAddMask) && (SPLIT == 1) && (H == 64) && (HV == 64);
  constexpr int kQT = 2;
  using C = Cfg<H, HV, kQT, kStage>;
  using Lay = Layout<kQT, SPLIT>;
  constexpr int kSplit = SPLIT;                     // softmax threads per query row
  constexpr int kHalf = kBN / kSplit;               // score columns per softmax thread
  constexpr int kSmxThreads = Lay::kSmxThreads;
  using T = typename std::conditional<kBF16, __nv_bfloat16, __half>::type;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_qfull, bar_qempty, bar_qready, bar_drain;
  __shared__ __align__(8) uint64_t bar_full[C::kStages], bar_empty[C::kStages];
  __shared__ __align__(8) uint64_t bar_sfull[2], bar_sfree[2], bar_pfull[2], bar_odone[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ float red_max[2][kQT][kSplit][kSplit == 2 ? kBM : 1];   // [tile parity][query tile][part][row]
  __shared__ float red_sum[kQT][kSplit][kSplit == 2 ? kBM : 1];      // [query tile][part][row]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  // the Q tiles need a prologue pass (projection bias) before the first MMA reads them
  const bool q_prologue = a.q_bias != nullptr;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::kQOff, sKV = sbase + C::kKVOff;
  const uint32_t b_qready = smem_u32(&bar_qready), b_drain = smem_u32(&bar_drain);
  const uint32_t b_qfull = smem_u32(&bar_qfull), b_qempty = smem_u32(&bar_qempty);
  auto b_full = [&](int s) { return smem_u32(&bar_full[s]); };
  auto b_empty = [&](int s) { return smem_u32(&bar_empty[s]); };
  auto b_sfull = [&](int x) { return smem_u32(&bar_sfull[x]); };
  auto b_sfree = [&](int x) { return smem_u32(&bar_sfree[x]); };
  auto b_pfull = [&](int x) { return smem_u32(&bar_pfull[x]); };
  auto b_odone = [&](int x) { return smem_u32(&bar_odone[x]); };
  volatile int* abortp = &abort_flag;
  constexpr uint64_t kDrainNs = 2000000000ull;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(b_qfull, 1);
    mbar_init(b_qempty, 1);
    mbar_init(b_qready, kSmxThreads);
    mbar_init(b_drain, 1);
    for (int s = 0; s < C::kStages; ++s) { mbar_init(b_full(s), 1); mbar_init(b_empty(s), 1); }
    for (int x = 0; x < kQT; ++x) {
      mbar_init(b_sfull(x), 1);
      mbar_init(b_sfree(x), kSplit * kBM);
      mbar_init(b_pfull(x), kSplit * kBM);
      mbar_init(b_odone(x), 1);
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
  // the control warpgroup hands registers to the softmax warpgroups
  if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Lay::kCtlRegs));

  // Every role walks the same unit sequence and skips the units with no admitted key.
  // Barrier phases are running counts over the CTA's lifetime.
  if (warp == 0) {
    // ================================================================ TMA producer
    // (the whole warp runs the loop and one elected lane issues the copies).  Ring order of
    // the K/V tiles follows their first use by the MMA warp: with P aliasing S (H = 128)
    // K_0, V_0, K_1, V_1, ...; otherwise S(j+1) is issued before PV(j), so the K tiles run one
    // step ahead: K_0, K_1, V_0, K_2, V_1, ...
    const uint32_t leader = elect_one();
    if (leader) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
    }
    int seq = 0, it = 0;
    bool ok = true;
    for (int ku = 0; ok; ++ku) {
      const int u = unit_at(ku, cta, G);
      if (u >= a.nunits) break;
      Unit w;
      decode_unit(a, u, w);
      if (w.n_tiles == 0) continue;
      auto load = [&](const CUtensorMap* map, int tile) -> bool {
        const int st = seq % C::kStages;
        if (seq >= C::kStages &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(b_empty(st), ((seq / C::kStages) - 1) & 1, abortp, a.wait_ns)))
          return false;
        if (leader && SDPA_IN_BOUNDS(w.kv_t0 + tile >= 0 && (int64_t)(w.kv_t0 + tile) * kBN < a.T && st < C::kStages &&
                                         w.kvh < a.Nkv && w.b < a.B, 101)) {
          const bool is_v = map == &tv;
          mbar_arrive_expect_tx(b_full(st), is_v ? C::kVTile : C::kKTile);
          int d1, d2, d3;
          perm_coords(a.kv_ds, a.kv_dn, a.kv_db, (w.kv_t0 + tile) * kBN, w.kvh, w.b, d1, d2, d3);
          for (int r = 0; r < (is_v ? C::kVRegions : C::kRegions); ++r)
            tma_load_4d(sKV + st * C::kKVTile + r * C::kRegionBytes, map, b_full(st), 64 * r, d1, d2, d3);
        }
        ++seq;
        return true;
      };
      // K_0 first: its ring slot frees up before the previous unit's last S MMAs have read Q
      ok = load(&tk, 0);
      // the previous unit's last S MMAs have read its Q tiles
      if (ok && it > 0) ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_qempty, (it - 1) & 1, abortp, a.wait_ns));
      if (!ok) break;
      if (leader && SDPA_IN_BOUNDS(w.m[0] >= 0 && w.m[0] < a.S && w.m[1] >= 0 && w.qh[0] < a.Nq && w.qh[1] < a.Nq, 102)) {
        mbar_arrive_expect_tx(b_qfull, kQT * C::kQTile);
        for (int x = 0; x < kQT; ++x) {
          int c1, c2, c3;
          perm_coords(a.q_ds, a.q_dn, a.q_db, w.m[x], w.qh[x], w.b, c1, c2, c3);
          for (int r = 0; r < C::kRegions; ++r)
            tma_load_4d(sQ + x * C::kQTile + r * C::kRegionBytes, &tq, b_qfull, 64 * r, c1, c2, c3);
        }
      }
      ++it;
      for (int j = 0; j < w.n_tiles && ok; ++j) {
        if constexpr (C::kAlias) {
          ok = load(&tv, j);
          if (ok && j + 1 < w.n_tiles) ok = load(&tk, j + 1);
        } else {
          if (j + 1 < w.n_tiles) ok = load(&tk, j + 1);
          if (ok) ok = load(&tv, j);
        }
      }
    }
    if (__any_sync(0xffffffffu, !ok || *abortp)) {
      // some role gave up: let every copy already issued land before the CTA can exit
      if (it > 0) mbar_wait_bounded(b_qfull, (it - 1) & 1, nullptr, kDrainNs);
      for (int s = 0; s < C::kStages && s < seq; ++s) {
        const int last = s + ((seq - 1 - s) / C::kStages) * C::kStages;
        mbar_wait_bounded(b_full(s), (last / C::kStages) & 1, nullptr, kDrainNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    // (the whole warp runs the loop; one elected lane issues every MMA and every commit, as a
    // commit tracks the MMAs of the thread that issues it)
    const uint32_t leader = elect_one();
    auto commit = [&](uint32_t bar) {
      if (leader) mma_commit(bar);
    };
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abortp, a.wait_ns));
    };
    constexpr uint32_t kIdQK = idesc_f16(kBF16, kBM, kBN, false);
    constexpr uint32_t kIdPV = idesc_f16(kBF16, kBM, HV, true);
    const uint32_t tS[2] = {tmem + C::kTmemS0, tmem + C::kTmemS1};
    const uint32_t tO[2] = {tmem + C::kTmemO0, tmem + C::kTmemO1};
    const uint32_t tP[2] = {tmem + C::kTmemP0, tmem + C::kTmemP1};
    int seq = 0, it = 0;
    int ns = 0;   // S batches issued (each covers both tiles)
    int np = 0;   // P batches consumed (each covers both tiles)
    auto wait_full = [&](int sq) -> bool {
      const bool ok = wait_all(b_full(sq % C::kStages), (sq / C::kStages) & 1);
      tc_fence_after();
      return ok;
    };
    // descriptors differ only in their start-address field: build them once
    const uint64_t dQ[2] = {desc_sw128(sQ, 16, 1024), desc_sw128(sQ + C::kQTile, 16, 1024)};
    const uint64_t dK0 = desc_sw128(sKV, 16, 1024);
    const uint64_t dV0 = desc_sw128(sKV, C::kRegionBytes, 1024);
    auto issue_S = [&](int x, int st) {
      const uint64_t dk = dK0 + (uint64_t)((st * C::kKVTile) >> 4);
#pragma unroll
      for (int kk = 0; kk < H / 16; ++kk) {
        const uint64_t off = (uint64_t)(((kk / 4) * C::kRegionBytes + (kk % 4) * 32) >> 4);
        if (leader) mma_f16_ss(tS[x], dQ[x] + off, dk + off, kIdQK, kk > 0);
      }
    };
    auto issue_PV = [&](int x, int st, bool acc) {
      const uint64_t dv = dV0 + (uint64_t)((st * C::kKVTile) >> 4);
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk)
        if (leader) mma_f16_ts(tO[x], tP[x] + kk * 8, dv + (uint64_t)((kk * 2048) >> 4), kIdPV, (acc || kk > 0) ? 1u : 0u);
    };
    // S_x may be overwritten once softmax x has taken the previous S_x into registers (with
    // P aliasing S, the in-order PV_x that read P_x already implies it)
    auto wait_sfree = [&](int x) -> bool {
      if (C::kAlias || ns == 0) return true;
      const bool ok = wait_all(b_sfree(x), (ns - 1) & 1);
      tc_fence_after();
      return ok;
    };
    bool ok = true;
    for (int ku = 0; ok; ++ku) {
      const int u = unit_at(ku, cta, G);
      if (u >= a.nunits) break;
      Unit w;
      decode_unit(a, u, w);
      const int n = w.n_tiles;
      if (n == 0) continue;
      if (!(ok = wait_all(q_prologue ? b_qready : b_qfull, it & 1))) break;
      tc_fence_after();
      ++it;
      if (!(ok = wait_full(seq))) break;
      {
        const int st = seq % C::kStages;
        for (int x = 0; x < kQT && ok; ++x) {
          if (!(ok = wait_sfree(x))) break;
          issue_S(x, st);
          commit(b_sfull(x));
        }
        if (!ok) break;
        ++ns;
        if (n == 1) commit(b_qempty);   // the unit's last S MMAs have been issued
        commit(b_empty(st));
        ++seq;
      }
      if constexpr (C::kAlias) {
        // P_X(j) lives in S_X's columns: PV_X(j) first, then S_X(j+1); one commit on
        // sfull_X then also tells softmax X that O_X holds PV_X(j).  The unit's last PV_X
        // commits on odone_X instead: the next unit's S_X(0) follows it without waiting for
        // the softmax, and a second sfull_X phase completing before the epilogue's wait
        // would leave that wait on the wrong parity.
        for (int j = 0; j < n && ok; ++j) {
          const bool more = j + 1 < n;
          const int vst = seq % C::kStages;
          if (!(ok = wait_full(seq))) break;
          ++seq;
          const int kst = seq % C::kStages;
          for (int x = 0; x < kQT && ok; ++x) {
            if (!(ok = wait_all(b_pfull(x), np & 1))) break;
            tc_fence_after();
            issue_PV(x, vst, j > 0);
            if (more) {
              if (x == 0 && !(ok = wait_full(seq))) break;
              issue_S(x, kst);
              commit(b_sfull(x));
            } else {
              commit(b_odone(x));
            }
          }
          if (!ok) break;
          ++np;
          if (more) ++ns;
          if (more && j + 2 == n) commit(b_qempty);
          commit(b_empty(vst));
          if (more) {
            commit(b_empty(kst));
            ++seq;
          }
        }
      } else {
        for (int j = 0; j < n && ok; ++j) {
          if (j + 1 < n) {
            // S_X(j+1) as soon as softmax X has taken S_X(j) out of tensor memory
            const int kst = seq % C::kStages;
            if (!(ok = wait_full(seq))) break;
            ++seq;
            for (int x = 0; x < kQT && ok; ++x) {
              if (!(ok = wait_sfree(x))) break;
              issue_S(x, kst);
              commit(b_sfull(x));
            }
            if (!ok) break;
            ++ns;
            if (j + 2 == n) commit(b_qempty);
            commit(b_empty(kst));
          }
          const int vst = seq % C::kStages;
          if (!(ok = wait_full(seq))) break;
          ++seq;
          for (int x = 0; x < kQT && ok; ++x) {
            if (!(ok = wait_all(b_pfull(x), np & 1))) break;
            tc_fence_after();
            issue_PV(x, vst, j > 0);
            commit(b_odone(x));
          }
          if (!ok) break;
          ++np;
          commit(b_empty(vst));
        }
      }
    }
    // every MMA this thread issued completes before the CTA frees its tensor memory
    commit(b_drain);
    mbar_wait_bounded(b_drain, 0, nullptr, kDrainNs);
    __syncwarp();
  } else if (warp >= 4) {
    // ================================================================ softmax warpgroups
    // (query tile 0 or 1) x (column part): one thread per row and part
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Lay::kSmxRegs));
    const int g = (warp - 4) >> 2;
    const int x = g / kSplit;                       // query tile
    const int hh = g % kSplit;                      // column part
    const int sub = warp & 3;                       // TMEM sub-partition of this warp
    const int row = sub * 32 + lane;                // row in the tile == TMEM lane
    const int pair_bar = 1 + x * 4 + sub;           // named barrier of the warps of these rows
    const uint32_t trow = tmem + ((uint32_t)(sub * 32) << 16);
    const uint32_t tS = trow + (x == 0 ? C::kTmemS0 : C::kTmemS1) + kHalf * hh;
    const uint32_t tO = trow + (x == 0 ? C::kTmemO0 : C::kTmemO1) + (HV / kSplit) * hh;
    const uint32_t tP = trow + (x == 0 ? C::kTmemP0 : C::kTmemP1) + (kHalf / 2) * hh;
    const uint32_t sMask = sbase + C::kMaskOff + (uint32_t)(x * 4 + sub) * C::kMaskWarpBytes;
    // log2-domain factor applied inside the exponent: raw scores (plain mode) carry the
    // scale or the softcap amplitude, additive-mask scores are in natural units, and the
    // generic mode produces log2-domain scores already
    const float kfac = (kMode == kPlain) ? (a.has_softcap ? a.cap_out_log2 : a.scale_log2)
                       : (kMode == kKeep) ? a.scale_log2
                                          : (kMode == kAddMask ? kLog2e : 1.f);
    int cs = 0;   // sfull phases waited
    int co = 0;   // odone phases waited
    int it = 0;   // units with work
    bool ok = true;
    // the unit whose epilogue is pending (e_real false: the dry pass before the first unit,
    // run in the interval-rule and softcap modes, where it measured faster; the mask modes
    // start their first unit at once)
    constexpr bool kPrimeEpilogue = (kMode == kPlain || kMode == kCapFixed);
    bool e_real = false;
    int e_tiles = 1, e_b = 0, e_qh = 0, e_mx0 = 0;
    float e_l = 0.f, e_m = -INFINITY;
    bool e_valid = false;
    int64_t e_i = 0;
    for (int ku = 0; ok; ++ku) {
      const int u = unit_at(ku, cta, G);
      if (e_real || kPrimeEpilogue) {
        const int n_tiles = e_tiles;
        const float l = e_l, m_use = e_m;
        const bool valid = e_valid;
        const int64_t i = e_i;
        const int b = e_b, qh = e_qh, mx0 = e_mx0;
        // ---- epilogue of the previous unit: O / (l + sink term), rounded once to the output
        // type; its last PV must be done (its odone commit).  Before the first unit the same code
        // runs once as a dry pass (no waits, nothing stored, results discarded): the CTA waits
        // for its first Q and K tiles then anyway, and the pass brings the epilogue's code into
        // the caches, where the first real epilogue, which every CTA reaches at about the same
        // time, would otherwise fetch it from memory.
        if (e_real && n_tiles > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_odone(x), co & 1, abortp, a.wait_ns));
          ++co;
          if (!ok) break;
        }
        tc_fence_after();
        float denom = l;
        if constexpr (kSplit == 2) {
          red_sum[x][hh][row] = l;
          named_bar_sync(pair_bar, 64);
          denom += red_sum[x][hh ^ 1][row];
        }
        if (a.head_sink && m_use != -INFINITY)
          denom += ex2_approx(Elem<T>::to_f32(reinterpret_cast<const T*>(a.head_sink)[qh]) * kLog2e - m_use);
        const float inv = (denom > 0.f && m_use != -INFINITY) ? 1.f / denom : 0.f;
        T* yrow = reinterpret_cast<T*>(a.y) + (int64_t)b * a.y_sb + (int64_t)qh * a.y_sh + i * a.y_ss +
                  (HV / kSplit) * hh;
        // y through shared memory: the warp's 32 rows, 64 columns at a time, one TMA store each
        // (rows past S are clipped by the tensor map); a unit with no admitted key writes its
        // zero rows directly
        const bool write_y = !kStats || a.y != nullptr;
        const uint32_t sY = kStage ? sMask : sbase + C::kYOff + (uint32_t)(x * 4 + sub) * C::kYWarpBytes;
        int yc1 = 0, yc2 = 0, yc3 = 0;
        if (write_y && n_tiles > 0) perm_coords(a.y_ds, a.y_dn, a.y_db, mx0 + sub * 32, qh, b, yc1, yc2, yc3);
        constexpr bool stats = kStats && kSplit == 1;   // the backward's statistics pass
        const T* dyrow = stats ? reinterpret_cast<const T*>(a.dy) + (int64_t)b * a.dy_sb + (int64_t)qh * a.dy_sh +
                                     i * a.dy_ss
                               : nullptr;
        float delta = 0.f;
  #pragma unroll
        for (int c = 0; c < HV / (32 * kSplit); ++c) {
          uint32_t o[32];
          if (n_tiles > 0) {
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait();
          } else {
  #pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
          }
          if (stats && valid) {
            // delta = dY . O with O = o / denom in fp32
  #pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 uv = *reinterpret_cast<const uint4*>(dyrow + c * 32 + q * 8);
              const T* e8 = reinterpret_cast<const T*>(&uv);
  #pragma unroll
              for (int e = 0; e < 8; ++e) delta = fmaf(Elem<T>::to_f32(e8[e]), __uint_as_float(o[q * 8 + e]) * inv, delta);
            }
          }
          if (n_tiles > 0) {
            if (write_y) {
              if ((c & 1) == 0) {
                // the warp's previous store has finished reading the staging buffer
                if (lane == 0) bulk_wait_read<0>();
                __syncwarp();
              }
  #pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint32_t wv[4];
  #pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float v0 = __uint_as_float(o[q * 8 + 2 * e]) * inv;
                  const float v1 = __uint_as_float(o[q * 8 + 2 * e + 1]) * inv;
                  wv[e] = kBF16 ? pack_bf16x2(v0, v1) : pack_f16x2(v0, v1);
                }
                const int c16 = (c & 1) * 4 + q;   // 16-byte piece of the row within the 64 columns
                if (SDPA_IN_BOUNDS(lane * 128 + (c16 << 4) + 16 <= C::kYWarpBytes || kStage, 104))
                  st_shared_v4(sY + lane * 128 + ((c16 ^ (lane & 7)) << 4), wv[0], wv[1], wv[2], wv[3]);
              }
              if ((c & 1) == 1) {
                fence_proxy_async_smem();
                __syncwarp();
                // a warp whose rows all lie past S has nothing to store
                if (e_real && lane == 0 && mx0 + sub * 32 < a.S && SDPA_IN_BOUNDS(mx0 + sub * 32 >= 0, 105)) {
                  tma_store_4d(&ty, sY, (c >> 1) * 64, yc1, yc2, yc3);
                  bulk_commit();
                }
              }
            }
          } else if (valid && write_y) {
  #pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t wv[4];
  #pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float v0 = __uint_as_float(o[q * 8 + 2 * e]) * inv;
                const float v1 = __uint_as_float(o[q * 8 + 2 * e + 1]) * inv;
                wv[e] = kBF16 ? pack_bf16x2(v0, v1) : pack_f16x2(v0, v1);
              }
              *reinterpret_cast<uint4*>(yrow + c * 32 + q * 8) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
          }
        }
        if (stats && valid) {
          const int64_t r_idx = ((int64_t)b * a.Nq + qh) * a.S + i;
          a.lse2_out[r_idx] = (denom > 0.f && m_use != -INFINITY) ? m_use + log2f(denom) : INFINITY;
          a.delta_out[r_idx] = delta;
        }
        // the epilogue's tensor-memory reads are complete before this thread's next P store,
        // which the MMA warp waits for before the next unit's first PV overwrites O
      }
      if (u >= a.nunits) break;
      Unit w;
      decode_unit(a, u, w);
      const int n_tiles = w.n_tiles;
      const int b = w.b;
      const int qh = x == 0 ? w.qh[0] : w.qh[1];
      const int mx0 = x == 0 ? w.m[0] : w.m[1];      // first row of this tile
      const int64_t len_b = w.len_b;
      const int64_t i = (int64_t)mx0 + row;          // query row
      const bool valid = i < a.S && SDPA_IN_BOUNDS(b < a.B && qh < a.Nq && i >= 0, 103);
      int64_t lo = 1, hi = 0;
      if (valid) key_bounds(a, len_b, i, lo, hi);
      // T <= 2^30, so the bounds fit 32 bits once clamped to [-1, T]
      const int lo32 = (int)max64(-1, min64(lo, a.T));
      const int hi32 = (int)max64(-1, min64(hi, a.T));
      RowCtx ctx;
      ctx.len = len_b;
      ctx.pos = pos_of(a, len_b, i);
      const void* mrow = nullptr;
      if (kMode == kKeep && valid && a.r.keep_kind != SDPA_KEEP_NONE) {
        const int esz = a.r.keep_kind == SDPA_KEEP_BOOL_U8 ? 1 : 4;
        mrow = reinterpret_cast<const char*>(a.r.keep) +
               (b * a.r.keep_sb + (int64_t)qh * a.r.keep_sh + i * a.r.keep_ss) * esz;
      }
      if (kMode == kAddMask && valid) {
        const int esz = a.r.add_dtype == SDPA_F32 ? 4 : 2;
        mrow = reinterpret_cast<const char*>(a.r.add) +
               (b * a.r.add_sb + (int64_t)qh * a.r.add_sh + i * a.r.add_ss) * esz;
      }
      // staged mask: the warp's first row, the row stride and how many of its 32 rows exist
      const int64_t wrow = (int64_t)mx0 + sub * 32;
      const char* mwarp = nullptr;
      int mrows = 0;
      if (kStage && a.add_stage) {
        mwarp = reinterpret_cast<const char*>(a.r.add) + (b * a.r.add_sb + (int64_t)qh * a.r.add_sh + wrow * a.r.add_ss) * 2;
        mrows = (int)max64(0, min64(32, (int64_t)a.S - wrow));
      }
      // kCapFixed: the fixed maximum (the cap, or the sink logit when that is larger)
      float m_fixed = a.cap_out_log2;
      if (kMode == kCapFixed && a.head_sink)
        m_fixed = fmaxf(m_fixed, Elem<T>::to_f32(reinterpret_cast<const T*>(a.head_sink)[qh]) * kLog2e);

      if (n_tiles > 0 && q_prologue) {
        // add the query segment of the projection bias to this row of Q (this thread's part
        // of the columns) in shared memory
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_qfull, it & 1, abortp, a.wait_ns));
        if (ok) {
          const uint32_t qRow = sQ + x * C::kQTile + row * 128;
          const T* qb = reinterpret_cast<const T*>(a.q_bias) + (int64_t)qh * H;
          const int swz = row & 7;
#pragma unroll
          for (int c16 = 0; c16 < H / (8 * kSplit); ++c16) {   // 16-byte chunks of this thread's part
            const int cidx = hh * (H / (8 * kSplit)) + c16;      // chunk index within the row
            const int r = cidx >> 3, c = cidx & 7;
            const uint32_t addr = qRow + r * C::kRegionBytes + ((c ^ swz) << 4);
            uint32_t wv[4];
            ld_shared_v4(addr, wv[0], wv[1], wv[2], wv[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int col = cidx * 8 + 2 * e;
              const T* pv = reinterpret_cast<const T*>(&wv[e]);
              const float lo_f = Elem<T>::to_f32(pv[0]) + Elem<T>::to_f32(qb[col]);
              const float hi_f = Elem<T>::to_f32(pv[1]) + Elem<T>::to_f32(qb[col + 1]);
              wv[e] = kBF16 ? pack_bf16x2(lo_f, hi_f) : pack_f16x2(lo_f, hi_f);
            }
            st_shared_v4(addr, wv[0], wv[1], wv[2], wv[3]);
          }
          fence_proxy_async_smem();
        }
        mbar_arrive(b_qready);
        if (!ok) break;
      }
      if (n_tiles > 0) ++it;

      if constexpr (kStage) {
        // the previous unit's y stores from this warp's mask region have read it
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
      }
      float m_use = (kMode == kCapFixed) ? m_fixed : -INFINITY, l = 0.f;
      for (int j = 0; j < n_tiles && ok; ++j) {
        bool staged = false;     // warp-uniform: the mask tile comes through shared memory
        if constexpr (kStage) {
          // copy the warp's mask rows for the tile now; the wait below hides the latency
          const int k0 = (w.kv_t0 + j) * kBN;
          staged = a.add_stage && (int64_t)k0 + kBN <= a.r.add_T;
          if (staged) stage_mask_tile(sMask, mwarp + (int64_t)k0 * 2, a.r.add_ss * 2, mrows, a.add_vec, lane);
        }
        uint32_t kb[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};   // keep bits
        if constexpr (kMode == kKeep) {
          if (mrow)
            keep_bits128(mrow, a.r.keep_kind == SDPA_KEEP_BOOL_U8, (w.kv_t0 + j) * kBN, a.r.keep_T, a.keep_vec != 0, kb);
        }
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_sfull(x), cs & 1, abortp, a.wait_ns)))) break;
        ++cs;
        tc_fence_after();
        float s[kHalf];
        {
          uint32_t uu[kHalf];
#pragma unroll
          for (int c = 0; c < kHalf / 32; ++c) tmem_ld32(tS + c * 32, uu + c * 32);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < kHalf; ++e) s[e] = __uint_as_float(uu[e]);
        }
        if constexpr (!C::kAlias) {
          // S_X(j) is in registers: the MMA warp may overwrite it with S_X(j+1)
          tc_fence_before();
          mbar_arrive(b_sfree(x));
        }
        if constexpr (kStage) {
          if (staged) {
            // the warp's copies have landed and are visible to every lane
            ptx::cp_async_wait_all();
            __syncwarp();
          }
        }

        const int key0 = (w.kv_t0 + j) * kBN + kHalf * hh;
        bool have_mx = false;       // set when the transform already produced this half's max
        float mx_own = -INFINITY;
        bool weights = false;       // kCapFixed: s already holds the weights p
        if constexpr (kMode == kCapFixed) {
          // s = raw q.k; the exponent c log2e tanh(s scale / c) - m, from the cubic when every
          // |s| of the segment is in its range (eight chains of three-input max of |s|)
          float am8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) am8[k] = fmaxf(fabsf(s[k]), fabsf(s[k + 8]));
#pragma unroll
          for (int e = 16; e < kHalf; e += 16)
#pragma unroll
            for (int k = 0; k < 8; ++k) am8[k] = fmax3(am8[k], fabsf(s[e + k]), fabsf(s[e + 8 + k]));
          const float amax = fmax3(fmax3(am8[0], am8[1], am8[2]), fmax3(am8[3], am8[4], am8[5]), fmaxf(am8[6], am8[7]));
          const float negm = -m_use;
          const bool full = (lo32 <= key0) && (key0 + kHalf - 1 <= hi32);
          if (amax <= a.fx_lim) {
            // exponent and weight in one pass, in place.  Tiles with excluded keys (the causal
            // diagonal, a length boundary) run the same pass, whose code the full tiles keep
            // hot, then set the excluded weights to 0: every score of the tile is finite and
            // inside the cubic's range, so the pass is defined for every key.
            const f2_t ca = f2_pack(a.fx_a, a.fx_a), cb = f2_pack(a.fx_b, a.fx_b), nm2 = f2_pack(negm, negm);
#pragma unroll
            for (int e = 0; e < kHalf; e += 2) {
              const f2_t x2 = f2_pack(s[e], s[e + 1]);
              const f2_t tt = f2_fma(f2_mul(x2, x2), cb, ca);
              float z0, z1;
              f2_unpack(f2_fma(x2, tt, nm2), z0, z1);
              s[e] = ex2_approx(z0);
              s[e + 1] = ex2_approx(z1);
            }
            if (!full) {
              // a suffix (causal diagonal, length boundary) and a prefix (window start) of
              // excluded keys, each with one compare and one select per key
              const int elo = lo32 - key0, ehi = hi32 - key0;
              if (ehi < kHalf - 1) {
#pragma unroll
                for (int e = 0; e < kHalf; ++e) s[e] = (e <= ehi) ? s[e] : 0.f;
              }
              if (elo > 0) {
#pragma unroll
                for (int e = 0; e < kHalf; ++e) s[e] = (e >= elo) ? s[e] : 0.f;
              }
            }
            weights = true;
          } else {
#pragma unroll
            for (int e = 0; e < kHalf; ++e) s[e] = fmaf(a.cap_out_log2, tanh_approx(s[e] * a.cap_in), negm);
            if (!full) clip_interval(s, lo32 - key0, hi32 - key0, -INFINITY);
          }
        } else if constexpr (kMode == kPlain) {
          const bool full = (lo32 <= key0) && (key0 + kHalf - 1 <= hi32);
          if (a.has_softcap) {
            const f2_t cin = f2_pack(a.cap_in, a.cap_in);
#pragma unroll
            for (int e = 0; e < kHalf; e += 2) f2_unpack(f2_mul(f2_pack(s[e], s[e + 1]), cin), s[e], s[e + 1]);
            bool poly = false;
            float umax = -INFINITY;
            if (full) {
              float hi8[4], lo8[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) { hi8[k] = fmaxf(s[k], s[k + 4]); lo8[k] = fminf(s[k], s[k + 4]); }
#pragma unroll
              for (int e = 8; e < kHalf; e += 8)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  hi8[k] = fmax3(hi8[k], s[e + k], s[e + 4 + k]);
                  lo8[k] = fminf(lo8[k], fminf(s[e + k], s[e + 4 + k]));
                }
              umax = fmaxf(fmaxf(hi8[0], hi8[1]), fmaxf(hi8[2], hi8[3]));
              const float umin = fminf(fminf(lo8[0], lo8[1]), fminf(lo8[2], lo8[3]));
              poly = fmaxf(umax, -umin) <= kTanhPolyLimit;
            }
            if (poly) {
              // small arguments: odd polynomial on the FMA pipe (monotonic here, so the
              // maximum is the polynomial of the largest argument)
              const f2_t a1 = f2_pack(kTanhA1, kTanhA1), a2 = f2_pack(kTanhA2, kTanhA2);
#pragma unroll
              for (int e = 0; e < kHalf; e += 2) {
                const f2_t uu = f2_pack(s[e], s[e + 1]);
                const f2_t z = f2_mul(uu, uu);
                const f2_t q = f2_fma(z, a2, a1);
                f2_unpack(f2_fma(f2_mul(uu, z), q, uu), s[e], s[e + 1]);
              }
              mx_own = tanh_poly(umax);
              have_mx = true;
            } else {
#pragma unroll
              for (int e = 0; e < kHalf; ++e) s[e] = tanh_approx(s[e]);
            }
          }
          if (!full) clip_interval(s, lo32 - key0, hi32 - key0, -INFINITY);
        } else if constexpr (kMode == kKeep) {
          // raw scores: a key the keep mask drops is excluded (bool) or gets the filter value
          // (binary), as does every key at or past a key-padding length; then the bounds
          const bool full = (lo32 <= key0) && (key0 + kHalf - 1 <= hi32);
          const bool all_keep = (kb[0] & kb[1] & kb[2] & kb[3]) == 0xffffffffu;
          const int len_e = (a.r.len_kind == SDPA_LEN_KEYLEN_I32) ? (int)max64(-1, min64(len_b - key0, kHalf)) : kHalf;
          if (!__all_sync(0xffffffffu, full && all_keep && len_e >= kHalf)) {
            const float fr = a.filter_raw;
            // dropped keys: one bit test and one predicated update per key
            if (!all_keep) {
              if (a.r.keep_kind == SDPA_KEEP_BOOL_U8) {
#pragma unroll
                for (int e = 0; e < kHalf; ++e)
                  if (!((kb[e >> 5] >> (e & 31)) & 1u)) s[e] = -INFINITY;
              } else {
#pragma unroll
                for (int e = 0; e < kHalf; ++e)
                  if (!((kb[e >> 5] >> (e & 31)) & 1u)) s[e] += fr;
              }
            }
            // keys at or past the key-padding length, 32 columns at a time
            if (len_e < kHalf) {
#pragma unroll
              for (int c0 = 0; c0 < kHalf; c0 += 32) {
                if (len_e <= c0) {
#pragma unroll
                  for (int e = c0; e < c0 + 32; ++e) s[e] += fr;
                } else if (len_e < c0 + 32) {
#pragma unroll
                  for (int e = c0; e < c0 + 32; ++e)
                    if (e >= len_e) s[e] += fr;
                }
              }
            }
            if (!full) clip_interval(s, lo32 - key0, hi32 - key0, -INFINITY);
          }
        } else if constexpr (kMode == kAddMask) {
          // additive mask / attention bias, then softcap (or the reverse), then the bounds;
          // scores stay in natural units here (kfac carries log2 e).  The mask is read eight
          // columns at a time: from the warp's staged rows, else from global memory.
          static_assert(kSplit == 1, "the additive-mask mode covers 128 columns per thread");
          auto run = [&](auto f) {
            if (staged) {
              const uint32_t rowp = sMask + lane * 256;
#pragma unroll
              for (int c = 0; c < kHalf / 8; ++c) {
                uint32_t w[4];
                ld_shared_v4(rowp + ((c ^ (lane & 15)) << 4), w[0], w[1], w[2], w[3]);
                if (!valid) w[0] = w[1] = w[2] = w[3] = 0u;
#pragma unroll
                for (int k = 0; k < 8; ++k) s[8 * c + k] = f(s[8 * c + k], mask_elem<T>(w, k));
              }
              __syncwarp();   // every lane has read its row: the region takes the next tile
            } else {
#pragma unroll
              for (int c = 0; c < kHalf / 8; ++c) {
                uint32_t w[4] = {0u, 0u, 0u, 0u};
                if (valid) load_mask_chunk(reinterpret_cast<const T*>(mrow), key0 + 8 * c, a.r.add_T, a.add_vec, w);
#pragma unroll
                for (int k = 0; k < 8; ++k) s[8 * c + k] = f(s[8 * c + k], mask_elem<T>(w, k));
              }
            }
          };
          if (!a.has_softcap) {
            const float sc = a.scale;
            run([sc](float sv, float mv) { return fmaf(sv, sc, mv); });
          } else if (!a.r.softcap_before_bias) {
            const float sc = a.scale, cap = a.r.softcap, cin = 1.f / a.r.softcap;
            run([sc, cap, cin](float sv, float mv) {
              const float v = fmaf(sv, sc, mv);
              return (v == -INFINITY) ? v : cap * tanh_approx(v * cin);
            });
          } else {
            const float cap = a.r.softcap, cin = a.cap_in;
            run([cap, cin](float sv, float mv) { return fmaf(cap, tanh_approx(sv * cin), mv); });
          }
          if (!((lo32 <= key0) && (key0 + kHalf - 1 <= hi32))) clip_interval(s, lo32 - key0, hi32 - key0, -INFINITY);
        } else {
#pragma unroll
          for (int e = 0; e < kHalf; ++e) {
            const int key = key0 + e;
            float v = -INFINITY;
            if (key >= lo32 && key <= hi32)
              v = generic_score(a.r, ctx, s[e] * a.scale, b, qh, (int)i, key) * kLog2e;
            s[e] = v;
          }
        }

        // row maximum: this half (eight chains of three-input max), then the partner's half
        if (kMode != kCapFixed && !have_mx) {
          float mx8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mx8[k] = fmax3(s[k], s[k + 8], -INFINITY);
#pragma unroll
          for (int e = 16; e < kHalf; e += 16)
#pragma unroll
            for (int k = 0; k < 8; ++k) mx8[k] = fmax3(mx8[k], s[e + k], s[e + 8 + k]);
          mx_own = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        }
        float mx = mx_own;
        if constexpr (kSplit == 2) {
          red_max[j & 1][x][hh][row] = mx_own;
          named_bar_sync(pair_bar, 64);
          mx = fmaxf(mx_own, red_max[j & 1][x][hh ^ 1][row]);
        }

        // move the running maximum only when it grows by more than 2^8 (both halves of a
        // row see the same maxima, so they take the same decision)
        bool need = false;
        float corr = 1.f;
        if constexpr (kMode != kCapFixed) {
          const float m_tile = mx * kfac;
          const float m_new = fmaxf(m_use, m_tile);
          need = m_new > m_use + kRescaleThreshold;
          if (need) {
            corr = ex2_approx(m_use - m_new);
            m_use = m_new;
          }
        }
        f2_t acc2[4] = {f2_zero(), f2_zero(), f2_zero(), f2_zero()};
        uint32_t pw[kHalf / 2];
        if constexpr (kMode == kCapFixed) {
          // s holds the exponents (masked keys: -inf), or the weights already
          if (!weights) {
#pragma unroll
            for (int e = 0; e < kHalf; ++e) s[e] = ex2_approx(s[e]);
          }
#pragma unroll
          for (int e = 0; e < kHalf; e += 2) {
            acc2[(e >> 1) & 3] = f2_add(acc2[(e >> 1) & 3], f2_pack(s[e], s[e + 1]));
            pw[e >> 1] = pack_bf16x2(s[e], s[e + 1]);
          }
        } else {
          // rows with nothing admitted yet get exponent -inf, hence p = 0
          const float negm = (m_use == -INFINITY) ? -INFINITY : -m_use;
          const f2_t kf2 = f2_pack(kfac, kfac), nm2 = f2_pack(negm, negm);
#pragma unroll
          for (int e = 0; e < kHalf; e += 2) {
            float z0, z1;
            f2_unpack(f2_fma(f2_pack(s[e], s[e + 1]), kf2, nm2), z0, z1);
            const float p0 = ex2_approx(z0), p1 = ex2_approx(z1);
            acc2[(e >> 1) & 3] = f2_add(acc2[(e >> 1) & 3], f2_pack(p0, p1));
            pw[e >> 1] = kBF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
          }
        }
        float r0, r1, r2, r3, r4, r5, r6, r7;
        f2_unpack(acc2[0], r0, r1);
        f2_unpack(acc2[1], r2, r3);
        f2_unpack(acc2[2], r4, r5);
        f2_unpack(acc2[3], r6, r7);
        l = l * corr + (((r0 + r1) + (r2 + r3)) + ((r4 + r5) + (r6 + r7)));

        // PV_X(j-1) must be done: it reads P_X and accumulates into O_X (with P aliasing S,
        // the sfull_X completion already implied it)
        if (j > 0) {
          if constexpr (!C::kAlias) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(b_odone(x), co & 1, abortp, a.wait_ns)))) break;
            ++co;
            tc_fence_after();
          }
          if (kMode != kCapFixed && __any_sync(0xffffffffu, need)) {
            // rescale this thread's half of its row of the accumulator (factor 1 for rows
            // that kept their maximum)
            const f2_t c2 = f2_pack(corr, corr);
#pragma unroll
            for (int c = 0; c < HV / (32 * kSplit); ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                float v0, v1;
                f2_unpack(f2_mul(f2_pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), c2), v0, v1);
                o[e] = __float_as_uint(v0);
                o[e + 1] = __float_as_uint(v1);
              }
              tmem_st32(tO + c * 32, o);
            }
            tmem_st_wait();
          }
        }
        // P_X(j) into tensor memory: lane = row, column c holds keys 2c and 2c+1
#pragma unroll
        for (int c = 0; c < kHalf / 64; ++c) tmem_st32(tP + c * 32, pw + c * 32);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_pfull(x));
      }
      // a loop left early may still have mask copies in flight into this warp's region
      if constexpr (kStage) ptx::cp_async_wait_all();
      if (!ok) break;

      // the epilogue of this unit runs at the top of the next pass
      e_real = true;
      e_tiles = n_tiles;
      e_l = l;
      e_m = m_use;
      e_valid = valid;
      e_i = i;
      e_b = b;
      e_qh = qh;
      e_mx0 = mx0;
    }
    // the warp's last stores have read shared memory before the CTA exits
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

// 4-D map over a (B, N, Seq, D) view: dim 0 = D (contiguous); dims 1..3 = the axes in
// tc_axis_order.  Box: 64 x 128 rows.
bool make_map(CUtensorMap* map, const View& v, sdpa_dtype dt, int64_t B, int64_t N, int64_t Sq, int D, int* ds,
              int* dn, int* db, int box_rows = kBN) {
  auto enc = encode_fn();
  if (!enc) return false;
  const int64_t ext[3] = {Sq, N, B};
  const int64_t str[3] = {v.ss, v.sh, v.sb};
  int order[3];
  tc_axis_order(v, B, N, Sq, order);
  const int64_t es = 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, 0, 0, 0};
  cuuint64_t strides[3];
  cuuint32_t box[4] = {64, 1, 1, 1};
  int64_t prev_end = (int64_t)D * es;  // bytes spanned so far
  for (int k = 0; k < 3; ++k) {
    const int id = order[k];
    dims[k + 1] = (cuuint64_t)ext[id];
    int64_t sb = str[id] * es;
    if (ext[id] == 1) sb = ((prev_end + 15) / 16) * 16;   // never stepped: any legal stride
    strides[k] = (cuuint64_t)sb;
    prev_end = std::max<int64_t>(prev_end, sb * ext[id]);
    if (id == 0) { box[k + 1] = (cuuint32_t)box_rows; *ds = k + 1; }
    if (id == 1) *dn = k + 1;
    if (id == 2) *db = k + 1;
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

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

template <int H, int HV, bool kBF16, int kMode, int SPLIT, bool kStats = false>
cudaError_t launch_mode(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& ty,
                        TcArgs a, cudaStream_t st) {
  using C = Cfg<H, HV, 2, (kMode == kAddMask) && (SPLIT == 1) && (H == 64) && (HV == 64)>;
  using Lay = Layout<2, SPLIT>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(prefill_tc_kernel<H, HV, kBF16, kMode, SPLIT, kStats>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    // the in-kernel register split assumes the block is launched with kLaunchRegs per
    // thread; with fewer, the softmax warps' request could never be met
    cudaFuncAttributes fa{};
    if (attr_err == cudaSuccess) attr_err = cudaFuncGetAttributes(&fa, prefill_tc_kernel<H, HV, kBF16, kMode, SPLIT, kStats>);
    if (attr_err == cudaSuccess && fa.numRegs < Lay::kLaunchRegs) attr_err = cudaErrorLaunchOutOfResources;
  });
  if (attr_err != cudaSuccess) return attr_err;
  // persistent: at most one CTA per SM (the tensor memory of a CTA fills the SM's), each
  // walking its share of the units
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = std::min(a.nunits, sms);
  prefill_tc_kernel<H, HV, kBF16, kMode, SPLIT, kStats><<<(unsigned)grid, Lay::kThreads, C::kSmem, st>>>(tq, tk, tv, ty, a);
  count_launch(1);
  return cudaGetLastError();
}

// Rule modes (additive mask, keep masks, bf16 softcap with a fixed maximum, per-element
// generic rules, plain interval rules), each a compile-time variant of the kernel.
template <int H, bool kBF16>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& ty,
                     const TcArgs& a, cudaStream_t st) {
  if (a.lse2_out) {
    // the backward's statistics pass, in the rule mode of the problem (no softcap: the
    // backward rejects it)
    if (a.has_softcap) return cudaErrorInvalidValue;
    if (a.generic) return launch_mode<H, H, kBF16, kGeneric, 1, true>(tq, tk, tv, ty, a, st);
    if (a.add_fast) return launch_mode<H, H, kBF16, kAddMask, 1, true>(tq, tk, tv, ty, a, st);
    if (a.keep_fast) return launch_mode<H, H, kBF16, kKeep, 1, true>(tq, tk, tv, ty, a, st);
    return launch_mode<H, H, kBF16, kPlain, 1, true>(tq, tk, tv, ty, a, st);
  }
  if (a.generic) return launch_mode<H, H, kBF16, kGeneric, 1>(tq, tk, tv, ty, a, st);
  if (a.keep_fast) return launch_mode<H, H, kBF16, kKeep, 1>(tq, tk, tv, ty, a, st);
  if (a.add_fast) return launch_mode<H, H, kBF16, kAddMask, 1>(tq, tk, tv, ty, a, st);
  if constexpr (kBF16)
    if (a.cap_fixed) return launch_mode<H, H, kBF16, kCapFixed, 1>(tq, tk, tv, ty, a, st);
  return launch_mode<H, H, kBF16, kPlain, 1>(tq, tk, tv, ty, a, st);
}

// A value head size different from the query/key one: the interval-rule mode when only
// structural rules (and softcap) apply, the per-element mode for everything else.
template <int H, int HV, bool kBF16>
cudaError_t launch_hv(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& ty,
                      const TcArgs& a, cudaStream_t st) {
  if (a.lse2_out) return cudaErrorInvalidValue;   // the backward takes H == Hv
  if (a.generic || a.keep_fast || a.add_fast) return launch_mode<H, HV, kBF16, kGeneric, 1>(tq, tk, tv, ty, a, st);
  return launch_mode<H, HV, kBF16, kPlain, 1>(tq, tk, tv, ty, a, st);
}

}  // namespace

void tc_axis_order(const View& v, int64_t B, int64_t N, int64_t S, int order[3]) {
  struct Ax { int64_t ext, stride; int id; };
  Ax ax[3] = {{S, v.ss, 0}, {N, v.sh, 1}, {B, v.sb, 2}};
  std::stable_sort(ax, ax + 3, [](const Ax& l, const Ax& r) {
    const bool l1 = l.ext == 1, r1 = r.ext == 1;
    if (l1 != r1) return r1;             // size-1 axes go last, in (seq, head, batch) order
    if (l1) return false;
    return l.stride < r.stride;
  });
  for (int k = 0; k < 3; ++k) order[k] = ax[k].id;
}

bool tc_same_axis_order(const View& k, const View& v, int64_t B, int64_t N, int64_t T) {
  int ok[3], ov[3];
  tc_axis_order(k, B, N, T, ok);
  tc_axis_order(v, B, N, T, ov);
  return ok[0] == ov[0] && ok[1] == ov[1] && ok[2] == ov[2];
}

bool tc_eligible(const Problem& p, sdpa_dtype dt) {
  if (dt != SDPA_F16 && dt != SDPA_BF16) return false;
  if ((p.H != 64 && p.H != 128) || (p.Hv != 64 && p.Hv != 128)) return false;
  if (p.T < 1 || p.S < 16) return false;
  if (p.T > (int64_t)1 << 30 || p.r.window > (int64_t)1 << 30) return false;
  for (const View* v : {&p.q, &p.k, &p.v})
    if (v->sb > ((int64_t)1 << 38) || v->sh > ((int64_t)1 << 38) || v->ss > ((int64_t)1 << 38)) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const Problem& p, sdpa_dtype dt, cudaStream_t st, const char** name) {
  return launch_prefill_tc_stats(p, dt, nullptr, nullptr, nullptr, st, name);
}

cudaError_t launch_prefill_tc_stats(const Problem& p, sdpa_dtype dt, float* lse2, float* delta, const View* dy,
                                    cudaStream_t st, const char** name) {
  TcArgs a{};
  a.B = p.B; a.Nq = p.Nq; a.Nkv = p.Nkv; a.S = p.S; a.T = (int)p.T; a.group = p.group;
  a.scale = p.scale;
  a.scale_log2 = p.scale * kLog2e;
  a.has_softcap = p.r.softcap > 0.f;
  a.cap_in = a.has_softcap ? p.scale / p.r.softcap : 0.f;
  a.cap_out_log2 = a.has_softcap ? p.r.softcap * kLog2e : 0.f;
  if (a.has_softcap) {
    // exponent = x (A + B x^2) - m on the raw product x = q.k, valid for |x scale / c| <= 0.25
    const double cin = (double)p.scale / p.r.softcap, K = (double)p.r.softcap * kLog2e;
    a.fx_a = (float)(kTanhMM1 * cin * K);
    a.fx_b = (float)(kTanhMM3 * cin * cin * cin * K);
    a.fx_lim = (float)(kTanhPolyLimit / std::fabs(cin));
  }
  a.causal = p.r.causal;
  a.window = (int)p.r.window;
  a.len_kind = p.r.len_kind;
  a.lens = p.r.lens;
  const bool other_rules = (p.r.keep_kind != SDPA_KEEP_NONE) || (p.r.len_kind == SDPA_LEN_KEYLEN_I32);
  a.keep_fast = other_rules && p.r.add == nullptr && !a.has_softcap;
  a.generic = other_rules && !a.keep_fast;
  if (a.keep_fast) {
    a.filter_raw = p.r.filter / p.scale;
    if (p.r.keep_kind != SDPA_KEEP_NONE) {
      // 16-byte loads need every row start 16-byte aligned (key offsets are multiples of 128)
      const int64_t esz = p.r.keep_kind == SDPA_KEEP_BOOL_U8 ? 1 : 4;
      uint64_t g = reinterpret_cast<uintptr_t>(p.r.keep);
      for (int64_t st : {p.r.keep_sb, p.r.keep_sh, p.r.keep_ss}) g |= (uint64_t)(st * esz);
      a.keep_vec = (g & 15u) == 0;
    }
  }
  a.add_fast = (p.r.add != nullptr) && !other_rules && p.r.add_dtype == (int)dt;
  if (p.r.add != nullptr && !a.add_fast) a.generic = 1;
  if (a.add_fast) {
    // widest load every mask row start allows (key offsets are multiples of 32 elements)
    const int64_t esz = p.r.add_dtype == SDPA_F32 ? 4 : 2;
    uint64_t g = reinterpret_cast<uintptr_t>(p.r.add) | 16u;
    for (int64_t st : {p.r.add_sb, p.r.add_sh, p.r.add_ss})
      if (st) g |= (uint64_t)(st * esz);
    a.add_vec = (int)(g & (~g + 1));   // lowest set bit
    if (a.add_vec > 16) a.add_vec = 16;
    // rows aligned to 4 bytes or more: coalesced copies through shared memory (cp.async
    // moves 4, 8 or 16 bytes); 2-byte-aligned rows keep the per-thread loads
    a.add_stage = esz == 2 && a.add_vec >= 4;
  }
  a.cap_fixed = dt == SDPA_BF16 && a.has_softcap && p.r.softcap <= 40.f && !a.generic && !a.add_fast && !a.keep_fast;
  a.r = p.r;
  a.y = const_cast<void*>(p.y.p);
  a.y_sb = p.y.sb; a.y_sh = p.y.sh; a.y_ss = p.y.ss;
  a.lse2_out = lse2;
  a.delta_out = delta;
  if (dy) { a.dy = dy->p; a.dy_sb = dy->sb; a.dy_sh = dy->sh; a.dy_ss = dy->ss; }
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
  // y: one 64-column x 32-row box per store; a statistics pass without y never stores and
  // takes Q's map as a stand-in
  CUtensorMap ty = tq;
  if (p.y.p && !make_map(&ty, p.y, dt, p.B, p.Nq, p.S, p.Hv, &a.y_ds, &a.y_dn, &a.y_db, 32))
    return cudaErrorInvalidValue;
  // work units: two heads of a group over one row block when the group is even, else two
  // consecutive row blocks of one head
  a.head_pairs = (p.group % 2) == 0;
  a.pairs = a.head_pairs ? p.group / 2 : p.group;
  a.nrow = a.head_pairs ? (p.S + kBM - 1) / kBM : (p.S + 2 * kBM - 1) / (2 * kBM);
  const int64_t units = (int64_t)a.nrow * p.B * p.Nkv * a.pairs;
  if (units > 0x7fffffff) return cudaErrorInvalidValue;
  a.nunits = (int)units;
  const bool bf = dt == SDPA_BF16;
  if (p.H != p.Hv) {
    if (a.keep_fast || a.add_fast) {   // per-element rules: the keep / additive-mask fast paths need H == Hv
      a.generic = 1;
      a.keep_fast = a.add_fast = 0;
    }
    a.cap_fixed = 0;
    if (p.H == 64) {
      *name = bf ? "prefill_tc_bf16_h64_hv128" : "prefill_tc_f16_h64_hv128";
      return bf ? launch_hv<64, 128, true>(tq, tk, tv, ty, a, st) : launch_hv<64, 128, false>(tq, tk, tv, ty, a, st);
    }
    *name = bf ? "prefill_tc_bf16_h128_hv64" : "prefill_tc_f16_h128_hv64";
    return bf ? launch_hv<128, 64, true>(tq, tk, tv, ty, a, st) : launch_hv<128, 64, false>(tq, tk, tv, ty, a, st);
  }
  if (p.H == 128) {
    *name = bf ? "prefill_tc_bf16_h128" : "prefill_tc_f16_h128";
    return bf ? launch_t<128, true>(tq, tk, tv, ty, a, st) : launch_t<128, false>(tq, tk, tv, ty, a, st);
  }
  *name = bf ? "prefill_tc_bf16_h64" : "prefill_tc_f16_h64";
  return bf ? launch_t<64, true>(tq, tk, tv, ty, a, st) : launch_t<64, false>(tq, tk, tv, ty, a, st);
}

PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn() { return encode_fn(); }

bool tc_make_map(CUtensorMap* map, const View& v, sdpa_dtype dt, int64_t B, int64_t N, int64_t Sq, int D, int* ds,
                 int* dn, int* db, int box_rows) {
  return make_map(map, v, dt, B, N, Sq, D, ds, dn, db, box_rows);
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

SDPA_DEFINE_BOUNDS_TAKE(take_bounds_prefill)

}  // namespace sdpa
