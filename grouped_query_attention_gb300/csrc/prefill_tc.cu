// Tensor-core flash prefill for GroupQueryAttention on sm_103a (fp16, head size 128).
//
// CTA = two 128-row query tiles of one KV head (b, g). Rows are the
// (position, grouped head) pairs of that KV head, so every K/V tile the CTA
// loads serves all G query heads of the group. Warp roles:
//   warp 0       TMA: both query tiles once, then K and V tiles of 128 keys
//                into a 2-stage ring (128-byte swizzle).
//   warp 1       MMA issue (one thread): S_q = Q_q K^T into tensor memory,
//                O_q += P_q V with P_q read from tensor memory; tensor-memory
//                allocation; zeroes V rows past the key range (no NaN * 0).
//   warps 2..5   softmax for query tile 0, warps 6..9 for query tile 1: one
//                thread per row; scores from tensor memory, causal / window /
//                live-length masks, softcap, bias, online max with lazy
//                rescaling of O in tensor memory, P written back over S as
//                fp16, epilogue O / l (+ sink term) to the output.
//                With a bias shared by all heads (G >= 8) warp 0 also copies
//                the bias block of each key tile (the CTA's distinct query
//                positions x 128 keys of the fp32 bias * log2(e) that a small
//                kernel stages before the launch) into a 2-stage shared ring
//                with one tensor copy; the softmax threads read it with
//                16-byte shared loads.
// The two softmax groups ping-pong: while one works on its tile the tensor
// core runs the other's MMAs. Tensor memory: S0 | S1 | O0 | O1 (512 columns).
// Every barrier wait is bounded; on expiry the CTA sets the TIMEOUT status
// bit, unwinds uniformly and still frees its tensor memory.
//
// com.microsoft.GroupQueryAttention, section Implementation variants
// (qkv_present_flash_cluster, past_kv_flash_prefill and its rotary / softcap
// / headsink / bias_headsink forms, share_append_split_flash_prefill:
// clustered online-softmax prefill over the cache as stored, causal bound
// right-aligned at the live length) and sections Inputs / Attributes.
#include <cuda_fp16.h>

#include "common.cuh"
#include "tcgen05.cuh"
#include "tma_host.h"

namespace gqa {
namespace {

using namespace tc;

constexpr int kBM = 128;                        // rows per query tile
constexpr int kBN = 128;                        // keys per K/V tile
constexpr int kHD = 128;                        // head size
constexpr int kNS = 2;                          // K/V stages
constexpr int kBiasRows = 33;                   // staged bias rows (distinct query positions of a CTA, G >= 8)
constexpr uint32_t kBiasBytes = kBiasRows * 128 * 4;   // one staged bias box (fp32)

// Kernel variants: scores without softcap and bias; softcap and/or bias read
// by each softmax thread; bias staged in shared memory by a loader warp.
enum PrefillMode { kPlain = 0, kGeneric = 1, kStagedBias = 2 };
__host__ __device__ constexpr int threads_for(int) { return 320; }
constexpr uint32_t kBox = 128u * 128u;          // one 64-column box of 128 rows (fp16) = 16 KB
constexpr uint32_t kTile = 2u * kBox;           // 128 rows x 128 columns = 32 KB
constexpr float kLazy = 8.0f;                   // log2 growth tolerated before rescaling O
constexpr uint32_t kIdS = idesc_f16(128, 128, 0, 0);   // Q (K-major) x K (K-major)
constexpr uint32_t kIdS64 = idesc_f16(128, 64, 0, 0);  // Q x half a K tile (64 keys)
constexpr uint32_t kIdO = idesc_f16(128, 128, 0, 1);   // P (tensor memory) x V (MN-major)

struct __align__(1024) TcSmem {
  uint8_t q[2][kTile];
  uint8_t k[kNS][kTile];
  uint8_t v[kNS][kTile];
  float bias[kNS][kBiasRows][kBN];                // staged bias rows, fp32 times log2(e)
  uint64_t q_land[2];           // query tile t copied (TMA)
  uint64_t q_ready[2];          // query tile t rewritten in place (norm / rotary by the softmax threads)
  uint64_t k_full[kNS], v_full[kNS], kv_empty[kNS];
  uint64_t bias_full[kNS], bias_empty[kNS];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t sb_full[2], sb_read[2];   // softcap / bias variants: second half of S landed / read (slab free)
  uint64_t drain;
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(TcSmem) + 1024 <= 232448, "shared memory per CTA");

__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           bool accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Constants of the transformed score in the log2 domain.
//   no softcap: x = raw * scale * log2(e) + bias * log2(e)
//   softcap c:  c * tanh(raw * scale / c) * log2(e) + bias * log2(e), with
//               tanh(u) = 1 - 2 / (exp(2u) + 1): e2 = exp2(raw * k_exp),
//               x = c log2(e) - 2 c log2(e) / (e2 + 1).
//   softcap, |u| = |raw * scale / c| <= 1/8 (every lane of a warp): the
//               same value on the FMA pipe, c tanh(u) log2(e) =
//               raw * scale * log2(e) * P(u^2), P below.
// tanh(u) / u = P(u^2) for |u| <= 1/8: degree-2 least-squares fit in z = u^2
// over [0, 1/64] (Chebyshev nodes, weighted for relative error), coefficients
// rounded to fp32: relative error 8.1e-9 in exact arithmetic.
constexpr float kTanhP1 = -3.3332762e-01f;
constexpr float kTanhP2 = 1.3216068e-01f;

struct ScoreConst {
  float k_raw;    // raw multiplier: scale * log2(e) (no softcap) or 2 * scale * log2(e) / c
  float k_mul;    // -2 c log2(e)
  float k_add;    // c log2(e)
  // Softcap on the FMA pipe in terms of the raw product x (u = x scale / c):
  // c tanh(u) log2(e) = x Q(x^2), Q(y) = sum_n C_n y^n with
  // C_n = scale log2(e) P_n (scale / c)^(2n) (P_0 = 1), so neither u nor the
  // final scale costs an operation per score.
  float cq[3];
  float yq;       // validity: x^2 <= (1/64) (c / scale)^2, i.e. |u| <= 1/8
};

__device__ __forceinline__ ScoreConst score_const(const Params& p) {
  ScoreConst k;
  k.k_raw = p.softcap > 0.f ? 2.0f * kLog2e * p.scale / p.softcap : p.scale * kLog2e;
  k.k_mul = -2.0f * p.softcap * kLog2e;
  k.k_add = p.softcap * kLog2e;
  const float ku = p.softcap > 0.f ? p.scale / p.softcap : 0.f;
  const float ku2 = ku * ku, kw = p.scale * kLog2e;
  const float pn[3] = {1.f, kTanhP1, kTanhP2};
  float pw = 1.f;
#pragma unroll
  for (int n = 0; n < 3; ++n) {
    k.cq[n] = kw * pn[n] * pw;
    pw *= ku2;
  }
  k.yq = ku2 > 0.f ? 0.015625f / ku2 : INFINITY;
  return k;
}

// Softcapped scores of two raw products on the FMA pipe, log2 domain, plus
// `add` (the bias in the log2 domain) in the last fused multiply-add; the
// squared raw products are returned for the validity check (x^2 <= yq).
__device__ __forceinline__ float2 softcap_poly2(float2 raw, const ScoreConst& k, float2& y, float2 add) {
  y = ffma2(raw, raw, make_float2(0.f, 0.f));
  float2 q = ffma2(y, make_float2(k.cq[2], k.cq[2]), make_float2(k.cq[1], k.cq[1]));
  q = ffma2(q, y, make_float2(k.cq[0], k.cq[0]));
  return ffma2(raw, q, add);
}



// Bias values of keys j .. j+31 (columns col0 .. col0+31 of the tile); zeros
// without a bias. 16-byte loads only where the address is 16-byte aligned and
// the whole 8-key group is visible; otherwise per-key loads of visible keys
// only (the bias row has total_sequence_length entries).
__device__ __forceinline__ void load_bias32(const __half* row, int j, int col0, int lo, int hi, float* out) {
  if (row == nullptr) {
#pragma unroll
    for (int e = 0; e < 32; ++e) out[e] = 0.f;
    return;
  }
#pragma unroll
  for (int g8 = 0; g8 < 32; g8 += 8) {
    const __half* src = row + j + g8;
    const int c0 = col0 + g8;
    if (c0 >= lo && c0 + 8 <= hi && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
      const uint4 u = *reinterpret_cast<const uint4*>(src);
      const __half2* h2 = reinterpret_cast<const __half2*>(&u);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(h2[e]);
        out[g8 + 2 * e] = f.x;
        out[g8 + 2 * e + 1] = f.y;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) out[g8 + e] = (c0 + e >= lo && c0 + e < hi) ? __half2float(src[e]) : 0.f;
    }
  }
}

// Query-block-major launch (prefill_prompt_qb_major) for prompts without a
// causal mask, where every block of a call is equally long: measured faster
// (202.7 against 208.9 us on a bidirectional B=4, S=2048 prompt). Causal
// prompts keep the KV-head-major order, in which the 64 blocks of a head run
// together over its K/V tiles (query-block-major measured 451 against 448 us
// on the causal B=4, S=4096 prompt).
__host__ __device__ inline bool tc_qb_major(const Params& p) { return prefill_prompt_qb_major(p) && !p.causal; }

// Causal prompts run KV-head-major, but the nqb / 8 shortest query blocks of
// every head are held back to the end of the grid, so that short blocks and
// not a late head's longest ones fill the tail while the long blocks keep
// starting at staggered times.
__host__ __device__ inline int tc_short_blocks(const Params& p, int nqb) {
  return p.mode == kPrompt && p.causal ? nqb / 8 : 0;
}

__device__ __forceinline__ bool aborted(const TcSmem& sm) {
  return *reinterpret_cast<const volatile int*>(&sm.abort) != 0;
}

__device__ __forceinline__ void set_abort(const Params& p, TcSmem& sm) {
  *reinterpret_cast<volatile int*>(&sm.abort) = 1;
  flag_status(p, GQA_DEVICE_TIMEOUT_BIT);
}

// All bits of `v` over the 128 threads of softmax group q (named barrier 1 + q).
__device__ __forceinline__ bool group_all(bool v, int q) {
  uint32_t r;
  asm volatile("{ .reg .pred p, c; setp.ne.u32 c, %1, 0; bar.red.and.pred p, %2, 128, c; selp.u32 %0, 1, 0, p; }"
               : "=r"(r)
               : "r"((uint32_t)v), "r"(1 + q)
               : "memory");
  return r != 0;
}

// Eight fp16 values (16 bytes) as fp32, and back (round to nearest).
__device__ __forceinline__ void ld_h8f(const __half* src, float* f) {
  const uint4 u = *reinterpret_cast<const uint4*>(src);
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 v = __half22float2(h[k]);
    f[2 * k] = v.x;
    f[2 * k + 1] = v.y;
  }
}

__device__ __forceinline__ uint4 f_to_h8(const float* f) {
  uint4 u;
  __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
  for (int k = 0; k < 4; ++k) h[k] = __floats2half2_rn(f[2 * k], f[2 * k + 1]);
  return u;
}

// RMS norm and rotary of one query row held by 8 lanes (lane l8: dims 8 l8 ..
// and 64 + 8 l8 ..), as packed fp32 pairs with fused multiply-adds: queries
// feed only the scores (no stored bytes depend on them), so they need no
// fixed rounding order. `ns` holds the negated sines.
__device__ __forceinline__ void norm_rope_q8(float2* lo, float2* hi, const float2* wlo, const float2* whi, bool norm,
                                             const float2* c, const float2* ns, float eps) {
  const float2 zero = make_float2(0.f, 0.f);
  if (norm) {
    float2 acc = zero;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc = ffma2(lo[k], lo[k], acc);
      acc = ffma2(hi[k], hi[k], acc);
    }
    float ss = acc.x + acc.y;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rn = rsqrtf(ss * (1.0f / 128.0f) + eps);
    const float2 rn2 = make_float2(rn, rn);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      lo[k] = ffma2(lo[k], ffma2(wlo[k], rn2, zero), zero);
      hi[k] = ffma2(hi[k], ffma2(whi[k], rn2, zero), zero);
    }
  }
  if (c) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 a = lo[k], b = hi[k];
      lo[k] = ffma2(b, ns[k], ffma2(a, c[k], zero));             // a c - b s
      hi[k] = ffma2(a, make_float2(-ns[k].x, -ns[k].y), ffma2(b, c[k], zero));   // b c + a s
    }
  }
}

// In-place query preparation (q_in_prefill with RMS norm and / or rotary):
// the TMA warp loads the raw query rows of the CTA's two tiles, row r of the
// (b, g) block = (position i = r / G, head g G + r % G), already in the
// 128-byte-swizzled K-major layout the S MMA reads; these threads rewrite
// them as norm, then rotary at the absolute position past + i, fp16
// (com.microsoft.GroupQueryAttention, section Inputs: q_norm_weight,
// cos/sin_cache; section Implementation variants: rotary flash prefill
// rotates query blocks at their absolute positions). `wt` = 0..255 over the
// softmax threads: 8 lanes per row, 32 rows per pass, four passes per tile;
// the cos/sin rows are loaded before the wait for the tile, and ready[t] is
// arrived (one arrival per warp) once tile t is rewritten. Rows past the
// block hold zeros (the copy's fill) and stay zero.
__device__ void transform_q_tiles(const Params& p, TcSmem& sm, int past, int r0, int nrows, int wt) {
  const int l8 = wt & 7, sub = wt >> 3, lane = wt & 31;
  float2 wlo[4], whi[4];
  if (p.has_norm) {
    ld_h8f(reinterpret_cast<const __half*>(p.qw) + 8 * l8, reinterpret_cast<float*>(wlo));
    ld_h8f(reinterpret_cast<const __half*>(p.qw) + 64 + 8 * l8, reinterpret_cast<float*>(whi));
  }
  const __half* cbase = reinterpret_cast<const __half*>(p.cos_c);
  const __half* sbase = reinterpret_cast<const __half*>(p.sin_c);
  for (int tile = 0; tile < 2; ++tile) {
    uint4 cs[4], sn[4];
    if (p.has_rotary) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = min(r0 + tile * kBM + k * 32 + sub, nrows - 1);
        const long long cb = (long long)(past + r / p.G) * (kHD / 2) + 8 * l8;
        cs[k] = __ldg(reinterpret_cast<const uint4*>(cbase + cb));
        sn[k] = __ldg(reinterpret_cast<const uint4*>(sbase + cb));
      }
    }
    if (!__all_sync(0xffffffffu, mbar_wait(&sm.q_land[tile], 0, p.wait_budget)) && lane == 0) set_abort(p, sm);
    uint8_t* qt = sm.q[tile];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int rl = k * 32 + sub;              // row inside the tile
      float2 lo[4], hi[4], c[4], ns[4];
      ld_h8f(reinterpret_cast<const __half*>(qt + sw128_offset(rl, l8)), reinterpret_cast<float*>(lo));
      ld_h8f(reinterpret_cast<const __half*>(qt + kBox + sw128_offset(rl, l8)), reinterpret_cast<float*>(hi));
      if (p.has_rotary) {
        const uint4 nsn = make_uint4(sn[k].x ^ 0x80008000u, sn[k].y ^ 0x80008000u, sn[k].z ^ 0x80008000u,
                                     sn[k].w ^ 0x80008000u);   // negated fp16 sines
        ld_h8f(reinterpret_cast<const __half*>(&cs[k]), reinterpret_cast<float*>(c));
        ld_h8f(reinterpret_cast<const __half*>(&nsn), reinterpret_cast<float*>(ns));
      }
      norm_rope_q8(lo, hi, wlo, whi, p.has_norm != 0, p.has_rotary ? c : nullptr, ns, p.eps);
      *reinterpret_cast<uint4*>(qt + sw128_offset(rl, l8)) = f_to_h8(reinterpret_cast<const float*>(lo));
      *reinterpret_cast<uint4*>(qt + kBox + sw128_offset(rl, l8)) = f_to_h8(reinterpret_cast<const float*>(hi));
    }
    fence_async_smem();   // rewritten tile (generic stores) -> async proxy: the S MMAs may read it
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.q_ready[tile]);
  }
}

// MODE (PrefillMode): kPlain has no softcap and no bias (the scores are the
// scaled products); kGeneric reads the bias per thread; kStagedBias adds the
// bias loader warp. CAP: softcap > 0 (compile-time, so that the 32 scores of
// a group are independent straight-line chains the scheduler can interleave).
template <int MODE, bool CAP>
__global__ void __launch_bounds__(threads_for(MODE), 1)
prefill_tc_kernel(const Params p, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmb,
                  const __grid_constant__ CUtensorMap tmo) {
  constexpr bool PLAIN = MODE == kPlain;
  constexpr bool STAGED = MODE == kStagedBias;
  constexpr int kThreads = threads_for(MODE);
  extern __shared__ uint8_t smem_raw[];
  TcSmem& sm = *reinterpret_cast<TcSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nrows = p.S * p.G;
  const int nqb = (nrows + 2 * kBM - 1) / (2 * kBM);
  int qb, bg;   // longest key ranges first
  if (tc_qb_major(p)) {
    qb = nqb - 1 - (int)blockIdx.y;
    bg = (int)blockIdx.x;
  } else {
    // KV-head-major; the ks shortest query blocks of every head follow all the others.
    const int ks = tc_short_blocks(p, nqb);
    const int lin = (int)(blockIdx.y * gridDim.x + blockIdx.x), n1 = (int)gridDim.y * (nqb - ks);
    if (lin < n1) {
      bg = lin / (nqb - ks);
      qb = nqb - 1 - lin % (nqb - ks);
    } else {
      bg = (lin - n1) / ks;
      qb = ks - 1 - (lin - n1) % ks;
    }
  }
  const int b = bg / p.Nkv, g = bg % p.Nkv;

  // ---- block-uniform checks before any barrier or tensor memory
  const int total = p.seqlens[b] + 1;
  const int past = batch_past(p, total);
  if (past < 0) {
    if (qb == nqb - 1 && g == 0 && tid == 0) flag_status(p, GQA_DEVICE_BAD_SEQLEN_BIT);
    return;
  }
  if (p.has_rotary && past + p.S > p.rotary_rows) return;  // flagged by the pre-pass
  const int live_i = p.mode == kPrompt ? min(p.S, total) : p.S;
  const int r0 = qb * 2 * kBM;
  const int i_lo = r0 / p.G;
  const int i_hi = min((min(r0 + 2 * kBM, nrows) - 1) / p.G, live_i - 1);
  if (i_lo > i_hi) {
    // Only prompt padding rows here: their output is 0.
    for (int x = tid; x < 2 * kBM * kHD; x += kThreads) {
      const int r = r0 + x / kHD, d = x % kHD;
      if (r >= nrows) continue;
      const int i = r / p.G, h = g * p.G + r % p.G;
      reinterpret_cast<__half*>(p.out)[((long long)(b * p.S + i) * p.N + h) * kHD + d] = __float2half_rn(0.f);
    }
    return;
  }
  const int kmax = p.causal ? min(total, past + i_hi + 1) : total;
  // First key of the tile grid, rounded down to a multiple of 8 so that bias
  // rows (when 16-byte aligned) are read with 16-byte loads; extra keys are masked.
  const int kmin = (p.window >= 0 ? max(0, past + i_lo - p.window) : 0) & ~7;
  const int ntiles = (kmax - kmin + kBN - 1) / kBN;

  if (warp == 1) tmem_alloc(&sm.tmem, 512);
  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.q_land[t], 1);
      mbar_init(&sm.q_ready[t], 8);   // one arrival per softmax warp
    }
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&sm.s_full[q], 1);
      mbar_init(&sm.p_full[q], kBM);
      mbar_init(&sm.o_done[q], 1);
      mbar_init(&sm.sb_full[q], 1);
      mbar_init(&sm.sb_read[q], 4);   // one arrival per softmax warp of the group
    }
    if constexpr (STAGED) {
      for (int s = 0; s < kNS; ++s) {
        mbar_init(&sm.bias_full[s], 1);           // the TMA warp's elected lane (with the copy's bytes)
        mbar_init(&sm.bias_empty[s], 8);          // one lane of every softmax warp
      }
    }
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  const int qrow0 = bg * nrows + r0;                 // row of Q0 in the prepared-query matrix
  const bool qx = p.q_in_prefill && (p.has_norm || p.has_rotary);   // query tiles rewritten in place
  const int krow0 = bg * (p.kv_separate ? p.S : p.C) + kmin;   // row of the first key in the K/V matrix

  if (warp == 0) {
    // ================================================================ TMA producer
    // The whole warp waits; one elected lane issues. With a staged bias the
    // warp then loads the bias block of the same key tile with one tensor
    // copy: stage s holds the staged bias rows bb*S + i_lo .. +kBiasRows-1
    // (fp32 times log2(e)), keys j0 .. j0+127; keys past the bias row read 0.
    const int brow0 = STAGED ? (p.bias_bdim > 1 ? b : 0) * p.S + i_lo : 0;
    if (elect_one()) {
      for (int q = 0; q < 2; ++q) {
        mbar_arrive_tx(&sm.q_land[q], kTile);
        for (int bx = 0; bx < 2; ++bx) {
          if (p.q_in_prefill)   // raw query rows: positions (r0 + 128 q) / G .., heads g G ..
            tma_load_4d(sm.q[q] + bx * kBox, &tmq, bx * 64, g * p.G, (r0 + q * kBM) / p.G, b, &sm.q_land[q]);
          else                  // queries prepared by the pre-pass
            tma_load_2d(sm.q[q] + bx * kBox, &tmq, bx * 64, qrow0 + q * kBM, &sm.q_land[q]);
        }
      }
    }
    __syncwarp();
    int issued = 0, issued_b = 0;
    for (int t = 0; t < ntiles; ++t) {
      if (t == p.withhold_tile) break;   // testing: no copy of this tile, its waits expire
      const int st = t % kNS;
      const uint32_t ph = (uint32_t)(t / kNS) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.kv_empty[st], ph ^ 1u, p.wait_budget)) || aborted(sm)) {
        if (lane == 0) set_abort(p, sm);
        break;
      }
      const int row = krow0 + t * kBN;
      if (elect_one()) {
        mbar_arrive_tx(&sm.k_full[st], kTile);
        for (int bx = 0; bx < 2; ++bx) tma_load_2d(sm.k[st] + bx * kBox, &tmk, bx * 64, row, &sm.k_full[st]);
        mbar_arrive_tx(&sm.v_full[st], kTile);
        for (int bx = 0; bx < 2; ++bx) tma_load_2d(sm.v[st] + bx * kBox, &tmv, bx * 64, row, &sm.v_full[st]);
      }
      __syncwarp();
      issued = t + 1;
      if constexpr (STAGED) {
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.bias_empty[st], ph ^ 1u, p.wait_budget)) || aborted(sm)) {
          if (lane == 0) set_abort(p, sm);
          break;
        }
        if (elect_one()) {
          mbar_arrive_tx(&sm.bias_full[st], kBiasBytes);
          tma_load_2d(&sm.bias[st][0][0], &tmb, kmin + t * kBN, brow0, &sm.bias_full[st]);
        }
        __syncwarp();
        issued_b = t + 1;
      }
    }
    // Drain: no copy of this CTA may still be landing when it exits.
    mbar_wait(&sm.q_land[0], 0, p.wait_budget);
    mbar_wait(&sm.q_land[1], 0, p.wait_budget);
    for (int t = max(0, issued_b - kNS); t < issued_b; ++t)
      mbar_wait(&sm.bias_full[t % kNS], (uint32_t)(t / kNS) & 1u, p.wait_budget);
    for (int t = max(0, issued - kNS); t < issued; ++t) {
      mbar_wait(&sm.k_full[t % kNS], (uint32_t)(t / kNS) & 1u, p.wait_budget);
      mbar_wait(&sm.v_full[t % kNS], (uint32_t)(t / kNS) & 1u, p.wait_budget);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    // Shared-memory descriptors built once; a K step adds its start-address
    // offset (16-byte units). One elected lane issues, the warp stays converged.
    // Stage s of the K (V) ring starts kTile bytes after stage s-1: its
    // descriptor is the stage-0 one plus that offset in 16-byte units (the
    // start-address field cannot overflow: shared addresses are below 256 KB).
    uint64_t dq[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) dq[i] = desc_kmajor_sw128(smem_addr(sm.q[i]));
    const uint64_t dk0 = desc_kmajor_sw128(smem_addr(sm.k[0]));
    const uint64_t dv0 = desc_mnmajor_sw128(smem_addr(sm.v[0]), kBox, 1024);
    auto issue_s = [&](int q, int st) {
      const uint32_t d = tmem + q * 128;
      const uint64_t a0 = dq[q], b0 = dk0 + (uint64_t)(st * (int)(kTile >> 4));
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t off = (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2);
        mma_f16_ss(d, a0 + off, b0 + off, kIdS, ks > 0);
      }
      mma_commit(&sm.s_full[q]);
    };
    auto issue_pv = [&](int q, int st, bool acc) {
      const uint32_t d = tmem + 256 + q * 128;
      const uint32_t pa = tmem + q * 128;  // P over the first 64 columns of S_q
      const uint64_t b0 = dv0 + (uint64_t)(st * (int)(kTile >> 4));
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) mma_f16_ts(d, pa + ks * 8, b0 + (uint64_t)(ks * 128), kIdO, acc || ks > 0);
      mma_commit(&sm.o_done[q]);
    };
    // Softcap / bias variants: S in two halves of 64 keys (N = 64) in the two
    // 64-column slabs of the group's tensor memory. Tile t: keys 0..63 in slab
    // t & 1 (A), keys 64..127 in the other (B); P of the whole tile is packed
    // into slab A. So slab B is free as soon as the softmax has read the second
    // half, and the first half of S(t+1) goes there while the softmax finishes
    // tile t; the second half follows P.V(t) into slab A.
    auto issue_s_half = [&](int q, int st, int half, int slab) {
      const uint32_t d = tmem + q * 128 + slab * 64;
      const uint64_t a0 = dq[q], b0 = dk0 + (uint64_t)(st * (int)(kTile >> 4) + half * 512);   // 64 key rows = 8 KB
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t off = (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2);
        mma_f16_ss(d, a0 + off, b0 + off, kIdS64, ks > 0);
      }
      mma_commit(half == 0 ? &sm.s_full[q] : &sm.sb_full[q]);
    };
    auto issue_pv_slab = [&](int q, int st, bool acc, int slab) {
      const uint32_t d = tmem + 256 + q * 128;
      const uint32_t pa = tmem + q * 128 + slab * 64;   // P packed over slab A of the tile
      const uint64_t b0 = dv0 + (uint64_t)(st * (int)(kTile >> 4));
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) mma_f16_ts(d, pa + ks * 8, b0 + (uint64_t)(ks * 128), kIdO, acc || ks > 0);
      mma_commit(&sm.o_done[q]);
    };
    // V rows past the key range (stale cache rows may hold any bits) are zeroed.
    auto wait_v = [&](int t, int st) {
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.v_full[st], (uint32_t)(t / kNS) & 1u, p.wait_budget))) return false;
      const int valid = kmax - (kmin + t * kBN);
      if (valid < kBN) {
        for (int x = lane; x < (kBN - valid) * 16; x += 32) {
          const int r = valid + x / 16, c = x % 16;
          *reinterpret_cast<uint4*>(sm.v[st] + (c >> 3) * kBox + r * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();
      }
      __syncwarp();
      return true;
    };
    // Query tile t is ready once copied, or once rewritten in place when the
    // softmax threads apply norm / rotary; S_0(0) may start before tile 1 is.
    uint64_t* qready = qx ? sm.q_ready : sm.q_land;
    bool ok = __all_sync(0xffffffffu, mbar_wait(&qready[0], 0, p.wait_budget) && mbar_wait(&sm.k_full[0], 0, p.wait_budget));
    for (int q = 0; q < 2 && ok; ++q) {
      if (q == 1) ok = __all_sync(0xffffffffu, mbar_wait(&qready[1], 0, p.wait_budget));
      if (!ok) break;
      if (elect_one()) {
        tc_fence_after();
        if constexpr (PLAIN) {
          issue_s(q, 0);
        } else {
          issue_s_half(q, 0, 0, 0);
          issue_s_half(q, 0, 1, 1);
        }
      }
      __syncwarp();
    }
    if constexpr (PLAIN) {
      for (int t = 0; t < ntiles && ok; ++t) {
        const int st = t % kNS;
        const uint32_t tp = (uint32_t)t & 1u;
        if (!wait_v(t, st)) {
          ok = false;
          break;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.p_full[0], tp, p.wait_budget))) {
          ok = false;
          break;
        }
        if (elect_one()) {
          tc_fence_after();
          issue_pv(0, st, t > 0);
        }
        __syncwarp();
        const bool more = t + 1 < ntiles;
        const int st1 = (t + 1) % kNS;
        if (more && !__all_sync(0xffffffffu, mbar_wait(&sm.k_full[st1], (uint32_t)((t + 1) / kNS) & 1u, p.wait_budget))) {
          ok = false;
          break;
        }
        if (more && elect_one()) issue_s(0, st1);
        __syncwarp();
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.p_full[1], tp, p.wait_budget))) {
          ok = false;
          break;
        }
        if (elect_one()) {
          tc_fence_after();
          issue_pv(1, st, t > 0);
          mma_commit(&sm.kv_empty[st]);
          if (more) issue_s(1, st1);
        }
        __syncwarp();
        if (__any_sync(0xffffffffu, aborted(sm))) ok = false;
      }
    } else {
      for (int t = 0; t < ntiles && ok; ++t) {
        const int st = t % kNS, slab_a = t & 1, slab_b = slab_a ^ 1;
        const uint32_t tp = (uint32_t)t & 1u;
        const bool more = t + 1 < ntiles;
        const int st1 = (t + 1) % kNS;
        for (int q = 0; q < 2 && ok; ++q) {
          // S_q(t+1), keys 0..63: slab B once the softmax has read the second half of S_q(t).
          if (more) {
            if (!__all_sync(0xffffffffu, mbar_wait(&sm.sb_read[q], tp, p.wait_budget) &&
                                             mbar_wait(&sm.k_full[st1], (uint32_t)((t + 1) / kNS) & 1u, p.wait_budget))) {
              ok = false;
              break;
            }
            if (elect_one()) {
              tc_fence_after();
              issue_s_half(q, st1, 0, slab_b);
            }
            __syncwarp();
          }
          if ((q == 0 && !wait_v(t, st)) ||
              !__all_sync(0xffffffffu, mbar_wait(&sm.p_full[q], tp, p.wait_budget))) {
            ok = false;
            break;
          }
          // P.V(t) reads P from slab A; S_q(t+1), keys 64..127, then overwrites it.
          if (elect_one()) {
            tc_fence_after();
            issue_pv_slab(q, st, t > 0, slab_a);
            if (q == 1) mma_commit(&sm.kv_empty[st]);
            if (more) issue_s_half(q, st1, 1, slab_a);
          }
          __syncwarp();
        }
        if (__any_sync(0xffffffffu, aborted(sm))) ok = false;
      }
    }
    if (!ok && lane == 0) set_abort(p, sm);
    // Drain: every MMA this thread issued has finished before tensor memory is freed.
    if (elect_one()) {
      mma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, p.wait_budget);
    }
    __syncwarp();
  } else {
    // ================================================================ softmax groups
    const int q = (warp - 2) >> 2;            // query tile of this group
    const int quarter = warp & 3;             // tensor-memory lane quarter of this warp
    const int rl = quarter * 32 + lane;       // row inside the tile
    const int r = r0 + q * kBM + rl;          // row of the (b, g) block
    const bool row_ok = r < nrows;
    const int i = row_ok ? r / p.G : 0;
    const int h = g * p.G + (row_ok ? r % p.G : 0);
    const int pos = past + i;
    const bool live = row_ok && i < live_i;
    const int hi_key = live ? (p.causal ? min(total, pos + 1) : total) : 0;   // visible keys [lo_key, hi_key)
    const int lo_key = p.window >= 0 ? max(0, pos - p.window) : 0;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + q * 128;
    const uint32_t o_addr = tmem + lane_addr + 256 + q * 128;
    const float qk_scale = p.softcap > 0.f ? p.scale : p.scale * kLog2e;
    const __half* bias_row = nullptr;
    if (!STAGED && p.has_bias && live)
      bias_row = reinterpret_cast<const __half*>(p.bias) +
                 (((long long)(p.bias_bdim > 1 ? b : 0) * p.bias_ndim + (p.bias_ndim > 1 ? h : 0)) * p.S + i) *
                     p.bias_ld;
    const int brow = live ? i - i_lo : 0;     // staged bias row of this thread (any in-range row when not live)
    if (qx) transform_q_tiles(p, sm, past, r0, nrows, tid - 64);
    const ScoreConst kc = score_const(p);
    float m_run = kNegBig, l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      bool got = mbar_wait(&sm.s_full[q], (uint32_t)t & 1u, p.wait_budget) && !aborted(sm);
      if constexpr (STAGED) got = got && mbar_wait(&sm.bias_full[t % kNS], (uint32_t)(t / kNS) & 1u, p.wait_budget);
      if (!__all_sync(0xffffffffu, got)) {   // the warp leaves together
        ok = false;
        break;
      }
      tc_fence_after();
      const int j0 = kmin + t * kBN;
      const int lo = max(lo_key - j0, 0), hi = min(hi_key - j0, kBN);   // visible columns [lo, hi)
      // Warp-uniform fast path: no row of this warp needs a mask on this tile.
      const bool full = __all_sync(0xffffffffu, lo == 0 && hi == kBN);
      // Plain scores: pass 1 takes the row max over the whole row (four loads
      // in flight, one wait, the raw products scaled once: the scale is
      // positive), pass 2 writes P = exp2(score - m) over S. Softcap / bias:
      // one pass per half of 64 columns: transform, half max, raise the
      // reference max when the half exceeds it by more than 2^8 (rescaling O,
      // l and the half already written), exp2 and pack P.
      float2 ls2 = make_float2(0.f, 0.f);
      if constexpr (PLAIN) {
        float mt = kNegBig;
        {
          uint32_t r[kBN];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, r + c * 32);
          tmem_ld_wait();
          float m4[4] = {kNegBig, kNegBig, kNegBig, kNegBig};   // four independent chains
          if (!full) {
            // Masked columns become -inf in tensor memory too, so pass 2 needs
            // no mask (the scale is positive: exp2 of -inf * scale - m is 0).
#pragma unroll
            for (int e = 0; e < kBN; ++e) r[e] = (e >= lo && e < hi) ? r[e] : 0xff800000u;
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_st32(s_addr + c * 32, r + c * 32);
            tmem_st_wait();
          }
#pragma unroll
          for (int e = 0; e < kBN; e += 2)
            m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], __uint_as_float(r[e]), __uint_as_float(r[e + 1]));
          const float m = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          mt = m > kNegBig ? m * qk_scale : kNegBig;
        }
        // Lazy rescale: a row moves its reference max only when the tile max
        // exceeds it by more than 2^8. The tensor-memory traffic is warp-wide,
        // so the whole warp takes the branch and lanes that keep their max use f = 1.
        const bool grow = mt > m_run + kLazy;
        const float m_new = grow ? mt : m_run;
        if (t > 0 && __any_sync(0xffffffffu, grow)) {
          // O_q is complete up to tile t-1 (its MMAs precede S_q(t)): rescale it in place.
          const float f = grow ? ex2(m_run - m_new) : 1.0f;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t raw[32];
            tmem_ld32(o_addr + c * 32, raw);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) raw[e] = __float_as_uint(__uint_as_float(raw[e]) * f);
            tmem_st32(o_addr + c * 32, raw);
          }
          l_run *= f;
        }
        m_run = m_new;
        // Pass 2: P = exp2(score - m) as fp16 pairs over the first 64 columns of
        // S_q, 64 scores per load batch; columns are overwritten only after read.
        const float neg_m = -m_run;
        const float2 scale2 = make_float2(qk_scale, qk_scale), negm2 = make_float2(neg_m, neg_m);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t r[64];
          tmem_ld32(s_addr + hf * 64, r);
          tmem_ld32(s_addr + hf * 64 + 32, r + 32);
          tmem_ld_wait();
          uint32_t packed[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float xa = __uint_as_float(r[2 * k]), xb = __uint_as_float(r[2 * k + 1]);
            const float2 arg = ffma2(make_float2(xa, xb), scale2, negm2);
            const float pa = ex2(arg.x), pb = ex2(arg.y);
            ls2 = ffma2(make_float2(pa, pb), make_float2(1.f, 1.f), ls2);
            const __half2 hp = __floats2half2_rn(pa, pb);
            packed[k] = *reinterpret_cast<const uint32_t*>(&hp);
          }
          tmem_st32(s_addr + hf * 32, packed);
        }
      } else {
        // Keys 0..63 of the tile in slab A = t & 1, keys 64..127 in slab B (the
        // other one, landing later); P of both halves is packed into slab A.
        const uint32_t s_a = s_addr + (uint32_t)(t & 1) * 64, s_b = s_addr + (uint32_t)((t & 1) ^ 1) * 64;
        bool half_ok = true;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          const uint32_t s_h = hf == 0 ? s_a : s_b;
          if (hf == 1 && !__all_sync(0xffffffffu, mbar_wait(&sm.sb_full[q], (uint32_t)t & 1u, p.wait_budget))) {
            half_ok = false;
            break;
          }
          tc_fence_after();
          uint32_t r[64];
          tmem_ld32(s_h, r);
          tmem_ld32(s_h + 32, r + 32);
          tmem_ld_wait();
          // Transform the half in place: scale, softcap, bias. With a softcap the
          // FMA-pipe polynomial goes first and is checked afterwards (|u| <= 1/8
          // on every lane of the warp, from the largest raw^2); otherwise the raw
          // scores are read again from tensor memory (intact: P of this half is
          // written after it) and take the exp2 / reciprocal form.
          auto transform = [&](bool poly) -> float {
            float zmax = 0.f;
#pragma unroll
            for (int c = 0; c < 64; c += 32) {
              float bv[32];
              if constexpr (!STAGED) load_bias32(bias_row, j0 + hf * 64 + c, hf * 64 + c, lo, hi, bv);
#pragma unroll
              for (int c16 = 0; c16 < 32; c16 += 16) {   // 16 independent chains at a time
                float x[16];
                if (CAP && poly) {   // bias added in the polynomial's last fused multiply-add
                  float ba[16];
                  if constexpr (STAGED) {
                    const float4* b4 = reinterpret_cast<const float4*>(&sm.bias[t % kNS][brow][hf * 64 + c + c16]);
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) {
                      const float4 bq = b4[e4];
                      ba[4 * e4] = bq.x;
                      ba[4 * e4 + 1] = bq.y;
                      ba[4 * e4 + 2] = bq.z;
                      ba[4 * e4 + 3] = bq.w;
                    }
                  } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) ba[e] = bv[c16 + e] * kLog2e;
                  }
#pragma unroll
                  for (int e = 0; e < 16; e += 2) {
                    float2 z;
                    const float2 raw2 = make_float2(__uint_as_float(r[c + c16 + e]), __uint_as_float(r[c + c16 + e + 1]));
                    const float2 bias2 = make_float2(ba[e], ba[e + 1]);
                    const float2 y = softcap_poly2(raw2, kc, z, bias2);
                    r[c + c16 + e] = __float_as_uint(y.x);
                    r[c + c16 + e + 1] = __float_as_uint(y.y);
                    zmax = fmax3(zmax, z.x, z.y);
                  }
                  continue;   // scores and bias done for this group
                } else {
#pragma unroll
                  for (int e = 0; e < 16; ++e) x[e] = __uint_as_float(r[c + c16 + e]) * kc.k_raw;
                  if constexpr (CAP) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = fmaf(rcp_approx(ex2(x[e]) + 1.0f), kc.k_mul, kc.k_add);
                  }
                }
                if constexpr (STAGED) {
                  // Staged bias: fp32, already times log2(e).
                  const float4* b4 = reinterpret_cast<const float4*>(&sm.bias[t % kNS][brow][hf * 64 + c + c16]);
#pragma unroll
                  for (int e4 = 0; e4 < 4; ++e4) {
                    const float4 bq = b4[e4];
                    x[4 * e4] += bq.x;
                    x[4 * e4 + 1] += bq.y;
                    x[4 * e4 + 2] += bq.z;
                    x[4 * e4 + 3] += bq.w;
                  }
                } else {
#pragma unroll
                  for (int e = 0; e < 16; ++e) x[e] = fmaf(bv[c16 + e], kLog2e, x[e]);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) r[c + c16 + e] = __float_as_uint(x[e]);
              }
            }
            return zmax;
          };
          if constexpr (CAP) {
            const float zmax = transform(true);
            if (__any_sync(0xffffffffu, !(zmax <= kc.yq))) {
              tmem_ld32(s_h, r);
              tmem_ld32(s_h + 32, r + 32);
              tmem_ld_wait();
              transform(false);
            }
          } else {
            transform(false);
          }
          if (hf == 1) {   // slab B read: the MMA may put the next tile's first half there
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.sb_read[q]);
          }
          if (!full) {   // warp-uniform: only tiles on a mask boundary pay for the selects
#pragma unroll
            for (int e = 0; e < 64; ++e) {
              const int col = hf * 64 + e;
              r[e] = (col >= lo && col < hi) ? r[e] : 0xff800000u;   // -inf
            }
          }
          float m4[4] = {kNegBig, kNegBig, kNegBig, kNegBig};   // four independent chains
#pragma unroll
          for (int e = 0; e < 64; e += 2)
            m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], __uint_as_float(r[e]), __uint_as_float(r[e + 1]));
          const float mh = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          const bool grow = mh > m_run + kLazy;
          if (__any_sync(0xffffffffu, grow)) {   // warp-wide tensor-memory traffic
            const float m_new = grow ? mh : m_run;
            const float f = grow ? ex2(m_run - m_new) : 1.0f;
            if (t > 0) {
              // Rescale O_q in place once it holds P.V up to tile t-1: the first
              // half of S_q(t) is issued before P.V(t-1), so that half waits for
              // it; the second half of S_q(t) is issued after it.
              if (hf == 0 && !__all_sync(0xffffffffu, mbar_wait(&sm.o_done[q], (uint32_t)(t - 1) & 1u, p.wait_budget)))
                half_ok = false;
              tc_fence_after();
#pragma unroll 1
              for (int c = 0; c < 8; ++c) {   // 16 columns at a time (the half's scores stay live)
                uint32_t raw[16];
                tmem_ld16(o_addr + c * 16, raw);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) raw[e] = __float_as_uint(__uint_as_float(raw[e]) * f);
                tmem_st16(o_addr + c * 16, raw);
              }
            }
            if (hf == 1) {
              // P of the first half was written with the old reference.
              tmem_st_wait();
              const float2 f2 = make_float2(f, f);
#pragma unroll 1
              for (int c = 0; c < 2; ++c) {
                uint32_t pk[16];
                tmem_ld16(s_a + c * 16, pk);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                  const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&pk[k]));
                  const float2 w = ffma2(v, f2, make_float2(0.f, 0.f));
                  const __half2 hw = __floats2half2_rn(w.x, w.y);
                  pk[k] = *reinterpret_cast<const uint32_t*>(&hw);
                }
                tmem_st16(s_a + c * 16, pk);
              }
            }
            l_run *= f;
            ls2.x *= f;
            ls2.y *= f;
            m_run = m_new;
          }
          // Masked scores are -inf: exp2 gives 0. P goes out 16 columns at a time.
          const float2 negm2 = make_float2(-m_run, -m_run);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t packed[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int e = 32 * h2 + 2 * k;
              const float2 arg = ffma2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                                       make_float2(1.f, 1.f), negm2);
              const float pa = ex2(arg.x), pb = ex2(arg.y);
              ls2 = ffma2(make_float2(pa, pb), make_float2(1.f, 1.f), ls2);
              const __half2 hp = __floats2half2_rn(pa, pb);
              packed[k] = *reinterpret_cast<const uint32_t*>(&hp);
            }
            tmem_st16(s_a + hf * 32 + 16 * h2, packed);
          }
        }
        if (!half_ok) {
          ok = false;
          break;
        }
        if constexpr (STAGED) {
          // The warp's bias reads have returned (their values are used above).
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.bias_empty[t % kNS]);
        }
      }
      const float ls = ls2.x + ls2.y;
      l_run += ls;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm.p_full[q]);
    }
    // ---- epilogue: O / l (+ sink), fp16, one row per thread. With raw query
    // tiles (the group size divides 128) the rows are staged in the group's
    // query tile (free: every S MMA of the group is done once its last P.V is),
    // in the copied layout, and one thread writes the tile with two tensor
    // stores (rows past S are skipped); otherwise each thread stores its row.
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&sm.o_done[q], (uint32_t)(ntiles - 1) & 1u, p.wait_budget) && !aborted(sm));
    float scale_out = 0.f;
    if (ok) {
      tc_fence_after();
      float mf = m_run, extra = 0.f;
      if (p.has_sink || p.smooth) {
        const float sg = (p.has_sink ? __half2float(reinterpret_cast<const __half*>(p.sink)[h]) : 0.f) * kLog2e;
        mf = fmaxf(m_run, sg);
        extra = ex2(sg - mf);
      }
      const float f = ex2(m_run - mf);
      const float den = l_run * f + extra;
      scale_out = (live && den > 0.f) ? f / den : 0.f;
    }
    if (p.q_in_prefill) {
      if (ok) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t raw[32];
          tmem_ld32(o_addr + c * 32, raw);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; e += 8) {   // dims 32 c + e .. : box (32 c + e) / 64, chunk ((32 c + e) % 64) / 8
            uint4 u;
            __half2* h2 = reinterpret_cast<__half2*>(&u);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              h2[k] = __floats2half2_rn(__uint_as_float(raw[e + 2 * k]) * scale_out,
                                        __uint_as_float(raw[e + 2 * k + 1]) * scale_out);
            const int d = c * 32 + e;
            *reinterpret_cast<uint4*>(sm.q[q] + (d >> 6) * kBox + sw128_offset(rl, (d & 63) >> 3)) = u;
          }
        }
        fence_async_smem();   // staged rows (generic stores) -> async proxy: the tensor stores read them
      }
      if (!group_all(ok, q)) {
        if (lane == 0) set_abort(p, sm);
      } else if (quarter == 2 && elect_one()) {   // warp 2 (group 0) or 6 (group 1)
        for (int bx = 0; bx < 2; ++bx) tma_store_4d(&tmo, sm.q[q] + bx * kBox, 64 * bx, g * p.G, (r0 + q * kBM) / p.G, b);
        bulk_commit();
        bulk_wait_read();   // the staged tile is read before the CTA may exit
      }
    } else if (!ok) {
      set_abort(p, sm);
    } else {
      __half* orow = reinterpret_cast<__half*>(p.out) + ((long long)(b * p.S + i) * p.N + h) * kHD;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t raw[32];
        tmem_ld32(o_addr + c * 32, raw);   // all lanes (warp-wide); only real rows store
        tmem_ld_wait();
        if (!row_ok) continue;
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 u;
          __half2* h2 = reinterpret_cast<__half2*>(&u);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            h2[k] = __floats2half2_rn(__uint_as_float(raw[e + 2 * k]) * scale_out,
                                      __uint_as_float(raw[e + 2 * k + 1]) * scale_out);
          *reinterpret_cast<uint4*>(orow + c * 32 + e) = u;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

// A bias shared by all heads is staged by TMA when a CTA's 256 rows span at
// most kBiasRows query positions (255 / G + 2 bounds the span).
bool prefill_tc_bias_staged(const Params& p) {
  return p.has_bias && p.bias_ndim == 1 && 255 / p.G + 2 <= kBiasRows;
}

bool prefill_tc_supported(const Params& p) {
  // With kv_separate attention reads the new rows in T (fp16 here).
  return p.t_type == kF16 && (p.cache_type == kF16 || p.kv_separate) && p.H == kHD;
}

cudaError_t prepare_prefill_tc(const Params& p, TmaMaps* maps) {
  const long long krows = (long long)p.B * p.Nkv * (p.kv_separate ? p.S : p.C);
  cudaError_t e;
  const void* ksrc = p.kv_separate ? p.kv_sep_k : p.present_k;
  const void* vsrc = p.kv_separate ? p.kv_sep_v : p.present_v;
  if ((e = encode_fp16_2d_sw128(&maps->m[1], ksrc, (uint64_t)krows, kHD, kHD * 2, 64, kBN)) != cudaSuccess)
    return e;
  if ((e = encode_fp16_2d_sw128(&maps->m[2], vsrc, (uint64_t)krows, kHD, kHD * 2, 64, kBN)) != cudaSuccess)
    return e;
  maps->m[4] = maps->m[2];   // a valid map in the output slot when the epilogue stores per thread (never read)
  if (p.q_in_prefill) {
    if ((e = encode_fp16_query_sw128(&maps->m[0], p.q, p.B, p.S, p.N, (uint32_t)p.G)) != cudaSuccess) return e;
    if ((e = encode_fp16_query_sw128(&maps->m[4], p.out, p.B, p.S, p.N, (uint32_t)p.G)) != cudaSuccess) return e;
  } else {
    const long long qrows = (long long)p.B * p.Nkv * p.S * p.G;
    if ((e = encode_fp16_2d_sw128(&maps->m[0], p.qprep, (uint64_t)qrows, kHD, kHD * 2, 64, kBM)) != cudaSuccess)
      return e;
  }
  maps->m[3] = maps->m[2];   // a valid map in the bias slot when nothing is staged (never read)
  if (!prefill_tc_bias_staged(p)) return cudaSuccess;
  return encode_f32_2d(&maps->m[3], p.bias_stage, (uint64_t)p.bias_bdim * p.S, (uint64_t)p.bias_ld,
                       (uint64_t)p.bias_stage_ld * 4, kBN, kBiasRows);
}

namespace {
// Dynamic shared memory opt-in, set once per device and kernel variant.
constexpr int kMaxDevices = 64;
bool g_smem_set[5][kMaxDevices];
}  // namespace

cudaError_t launch_prefill_tc(const Params& p, cudaStream_t st, const TmaMaps& maps) {
  const int smem = (int)sizeof(TcSmem) + 1024;
  // The plain kernel scales the row max once, which needs a positive scale.
  const bool plain = p.softcap <= 0.f && !p.has_bias && p.scale > 0.f;
  const bool staged = prefill_tc_bias_staged(p);
  const int mode = plain ? kPlain : staged ? kStagedBias : kGeneric;
  const bool cap = p.softcap > 0.f;
  auto kern = mode == kPlain ? prefill_tc_kernel<kPlain, false>
              : mode == kStagedBias ? (cap ? prefill_tc_kernel<kStagedBias, true> : prefill_tc_kernel<kStagedBias, false>)
                                    : (cap ? prefill_tc_kernel<kGeneric, true> : prefill_tc_kernel<kGeneric, false>);
  const int variant = mode == kPlain ? 0 : 1 + 2 * (mode == kStagedBias) + cap;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!g_smem_set[variant][dev]) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
    g_smem_set[variant][dev] = true;
  }
  const int nrows = p.S * p.G;
  const unsigned nqb = (unsigned)((nrows + 2 * kBM - 1) / (2 * kBM)), nbg = (unsigned)(p.B * p.Nkv);
  const dim3 grid = tc_qb_major(p) ? dim3(nbg, nqb) : dim3(nqb, nbg);
  kern<<<grid, threads_for(mode), smem, st>>>(p, maps.m[0], maps.m[1], maps.m[2], maps.m[3], maps.m[4]);
  return cudaGetLastError();
}

}  // namespace gqa
