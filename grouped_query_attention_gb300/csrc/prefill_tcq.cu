// Tensor-core flash prefill over an int8 or 4-bit cache with fp32 queries,
// keys, values and output (sm_103a, head size 128).
//
// The cache codes are small integers, exact in fp16; the channel scales are
// folded into the query (K) and into the output (V). fp32 accuracy on fp16
// tensor cores comes from splitting each fp32 operand that is not exact in
// fp16 into two fp16 parts:
//   q' = rotary(norm(q)) * scale (log2 domain unless softcap) * K channel
//        scale, times 2^-e (2^e the power of two at or below the row's
//        largest |q'|); hi = fp16(q' 2^-e), lo = fp16(q' 2^-e - hi), so
//        hi + lo keeps about 22 bits and S = (hi + lo) . codes is accumulated
//        in fp32 by two MMA chains into the same tensor-memory columns;
//   P    = exp2(s - m) is split the same way, O += P_hi V + P_lo V.
// That is twice the tensor work of the fp16 prefill per visible pair.
//
// CTA = two 128-row query tiles of one KV head (b, g), rows = (position,
// grouped head) as in the fp16 prefill. Warp roles (384 threads):
//   warp 0       TMA: the raw fp32 query rows of both tiles (four boxes of 32
//                dimensions, 128-byte swizzle).
//   warp 1       MMA issue and tensor-memory allocation.
//   warps 2..9   all eight first rewrite the two query tiles in place as the
//                hi and lo fp16 operand tiles (8 lanes per row); then softmax,
//                one thread per row of query tile (warp - 2) / 4, and the
//                epilogue, which stages O in the group's query region and
//                writes it with tensor stores.
//   warps 10..13 converters, 32 key rows each: the codes of the next K or V
//                tile are loaded from global memory into registers while the
//                current one is converted to its fp16 operand tile (K-major
//                K, two buffers; MN-major V, one buffer; 128-byte swizzle).
// Shared memory: query tiles 128 KB, fp16 K 2 x 32 KB, fp16 V 32 KB.
// Tensor memory: S0 | S1 | O0 | O1. The MMA order is the fp16 prefill's (P.V
// of one tile, then S of the other tile's next key tile); K(t+1) may be
// converted from the moment S_1(t-1) is done, V(t) while S_1(t) runs. Every
// barrier wait is bounded.
//
// com.microsoft.GroupQueryAttention, section Implementation variants
// (quant_int8_flash_prefill, quant_int4_flash_prefill: attention over the
// stored codes times their per-tensor or per-channel scales) and sections
// Inputs / Attributes (k_scale, v_scale, kv_cache_bit_width).
#include <cuda_fp16.h>

#include "common.cuh"
#include "tcgen05.cuh"
#include "tma_host.h"

namespace gqa {
namespace {

using namespace tc;

constexpr int kBM = 128;                       // rows per query tile
constexpr int kBN = 128;                       // keys per K/V tile
constexpr int kHD = 128;                       // head size
constexpr int kThreads = 448;
constexpr int kConvWarp0 = 10;                 // first converter warp
constexpr int kConvWarps = 4;                  // converter warps, 32 key rows each
constexpr int kConvRows = kBN / kConvWarps;
constexpr uint32_t kBox = 128u * 128u;         // 128 rows x 128 bytes = 16 KB
constexpr uint32_t kTile = 2u * kBox;          // fp16 operand tile, 128 x 128
constexpr uint32_t kQRegion = 4u * kBox;       // fp32 query tile = hi and lo fp16 tiles
constexpr float kLazy = 8.0f;                  // log2 growth tolerated before rescaling O
constexpr uint32_t kIdS = idesc_f16(128, 128, 0, 0);   // Q (K-major) x K (K-major)
constexpr uint32_t kIdO = idesc_f16(128, 128, 0, 1);   // P (tensor memory) x V (MN-major)

struct __align__(1024) QcSmem {
  // Per query tile: box k holds dims 32k .. 32k+31 (fp32) as copied; after the
  // rewrite boxes 0, 1 are the hi fp16 tile (dims 0..63, 64..127) and boxes
  // 2, 3 the lo fp16 tile; after the last S MMA the epilogue stages O here
  // (fp32, the copied layout).
  uint8_t q[2][kQRegion];
  uint8_t kf[2][kTile];         // K codes as fp16, K-major (the B operand of S), tile t in buffer t & 1
  uint8_t vf[kTile];            // V codes as fp16, MN-major (the B operand of O)
  float rho[2][kBM];            // 2^e of each query row (S 2^e is the scaled score)
  uint64_t q_land[2], q_ready[2];
  uint64_t kf_full[2], kf_empty[2], vf_full, vf_empty;   // fp16 tiles: converters <-> MMA
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t drain;
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(QcSmem) + 1024 <= 232448, "shared memory per CTA");

__device__ __forceinline__ bool aborted(const QcSmem& sm) {
  return *reinterpret_cast<const volatile int*>(&sm.abort) != 0;
}

__device__ __forceinline__ void set_abort(const Params& p, QcSmem& sm) {
  *reinterpret_cast<volatile int*>(&sm.abort) = 1;
  flag_status(p, GQA_DEVICE_TIMEOUT_BIT);
}

// Sixteen int8 codes (one 16-byte chunk) as sixteen fp16 values: the byte
// x ^ 0x80 placed under the fp16 exponent of 1024 gives 1024 + x + 128
// exactly, and 1152 is subtracted (exact: small integers).
__device__ __forceinline__ void i8x16_to_h16(uint4 w, uint32_t* h) {
  const __half2 bias = __floats2half2_rn(1152.f, 1152.f);
  const uint32_t wv[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t p01 = __byte_perm(wv[k], 0x64646464u, 0x4140u);
    const uint32_t p23 = __byte_perm(wv[k], 0x64646464u, 0x4342u);
    const __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&p01), bias);
    const __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&p23), bias);
    h[2 * k] = *reinterpret_cast<const uint32_t*>(&a);
    h[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&c);
  }
}

// Thirty-two 4-bit codes (16 bytes; byte k holds coordinates 2k (low nibble)
// and 2k+1, each +8-biased) as thirty-two fp16 values. Per byte n the pair
// (n & 15, n & 0xF0) goes under the fp16 exponent of 1024: 1024 + lo and
// 1024 + 16 hi; one fused multiply-add by (1, 1/16) and (-1032, -72) leaves
// lo - 8 and hi - 8 (every step exact).
__device__ __forceinline__ void i4x32_to_h32(uint4 w, uint32_t* h) {
  const __half2 mul = __floats2half2_rn(1.0f, 0.0625f);
  const __half2 add = __floats2half2_rn(-1032.0f, -72.0f);
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int by = 0; by < 4; ++by) {
      const uint32_t t = __byte_perm(wv[k], 0u, 0x4040u | (uint32_t)by | ((uint32_t)by << 8));
      const uint32_t u = (t & 0x00F0000Fu) | 0x64006400u;
      const __half2 v = __hfma2(*reinterpret_cast<const __half2*>(&u), mul, add);
      h[4 * k + by] = *reinterpret_cast<const uint32_t*>(&v);
    }
  }
}

// Codes of key rows [row0, row0 + 32) of a tile whose first cache row is
// `grow0`: lane l takes 16-byte chunk x = 32 s + l of the 32-row block in step
// s (row x / chunks, chunk x % chunks); rows past the cache read as zeros.
template <int BITS>
__device__ __forceinline__ void load_codes(const uint8_t* cache, long long grow0, long long nrows_cache, int row0,
                                           int lane, uint4* w) {
  constexpr int kRowBytes = BITS == 8 ? 128 : 64;
  constexpr int kChunks = kRowBytes / 16;
  constexpr int kSteps = kConvRows * kChunks / 32;
#pragma unroll
  for (int s = 0; s < kSteps; ++s) {
    const int x = s * 32 + lane, row = row0 + x / kChunks, j = x % kChunks;
    const long long gr = grow0 + row;
    w[s] = gr < nrows_cache ? __ldg(reinterpret_cast<const uint4*>(cache + gr * kRowBytes + j * 16))
                            : make_uint4(0u, 0u, 0u, 0u);
  }
}

// The codes of load_codes as fp16 into the operand tile `dst` (128-byte
// swizzle; box bx = dims 64 bx .. 64 bx + 63).
template <int BITS>
__device__ __forceinline__ void store_codes_h(const uint4* w, uint8_t* dst, int row0, int lane) {
  constexpr int kRowBytes = BITS == 8 ? 128 : 64;
  constexpr int kChunks = kRowBytes / 16;
  constexpr int kSteps = kConvRows * kChunks / 32;
#pragma unroll
  for (int s = 0; s < kSteps; ++s) {
    const int x = s * 32 + lane, row = row0 + x / kChunks, j = x % kChunks;
    if constexpr (BITS == 8) {
      // chunk j: dims 16 j .. 16 j + 15 = fp16 chunks 2 (j % 4), +1 of box j / 4
      uint32_t h[8];
      i8x16_to_h16(w[s], h);
      uint8_t* b = dst + (j >> 2) * kBox;
      *reinterpret_cast<uint4*>(b + sw128_offset(row, 2 * (j & 3))) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(b + sw128_offset(row, 2 * (j & 3) + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
    } else {
      // chunk j: dims 32 j .. 32 j + 31 = fp16 chunks 4 (j % 2) .. +3 of box j / 2
      uint32_t h[16];
      i4x32_to_h32(w[s], h);
      uint8_t* b = dst + (j >> 1) * kBox;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(b + sw128_offset(row, 4 * (j & 1) + c)) =
            make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
    }
  }
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

__device__ __forceinline__ void ld_f8(const float* src, float* f) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(src));
  const float4 b = __ldg(reinterpret_cast<const float4*>(src) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ void lds_f8(const uint8_t* line, int c0, int rl, float* f) {
  const float4 a = *reinterpret_cast<const float4*>(line + sw128_offset(rl, c0));
  const float4 b = *reinterpret_cast<const float4*>(line + sw128_offset(rl, c0 + 1));
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// Both query tiles, in place, by the 256 softmax threads (wt = 0..255): 8
// lanes per row (lane l8: dims 8 l8 .. and 64 + 8 l8 .., so the rotary
// partner is in the lane), 32 rows per pass, four passes per tile. A row is
// normalised (q_norm_weight), rotated at its absolute position (cos/sin_cache),
// scaled (score scale, K channel scale), brought to [1, 2) by 2^-e and split
// into hi = fp16(x) and lo = fp16(x - hi), written over the same four 128-byte
// lines that held it (hi: boxes 0, 1; lo: boxes 2, 3); 2^e goes to rho. The
// lanes of a row read before any of them writes (__syncwarp). Queries feed
// only the scores, so the rounding order is free (fused multiply-adds).
// Rows past the block were filled with zeros by the copy and stay zero.
__device__ void split_query_tiles(const Params& p, QcSmem& sm, int past, int r0, int nrows, int g, int wt,
                                  float qscale) {
  const int l8 = wt & 7, sub = wt >> 3, lane = wt & 31;
  float wlo[8], whi[8], klo[8], khi[8];
  if (p.has_norm) {
    ld_f8(reinterpret_cast<const float*>(p.qw) + 8 * l8, wlo);
    ld_f8(reinterpret_cast<const float*>(p.qw) + 64 + 8 * l8, whi);
  }
  if (p.k_scale_n == 1) {
#pragma unroll
    for (int k = 0; k < 8; ++k) klo[k] = khi[k] = qscale * p.k_scale[0];
  } else {
    ld_f8(p.k_scale + g * kHD + 8 * l8, klo);
    ld_f8(p.k_scale + g * kHD + 64 + 8 * l8, khi);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      klo[k] *= qscale;
      khi[k] *= qscale;
    }
  }
  const float* cbase = reinterpret_cast<const float*>(p.cos_c);
  const float* sbase = reinterpret_cast<const float*>(p.sin_c);
  for (int tile = 0; tile < 2; ++tile) {
    if (!__all_sync(0xffffffffu, mbar_wait(&sm.q_land[tile], 0, p.wait_budget)) && lane == 0) set_abort(p, sm);
    uint8_t* qt = sm.q[tile];
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
      const int rl = k * 32 + sub;                               // row inside the tile
      const int r = min(r0 + tile * kBM + rl, nrows - 1);
      float lo[8], hi[8];
      lds_f8(qt + (l8 >> 2) * kBox, 2 * (l8 & 3), rl, lo);
      lds_f8(qt + (2 + (l8 >> 2)) * kBox, 2 * (l8 & 3), rl, hi);
      if (p.has_norm) {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(hi[e], hi[e], fmaf(lo[e], lo[e], ss));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float rn = rsqrtf(ss * (1.0f / kHD) + p.eps);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          lo[e] *= rn * wlo[e];
          hi[e] *= rn * whi[e];
        }
      }
      if (p.has_rotary) {
        float c[8], sn[8];
        const long long cb = (long long)(past + r / p.G) * (kHD / 2) + 8 * l8;
        ld_f8(cbase + cb, c);
        ld_f8(sbase + cb, sn);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float a = lo[e], b = hi[e];
          lo[e] = fmaf(a, c[e], -b * sn[e]);
          hi[e] = fmaf(b, c[e], a * sn[e]);
        }
      }
      float mx = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        lo[e] *= klo[e];
        hi[e] *= khi[e];
        mx = fmax3(mx, fabsf(lo[e]), fabsf(hi[e]));
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      // 2^e <= mx < 2^(e+1) from the exponent bits (mx = 0 or subnormal: e = 0).
      const int ebits = (__float_as_int(mx) >> 23) & 0xff;
      const int e = ebits == 0 ? 0 : ebits - 127;
      const float down = __int_as_float((127 - e) << 23);
      uint32_t hw[2][4], lw[2][4];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float* x = half == 0 ? lo : hi;
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          const float a = x[2 * k2] * down, b = x[2 * k2 + 1] * down;
          const __half2 hh = __floats2half2_rn(a, b);
          const float2 hf = __half22float2(hh);
          const __half2 ll = __floats2half2_rn(a - hf.x, b - hf.y);
          hw[half][k2] = *reinterpret_cast<const uint32_t*>(&hh);
          lw[half][k2] = *reinterpret_cast<const uint32_t*>(&ll);
        }
      }
      __syncwarp();   // every lane of the row has read its values
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        *reinterpret_cast<uint4*>(qt + half * kBox + sw128_offset(rl, l8)) =
            make_uint4(hw[half][0], hw[half][1], hw[half][2], hw[half][3]);
        *reinterpret_cast<uint4*>(qt + (2 + half) * kBox + sw128_offset(rl, l8)) =
            make_uint4(lw[half][0], lw[half][1], lw[half][2], lw[half][3]);
      }
      if (l8 == 0) sm.rho[tile][rl] = __int_as_float((127 + e) << 23);
    }
    fence_async_smem();   // rewritten tile (generic stores) -> async proxy: the S MMAs may read it
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.q_ready[tile]);
  }
}

// BITS: 8 (int8 cache) or 4 (4-bit cache). PLAIN: no softcap and no bias
// (the scores are S 2^e, already in the log2 domain); otherwise softcap and
// bias are applied per thread in the max pass and written back to tensor memory.
template <int BITS, bool PLAIN>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tcq_kernel(const Params p, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmo) {
  extern __shared__ uint8_t smem_raw[];
  QcSmem& sm = *reinterpret_cast<QcSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nrows = p.S * p.G;
  const int nqb = (nrows + 2 * kBM - 1) / (2 * kBM);
  // Query-block-major for prompts (127 against 145 us on the causal int8
  // B=2, S=2048 prompt: with three to four waves of CTAs the tail counts).
  const bool qbm = prefill_prompt_qb_major(p);
  const int qb = nqb - 1 - (int)(qbm ? blockIdx.y : blockIdx.x);  // longest key ranges first
  const int bg = (int)(qbm ? blockIdx.x : blockIdx.y), b = bg / p.Nkv, g = bg % p.Nkv;

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
      reinterpret_cast<float*>(p.out)[((long long)(b * p.S + i) * p.N + h) * kHD + d] = 0.f;
    }
    return;
  }
  const int kmax = p.causal ? min(total, past + i_hi + 1) : total;
  const int kmin = p.window >= 0 ? max(0, past + i_lo - p.window) : 0;
  const int ntiles = (kmax - kmin + kBN - 1) / kBN;

  if (warp == 1) tmem_alloc(&sm.tmem, 512);
  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.q_land[t], 1);
      mbar_init(&sm.q_ready[t], 8);   // one arrival per softmax warp
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.p_full[t], kBM);
      mbar_init(&sm.o_done[t], 1);
      mbar_init(&sm.kf_full[t], kConvWarps);   // one arrival per converter warp
      mbar_init(&sm.kf_empty[t], 1);  // MMA commits
    }
    mbar_init(&sm.vf_full, kConvWarps);
    mbar_init(&sm.vf_empty, 1);
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  const long long krow0 = (long long)bg * p.C + kmin;   // cache row of the first key

  if (warp == 0) {
    // ================================================================ TMA: query tiles
    if (elect_one()) {
      for (int q = 0; q < 2; ++q) {
        mbar_arrive_tx(&sm.q_land[q], kQRegion);
        for (int k = 0; k < 4; ++k)
          tma_load_4d(sm.q[q] + k * kBox, &tmq, 32 * k, g * p.G, (r0 + q * kBM) / p.G, b, &sm.q_land[q]);
      }
    }
    __syncwarp();
    // No copy of this CTA may still be landing when it exits.
    mbar_wait(&sm.q_land[0], 0, p.wait_budget);
    mbar_wait(&sm.q_land[1], 0, p.wait_budget);
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    uint64_t dk[2], dq[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      dk[i] = desc_kmajor_sw128(smem_addr(sm.kf[i]));
      dq[i] = desc_kmajor_sw128(smem_addr(sm.q[i]));
    }
    const uint64_t dv = desc_mnmajor_sw128(smem_addr(sm.vf), kBox, 1024);
    // S_q = Q_hi K^T + Q_lo K^T (the lo tile starts 32 KB after the hi tile).
    auto issue_s = [&](int q, int kb) {
      const uint32_t d = tmem + q * 128;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint64_t a0 = dq[q] + (uint64_t)(part * (int)((2 * kBox) >> 4));
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t off = (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2);
          mma_f16_ss(d, a0 + off, dk[kb] + off, kIdS, part > 0 || ks > 0);
        }
      }
      mma_commit(&sm.s_full[q]);
    };
    // O_q += P_hi V + P_lo V. Keys 64 h .. 64 h + 63 of P: hi pairs in columns
    // 64 h .. 64 h + 31 of S_q, lo pairs in the next 32.
    auto issue_pv = [&](int q, bool acc) {
      const uint32_t d = tmem + 256 + q * 128;
      const uint32_t pa = tmem + q * 128;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t col = (uint32_t)((ks >> 2) * 64 + (ks & 3) * 8);
        const uint64_t bv = dv + (uint64_t)(ks * 128);
        mma_f16_ts(d, pa + col, bv, kIdO, acc || ks > 0);
        mma_f16_ts(d, pa + col + 32, bv, kIdO, true);
      }
      mma_commit(&sm.o_done[q]);
    };
    bool ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_ready[0], 0, p.wait_budget) &&
                                          mbar_wait(&sm.kf_full[0], 0, p.wait_budget));
    if (ok && elect_one()) {
      tc_fence_after();
      issue_s(0, 0);
    }
    __syncwarp();
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_ready[1], 0, p.wait_budget));
    if (ok && elect_one()) {
      tc_fence_after();
      issue_s(1, 0);
      mma_commit(&sm.kf_empty[0]);
    }
    __syncwarp();
    for (int t = 0; t < ntiles && ok; ++t) {
      const uint32_t tp = (uint32_t)t & 1u;
      const bool more = t + 1 < ntiles;
      const int kb1 = (t + 1) & 1;                                 // K buffer of tile t+1
      const uint32_t kp1 = (uint32_t)((t + 1) >> 1) & 1u;          // its use parity
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.vf_full, tp, p.wait_budget) &&
                                       mbar_wait(&sm.p_full[0], tp, p.wait_budget))) {
        ok = false;
        break;
      }
      if (elect_one()) {
        tc_fence_after();
        issue_pv(0, t > 0);
      }
      __syncwarp();
      if (more && !__all_sync(0xffffffffu, mbar_wait(&sm.kf_full[kb1], kp1, p.wait_budget))) {
        ok = false;
        break;
      }
      if (more && elect_one()) {
        tc_fence_after();
        issue_s(0, kb1);
      }
      __syncwarp();
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.p_full[1], tp, p.wait_budget))) {
        ok = false;
        break;
      }
      if (elect_one()) {
        tc_fence_after();
        issue_pv(1, t > 0);
        mma_commit(&sm.vf_empty);
        if (more) {
          issue_s(1, kb1);
          mma_commit(&sm.kf_empty[kb1]);
        }
      }
      __syncwarp();
      if (__any_sync(0xffffffffu, aborted(sm))) ok = false;
    }
    if (!ok && lane == 0) set_abort(p, sm);
    // Drain: every MMA this thread issued has finished before tensor memory is freed.
    if (elect_one()) {
      mma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, p.wait_budget);
    }
    __syncwarp();
  } else if (warp >= kConvWarp0) {
    // ================================================================ converters
    // Conversion order: K(0), then K(t+1) (its buffer is free once S_1(t-1)
    // is done), V(t) (free once P_1.V(t-1) is done). The codes of the next
    // conversion are loaded while the current one waits and converts.
    constexpr int kSteps = kConvRows * (BITS == 8 ? 8 : 4) / 32;
    const int row0 = (warp - kConvWarp0) * kConvRows;
    const long long ncache = (long long)p.B * p.Nkv * p.C;
    const uint8_t* kcache = static_cast<const uint8_t*>(p.present_k);
    const uint8_t* vcache = static_cast<const uint8_t*>(p.present_v);
    const int nconv = 2 * ntiles;
    // item n: 0 -> K(0); 2t+1 -> K(t+1) (V(t) when t is the last tile); 2t+2 -> V(t)
    auto item = [&](int n, bool& is_k) -> int {
      if (n == 0) {
        is_k = true;
        return 0;
      }
      const int t = (n - 1) >> 1;
      is_k = ((n - 1) & 1) == 0 && t + 1 < ntiles;
      return is_k ? t + 1 : t;
    };
    auto load = [&](int n, uint4* w) {
      bool is_k;
      const int u = item(n, is_k);
      load_codes<BITS>(is_k ? kcache : vcache, krow0 + (long long)u * kBN, ncache, row0, lane, w);
    };
    bool withheld = false;
    auto convert = [&](int n, const uint4* w) -> bool {
      bool is_k;
      const int u = item(n, is_k);
      if (u == p.withhold_tile) {   // testing: this tile is never converted, the waits for it expire
        withheld = true;
        return false;
      }
      uint64_t* empty = is_k ? &sm.kf_empty[u & 1] : &sm.vf_empty;
      const uint32_t pe = (is_k ? (uint32_t)(u >> 1) : (uint32_t)u) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(empty, pe ^ 1u, p.wait_budget)) || aborted(sm)) return false;
      store_codes_h<BITS>(w, is_k ? sm.kf[u & 1] : sm.vf, row0, lane);
      fence_async_smem();   // fp16 tile (generic stores) -> async proxy: the MMAs may read it
      __syncwarp();
      if (lane == 0) mbar_arrive(is_k ? &sm.kf_full[u & 1] : &sm.vf_full);
      return true;
    };
    uint4 wa[kSteps], wb[kSteps];
    bool ok = true;
    load(0, wa);
    for (int n = 0; n < nconv && ok; n += 2) {
      if (n + 1 < nconv) load(n + 1, wb);
      ok = convert(n, wa);
      if (!ok || n + 1 >= nconv) break;
      if (n + 2 < nconv) load(n + 2, wa);
      ok = convert(n + 1, wb);
    }
    if (!ok && !withheld && lane == 0) set_abort(p, sm);
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
    const bool cap = p.softcap > 0.f;
    const float* bias_row = nullptr;
    if (!PLAIN && p.has_bias && live)
      bias_row = reinterpret_cast<const float*>(p.bias) +
                 (((long long)(p.bias_bdim > 1 ? b : 0) * p.bias_ndim + (p.bias_ndim > 1 ? h : 0)) * p.S + i) *
                     p.bias_ld;

    split_query_tiles(p, sm, past, r0, nrows, g, tid - 64, cap ? p.scale : p.scale * kLog2e);
    bool ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_ready[q], 0, p.wait_budget));   // rho of every row written
    const float rho = sm.rho[q][rl];

    // Score of column e in the log2 domain: S rho (plain); with softcap c the
    // tanh form on S rho = scale q.k, then + bias log2(e).
    const float k_raw = cap ? rho * 2.0f * kLog2e / p.softcap : rho;
    const float k_mul = -2.0f * p.softcap * kLog2e, k_add = p.softcap * kLog2e;
    float m_run = kNegBig, l_run = 0.f;
    for (int t = 0; t < ntiles && ok; ++t) {
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_full[q], (uint32_t)t & 1u, p.wait_budget) && !aborted(sm))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int j0 = kmin + t * kBN;
      const int lo = max(lo_key - j0, 0), hi = min(hi_key - j0, kBN);   // visible columns [lo, hi)
      const bool full = __all_sync(0xffffffffu, lo == 0 && hi == kBN);
      // Pass 1: row max, 64 columns at a time. Masked columns (and, with
      // softcap / bias, every transformed score) are written back so that
      // pass 2 is the same for all.
      float mt;
      {
        float m4[4] = {kNegBig, kNegBig, kNegBig, kNegBig};   // four independent chains
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t x[64];
          tmem_ld32(s_addr + hf * 64, x);
          tmem_ld32(s_addr + hf * 64 + 32, x + 32);
          tmem_ld_wait();
          if constexpr (!PLAIN) {
#pragma unroll
            for (int e = 0; e < 64; ++e) {
              const int col = hf * 64 + e;
              float v = __uint_as_float(x[e]) * k_raw;
              if (cap) v = fmaf(__frcp_rn(ex2(v) + 1.0f), k_mul, k_add);
              if (bias_row != nullptr && col >= lo && col < hi) v = fmaf(bias_row[j0 + col], kLog2e, v);
              x[e] = __float_as_uint(v);
            }
          }
          if (!PLAIN || !full) {
#pragma unroll
            for (int e = 0; e < 64; ++e) {
              const int col = hf * 64 + e;
              x[e] = (col >= lo && col < hi) ? x[e] : 0xff800000u;   // -inf
            }
            tmem_st32(s_addr + hf * 64, x);
            tmem_st32(s_addr + hf * 64 + 32, x + 32);
          }
#pragma unroll
          for (int e = 0; e < 64; e += 2)
            m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], __uint_as_float(x[e]), __uint_as_float(x[e + 1]));
        }
        if (!PLAIN || !full) tmem_st_wait();
        const float m = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        mt = m > kNegBig ? (PLAIN ? m * k_raw : m) : kNegBig;   // k_raw = rho > 0 in the plain form
      }
      // Lazy rescale: the reference max moves only when the tile max exceeds
      // it by more than 2^8; O_q is complete up to tile t-1 (its MMAs precede S_q(t)).
      const bool grow = mt > m_run + kLazy;
      const float m_new = grow ? mt : m_run;
      if (t > 0 && __any_sync(0xffffffffu, grow)) {
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
      // Pass 2: P = exp2(score - m), split into fp16 hi and lo; keys 64 hf ..
      // of the half: hi pairs over columns 64 hf .. 64 hf + 31, lo pairs over
      // the next 32 (only columns of the half just read are overwritten).
      const float mul2 = PLAIN ? k_raw : 1.0f;
      const float2 mul22 = make_float2(mul2, mul2), negm2 = make_float2(-m_run, -m_run);
      float2 ls2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t x[64];
        tmem_ld32(s_addr + hf * 64, x);
        tmem_ld32(s_addr + hf * 64 + 32, x + 32);
        tmem_ld_wait();
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {   // keys 32 qq .. 32 qq + 31 of the half
          uint32_t ph[16], pl[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int e = 32 * qq + 2 * k;
            const float2 arg = ffma2(make_float2(__uint_as_float(x[e]), __uint_as_float(x[e + 1])), mul22, negm2);
            const float pa = ex2(arg.x), pb = ex2(arg.y);
            ls2 = ffma2(make_float2(pa, pb), make_float2(1.f, 1.f), ls2);
            const __half2 hp = __floats2half2_rn(pa, pb);
            const float2 hf2 = __half22float2(hp);
            const __half2 lp = __floats2half2_rn(pa - hf2.x, pb - hf2.y);
            ph[k] = *reinterpret_cast<const uint32_t*>(&hp);
            pl[k] = *reinterpret_cast<const uint32_t*>(&lp);
          }
          tmem_st16(s_addr + hf * 64 + 16 * qq, ph);
          tmem_st16(s_addr + hf * 64 + 32 + 16 * qq, pl);
        }
      }
      l_run += ls2.x + ls2.y;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm.p_full[q]);
    }
    // ---- epilogue: O / l (+ sink) times the V channel scales, fp32. Each
    // thread stages its row in the group's query region (free: every S MMA of
    // the group is done once its last P.V is) in the copied layout, and one
    // thread writes the tile with four tensor stores (rows past S are skipped).
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&sm.o_done[q], (uint32_t)(ntiles - 1) & 1u, p.wait_budget) && !aborted(sm));
    if (ok) {
      tc_fence_after();
      float mf = m_run, extra = 0.f;
      if (p.has_sink || p.smooth) {
        const float sg = (p.has_sink ? reinterpret_cast<const float*>(p.sink)[h] : 0.f) * kLog2e;
        mf = fmaxf(m_run, sg);
        extra = ex2(sg - mf);
      }
      const float f = ex2(m_run - mf);
      const float den = l_run * f + extra;
      const float scale_out = (live && den > 0.f) ? f / den : 0.f;
      const bool vch = p.v_scale_n != 1;
      const float so = vch ? scale_out : scale_out * p.v_scale[0];
      const float4* vs4 = reinterpret_cast<const float4*>(p.v_scale + (vch ? g * kHD : 0));
      uint8_t* stage = sm.q[q];
#pragma unroll
      for (int c = 0; c < 4; ++c) {          // box c: dims 32 c .. 32 c + 31
        uint32_t raw[32];
        tmem_ld32(o_addr + c * 32, raw);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 v = vch ? __ldg(vs4 + (c * 32 + e) / 4) : make_float4(1.f, 1.f, 1.f, 1.f);
          float4 o;
          o.x = __uint_as_float(raw[e]) * so * v.x;
          o.y = __uint_as_float(raw[e + 1]) * so * v.y;
          o.z = __uint_as_float(raw[e + 2]) * so * v.z;
          o.w = __uint_as_float(raw[e + 3]) * so * v.w;
          *reinterpret_cast<float4*>(stage + c * kBox + sw128_offset(rl, e >> 2)) = o;
        }
      }
      fence_async_smem();   // staged rows (generic stores) -> async proxy: the tensor stores read them
    }
    const bool all_ok = group_all(ok, q);
    if (!all_ok) {
      if (lane == 0) set_abort(p, sm);
    } else if (quarter == 2 && elect_one()) {   // warp 2 (group 0) or 6 (group 1)
      for (int k = 0; k < 4; ++k) tma_store_4d(&tmo, sm.q[q] + k * kBox, 32 * k, g * p.G, (r0 + q * kBM) / p.G, b);
      bulk_commit();
      bulk_wait_read();   // the staged tile is read before the CTA may exit
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

bool prefill_tcq_supported(const Params& p) {
  return p.t_type == kF32 && (p.cache_type == kI8 || p.cache_type == kI4) && p.H == kHD && 128 % p.G == 0 &&
         !p.kv_separate && !p.window_cache;
}

cudaError_t prepare_prefill_tcq(const Params& p, TmaMaps* maps) {
  cudaError_t e;
  if ((e = encode_f32_query_sw128(&maps->m[0], p.q, p.B, p.S, p.N, (uint32_t)p.G)) != cudaSuccess) return e;
  if ((e = encode_f32_query_sw128(&maps->m[1], p.out, p.B, p.S, p.N, (uint32_t)p.G)) != cudaSuccess) return e;
  maps->m[2] = maps->m[3] = maps->m[1];
  return cudaSuccess;
}

namespace {
constexpr int kMaxDevices = 64;
bool g_smem_set[4][kMaxDevices];
}  // namespace

cudaError_t launch_prefill_tcq(const Params& p, cudaStream_t st, const TmaMaps& maps) {
  const int smem = (int)sizeof(QcSmem) + 1024;
  const bool plain = p.softcap <= 0.f && !p.has_bias;
  const bool i8 = p.cache_type == kI8;
  auto kern = i8 ? (plain ? prefill_tcq_kernel<8, true> : prefill_tcq_kernel<8, false>)
                 : (plain ? prefill_tcq_kernel<4, true> : prefill_tcq_kernel<4, false>);
  const int variant = (i8 ? 0 : 2) + (plain ? 0 : 1);
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
  const dim3 grid = prefill_prompt_qb_major(p) ? dim3(nbg, nqb) : dim3(nqb, nbg);
  kern<<<grid, kThreads, smem, st>>>(p, maps.m[0], maps.m[1]);
  return cudaGetLastError();
}

}  // namespace gqa
