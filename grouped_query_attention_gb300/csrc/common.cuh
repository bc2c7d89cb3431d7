// Device helpers shared by the GQA kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

#include "gqa_internal.h"

namespace gqa {

#define GQA_DEVICE_BAD_SEQLEN_BIT 1u
#define GQA_DEVICE_BAD_ROTARY_BIT 2u
#define GQA_DEVICE_TIMEOUT_BIT 4u

constexpr float kLog2e = 1.4426950408889634f;
// Finite stand-in for -inf in running maxima: exp2 of (kNegBig - finite) is 0
// and kNegBig - kNegBig is 0, so no NaN appears when a row sees no key.
constexpr float kNegBig = -1.0e30f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void flag_status(const Params& p, unsigned int bit) {
  atomicOr(p.status, bit);
}

// fp32 view of one element of a T tensor.
__device__ __forceinline__ float load_t(const void* base, long long idx, int t_type) {
  if (t_type == kF16) return __half2float(reinterpret_cast<const __half*>(base)[idx]);
  return reinterpret_cast<const float*>(base)[idx];
}

// Packed fp32x2 fused multiply-add (Blackwell FFMA2): d = a * b + c per lane pair.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long av = *reinterpret_cast<unsigned long long*>(&a);
  unsigned long long bv = *reinterpret_cast<unsigned long long*>(&b);
  unsigned long long cv = *reinterpret_cast<unsigned long long*>(&c);
  unsigned long long dv;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(dv) : "l"(av), "l"(bv), "l"(cv));
  return *reinterpret_cast<float2*>(&dv);
}

// Maximum of three values (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Rotary table row element (T) as fp32.
__device__ __forceinline__ float rot_t(const void* base, long long idx, int t_type) {
  return load_t(base, idx, t_type);
}

// Symmetric int8 code of an fp32 value: clamp(rint(x / s), -127, 127) with the
// division correctly rounded (IEEE), ties to even.
__device__ __forceinline__ int8_t quant_i8(float x, float s) {
  float t = __fdiv_rn(x, s);
  t = rintf(t);
  t = fminf(fmaxf(t, -127.0f), 127.0f);
  return static_cast<int8_t>(static_cast<int>(t));
}

// 4-bit cache code as its stored nibble: clamp(rint(x / s), -7, 7) + 8, the
// division in IEEE fp32 (com.microsoft.GroupQueryAttention, section Inputs:
// +8-biased nibbles; section Attributes: kv_cache_bit_width).
__device__ __forceinline__ unsigned quant_i4_nibble(float x, float s) {
  float t = __fdiv_rn(x, s);
  t = rintf(t);
  t = fminf(fmaxf(t, -7.0f), 7.0f);
  return static_cast<unsigned>(static_cast<int>(t) + 8);
}

// ---- fp32 recipe of the rows stored in the cache (RMS norm, then NeoX rotary)
// Every operation is one IEEE fp32 rounding and none is fused, so the stored
// bytes do not depend on which kernel (or lane layout) appends a row: the
// squares of four consecutive coordinates are summed left to right, the H/4
// group sums are added as a pairwise tree (neighbours first; a lane butterfly
// with rising xor distance over lanes that hold consecutive groups computes
// exactly that tree, zero groups padding it to a power of two),
// r = 1 / sqrt(ss / H + eps), y = (x r) w, and rotary
// y[d] = x[d] c - x[d+H/2] s, y[d+H/2] = x[d+H/2] c + x[d] s with each product
// rounded before the add (com.microsoft.GroupQueryAttention, section Inputs:
// q/k_norm_weight, cos/sin_cache; section Attributes: qk_norm_epsilon).
__device__ __forceinline__ float sumsq4_rn(float a, float b, float c, float d) {
  float s = __fmul_rn(a, a);
  s = __fadd_rn(s, __fmul_rn(b, b));
  s = __fadd_rn(s, __fmul_rn(c, c));
  return __fadd_rn(s, __fmul_rn(d, d));
}

// Sum of squares of eight consecutive coordinates (two groups, one tree node).
__device__ __forceinline__ float sumsq8_rn(const float* x) {
  return __fadd_rn(sumsq4_rn(x[0], x[1], x[2], x[3]), sumsq4_rn(x[4], x[5], x[6], x[7]));
}

// 1 / sqrt(ss / H + eps), each step one IEEE rounding. For a power-of-two H
// the division is the (exact) product with 1/H, and 1 / x rounded to nearest
// is the correctly rounded reciprocal: the same values with fewer instructions.
__device__ __forceinline__ float rms_inv_rn(float ss, int H, float eps) {
  const float ms = (H & (H - 1)) == 0 ? __fmul_rn(ss, 1.0f / (float)H) : __fdiv_rn(ss, (float)H);
  return __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
}

__device__ __forceinline__ float norm_rn(float x, float r, float w) { return __fmul_rn(__fmul_rn(x, r), w); }

// Rotary of coordinate d < H/2 (x = x[d], partner = x[d+H/2]) and of
// coordinate d + H/2 (x = x[d+H/2], partner = x[d]).
__device__ __forceinline__ float rope_first_rn(float x, float partner, float c, float s) {
  return __fsub_rn(__fmul_rn(x, c), __fmul_rn(partner, s));
}
__device__ __forceinline__ float rope_second_rn(float x, float partner, float c, float s) {
  return __fadd_rn(__fmul_rn(x, c), __fmul_rn(partner, s));
}

// Sum of squares of a row of H <= 256 fp32 values in shared memory, by one
// whole warp: lane l holds groups l and l + 32.
__device__ __forceinline__ float row_sum_squares_warp(const float* row, int H) {
  const int lane = threadIdx.x & 31;
  float part[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int d = 4 * (j * 32 + lane);
    part[j] = d < H ? sumsq4_rn(row[d], row[d + 1], row[d + 2], row[d + 3]) : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) part[j] = __fadd_rn(part[j], __shfl_xor_sync(0xffffffffu, part[j], o));
  }
  return __fadd_rn(part[0], part[1]);
}

// RMS norm (weights wlo / whi, when `norm`) and then rotary (cos c / sin s,
// when c is not null) of one 128-value row spread over 8 lanes: lane l8 of the
// row holds dims 8 l8 .. 8 l8 + 7 (lo) and 64 + 8 l8 .. (hi), so the NeoX
// partner of every value is in the same lane. The 8 lanes are consecutive
// lanes of the warp and every lane of the warp calls (shuffles). Same fp32
// recipe as the stored rows (groups of four, pairwise tree).
__device__ __forceinline__ void norm_rope_row8(float* lo, float* hi, const float* wlo, const float* whi, bool norm,
                                               const float* c, const float* s, float eps) {
  if (norm) {
    float slo = sumsq8_rn(lo), shi = sumsq8_rn(hi);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      slo = __fadd_rn(slo, __shfl_xor_sync(0xffffffffu, slo, o));
      shi = __fadd_rn(shi, __shfl_xor_sync(0xffffffffu, shi, o));
    }
    const float rn = rms_inv_rn(__fadd_rn(slo, shi), 128, eps);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      lo[k] = norm_rn(lo[k], rn, wlo[k]);
      hi[k] = norm_rn(hi[k], rn, whi[k]);
    }
  }
  if (c) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float a = lo[k], b = hi[k];
      lo[k] = rope_first_rn(a, b, c[k], s[k]);
      hi[k] = rope_second_rn(b, a, c[k], s[k]);
    }
  }
}

__device__ __forceinline__ float channel_scale(const float* sc, int n, int c) {
  return n == 1 ? sc[0] : sc[c];
}

}  // namespace gqa
