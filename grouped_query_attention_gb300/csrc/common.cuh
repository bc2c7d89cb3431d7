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

__device__ __forceinline__ float channel_scale(const float* sc, int n, int c) {
  return n == 1 ? sc[0] : sc[c];
}

}  // namespace gqa
