// Split-KV decode for GroupQueryAttention on sm_103a (CUDA cores, HBM-bound).
//
// One launch per call. CTA (split s, KV head g, batch b) streams keys
// [kstart + s*L, kstart + (s+1)*L) of cache row block (b, g) once and scores
// them against all R = S*G query rows of the group (GQA: one K/V stream serves
// every grouped query head). The CTA that owns a new row position appends it
// (norm -> rotary -> cast / int8 code) before reading it back as stored.
// Each split leaves a partial (m, l, o) in the workspace; the last split of a
// (b, g) to finish, known from an atomic ticket (no waiting), merges them with
// a log-sum-exp combine and writes the output rows.
//
// com.microsoft.GroupQueryAttention, section Implementation variants:
// share_append_split_decode_splitk / past_kv_decode_splitk (append, then
// partition the key axis and merge partial online-softmax results),
// quant_int8_decode_splitk (int8 rows appended, attention over the stored
// codes); sections Inputs and Attributes for the features.
//
// Lane layout: a warp is 4 groups of 8 lanes. In the score phase each group
// owns 4 keys per iteration and lane c of a group holds 16-byte chunks
// c, c+8, ... of each key row (coalesced 128-byte segments); a transposed
// reduce-scatter over the 8 lanes leaves key (c >> 1)'s scores in lane c.
// In the P.V phase every lane owns H/32 consecutive dims of all 16 keys of the
// warp-iteration, with the probabilities broadcast through shared memory.
#include <mutex>

#include "common.cuh"

namespace gqa {

// Fixed scratch for gqa_forward_noalloc: callers that cannot allocate device
// memory get the decode kernel's status word, merge tickets and split
// partials from this array instead of a workspace. Every GPU that loads the
// library holds it until the process exits. Zero-initialised at load.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kKPG = 4;                  // keys per 8-lane group per iteration
constexpr int kKW = 4 * kKPG;            // keys per warp per iteration
constexpr float kLazyRescale = 8.0f;     // log2 growth tolerated before rescaling o, l

template <typename CacheT>
struct CacheTraits;
template <>
struct CacheTraits<__half> {
  static constexpr int es = 2;
};
template <>
struct CacheTraits<float> {
  static constexpr int es = 4;
};
template <>
struct CacheTraits<int8_t> {
  static constexpr int es = 1;
};

template <int BYTES>
struct RawVec;
template <>
struct RawVec<16> {
  using type = uint4;
};
template <>
struct RawVec<8> {
  using type = uint2;
};
template <>
struct RawVec<4> {
  using type = uint32_t;
};
template <>
struct RawVec<2> {
  using type = uint16_t;
};

// Expand the raw bytes of one chunk into fp32 values.
template <typename CacheT, int N>
__device__ __forceinline__ void expand(const void* raw, float* out) {
  if constexpr (CacheTraits<CacheT>::es == 2) {
    const __half2* h = reinterpret_cast<const __half2*>(raw);
#pragma unroll
    for (int k = 0; k < N / 2; ++k) {
      float2 f = __half22float2(h[k]);
      out[2 * k] = f.x;
      out[2 * k + 1] = f.y;
    }
  } else if constexpr (CacheTraits<CacheT>::es == 4) {
    const float* f = reinterpret_cast<const float*>(raw);
#pragma unroll
    for (int k = 0; k < N; ++k) out[k] = f[k];
  } else {
    const int8_t* q = reinterpret_cast<const int8_t*>(raw);
#pragma unroll
    for (int k = 0; k < N; ++k) out[k] = (float)q[k];
  }
}

// Append new row i of (b, g) at cache position j: one warp.
template <typename T, typename CacheT>
__device__ void append_row(const Params& p, int b, int g, int i, int j, float* buf) {
  const int lane = threadIdx.x & 31, H = p.H, half = H >> 1;
  const long long src = ((long long)(b * p.S + i) * p.Nkv + g) * H;
  const long long dst = (((long long)b * p.Nkv + g) * p.C + j) * H;
  // K: RMS norm, rotary at position j, cast or int8 code (the stored-row fp32 recipe).
  for (int d = lane; d < H; d += 32) buf[d] = load_t(p.k, src + d, p.t_type);
  __syncwarp();
  const float r = p.has_norm ? rms_inv_rn(row_sum_squares_warp(buf, H), H, p.eps) : 1.f;
  for (int d = lane; d < H; d += 32) {
    float x = buf[d];
    if (p.has_norm) x = norm_rn(x, r, load_t(p.kw, d, p.t_type));
    if (p.has_rotary) {
      const int dp = d < half ? d + half : d - half;
      float xp = buf[dp];
      if (p.has_norm) xp = norm_rn(xp, r, load_t(p.kw, dp, p.t_type));
      const int dc = d < half ? d : d - half;
      const float c = load_t(p.cos_c, (long long)j * half + dc, p.t_type);
      const float s = load_t(p.sin_c, (long long)j * half + dc, p.t_type);
      x = d < half ? rope_first_rn(x, xp, c, s) : rope_second_rn(x, xp, c, s);
    }
    if constexpr (CacheTraits<CacheT>::es == 1)
      reinterpret_cast<int8_t*>(p.present_k)[dst + d] =
          quant_i8(x, channel_scale(p.k_scale, p.k_scale_n, g * H + d));
    else if constexpr (CacheTraits<CacheT>::es == 2)
      reinterpret_cast<__half*>(p.present_k)[dst + d] = __float2half_rn(x);
    else
      reinterpret_cast<float*>(p.present_k)[dst + d] = x;
  }
  __syncwarp();
  // V: cast or int8 code.
  for (int d = lane; d < H; d += 32) {
    float x = load_t(p.v, src + d, p.t_type);
    if constexpr (CacheTraits<CacheT>::es == 1)
      reinterpret_cast<int8_t*>(p.present_v)[dst + d] =
          quant_i8(x, channel_scale(p.v_scale, p.v_scale_n, g * H + d));
    else if constexpr (CacheTraits<CacheT>::es == 2)
      reinterpret_cast<__half*>(p.present_v)[dst + d] = __float2half_rn(x);
    else
      reinterpret_cast<float*>(p.present_v)[dst + d] = x;
  }
}

template <int H, int R>
struct __align__(16) DecodeSmem {
  float q[R][H];                // prepared, pre-scaled query rows
  float praw[kWarps][H];        // per-warp row buffer (norm / rotary partner lookups)
  float p[kWarps][kKW][R];      // probabilities of the warp's current keys
  float m[kWarps][R];
  float l[kWarps][R];
  float o[kWarps][R][H];
  int last;
};

template <typename T, typename CacheT, int H, int R>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const Params p) {
  constexpr int ES = CacheTraits<CacheT>::es;
  constexpr int CB = (H * ES / 8) < 16 ? (H * ES / 8) : 16;  // bytes per chunk
  constexpr int VEC = CB / ES;                               // elements per chunk
  constexpr int NC = H / VEC;                                // chunks per row
  constexpr int CPL = NC / 8;                                // chunks per lane
  constexpr int DPV = H / 32;                                // P.V dims per lane
  static_assert(CPL >= 1 && NC % 8 == 0, "head size too small for the lane layout");
  static_assert(DPV % 2 == 0, "P.V dims per lane must be even");
  using Raw = typename RawVec<CB>::type;
  using RawV = typename RawVec<DPV * ES>::type;

  __shared__ DecodeSmem<H, R> sm;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = lane >> 3, c = lane & 7;

  const int total = p.seqlens[b] + 1;
  const int past = batch_past(p, total);
  const int rows = p.S * p.G;
  if (past < 0 || (p.has_rotary && past + p.S > p.rotary_rows)) {
    if (split == 0 && g == 0 && tid == 0)
      flag_status(p, past < 0 ? GQA_DEVICE_BAD_SEQLEN_BIT : GQA_DEVICE_BAD_ROTARY_BIT);
    return;
  }
  const int kstart = p.window >= 0 ? max(0, past - p.window) : 0;
  const int L = p.split_len;
  const int nsplit = (total - kstart + L - 1) / L;
  if (split >= nsplit) return;
  const int j0 = kstart + split * L;
  const int j1 = min(j0 + L, total);

  // ---- append the new rows this split owns (prompt padding rows go to the last split)
  for (int i = warp; i < p.S; i += kWarps) {
    const int j = past + i;
    const int owner = j < total ? (j - kstart) / L : nsplit - 1;
    if (owner == split) append_row<T, CacheT>(p, b, g, i, j, sm.praw[warp]);
  }

  // ---- prepared queries: norm -> rotary -> scale (log2 domain unless softcap)
  const float qscale = p.softcap > 0.f ? p.scale : p.scale * kLog2e;
  for (int r = warp; r < R; r += kWarps) {
    float* buf = sm.praw[warp];
    __syncwarp();
    if (r >= rows) {
      for (int d = lane; d < H; d += 32) sm.q[r][d] = 0.f;
      continue;
    }
    const int i = r / p.G, h = g * p.G + r % p.G;
    const long long src = ((long long)(b * p.S + i) * p.N + h) * H;
    for (int d = lane; d < H; d += 32) buf[d] = load_t(p.q, src + d, p.t_type);
    __syncwarp();
    const float rn = p.has_norm ? rms_inv_rn(row_sum_squares_warp(buf, H), H, p.eps) : 1.f;
    const int pos = past + i, half = H >> 1;
    for (int d = lane; d < H; d += 32) {
      float x = buf[d];
      if (p.has_norm) x = norm_rn(x, rn, load_t(p.qw, d, p.t_type));
      if (p.has_rotary) {
        const int dp = d < half ? d + half : d - half;
        float xp = buf[dp];
        if (p.has_norm) xp = norm_rn(xp, rn, load_t(p.qw, dp, p.t_type));
        const int dc = d < half ? d : d - half;
        const float cs = load_t(p.cos_c, (long long)pos * half + dc, p.t_type);
        const float sn = load_t(p.sin_c, (long long)pos * half + dc, p.t_type);
        x = d < half ? rope_first_rn(x, xp, cs, sn) : rope_second_rn(x, xp, cs, sn);
      }
      x *= qscale;
      if constexpr (ES == 1) x *= channel_scale(p.k_scale, p.k_scale_n, g * H + d);  // int8 K dequant folded in
      sm.q[r][d] = x;
    }
  }
  __syncthreads();

  // Per-row constants of this lane's score slot.
  int pos_r[R], ih_r[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int i = r < rows ? r / p.G : 0;
    pos_r[r] = past + i;
    ih_r[r] = r < rows ? i * p.N + g * p.G + r % p.G : -1;  // i*N + h
  }

  const CacheT* kbase = reinterpret_cast<const CacheT*>(p.present_k) + ((long long)b * p.Nkv + g) * p.C * H;
  const CacheT* vbase = reinterpret_cast<const CacheT*>(p.present_v) + ((long long)b * p.Nkv + g) * p.C * H;

  float m_run[R], l_part[R];
  float2 o2[R][DPV / 2];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m_run[r] = kNegBig;
    l_part[r] = 0.f;
#pragma unroll
    for (int e = 0; e < DPV / 2; ++e) o2[r][e] = make_float2(0.f, 0.f);
  }

  float vsc[DPV];  // int8 V channel scales of this lane's P.V dims, applied once at the end
  if constexpr (ES == 1) {
#pragma unroll
    for (int e = 0; e < DPV; ++e) vsc[e] = channel_scale(p.v_scale, p.v_scale_n, g * H + lane * DPV + e);
  }

  for (int base = j0 + warp * kKW; base < j1; base += kWarps * kKW) {
    // ---- scores: K chunks of this lane's 4 keys
    Raw kr[kKPG][CPL];
#pragma unroll
    for (int t = 0; t < kKPG; ++t) {
      const int j = base + grp * kKPG + t;
#pragma unroll
      for (int s = 0; s < CPL; ++s) {
        if (j < j1)
          kr[t][s] = *reinterpret_cast<const Raw*>(kbase + (long long)j * H + (c + 8 * s) * VEC);
        else
          kr[t][s] = Raw{};
      }
    }
    // V loads of the P.V phase are issued early to overlap the score math.
    RawV vr[kKW];
#pragma unroll
    for (int t = 0; t < kKW; ++t) {
      const int j = base + t;
      if (j < j1)
        vr[t] = *reinterpret_cast<const RawV*>(vbase + (long long)j * H + lane * DPV);
      else
        vr[t] = RawV{};
    }

    float2 acc2[kKPG][R];
#pragma unroll
    for (int t = 0; t < kKPG; ++t)
#pragma unroll
      for (int r = 0; r < R; ++r) acc2[t][r] = make_float2(0.f, 0.f);
#pragma unroll
    for (int s = 0; s < CPL; ++s) {
      float kv[kKPG][VEC];
#pragma unroll
      for (int t = 0; t < kKPG; ++t) expand<CacheT, VEC>(&kr[t][s], kv[t]);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float* qrow = &sm.q[r][(c + 8 * s) * VEC];
#pragma unroll
        for (int e = 0; e < VEC; e += 4) {
          const float4 q4 = *reinterpret_cast<const float4*>(qrow + e);
#pragma unroll
          for (int t = 0; t < kKPG; ++t) {
            acc2[t][r] = ffma2(make_float2(q4.x, q4.y), make_float2(kv[t][e], kv[t][e + 1]), acc2[t][r]);
            acc2[t][r] = ffma2(make_float2(q4.z, q4.w), make_float2(kv[t][e + 2], kv[t][e + 3]), acc2[t][r]);
          }
        }
      }
    }
    float acc[kKPG][R];
#pragma unroll
    for (int t = 0; t < kKPG; ++t)
#pragma unroll
      for (int r = 0; r < R; ++r) acc[t][r] = acc2[t][r].x + acc2[t][r].y;
    // ---- reduce-scatter over the 8 lanes: lane c ends with key (c >> 1)
    float sc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const bool hi4 = c & 4;
      float s0 = hi4 ? acc[0][r] : acc[2][r];
      float s1 = hi4 ? acc[1][r] : acc[3][r];
      float k0 = hi4 ? acc[2][r] : acc[0][r];
      float k1 = hi4 ? acc[3][r] : acc[1][r];
      k0 += __shfl_xor_sync(0xffffffffu, s0, 4);
      k1 += __shfl_xor_sync(0xffffffffu, s1, 4);
      const bool hi2 = c & 2;
      float snd = hi2 ? k0 : k1;
      float kp = hi2 ? k1 : k0;
      kp += __shfl_xor_sync(0xffffffffu, snd, 2);
      kp += __shfl_xor_sync(0xffffffffu, kp, 1);
      sc[r] = kp;
    }
    // ---- masks, softcap, bias; running max
    const int jk = base + grp * kKPG + (c >> 1);
    float mt[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float s = sc[r];
      bool vis = jk < j1 && ih_r[r] >= 0;
      if (p.causal) vis = vis && jk <= pos_r[r];
      if (p.window >= 0) vis = vis && jk >= pos_r[r] - p.window;
      if (p.softcap > 0.f) s = p.softcap * tanhf(s / p.softcap) * kLog2e;
      if (p.has_bias && vis) {
        const int i = ih_r[r] / p.N, h = ih_r[r] % p.N;
        const long long bi = (((long long)(p.bias_bdim > 1 ? b : 0) * p.bias_ndim + (p.bias_ndim > 1 ? h : 0)) *
                                  p.S + i) * p.bias_ld + jk;
        s += load_t(p.bias, bi, p.t_type) * kLog2e;
      }
      s = vis ? s : kNegBig;
      sc[r] = s;
      float m = s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      mt[r] = m;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (mt[r] > m_run[r] + kLazyRescale) {   // warp-uniform
        const float f = ex2(m_run[r] - mt[r]);
        l_part[r] *= f;
#pragma unroll
        for (int e = 0; e < DPV / 2; ++e) {
          o2[r][e].x *= f;
          o2[r][e].y *= f;
        }
        m_run[r] = mt[r];
      }
      const float pr = sc[r] <= kNegBig ? 0.f : ex2(sc[r] - m_run[r]);
      if ((c & 1) == 0) {
        l_part[r] += pr;
        sm.p[warp][grp * kKPG + (c >> 1)][r] = pr;
      }
    }
    __syncwarp();
    // ---- P.V over the warp's 16 keys; this lane owns dims lane*DPV .. +DPV-1
#pragma unroll
    for (int t = 0; t < kKW; ++t) {
      float vv[DPV];
      expand<CacheT, DPV>(&vr[t], vv);
      float pr[R];
#pragma unroll
      for (int r = 0; r < R; ++r) pr[r] = sm.p[warp][t][r];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int e = 0; e < DPV / 2; ++e)
          o2[r][e] = ffma2(make_float2(pr[r], pr[r]), make_float2(vv[2 * e], vv[2 * e + 1]), o2[r][e]);
    }
    __syncwarp();
  }

  // ---- combine the 4 warps of this split
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float l = l_part[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) {
      sm.m[warp][r] = m_run[r];
      sm.l[warp][r] = l;
    }
#pragma unroll
    for (int e = 0; e < DPV / 2; ++e) {
      float ox = o2[r][e].x, oy = o2[r][e].y;
      if constexpr (ES == 1) {
        ox *= vsc[2 * e];
        oy *= vsc[2 * e + 1];
      }
      sm.o[warp][r][lane * DPV + 2 * e] = ox;
      sm.o[warp][r][lane * DPV + 2 * e + 1] = oy;
    }
  }
  __syncthreads();

  const int bg = b * p.Nkv + g;
  auto finalize = [&](int r, float m, float l, float o, int d) {
    const int i = r / p.G, h = g * p.G + r % p.G;
    const long long oi = ((long long)(b * p.S + i) * p.N + h) * H + d;
    float val;
    if (p.mode == kPrompt && i >= total) {
      val = 0.f;
    } else {
      float mf = m, extra = 0.f;
      if (p.has_sink || p.smooth) {
        const float sg = (p.has_sink ? load_t(p.sink, h, p.t_type) : 0.f) * kLog2e;
        mf = fmaxf(m, sg);
        extra = ex2(sg - mf);
      }
      const float f = ex2(m - mf);
      const float den = l * f + extra;
      val = den > 0.f ? o * f / den : 0.f;
    }
    if (p.t_type == kF16) reinterpret_cast<__half*>(p.out)[oi] = __float2half_rn(val);
    else reinterpret_cast<float*>(p.out)[oi] = val;
  };

  if (nsplit == 1) {
    for (int x = tid; x < rows * H; x += kThreads) {
      const int r = x / H, d = x % H;
      float M = kNegBig;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.m[w][r]);
      float l = 0.f, o = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = ex2(sm.m[w][r] - M);
        l += sm.l[w][r] * f;
        o += sm.o[w][r][d] * f;
      }
      finalize(r, M, l, o, d);
    }
    return;
  }

  // Partial of this split.
  const long long pbase = ((long long)bg * p.max_splits + split) * p.rows_pad;
  for (int x = tid; x < rows * H; x += kThreads) {
    const int r = x / H, d = x % H;
    float M = kNegBig;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.m[w][r]);
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) o += sm.o[w][r][d] * ex2(sm.m[w][r] - M);
    p.part_o[(pbase + r) * H + d] = o;
    if (d == 0) {
      float l = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) l += sm.l[w][r] * ex2(sm.m[w][r] - M);
      p.part_ml[(pbase + r) * 2] = M;
      p.part_ml[(pbase + r) * 2 + 1] = l;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned ticket = atomicAdd(&p.counters[bg], 1u);
    sm.last = ticket == (unsigned)(nsplit - 1);
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();

  // Last split of (b, g): log-sum-exp merge of all partials.
  const long long b0 = (long long)bg * p.max_splits * p.rows_pad;
  for (int x = tid; x < rows * H; x += kThreads) {
    const int r = x / H, d = x % H;
    float M = kNegBig;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, __ldcg(&p.part_ml[(b0 + (long long)s * p.rows_pad + r) * 2]));
    float l = 0.f, o = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const long long idx = b0 + (long long)s * p.rows_pad + r;
      const float f = ex2(__ldcg(&p.part_ml[idx * 2]) - M);
      l += __ldcg(&p.part_ml[idx * 2 + 1]) * f;
      o += __ldcg(&p.part_o[idx * H + d]) * f;
    }
    finalize(r, M, l, o, d);
  }
  if (tid == 0) p.counters[bg] = 0;  // ready for the next call
}

template <typename T, typename CacheT, int H>
cudaError_t launch_h(const Params& p, cudaStream_t st) {
  dim3 grid(p.max_splits, p.Nkv, p.B), block(kThreads);
  switch (p.rows_pad) {
    case 1: decode_kernel<T, CacheT, H, 1><<<grid, block, 0, st>>>(p); break;
    case 2: decode_kernel<T, CacheT, H, 2><<<grid, block, 0, st>>>(p); break;
    case 4: decode_kernel<T, CacheT, H, 4><<<grid, block, 0, st>>>(p); break;
    case 8: decode_kernel<T, CacheT, H, 8><<<grid, block, 0, st>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <typename T, typename CacheT>
cudaError_t launch_t(const Params& p, cudaStream_t st) {
  if (p.H == 128) return launch_h<T, CacheT, 128>(p, st);
  if (p.H == 64) return launch_h<T, CacheT, 64>(p, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t noalloc_scratch(void** ptr) {
  // Device address of g_noalloc_scratch for the current device, looked up
  // once per device (host code may not use the array's name as an address).
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = a;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

bool decode_supported(const Params& p) {
  return (p.H == 128 || p.H == 64) && p.S * p.G <= 8;
}

cudaError_t launch_decode(const Params& p, cudaStream_t st) {
  if (p.t_type == kF16) return launch_t<__half, __half>(p, st);
  if (p.cache_type == kI8) return launch_t<float, int8_t>(p, st);
  return launch_t<float, float>(p, st);
}

}  // namespace gqa
