// CUDA-core flash prefill for GroupQueryAttention: float32 Q/K/V (including
// an int8 or 4-bit cache read back through its scales), head sizes the
// tensor-core kernel does not take, sliding-window caches. Reads the
// prepared queries the pre-pass left in the workspace and the present cache
// after the append (or the query-dtype rows of a prompt whose cache has the
// other float dtype).
//
// com.microsoft.GroupQueryAttention, section Implementation variants
// (qkv_present_flash_cluster / past_kv_flash_prefill / new_kv_past_flash_prefill
// / quant_int8_flash_prefill / quant_int4_flash_prefill / window_shift_flash_prefill:
// online-softmax prefill over the cache as stored, causal bound right-aligned
// at the live length, window floor, softcap, bias and head sink) and sections
// Inputs / Attributes.
//
// CTA = 32 consecutive rows of the (position, grouped head) row list of one
// KV head (b, g), so every K/V tile staged in shared memory serves all G
// query heads; 128 threads, register-blocked so that the fp32 FMA pipe, not
// shared memory, sets the pace:
//   scores  thread (rg, kg) = (tid / 16, tid % 16) computes the 4 x 4 block of
//           rows 4rg.. and keys 4kg.. of a 64-key tile: per head coordinate one
//           16-byte load of Q^T, one of K^T, 16 FMAs;
//   softmax the 16 threads of a row group hold a row's 64 scores; max and sum
//           by shuffles within the half warp; P goes to shared memory (P^T);
//   P.V     the same thread owns rows 4rg.. x dims {64c + 4kg .. +3}: per key one
//           16-byte load of P^T and HMAX/64 of V, 16 FMAs each.
#include "common.cuh"

namespace gqa {
namespace {

constexpr int kThreads = 128;
constexpr int kR = 32;          // rows per CTA
constexpr int kK = 64;          // keys per tile
constexpr int kKP = kK + 4;     // padded K^T row (keeps 16-byte alignment)
constexpr int kMaxH = 256;

// Launch order: prompt calls (no past: a block's key range depends only on
// its row block) run row-block-major over all KV heads, so the longest blocks
// of every head start first; otherwise one grid row per KV head, its longest
// blocks first. (Row blocks in rising order, shortest first, took 427-431
// against 342 us on a causal fp32 B=2, S=1024, 16-head prompt.)
__host__ __device__ inline bool simt_rb_major(const Params& p) {
  return p.mode == kPrompt && (p.S * p.G + kR - 1) / kR <= 65535;
}

template <int HMAX>
constexpr size_t smem_floats() {
  return (size_t)HMAX * kR + (size_t)HMAX * kKP + (size_t)kK * HMAX + (size_t)kR * kKP;
}

// Four consecutive head coordinates d .. d+3 of one cache row as fp32
// (int8 / 4-bit codes times their channel scales).
template <typename CacheT>
__device__ __forceinline__ float4 load4(const CacheT* row, int d, const float* sc, int nsc, int ch0) {
  float4 v;
  if constexpr (std::is_same<CacheT, float>::value) {
    v = *reinterpret_cast<const float4*>(row + d);
  } else if constexpr (std::is_same<CacheT, __half>::value) {
    const uint2 u = *reinterpret_cast<const uint2*>(row + d);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    v = make_float4(a.x, a.y, c.x, c.y);
  } else if constexpr (std::is_same<CacheT, int8_t>::value) {
    const char4 q = *reinterpret_cast<const char4*>(row + d);
    v = make_float4((float)q.x * channel_scale(sc, nsc, ch0), (float)q.y * channel_scale(sc, nsc, ch0 + 1),
                    (float)q.z * channel_scale(sc, nsc, ch0 + 2), (float)q.w * channel_scale(sc, nsc, ch0 + 3));
  } else {   // uint8_t: 4-bit cache, d/2 .. d/2+1 bytes, +8-biased nibbles, even coordinate low
    const unsigned short u = *reinterpret_cast<const unsigned short*>(reinterpret_cast<const uint8_t*>(row) + d / 2);
    v = make_float4((float)((int)(u & 15) - 8) * channel_scale(sc, nsc, ch0),
                    (float)((int)((u >> 4) & 15) - 8) * channel_scale(sc, nsc, ch0 + 1),
                    (float)((int)((u >> 8) & 15) - 8) * channel_scale(sc, nsc, ch0 + 2),
                    (float)((int)(u >> 12) - 8) * channel_scale(sc, nsc, ch0 + 3));
  }
  return v;
}

// Two CTAs per SM (register budget 255 per thread; shared memory 91 KB per CTA
// at HMAX = 128).
template <typename T, typename CacheT, int HMAX>
__global__ void __launch_bounds__(kThreads, 2)
prefill_simt_kernel(const Params p) {
  constexpr int NC = HMAX / 64;            // 4-dim chunks per thread in P.V: dims 64c + 4kg .. +3
  extern __shared__ __align__(16) float smem[];
  float* qT = smem;                        // [HMAX][kR]   prepared queries, transposed
  float* kT = qT + HMAX * kR;              // [HMAX][kKP]  key tile, transposed
  float* vs = kT + HMAX * kKP;             // [kK][HMAX]   value tile
  float* ps = vs + kK * HMAX;              // [kR][kKP]    probabilities

  const int H = p.H;
  const int tid = threadIdx.x, rg = tid >> 4, kg = tid & 15;
  // Row blocks from the last (longest key ranges first), in the order of
  // simt_rb_major.
  const int nrb = (p.S * p.G + kR - 1) / kR;
  const bool rbm = simt_rb_major(p);
  const int rb = nrb - 1 - (int)(rbm ? blockIdx.y : blockIdx.x);
  const int g = rbm ? (int)(blockIdx.x % p.Nkv) : (int)blockIdx.y;
  const int b = rbm ? (int)(blockIdx.x / p.Nkv) : (int)blockIdx.z;
  const int total = p.seqlens[b] + 1;
  const int past = batch_past(p, total);
  if (past < 0) {
    if (rb == 0 && g == 0 && tid == 0) flag_status(p, GQA_DEVICE_BAD_SEQLEN_BIT);
    return;
  }
  if (p.has_rotary && past + p.S > p.rotary_rows) return;  // flagged by the pre-pass
  const int nrows = p.S * p.G;
  const int r0 = rb * kR;
  const int live_i = p.mode == kPrompt ? min(p.S, total) : p.S;  // rows i >= live_i are padding

  // Prepared query rows (fp32, layout [B][N_kv][S*G][H]) into Q^T.
  const float* qp = reinterpret_cast<const float*>(p.qprep) + ((long long)(b * p.Nkv + g) * nrows) * H;
  for (int x = tid; x < kR * H; x += kThreads) {
    const int r = x % kR, d = x / kR;
    qT[d * kR + r] = r0 + r < nrows ? qp[(long long)(r0 + r) * H + d] : 0.f;
  }
  // Key range of the block in cache rows: [kmin, kmax). Cache row j holds
  // absolute position off + j (off = 0 except for a sliding-window cache).
  const BatchRows br = batch_rows(p, total, past);
  const int off = br.off, past_row = past - off;
  const int i_lo = r0 / p.G;
  const int i_hi = min((min(r0 + kR, nrows) - 1) / p.G, live_i - 1);
  int kmin = 0, kmax = br.live;
  if (p.causal) kmax = min(br.live, past_row + i_hi + 1);
  if (p.window >= 0) kmin = max(0, past_row + i_lo - p.window);

  // This thread's rows 4rg .. 4rg+3.
  int pos_r[4], head_r[4], i_r[4];
  bool live_r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + 4 * rg + i;
    const bool ok = r < nrows;
    i_r[i] = ok ? r / p.G : 0;
    head_r[i] = g * p.G + (ok ? r % p.G : 0);
    live_r[i] = ok && i_r[i] < live_i;
    pos_r[i] = past_row + i_r[i];          // position in cache rows
  }
  const float qscale = p.softcap > 0.f ? p.scale : p.scale * kLog2e;
  float m[4], l[4];
  float2 o2[4][NC][2];   // rows x chunks x dim pairs
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = kNegBig;
    l[i] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) o2[i][c][0] = o2[i][c][1] = make_float2(0.f, 0.f);
  }

  // Attention reads the present cache, or the new rows in T when a prompt's
  // cache has another float dtype (kv_separate: [B][N_kv][S][H], S rows).
  // CacheT = uint8_t: 4-bit cache, H/2 bytes per row.
  constexpr bool i4 = std::is_same<CacheT, uint8_t>::value;
  const long long row_elems = i4 ? H / 2 : H;
  const void* ksrc = p.kv_separate ? p.kv_sep_k : p.present_k;
  const void* vsrc = p.kv_separate ? p.kv_sep_v : p.present_v;
  const long long rows = p.kv_separate ? p.S : p.C;
  const CacheT* kb = reinterpret_cast<const CacheT*>(ksrc) + ((long long)b * p.Nkv + g) * rows * row_elems;
  const CacheT* vb = reinterpret_cast<const CacheT*>(vsrc) + ((long long)b * p.Nkv + g) * rows * row_elems;
  const int H4 = H / 4;

  for (int t0 = kmin; t0 < kmax; t0 += kK) {
    __syncthreads();   // the previous tile's reads of kT / vs / ps are done
    // K tile transposed (consecutive threads take consecutive keys: conflict-free
    // stores), V tile as rows (consecutive threads take consecutive dims). Keys
    // past kmax are zero.
    for (int x = tid; x < kK * H4; x += kThreads) {
      const int j = x % kK, d = (x / kK) * 4;
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t0 + j < kmax) kv = load4<CacheT>(kb + (long long)(t0 + j) * row_elems, d, p.k_scale, p.k_scale_n, g * H + d);
      kT[(d + 0) * kKP + j] = kv.x;
      kT[(d + 1) * kKP + j] = kv.y;
      kT[(d + 2) * kKP + j] = kv.z;
      kT[(d + 3) * kKP + j] = kv.w;
    }
    for (int x = tid; x < kK * H4; x += kThreads) {
      const int j = x / H4, d = (x - j * H4) * 4;
      float4 vv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t0 + j < kmax) vv = load4<CacheT>(vb + (long long)(t0 + j) * row_elems, d, p.v_scale, p.v_scale_n, g * H + d);
      *reinterpret_cast<float4*>(&vs[j * HMAX + d]) = vv;
    }
    __syncthreads();

    // Scores of rows 4rg.. x keys 4kg.. : one 16-byte load of Q^T and of K^T per
    // coordinate, 16 FMAs as 8 packed fp32x2 ones (key pairs).
    float2 s2[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) s2[i][0] = s2[i][1] = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int d = 0; d < H; ++d) {
      const float4 qv = *reinterpret_cast<const float4*>(&qT[d * kR + 4 * rg]);
      const float4 kv = *reinterpret_cast<const float4*>(&kT[d * kKP + 4 * kg]);
      const float qa[4] = {qv.x, qv.y, qv.z, qv.w};
      const float2 k01 = make_float2(kv.x, kv.y), k23 = make_float2(kv.z, kv.w);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 qq = make_float2(qa[i], qa[i]);
        s2[i][0] = ffma2(qq, k01, s2[i][0]);
        s2[i][1] = ffma2(qq, k23, s2[i][1]);
      }
    }
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s[i][0] = s2[i][0].x;
      s[i][1] = s2[i][0].y;
      s[i][2] = s2[i][1].x;
      s[i][3] = s2[i][1].y;
    }
    // Scale, softcap, bias (log2 domain), masks: causal / window in cache rows,
    // bias columns at absolute positions.
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int jj = t0 + 4 * kg + j;
        bool vis = live_r[i] && jj < kmax;
        if (p.causal) vis = vis && jj <= pos_r[i];
        if (p.window >= 0) vis = vis && jj >= pos_r[i] - p.window;
        float x = s[i][j] * qscale;
        if (p.softcap > 0.f) x = p.softcap * tanhf(x / p.softcap) * kLog2e;
        if (p.has_bias && vis) {
          const long long bi = (((long long)(p.bias_bdim > 1 ? b : 0) * p.bias_ndim + (p.bias_ndim > 1 ? head_r[i] : 0)) *
                                    p.S + i_r[i]) * p.bias_ld + jj + off;
          x += load_t(p.bias, bi, p.t_type) * kLog2e;
        }
        s[i][j] = vis ? x : -INFINITY;
      }
    }
    // Online softmax: a row's 64 scores live in the 16 threads of its half warp.
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float mt = fmaxf(fmaxf(s[i][0], s[i][1]), fmaxf(s[i][2], s[i][3]));
#pragma unroll
      for (int o16 = 8; o16 > 0; o16 >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o16, 16));
      const float mn = fmaxf(m[i], mt);
      const float f = ex2(m[i] - mn);
      m[i] = mn;
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        s[i][j] = ex2(s[i][j] - mn);   // masked (-inf) scores give 0
        sum += s[i][j];
      }
#pragma unroll
      for (int o16 = 8; o16 > 0; o16 >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o16, 16);
      l[i] = l[i] * f + sum;
      const float2 f2 = make_float2(f, f), z2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        o2[i][c][0] = ffma2(o2[i][c][0], f2, z2);
        o2[i][c][1] = ffma2(o2[i][c][1], f2, z2);
      }
      *reinterpret_cast<float4*>(&ps[(4 * rg + i) * kKP + 4 * kg]) = make_float4(s[i][0], s[i][1], s[i][2], s[i][3]);
    }
    __syncthreads();

    // P.V over the 64 keys, four at a time: one 16-byte load of P per row and
    // NC of V per key.
#pragma unroll 2
    for (int j4 = 0; j4 < kK; j4 += 4) {
      float pr[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 pv = *reinterpret_cast<const float4*>(&ps[(4 * rg + i) * kKP + j4]);
        pr[i][0] = pv.x;
        pr[i][1] = pv.y;
        pr[i][2] = pv.z;
        pr[i][3] = pv.w;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float4 vv = *reinterpret_cast<const float4*>(&vs[(j4 + k) * HMAX + 64 * c + 4 * kg]);
          const float2 v01 = make_float2(vv.x, vv.y), v23 = make_float2(vv.z, vv.w);
#pragma unroll
          for (int i = 0; i < 4; ++i) {   // packed fp32x2 FMAs over dim pairs
            const float2 pp = make_float2(pr[i][k], pr[i][k]);
            o2[i][c][0] = ffma2(pp, v01, o2[i][c][0]);
            o2[i][c][1] = ffma2(pp, v23, o2[i][c][1]);
          }
        }
      }
    }
  }

  // Epilogue: out = o / (l + sink term), cast to T; padding rows get 0.
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + 4 * rg + i;
    if (r >= nrows) continue;
    const int h = head_r[i];
    float mf = m[i], extra = 0.f;
    if (p.has_sink || p.smooth) {
      const float sg = (p.has_sink ? load_t(p.sink, h, p.t_type) : 0.f) * kLog2e;
      mf = fmaxf(m[i], sg);
      extra = ex2(sg - mf);
    }
    const float f = ex2(m[i] - mf);
    const float den = l[i] * f + extra;
    const float sc = (!live_r[i] || den <= 0.f) ? 0.f : f / den;
    const long long ob = ((long long)(b * p.S + i_r[i]) * p.N + h) * H;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int d = 64 * c + 4 * kg;
      if (d >= H) continue;
      const float4 v = make_float4(o2[i][c][0].x * sc, o2[i][c][0].y * sc, o2[i][c][1].x * sc, o2[i][c][1].y * sc);
      if constexpr (sizeof(T) == 2) {
        uint2 u;
        *reinterpret_cast<__half2*>(&u.x) = __floats2half2_rn(v.x, v.y);
        *reinterpret_cast<__half2*>(&u.y) = __floats2half2_rn(v.z, v.w);
        *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(p.out) + ob + d) = u;
      } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + ob + d) = v;
      }
    }
  }
}

// Dynamic shared memory opt-in, set once per device and kernel variant.
constexpr int kMaxDevices = 64;

template <typename T, typename CacheT, int HMAX>
cudaError_t launch_h(const Params& p, cudaStream_t st) {
  static bool set[kMaxDevices];
  const size_t smem = smem_floats<HMAX>() * sizeof(float);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!set[dev]) {
    e = cudaFuncSetAttribute(prefill_simt_kernel<T, CacheT, HMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    set[dev] = true;
  }
  const unsigned nrb = (unsigned)((p.S * p.G + kR - 1) / kR);
  const dim3 grid = simt_rb_major(p) ? dim3((unsigned)(p.B * p.Nkv), nrb) : dim3(nrb, p.Nkv, p.B), block(kThreads);
  prefill_simt_kernel<T, CacheT, HMAX><<<grid, block, smem, st>>>(p);
  return cudaGetLastError();
}

template <typename T, typename CacheT>
cudaError_t launch_t(const Params& p, cudaStream_t st) {
  if (p.H <= 64) return launch_h<T, CacheT, 64>(p, st);
  if (p.H <= 128) return launch_h<T, CacheT, 128>(p, st);
  return launch_h<T, CacheT, 256>(p, st);
}

}  // namespace

bool prefill_simt_supported(const Params& p) { return p.H <= kMaxH && p.H % 16 == 0 && p.H >= 16; }

cudaError_t launch_prefill_simt(const Params& p, cudaStream_t st) {
  // With kv_separate the rows attention reads have the query dtype.
  const int src = p.kv_separate ? p.t_type : p.cache_type;
  if (p.t_type == kF16) return launch_t<__half, __half>(p, st);
  if (src == kI8) return launch_t<float, int8_t>(p, st);
  if (src == kI4) return launch_t<float, uint8_t>(p, st);
  return launch_t<float, float>(p, st);
}

}  // namespace gqa
