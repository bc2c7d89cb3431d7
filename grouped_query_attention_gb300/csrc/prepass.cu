// Pre-pass of the prefill path: appends the new K/V rows to the present cache
// (RMS norm -> NeoX rotary -> cast, int8 code or packed 4-bit code for K;
// the same store for V) and
// writes the prepared queries (norm -> rotary) to the workspace for the
// attention kernel. One warp per row, 16-byte vector loads and stores.
//
// com.microsoft.GroupQueryAttention: section Inputs (q/k_norm_weight applied
// before rotary; cos/sin_cache; k/v_scale), section Attributes
// (qk_norm_epsilon, do_rotary, k/v_quant_type) and section Implementation
// variants (new rows are appended at the live length before attention reads
// the cache; copy mode keeps the live past rows).
#include "common.cuh"

namespace gqa {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kMaxH = 256;

template <typename T>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int n = 4;
};
template <>
struct Vec<__half> {
  static constexpr int n = 8;
};

template <typename T>
__device__ __forceinline__ void load_vec(const T* src, float* dst);
template <>
__device__ __forceinline__ void load_vec<float>(const float* src, float* dst) {
  float4 v = *reinterpret_cast<const float4*>(src);
  dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
}
template <>
__device__ __forceinline__ void load_vec<__half>(const __half* src, float* dst) {
  uint4 u = *reinterpret_cast<const uint4*>(src);
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 f = __half22float2(h[k]);
    dst[2 * k] = f.x;
    dst[2 * k + 1] = f.y;
  }
}

// Store V consecutive fp32 values as DstT (round to nearest), 16/8-byte stores.
template <typename DstT, int V>
__device__ __forceinline__ void store_n(DstT* dst, const float* src) {
  static_assert(V % 4 == 0, "vector width");
  if constexpr (sizeof(DstT) == 4) {
#pragma unroll
    for (int k = 0; k < V; k += 4)
      *reinterpret_cast<float4*>(dst + k) = make_float4(src[k], src[k + 1], src[k + 2], src[k + 3]);
  } else {
#pragma unroll
    for (int k = 0; k < V; k += 4) {
      uint2 u;
      __half2* h = reinterpret_cast<__half2*>(&u);
      h[0] = __floats2half2_rn(src[k], src[k + 1]);
      h[1] = __floats2half2_rn(src[k + 2], src[k + 3]);
      *reinterpret_cast<uint2*>(dst + k) = u;
    }
  }
}

// Row roles of the flattened row index.
enum Role { kKey = 0, kValue = 1, kQuery = 2 };

// A prompt's float cache of another dtype than T: attention reads the new rows
// in T from the workspace (kv_sep_k / kv_sep_v) instead of the cache.
template <typename T, typename CacheT>
constexpr bool kSeparate = (std::is_same<CacheT, float>::value || std::is_same<CacheT, __half>::value) &&
                           !std::is_same<T, CacheT>::value;

// Appends V consecutive values (head coordinates d0 .. d0+V-1 of cache row pos of KV
// head `head`) to the present K or V cache: a cast for a float cache, int8
// codes, or for a 4-bit cache (CacheT = uint8_t) V/2 bytes of +8-biased
// nibbles with the even coordinate in the low nibble. With a separate cache
// dtype the values are also stored in T for attention.
template <typename T, typename CacheT, int V>
__device__ __forceinline__ void append_chunk(const Params& p, int role, int b, int head, int pos, int d0,
                                             const float* y) {
  const int H = p.H;
  const long long row = ((long long)b * p.Nkv + head) * p.C + pos;
  void* base = role == kKey ? p.present_k : p.present_v;
  if constexpr (std::is_same<CacheT, uint8_t>::value) {
    static_assert(V == 4, "4-bit cache: fp32 rows, four values per chunk");
    const float* sc = role == kKey ? p.k_scale : p.v_scale;
    const int nsc = role == kKey ? p.k_scale_n : p.v_scale_n;
    unsigned n[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) n[k] = quant_i4_nibble(y[k], channel_scale(sc, nsc, head * H + d0 + k));
    const unsigned short packed = (unsigned short)(n[0] | (n[1] << 4) | (n[2] << 8) | (n[3] << 12));
    *reinterpret_cast<unsigned short*>(reinterpret_cast<uint8_t*>(base) + row * (H / 2) + d0 / 2) = packed;
  } else if constexpr (sizeof(CacheT) == 1) {
    const float* sc = role == kKey ? p.k_scale : p.v_scale;
    const int nsc = role == kKey ? p.k_scale_n : p.v_scale_n;
    char4 q4[V / 4];
    int8_t* qb = reinterpret_cast<int8_t*>(q4);
#pragma unroll
    for (int k = 0; k < V; ++k) qb[k] = quant_i8(y[k], channel_scale(sc, nsc, head * H + d0 + k));
    int8_t* dst = reinterpret_cast<int8_t*>(base) + row * H + d0;
    if constexpr (V == 4) *reinterpret_cast<char4*>(dst) = q4[0];
    else *reinterpret_cast<int2*>(dst) = *reinterpret_cast<int2*>(q4);
  } else {
    store_n<CacheT, V>(reinterpret_cast<CacheT*>(base) + row * H + d0, y);
  }
  if constexpr (kSeparate<T, CacheT>) {
    T* sep = reinterpret_cast<T*>(role == kKey ? p.kv_sep_k : p.kv_sep_v);
    store_n<T, V>(sep + (((long long)b * p.Nkv + head) * p.S + pos) * H + d0, y);
  }
}

// T: element type of query/key/value. CacheT: element type of the cache
// (T, int8_t for an int8 cache, uint8_t for a 4-bit cache). QT: element type
// of prepared queries.
template <typename T, typename CacheT, typename QT>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
prepass_kernel(const Params p) {
  __shared__ float rowbuf[kWarpsPerBlock][kMaxH];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long kv_rows = (long long)p.B * p.S * p.Nkv;
  const long long q_rows = (long long)p.B * p.S * p.N;
  const long long row = (long long)blockIdx.x * kWarpsPerBlock + warp;
  if (row >= 2 * kv_rows + q_rows) return;

  int role, b, i, head;
  if (row < 2 * kv_rows) {
    role = row < kv_rows ? kKey : kValue;
    long long r = row - (role == kValue ? kv_rows : 0);
    head = (int)(r % p.Nkv);
    i = (int)((r / p.Nkv) % p.S);
    b = (int)(r / ((long long)p.Nkv * p.S));
  } else {
    role = kQuery;
    long long r = row - 2 * kv_rows;
    head = (int)(r % p.N);
    i = (int)((r / p.N) % p.S);
    b = (int)(r / ((long long)p.N * p.S));
  }
  const int H = p.H;
  const int total = p.seqlens[b] + 1;
  const int past = batch_past(p, total);
  if (past < 0) {
    if (role == kKey && i == 0 && head == 0 && lane == 0) flag_status(p, GQA_DEVICE_BAD_SEQLEN_BIT);
    return;
  }
  const int pos = past + i;                                 // absolute position (rotary)
  const int crow = batch_rows(p, total, past).keep + i;     // cache row
  const bool rotate = p.has_rotary && role != kValue;
  if (rotate && pos >= p.rotary_rows) {
    if (lane == 0) flag_status(p, GQA_DEVICE_BAD_ROTARY_BIT);
    return;
  }

  constexpr int V = Vec<T>::n;
  const T* src;
  if (role == kQuery)
    src = reinterpret_cast<const T*>(p.q) + ((long long)(b * p.S + i) * p.N + head) * H;
  else
    src = reinterpret_cast<const T*>(role == kKey ? p.k : p.v) + ((long long)(b * p.S + i) * p.Nkv + head) * H;

  float* buf = rowbuf[warp];
  for (int d0 = lane * V; d0 < H; d0 += 32 * V) {
    float x[V];
    load_vec<T>(src + d0, x);
#pragma unroll
    for (int k = 0; k < V; ++k) buf[d0 + k] = x[k];
  }
  __syncwarp();
  const bool norm = p.has_norm && role != kValue;
  const float r = norm ? rms_inv_rn(row_sum_squares_warp(buf, H), H, p.eps) : 1.f;
  const T* w = reinterpret_cast<const T*>(role == kQuery ? p.qw : p.kw);
  const int half = H >> 1;
  for (int d0 = lane * V; d0 < H; d0 += 32 * V) {
    float y[V];
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int d = d0 + k;
      float x = buf[d];
      if (norm) x = norm_rn(x, r, load_t(w, d, p.t_type));
      if (rotate) {
        const int dp = d < half ? d + half : d - half;
        float xp = buf[dp];
        if (norm) xp = norm_rn(xp, r, load_t(w, dp, p.t_type));
        const int dc = d < half ? d : d - half;
        const float c = rot_t(p.cos_c, (long long)pos * half + dc, p.t_type);
        const float s = rot_t(p.sin_c, (long long)pos * half + dc, p.t_type);
        x = d < half ? rope_first_rn(x, xp, c, s) : rope_second_rn(x, xp, c, s);
      }
      y[k] = x;
    }
    if (role == kQuery) {
      const int g = head / p.G, gi = head % p.G;
      QT* dst = reinterpret_cast<QT*>(p.qprep) +
                (((long long)(b * p.Nkv + g) * p.S + i) * p.G + gi) * H + d0;
      store_n<QT, V>(dst, y);
    } else {
      append_chunk<T, CacheT, V>(p, role, b, head, crow, d0, y);
    }
  }
}

// Vectorised pre-pass for rows of at most 32 16-byte chunks. One block per
// token (b, i) handles its 2*N_kv + N_q rows (K rows, V rows, query rows);
// LPR = H / V lanes per row (V elements per 16-byte chunk), 256 / LPR row
// groups per block, each taking kUnroll rows per pass with their loads issued
// together. The rotary partner (d +- H/2) is chunk lane ^ LPR/2, read with one
// shuffle per element; norm weights and cos/sin rows are 16-byte vector loads.
constexpr int kUnroll = 4;

template <typename T, typename CacheT, typename QT, int H>
__global__ void __launch_bounds__(256, 4)
prepass_vec_kernel(const Params p) {
  constexpr int V = Vec<T>::n;
  constexpr int LPR = H / V;            // lanes per row (power of two, <= 32)
  constexpr int GROUPS = 256 / LPR;     // row groups per block
  static_assert(LPR >= 2 && LPR <= 32 && (LPR & (LPR - 1)) == 0, "row layout");
  const int lane = threadIdx.x & 31;
  const int grp = threadIdx.x / LPR, cl = threadIdx.x % LPR;
  const unsigned gmask = (LPR == 32) ? 0xffffffffu : (((1u << LPR) - 1u) << ((lane / LPR) * LPR));
  const int tok = blockIdx.x;
  const int b = tok / p.S, i = tok - b * p.S;
  const int nrow = 2 * p.Nkv + p.N;
  const int d0 = cl * V;
  const T* qsrc = reinterpret_cast<const T*>(p.q) + (long long)tok * p.N * H + d0;
  const T* ksrc = reinterpret_cast<const T*>(p.k) + (long long)tok * p.Nkv * H + d0;
  const T* vsrc = reinterpret_cast<const T*>(p.v) + (long long)tok * p.Nkv * H + d0;
  const int total = p.seqlens[b] + 1;

  for (int r0 = grp; r0 < nrow; r0 += GROUPS * kUnroll) {
    // Loads of all rows of this pass first (addresses need no lengths), kept
    // as raw 16-byte chunks until used.
    uint4 raw[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int r = r0 + u * GROUPS;
      if (r >= nrow) continue;
      const T* src = r < p.Nkv ? ksrc + (long long)r * H
                     : r < 2 * p.Nkv ? vsrc + (long long)(r - p.Nkv) * H
                                     : qsrc + (long long)(r - 2 * p.Nkv) * H;
      raw[u] = *reinterpret_cast<const uint4*>(src);
    }
    const int past = batch_past(p, total);
    if (past < 0) {
      if (i == 0 && threadIdx.x == 0 && r0 == grp) flag_status(p, GQA_DEVICE_BAD_SEQLEN_BIT);
      return;   // the whole block (one token) is skipped
    }
    const int pos = past + i;                                 // absolute position (rotary)
    const int crow = batch_rows(p, total, past).keep + i;     // cache row
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int r = r0 + u * GROUPS;
      if (r >= nrow) continue;
      const int role = r < p.Nkv ? kKey : (r < 2 * p.Nkv ? kValue : kQuery);
      const int head = role == kKey ? r : (role == kValue ? r - p.Nkv : r - 2 * p.Nkv);
      if (role != kValue && p.has_rotary && pos >= p.rotary_rows) {
        if (cl == 0) flag_status(p, GQA_DEVICE_BAD_ROTARY_BIT);
        continue;   // every lane of the row group takes this branch together
      }
      float xr[V];
      load_vec<T>(reinterpret_cast<const T*>(&raw[u]), xr);
      if (role != kValue && p.has_norm) {
        // Lane cl holds the groups of coordinates 4 * (V/4 * cl) ..: the rising
        // xor distances add neighbouring subtrees (the stored-row recipe).
        float ss = V == 8 ? sumsq8_rn(xr) : sumsq4_rn(xr[0], xr[1], xr[2], xr[3]);
#pragma unroll
        for (int o = 1; o < LPR; o <<= 1) ss = __fadd_rn(ss, __shfl_xor_sync(gmask, ss, o));
        const float rn = rms_inv_rn(ss, H, p.eps);
        float w[V];
        load_vec<T>(reinterpret_cast<const T*>(role == kQuery ? p.qw : p.kw) + d0, w);
#pragma unroll
        for (int k = 0; k < V; ++k) xr[k] = norm_rn(xr[k], rn, w[k]);
      }
      if (role != kValue && p.has_rotary) {
        const bool first = cl < LPR / 2;
        const int dc = (first ? cl : cl - LPR / 2) * V;
        float c[V], sn[V];
        load_vec<T>(reinterpret_cast<const T*>(p.cos_c) + (long long)pos * (H / 2) + dc, c);
        load_vec<T>(reinterpret_cast<const T*>(p.sin_c) + (long long)pos * (H / 2) + dc, sn);
        float y[V];
#pragma unroll
        for (int k = 0; k < V; ++k) {
          const float xp = __shfl_xor_sync(gmask, xr[k], LPR / 2);
          y[k] = first ? rope_first_rn(xr[k], xp, c[k], sn[k]) : rope_second_rn(xr[k], xp, c[k], sn[k]);
        }
#pragma unroll
        for (int k = 0; k < V; ++k) xr[k] = y[k];
      }
      if (role == kQuery) {
        const int g = head / p.G, gi = head - g * p.G;
        QT* dst = reinterpret_cast<QT*>(p.qprep) + (((long long)(b * p.Nkv + g) * p.S + i) * p.G + gi) * H + d0;
        store_n<QT, V>(dst, xr);
      } else {
        append_chunk<T, CacheT, V>(p, role, b, head, crow, d0, xr);
      }
    }
  }
}

template <typename T, typename CacheT, typename QT>
cudaError_t launch_vec(const Params& p, cudaStream_t st, bool* done) {
  constexpr int V = Vec<T>::n;
  const long long tokens = (long long)p.B * p.S;
  auto go = [&](auto kern) {
    *done = true;
    if (tokens == 0) return cudaSuccess;
    kern<<<(unsigned)tokens, 256, 0, st>>>(p);
    return cudaGetLastError();
  };
  switch (p.H / V) {
    case 2: return go(prepass_vec_kernel<T, CacheT, QT, 2 * V>);
    case 4: return go(prepass_vec_kernel<T, CacheT, QT, 4 * V>);
    case 8: return go(prepass_vec_kernel<T, CacheT, QT, 8 * V>);
    case 16: return go(prepass_vec_kernel<T, CacheT, QT, 16 * V>);
    case 32: return go(prepass_vec_kernel<T, CacheT, QT, 32 * V>);
    default: return cudaSuccess;  // not a power-of-two chunk count: the generic kernel runs
  }
}

// Copy mode: present[b, g, 0:past_b] = past[b, g, 0:past_b] with 16-byte moves.
__global__ void copy_past_kernel(const Params p, int esize) {
  const int bg = blockIdx.y;
  const int b = bg / p.Nkv, g = bg % p.Nkv;
  const int total = p.seqlens[b] + 1;
  const int past = batch_past(p, total);
  if (past <= 0) return;
  const long long row_bytes = (long long)p.H * esize;
  const long long n16 = (long long)past * row_bytes / 16;
  const uint4* src = reinterpret_cast<const uint4*>(
      reinterpret_cast<const char*>(p.past_k) + ((long long)b * p.Nkv + g) * p.past_cap * row_bytes);
  uint4* dst = reinterpret_cast<uint4*>(
      reinterpret_cast<char*>(p.present_k) + ((long long)b * p.Nkv + g) * p.C * row_bytes);
  const uint4* srcv = reinterpret_cast<const uint4*>(
      reinterpret_cast<const char*>(p.past_v) + ((long long)b * p.Nkv + g) * p.past_cap * row_bytes);
  uint4* dstv = reinterpret_cast<uint4*>(
      reinterpret_cast<char*>(p.present_v) + ((long long)b * p.Nkv + g) * p.C * row_bytes);
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n16;
       x += (long long)gridDim.x * blockDim.x) {
    dst[x] = src[x];
    dstv[x] = srcv[x];
  }
}

// Window-shift update of a sliding-window cache: present rows [0, keep) =
// past rows [n_old - keep, n_old) (the most recent ones; the older rows are
// evicted from the front). One CTA per (batch, KV head, K or V) moves the rows
// in order, 16-byte vectors, a chunk of kShiftVec vectors per thread at a
// time: each chunk is read completely before any of it is written, and a
// chunk's destination lies below the source of every later chunk, so the
// in-place move of a shared buffer (toward the front) is safe.
constexpr int kShiftThreads = 256, kShiftVec = 8;

__global__ void __launch_bounds__(kShiftThreads) window_shift_kernel(const Params p, int esize) {
  const int bg = blockIdx.x, b = bg / p.Nkv;
  const bool is_v = blockIdx.y == 1;
  const int total = p.seqlens[b] + 1;
  const int past = batch_past(p, total);
  if (past < 0) return;   // the pre-pass reports the bad length
  const BatchRows r = batch_rows(p, total, past);
  const int src0 = r.n_old - r.keep;
  if (r.keep <= 0 || (p.mode == kShared && src0 == 0)) return;   // nothing moves
  const long long row_bytes = (long long)p.H * esize;
  const int L = p.mode == kShared ? p.C : p.past_cap;
  const char* src = reinterpret_cast<const char*>(is_v ? p.past_v : p.past_k) + ((long long)bg * L + src0) * row_bytes;
  char* dst = reinterpret_cast<char*>(is_v ? p.present_v : p.present_k) + (long long)bg * p.C * row_bytes;
  const uint4* s16 = reinterpret_cast<const uint4*>(src);
  uint4* d16 = reinterpret_cast<uint4*>(dst);
  const long long n16 = (long long)r.keep * row_bytes / 16;
  for (long long base = 0; base < n16; base += kShiftThreads * kShiftVec) {
    uint4 v[kShiftVec];
#pragma unroll
    for (int k = 0; k < kShiftVec; ++k) {
      const long long x = base + k * kShiftThreads + threadIdx.x;
      if (x < n16) v[k] = s16[x];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kShiftVec; ++k) {
      const long long x = base + k * kShiftThreads + threadIdx.x;
      if (x < n16) d16[x] = v[k];
    }
    __syncthreads();
  }
}

// Bias staging for the tensor-core prefill: bias[bb, 0, i, j] * log2(e) as fp32
// rows of bias_stage_ld floats (16-byte stride), so that the prefill's TMA warp
// loads a (positions x 128 keys) block with one tensor copy. A thread converts
// four consecutive keys of a row (one 16-byte store; the row's tail past T is
// never read by the copies, which stop at T).
__global__ void __launch_bounds__(256) bias_stage_kernel(const Params p) {
  const long long rows = (long long)p.bias_bdim * p.S;
  const int T = p.bias_ld, q4 = (T + 3) / 4;
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < rows * q4;
       x += (long long)gridDim.x * blockDim.x) {
    const long long r = x / q4;
    const int j = (int)(x - r * q4) * 4;
    float v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = j + k < T ? load_t(p.bias, r * T + j + k, p.t_type) * kLog2e : 0.f;
    *reinterpret_cast<float4*>(p.bias_stage + r * p.bias_stage_ld + j) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

}  // namespace

cudaError_t launch_bias_stage(const Params& p, cudaStream_t st) {
  const long long n = (long long)p.bias_bdim * p.S * ((p.bias_ld + 3) / 4);
  const unsigned blocks = (unsigned)min((n + 255) / 256, 152LL * 16);
  if (blocks == 0) return cudaSuccess;
  bias_stage_kernel<<<blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_window_shift(const Params& p, cudaStream_t st) {
  const int esize = p.cache_type == kF32 ? 4 : (p.cache_type == kF16 ? 2 : 1);
  dim3 grid(p.B * p.Nkv, 2), block(kShiftThreads);
  window_shift_kernel<<<grid, block, 0, st>>>(p, esize);
  return cudaGetLastError();
}

bool prepass_supported(const Params& p) {
  return p.H % 16 == 0 && p.H <= kMaxH && p.H >= 16;
}

cudaError_t launch_prepass(const Params& p, cudaStream_t st) {
  // Vectorised kernel whenever a row is a power-of-two count (<= 32) of 16-byte chunks.
  bool done = false;
  cudaError_t ev;
  if (p.t_type == kF16 && p.cache_type == kF32)
    ev = p.qprep_type == kF16 ? launch_vec<__half, float, __half>(p, st, &done)
                              : launch_vec<__half, float, float>(p, st, &done);
  else if (p.t_type == kF16)
    ev = p.qprep_type == kF16 ? launch_vec<__half, __half, __half>(p, st, &done)
                              : launch_vec<__half, __half, float>(p, st, &done);
  else if (p.cache_type == kF16)
    ev = launch_vec<float, __half, float>(p, st, &done);
  else if (p.cache_type == kI8)
    ev = launch_vec<float, int8_t, float>(p, st, &done);
  else if (p.cache_type == kI4)
    ev = launch_vec<float, uint8_t, float>(p, st, &done);
  else
    ev = launch_vec<float, float, float>(p, st, &done);
  if (done || ev != cudaSuccess) return ev;
  const long long rows = (long long)p.B * p.S * (2 * p.Nkv + p.N);
  const unsigned blocks = (unsigned)((rows + kWarpsPerBlock - 1) / kWarpsPerBlock);
  if (blocks == 0) return cudaSuccess;
  dim3 grid(blocks), block(kWarpsPerBlock * 32);
  const bool q16 = p.qprep_type == kF16;
  if (p.t_type == kF16 && p.cache_type == kF32) {
    if (q16) prepass_kernel<__half, float, __half><<<grid, block, 0, st>>>(p);
    else prepass_kernel<__half, float, float><<<grid, block, 0, st>>>(p);
  } else if (p.t_type == kF16) {
    if (q16) prepass_kernel<__half, __half, __half><<<grid, block, 0, st>>>(p);
    else prepass_kernel<__half, __half, float><<<grid, block, 0, st>>>(p);
  } else if (p.cache_type == kF16) {
    prepass_kernel<float, __half, float><<<grid, block, 0, st>>>(p);
  } else if (p.cache_type == kI8) {
    prepass_kernel<float, int8_t, float><<<grid, block, 0, st>>>(p);
  } else if (p.cache_type == kI4) {
    prepass_kernel<float, uint8_t, float><<<grid, block, 0, st>>>(p);
  } else {
    prepass_kernel<float, float, float><<<grid, block, 0, st>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_copy_past(const Params& p, cudaStream_t st) {
  if (p.cache_type == kI4) return cudaErrorNotSupported;   // a 4-bit cache has no past
  const int esize = p.cache_type == kF32 ? 4 : (p.cache_type == kF16 ? 2 : 1);
  dim3 grid(64, p.B * p.Nkv), block(256);
  copy_past_kernel<<<grid, block, 0, st>>>(p, esize);
  return cudaGetLastError();
}

}  // namespace gqa
