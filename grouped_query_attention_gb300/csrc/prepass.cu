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

// The same from a 16-byte chunk already in registers (passed by value, so no
// local-memory copy is needed).
template <typename T>
__device__ __forceinline__ void unpack_vec(uint4 v, float* dst);
template <>
__device__ __forceinline__ void unpack_vec<float>(uint4 v, float* dst) {
  dst[0] = __uint_as_float(v.x); dst[1] = __uint_as_float(v.y); dst[2] = __uint_as_float(v.z); dst[3] = __uint_as_float(v.w);
}
template <>
__device__ __forceinline__ void unpack_vec<__half>(uint4 v, float* dst) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
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
  const long long q_rows = p.q_in_prefill ? 0 : (long long)p.B * p.S * p.N;   // the prefill may prepare its queries
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

// Vectorised pre-pass. Rows are numbered token-major, row = token * nrow + r
// with r < N_kv a K row, N_kv <= r < 2 N_kv a V row and the rest query rows
// (none when the prefill prepares its own); nrow = 2*N_kv + N_q. A row group
// of LPR = H / (2 V) lanes (V elements per 16-byte chunk) takes one row at a
// time, striding over the grid's row groups; lane l holds the chunk of dims
// l V .. (lo) and the one of dims H/2 + l V .. (hi), so the NeoX rotary
// partner of every value is in the same lane and one cos / sin chunk serves
// both. The loads of the group's next row are issued before the current row
// is computed. Norm weights are loaded once.
__host__ __device__ inline int prepass_rows_per_token(const Params& p) { return 2 * p.Nkv + (p.q_in_prefill ? 0 : p.N); }
constexpr int kPrepassBlocksPerSm = 3;

// Where a row is: row = tok * nrow + r, tok = b * S + i. Kept incrementally
// (no integer division per row).
struct RowPos {
  int tok, r, b, i;
};

__device__ __forceinline__ RowPos row_pos(long long row, int nrow, int S) {
  RowPos q;
  q.tok = (int)(row / nrow);
  q.r = (int)(row - (long long)q.tok * nrow);
  q.b = q.tok / S;
  q.i = q.tok - q.b * S;
  return q;
}

// The position `stride` rows further, stride = st_tok * nrow + st_r.
__device__ __forceinline__ RowPos row_advance(RowPos q, int st_tok, int st_r, int nrow, int S) {
  q.r += st_r;
  int dt = st_tok;
  if (q.r >= nrow) {
    q.r -= nrow;
    ++dt;
  }
  q.tok += dt;
  q.i += dt;
  if (q.i >= S) {
    q.b += q.i / S;
    q.i %= S;
  }
  return q;
}

// A lane's part of one row: its lo and hi chunks and the batch length.
struct RowLoads {
  uint4 lo, hi;
  int total;        // seqlens_k[b] + 1
};

template <typename T, typename CacheT, typename QT, int H>
__global__ void __launch_bounds__(256, kPrepassBlocksPerSm)
prepass_vec_kernel(const Params p) {
  constexpr int V = Vec<T>::n;
  constexpr int LPR = H / (2 * V);      // lanes per row (power of two, <= 16)
  constexpr int GROUPS = 256 / LPR;     // row groups per block
  static_assert(LPR >= 1 && LPR <= 16 && (LPR & (LPR - 1)) == 0, "row layout");
  const int lane = threadIdx.x & 31;
  const int cl = threadIdx.x % LPR;
  const unsigned gmask = LPR == 32 ? 0xffffffffu : (((1u << LPR) - 1u) << ((lane / LPR) * LPR));
  const int nrow = prepass_rows_per_token(p);
  const long long nrows = (long long)p.B * p.S * nrow;
  const long long stride = (long long)gridDim.x * GROUPS;
  const int dlo = cl * V, dhi = H / 2 + cl * V;   // this lane's dims, and the cos / sin columns dlo ..
  // Norm weights of this lane's chunks (K and query rows), loaded once, kept raw.
  uint4 wk_lo = make_uint4(0, 0, 0, 0), wk_hi = wk_lo, wq_lo = wk_lo, wq_hi = wk_lo;
  if (p.has_norm) {
    wk_lo = *reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.kw) + dlo);
    wk_hi = *reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.kw) + dhi);
    if (!p.q_in_prefill) {
      wq_lo = *reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.qw) + dlo);
      wq_hi = *reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.qw) + dhi);
    }
  }
  auto issue = [&](const RowPos& q, RowLoads& l) {
    const int r = q.r;
    const T* src = r < p.Nkv ? reinterpret_cast<const T*>(p.k) + ((long long)q.tok * p.Nkv + r) * H
                   : r < 2 * p.Nkv ? reinterpret_cast<const T*>(p.v) + ((long long)q.tok * p.Nkv + r - p.Nkv) * H
                                   : reinterpret_cast<const T*>(p.q) + ((long long)q.tok * p.N + r - 2 * p.Nkv) * H;
    l.lo = *reinterpret_cast<const uint4*>(src + dlo);
    l.hi = *reinterpret_cast<const uint4*>(src + dhi);
    l.total = p.seqlens[q.b] + 1;
  };

  long long row = (long long)blockIdx.x * GROUPS + threadIdx.x / LPR;
  const int st_tok = (int)(stride / nrow), st_r = (int)(stride - (long long)st_tok * nrow);
  RowPos pc = row_pos(row, nrow, p.S), pn = pc;
  RowLoads cur, nxt;
  if (row < nrows) issue(pc, cur);
  for (; row < nrows; row += stride) {   // uniform over the row group
    if (row + stride < nrows) {
      pn = row_advance(pc, st_tok, st_r, nrow, p.S);
      issue(pn, nxt);
    }
    const int r = pc.r, b = pc.b, i = pc.i;
    const int past = batch_past(p, cur.total);
    const int role = r < p.Nkv ? kKey : (r < 2 * p.Nkv ? kValue : kQuery);
    const int head = role == kKey ? r : (role == kValue ? r - p.Nkv : r - 2 * p.Nkv);
    const int pos = past + i;                                 // absolute position (rotary)
    const bool rot = p.has_rotary && role != kValue;
    if (past < 0) {   // the token is skipped
      if (i == 0 && r == 0 && cl == 0) flag_status(p, GQA_DEVICE_BAD_SEQLEN_BIT);
    } else if (rot && pos >= p.rotary_rows) {
      if (cl == 0) flag_status(p, GQA_DEVICE_BAD_ROTARY_BIT);
    } else {
      uint4 cr = make_uint4(0, 0, 0, 0), sr = cr;
      if (rot) {   // cos / sin rows are shared by the heads of a token (cache hits after the first)
        cr = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.cos_c) + (long long)pos * (H / 2) + dlo));
        sr = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.sin_c) + (long long)pos * (H / 2) + dlo));
      }
      const int crow = batch_rows(p, cur.total, past).keep + i;   // cache row
      float lo[V], hi[V];
      unpack_vec<T>(cur.lo, lo);
      unpack_vec<T>(cur.hi, hi);
      if (role != kValue && p.has_norm) {
        // The stored-row recipe: the lo chunks of the row's lanes are the
        // groups of the first half, the hi chunks those of the second; rising
        // xor distances add neighbouring subtrees of each half, then the halves.
        float slo = V == 8 ? sumsq8_rn(lo) : sumsq4_rn(lo[0], lo[1], lo[2], lo[3]);
        float shi = V == 8 ? sumsq8_rn(hi) : sumsq4_rn(hi[0], hi[1], hi[2], hi[3]);
#pragma unroll
        for (int o = 1; o < LPR; o <<= 1) {
          slo = __fadd_rn(slo, __shfl_xor_sync(gmask, slo, o));
          shi = __fadd_rn(shi, __shfl_xor_sync(gmask, shi, o));
        }
        const float rn = rms_inv_rn(__fadd_rn(slo, shi), H, p.eps);
        float wl[V], wh[V];
        unpack_vec<T>(role == kQuery ? wq_lo : wk_lo, wl);
        unpack_vec<T>(role == kQuery ? wq_hi : wk_hi, wh);
#pragma unroll
        for (int k = 0; k < V; ++k) {
          lo[k] = norm_rn(lo[k], rn, wl[k]);
          hi[k] = norm_rn(hi[k], rn, wh[k]);
        }
      }
      if (rot) {
        float c[V], sn[V];
        unpack_vec<T>(cr, c);
        unpack_vec<T>(sr, sn);
#pragma unroll
        for (int k = 0; k < V; ++k) {
          const float a = lo[k], bb = hi[k];
          lo[k] = rope_first_rn(a, bb, c[k], sn[k]);
          hi[k] = rope_second_rn(bb, a, c[k], sn[k]);
        }
      }
      if (role == kQuery) {
        const int g = head / p.G, gi = head - g * p.G;
        QT* dst = reinterpret_cast<QT*>(p.qprep) + (((long long)(b * p.Nkv + g) * p.S + i) * p.G + gi) * H;
        store_n<QT, V>(dst + dlo, lo);
        store_n<QT, V>(dst + dhi, hi);
      } else {
        append_chunk<T, CacheT, V>(p, role, b, head, crow, dlo, lo);
        append_chunk<T, CacheT, V>(p, role, b, head, crow, dhi, hi);
      }
    }
    cur = nxt;
    pc = pn;
  }
}

template <typename T, typename CacheT, typename QT>
cudaError_t launch_vec(const Params& p, cudaStream_t st, bool* done) {
  constexpr int V = Vec<T>::n;
  const long long rows = (long long)p.B * p.S * prepass_rows_per_token(p);
  auto go = [&](auto kern) {
    *done = true;
    if (rows == 0) return cudaSuccess;
    // One row group per row up to kPrepassBlocksPerSm resident blocks per SM
    // (152 SMs); beyond that the groups stride over the rows.
    const long long groups = 256 / (p.H / (2 * V));
    const long long want = (rows + groups - 1) / groups;
    const long long cap = 152LL * kPrepassBlocksPerSm;
    kern<<<(unsigned)(want < cap ? want : cap), 256, 0, st>>>(p);
    return cudaGetLastError();
  };
  switch (p.H / (2 * V)) {   // lanes per row
    case 1: return go(prepass_vec_kernel<T, CacheT, QT, 2 * V>);
    case 2: return go(prepass_vec_kernel<T, CacheT, QT, 4 * V>);
    case 4: return go(prepass_vec_kernel<T, CacheT, QT, 8 * V>);
    case 8: return go(prepass_vec_kernel<T, CacheT, QT, 16 * V>);
    case 16: return go(prepass_vec_kernel<T, CacheT, QT, 32 * V>);
    default: return cudaSuccess;  // not a power of two: the generic kernel runs
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
  const long long rows = (long long)p.B * p.S * prepass_rows_per_token(p);
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
