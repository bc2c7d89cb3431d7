// Tensor-core split-KV decode for GroupQueryAttention on sm_103a, head size
// 128: an fp16 cache with fp16 queries (at most 16 query rows per KV head) and
// an int8 cache with fp32 queries and output (at most 8), one kernel template
// (I8) whose two forms differ only in how K / V tiles reach the MMAs and in
// the precision of the query and probability operands.
//
// The R = S*G query rows of one KV head share every key, so each 128-key tile
// is two small MMAs: S^T = K Q^T (M = 128 keys, N = 16 padded rows, K = 128
// dims) and O^T += V^T P^T (M = 128 dims, V read as an MN-major operand,
// N = 16, K = 128 keys). The CUDA cores only run the softmax (one thread per
// key), so the kernel streams the cache at the memory rate.
//
// Work is balanced statically: the key range of every (batch b, KV head g)
// is cut into 128-key tiles, the tiles of all (b, g) are laid end to end, and
// persistent CTA c (one per SM) takes the c-th equal share of that sequence.
// A share covers one or a few segments (the tiles of one (b, g) inside it);
// only a share's first and last segment can be split with a neighbour CTA, so
// a CTA writes at most two partial results. Warp roles:
//   warp 2      preparer: maps the CTA's segments, prepares Q^T (norm, rotary,
//               scale, fp16, 128-byte swizzle) in one of two item slots and
//               appends the new rows that fall in the segment (then an
//               async-proxy fence so TMA reads them); it runs one item ahead.
//   warp 0      TMA: streams each published item's 128-key K and V tiles into
//               a 3-stage ring.
//   warp 1      MMA issue: S^T(t) into one of two tensor-memory buffers, then
//               O^T += V^T P^T(t-1), so scores of the next tile are ready
//               while the softmax works.
//   warps 3..6  softmax: a thread holds one key's R scores (tensor-memory lane
//               = key), masks / softcap / bias, cross-warp row max, lazy
//               rescaling of O^T, P^T (fp16) into one of two shared buffers,
//               zeroed V rows past the key range; at the end of an item one
//               thread per dim writes the partial (or the output) and the last
//               CTA to finish a shared (b, g) merges its partials (atomic
//               ticket, no wait).
// Every mbarrier wait is bounded; a timed-out consumer sets an abort flag that
// all softmax warps check right after a shared named barrier, so they leave
// together; tensor memory is always freed.
//
// The int8 form (I8) adds:
//   - int8 codes are exact in fp16, so TMA brings the int8 K / V tiles (5 and
//     4 stages) and four converter warps (7..10, thread = tensor-memory lane =
//     key row of the tile) rewrite them in fp16: K straight into tensor
//     memory (the A operand of S^T, one key per lane), V into one of two
//     shared-memory operand tiles; one converter step turns K(u) and V(u-1);
//   - fp32 accuracy: each prepared query row q' (norm, rotary, scale, K
//     channel scale folded in, times a power of two 2^-e that brings its
//     largest value to [1, 2)) is split into two fp16 rows hi = fp16(q'),
//     lo = fp16(q' - hi), placed as MMA rows r and r+R; the products with the
//     codes are exact and accumulate in fp32, so S = (S_hi + S_lo) 2^e holds
//     q' to about 2^-22. Probabilities are split the same way for P.V, and
//     the V channel scale multiplies O once at the end; the appended rows are
//     stored as int8 codes.
//
// com.microsoft.GroupQueryAttention, section Implementation variants
// (share_append_split_decode_splitk / past_kv_decode_splitk: append, then
// partition the key axis and merge partial online-softmax results;
// quant_int8_decode_splitk: int8 rows appended with k/v_scale, attention over
// the stored codes times the scales) and sections Inputs (k_scale, v_scale) /
// Attributes (k/v_quant_type).
#include <cuda_fp16.h>

#include "common.cuh"
#include "tcgen05.cuh"
#include "tma_host.h"

namespace gqa {
namespace {

using namespace tc;

constexpr int kHD = 128;
constexpr int kKT = kTcDecodeTile;       // keys per tile (128)
constexpr int kNR = 16;                  // MMA N: query rows of the group (int8: hi and lo rows), padded
constexpr int kSoftWarp0 = 3;            // first softmax warp
constexpr int kConvWarp0 = 7;            // first converter warp (int8 cache)
constexpr int kSoft = 128;               // softmax threads
constexpr int kConv = 128;               // converter threads (int8 cache)
constexpr uint32_t kBox = 128u * 128u;   // 64 columns x 128 rows (fp16) = 16 KB
constexpr uint32_t kTile = 2u * kBox;    // fp16 K or V tile: 128 keys x 128 dims
constexpr uint32_t kTile8 = 128u * 128u; // int8 K or V tile: 128 keys x 128 dims
constexpr uint32_t kRowBox = 16u * 128u; // 64 columns x 16 rows = 2 KB
constexpr float kLazy = 8.0f;            // log2 growth tolerated before rescaling O
constexpr uint32_t kIdS = idesc_f16(128, kNR, 0, 0);   // K (K-major) x Q^T rows (K-major)
constexpr uint32_t kIdO = idesc_f16(128, kNR, 1, 0);   // V (MN-major) x P^T rows (K-major)
// Tensor memory: S^T buffers at columns 0 and 16, O^T at 32 (16 columns
// each); int8 cache: fp16 K tiles (A operand of S^T, one key per lane, two
// dims per column) at columns 64 and 128.
constexpr uint32_t kKCol = 64;

// The two forms: K / V stages, threads, tensor-memory columns.
template <bool I8>
struct DCfg {
  static constexpr int kNS = 3;          // K / V stages (fp16 tiles)
  static constexpr int kNSV = 3;
  static constexpr int kThreads = 224;   // TMA, MMA, preparer, 4 softmax warps
  static constexpr uint32_t kTmemCols = 64;
};
template <>
struct DCfg<true> {
  static constexpr int kNS = 5;          // int8 K stages
  static constexpr int kNSV = 4;         // int8 V stages
  static constexpr int kThreads = 352;   // TMA, MMA, preparer, 4 softmax, 4 converter warps
  static constexpr uint32_t kTmemCols = 256;
};

struct DItem {
  int b, g;
  int split, nsplit;     // this segment's index among the CTAs sharing (b, g), their count
  int slot, slot0;       // partial slot of this segment / of the first segment of (b, g)
  int cfirst;            // first CTA of (b, g)
  int j0, jend;          // keys of this segment: [j0, jend)
  int last;              // the segment holds the last tile of (b, g)
  int past, total, ntiles, end;   // past / total in cache rows (see batch_tiles)
  int off;                        // absolute position of cache row 0 (rotary, bias columns)
};

// K / V tiles as the TMA writes them (and, int8 cache, the fp16 V operand tiles).
template <bool I8>
struct __align__(1024) DTiles {
  uint8_t k[DCfg<I8>::kNS][kTile];
  uint8_t v[DCfg<I8>::kNSV][kTile];
};
template <>
struct __align__(1024) DTiles<true> {
  uint8_t k8[DCfg<true>::kNS][kTile8];   // int8 tiles as loaded (128-byte swizzle)
  uint8_t v8[DCfg<true>::kNSV][kTile8];
  uint8_t v[2][kTile];                  // fp16 V operand tiles (two buffers)
};

template <bool I8>
struct __align__(1024) DSmem : DTiles<I8> {
  uint8_t qt[2][2 * kRowBox];   // per item slot: the group's query rows (int8: hi / lo rows), 16 x 128 fp16, swizzled
  uint8_t pt[2][2 * kRowBox];   // P^T buffers: 16 rows x 128 keys (fp16, swizzled)
  float red[2][4][kNR];         // cross-warp row max, double-buffered by tile parity
  float redl[4][kNR];           // cross-warp row sum
  float qpow[2][8];             // int8 cache, per item slot: 2^e of each query row
  DItem item[2];
  uint64_t kfull[DCfg<I8>::kNS], kempty[DCfg<I8>::kNS], vfull[DCfg<I8>::kNSV], vempty[DCfg<I8>::kNSV];
  uint64_t k16full[2], k16empty[2], v16full[2], v16empty[2];      // int8 cache: fp16 operand tiles
  uint64_t imap[2], qready[2], iready[2], iempty[2];   // item mapped / query rows / appended rows / slot free
  uint64_t s_full[2], s_free[2], p_full[2], p_free[2];
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem;
  int abort;
  int last;
};

__device__ __forceinline__ void named_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kSoft) : "memory"); }

// Named barrier of the softmax threads that also returns the OR of `v` over them.
__device__ __forceinline__ bool named_sync_or(bool v) {
  uint32_t r;
  asm volatile("{ .reg .pred p, q; setp.ne.u32 q, %1, 0; bar.red.or.pred p, 1, %2, q; selp.u32 %0, 1, 0, p; }"
               : "=r"(r)
               : "r"((uint32_t)v), "n"(kSoft)
               : "memory");
  return r != 0;
}

// Merge ticket with acquire-release ordering at GPU scope: after the named
// barrier, the release covers every softmax thread's partial stores, and the
// acquire makes the other splits' partials visible to the last one.
__device__ __forceinline__ unsigned ticket_acq_rel(unsigned* addr) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(addr) : "memory");
  return old;
}

__device__ __forceinline__ void fence_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

template <class SM>
__device__ __forceinline__ bool aborted(const SM& sm) {
  return *reinterpret_cast<const volatile int*>(&sm.abort) != 0;
}

template <class SM>
__device__ __forceinline__ void set_abort(const Params& p, SM& sm) {
  *reinterpret_cast<volatile int*>(&sm.abort) = 1;
  flag_status(p, GQA_DEVICE_TIMEOUT_BIT);
}

// Byte offset of element (row, col) in a [rows][128] fp16 matrix stored as two
// 64-column boxes of `box` bytes with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw_elem(uint32_t row, uint32_t col, uint32_t box) {
  return (col >> 6) * box + sw128_offset(row, (col & 63) >> 3) + (col & 7) * 2;
}

// ---------------------------------------------------------------- producer helpers

// Tiles of batch b (its key range [kstart, total) in 128-key tiles, for each
// KV head); 0 for a batch whose lengths are inconsistent.
__device__ __forceinline__ int batch_tiles(const Params& p, int b, int& past, int& total, int& off, bool flag_bad) {
  total = p.seqlens[b] + 1;
  past = batch_past(p, total);
  off = 0;
  if (past >= 0 && p.has_rotary && past + p.S > p.rotary_rows) {
    if (flag_bad) flag_status(p, GQA_DEVICE_BAD_ROTARY_BIT);
    past = -1;
  } else if (past < 0 && flag_bad) {
    flag_status(p, GQA_DEVICE_BAD_SEQLEN_BIT);
  }
  if (past < 0) return 0;
  // From here on in cache rows: a sliding-window cache keeps the most recent
  // rows at the front (row r holds absolute position off + r); else off = 0.
  const BatchRows br = batch_rows(p, total, past);
  off = br.off;
  past = br.keep;
  total = br.live;
  const int kstart = p.window >= 0 ? max(0, past - p.window) : 0;
  return (total - kstart + kKT - 1) / kKT;
}

// Work units of a (b, g) with `tiles` tiles: one per tile plus kEndUnits for
// the end of its key range (the epilogue that writes the output or a partial
// costs about as much as that many tiles). Shares are equal in units, so a
// CTA that ends more key ranges gets fewer tiles. (A weight of 2 measured
// 56.4-56.6 us against 54.4-55.4 with 5 on the fp16 B=16, C=8192 decode.)
constexpr int kEndUnits = 5;
__device__ __forceinline__ long long bg_units(int tiles) { return tiles > 0 ? tiles + kEndUnits : 0; }

// Number of work units over all (b, g) (whole warp).
__device__ long long count_units(const Params& p, bool flag_bad) {
  const int lane = threadIdx.x & 31;
  long long n = 0;
  for (int b = lane; b < p.B; b += 32) {
    int past, total, off;
    n += bg_units(batch_tiles(p, b, past, total, off, flag_bad)) * p.Nkv;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  return n;
}

// CTA owning global unit t when `ntot` units are shared by `nc` <= ntot CTAs
// (CTA c owns [c*ntot/nc, (c+1)*ntot/nc), never empty).
__device__ __forceinline__ long long share_start(long long c, long long ntot, long long nc) { return c * ntot / nc; }
__device__ __forceinline__ int tile_owner(long long t, long long ntot, long long nc) {
  return (int)(((t + 1) * nc - 1) / ntot);
}

// The segment that starts at global unit t and ends at min(tend, last tile of
// its (b, g)), with a warp-wide prefix scan of the per-batch unit counts. A
// unit past the last tile of its (b, g) gives end = 2 and, in ntiles, the
// units to skip to the next (b, g).
__device__ void map_segment(const Params& p, long long t, long long tend, long long ntot, long long nc,
                            DItem& it) {
  const int lane = threadIdx.x & 31;
  long long base = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    int past = -1, total = 0, off = 0, tb = 0;
    if (b < p.B) tb = batch_tiles(p, b, past, total, off, false);
    const long long n = bg_units(tb) * p.Nkv;
    long long incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const long long excl = base + incl - n;
    const unsigned ballot = __ballot_sync(0xffffffffu, n > 0 && t >= excl && t < excl + n);
    if (ballot) {
      const int src = __ffs(ballot) - 1;
      const int pp = __shfl_sync(0xffffffffu, past, src);
      const int tt = __shfl_sync(0xffffffffu, total, src);
      const int tiles = __shfl_sync(0xffffffffu, tb, src);
      const long long r = t - __shfl_sync(0xffffffffu, excl, src);
      const int blk = (int)bg_units(tiles);
      it.b = __shfl_sync(0xffffffffu, b, src);
      it.g = (int)(r / blk);
      const int lt = (int)(r % blk);
      if (lt >= tiles) {   // end units of the (b, g): nothing to load
        it.end = 2;
        it.ntiles = blk - lt;
        return;
      }
      const long long first = t - lt, bg_end = first + tiles;
      const long long seg_end = tend < bg_end ? tend : bg_end;
      const int kstart = p.window >= 0 ? max(0, pp - p.window) : 0;
      it.past = pp;
      it.total = tt;
      it.off = __shfl_sync(0xffffffffu, off, src);
      it.j0 = kstart + lt * kKT;
      it.jend = min(tt, kstart + (int)(seg_end - first) * kKT);
      it.ntiles = (int)(seg_end - t);
      it.last = seg_end == bg_end;
      it.cfirst = tile_owner(first, ntot, nc);
      it.nsplit = tile_owner(bg_end - 1, ntot, nc) - it.cfirst + 1;
      it.split = (int)blockIdx.x - it.cfirst;
      it.slot0 = 2 * it.cfirst + (share_start(it.cfirst, ntot, nc) != first ? 1 : 0);
      it.slot = it.split == 0 ? it.slot0 : 2 * (int)blockIdx.x;
      it.end = 0;
      return;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  it.end = 1;   // not reached for t < ntot
}

// Rows of H = 128 values, eight lanes per row and four rows per warp pass:
// lane part l8 = lane & 7 holds dims 8*l8 .. 8*l8+7 (lo) and 64+8*l8 ..
// 64+8*l8+7 (hi), so the NeoX rotary partner of every value is in the same
// lane and each half is one 16-byte chunk (fp16) or two (fp32).
__device__ __forceinline__ void h8_to_f(const uint4& u, float* f) {
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 v = __half22float2(h[k]);
    f[2 * k] = v.x;
    f[2 * k + 1] = v.y;
  }
}

__device__ __forceinline__ void load8f(const float* src, float* f) {
  const float4 a = *reinterpret_cast<const float4*>(src);
  const float4 c = *reinterpret_cast<const float4*>(src + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = c.x; f[5] = c.y; f[6] = c.z; f[7] = c.w;
}

__device__ __forceinline__ uint4 f_to_h8(const float* f) {
  uint4 u;
  __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
  for (int k = 0; k < 4; ++k) h[k] = __floats2half2_rn(f[2 * k], f[2 * k + 1]);
  return u;
}

__device__ __forceinline__ uint4 f_to_h8(const float* f, float scale) {
  uint4 u;
  __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
  for (int k = 0; k < 4; ++k) h[k] = __floats2half2_rn(f[2 * k] * scale, f[2 * k + 1] * scale);
  return u;
}

// RMS norm (weights w) and / or rotary (cos c, sin s) of one row held as lo /
// hi halves; the row's 8 lanes reduce together (every lane must call).
__device__ __forceinline__ void norm_rope8(const Params& p, float* lo, float* hi, const float* wlo, const float* whi,
                                           bool norm, bool rope, const float* c, const float* sv) {
  if (norm) {
    // The stored-row fp32 recipe: lane l8 holds groups 2 l8, 2 l8 + 1 (lo) and
    // 16 + 2 l8, 17 + 2 l8 (hi); xor distances 1, 2, 4 build the subtrees of
    // the two halves, which are added last.
    float slo = sumsq8_rn(lo), shi = sumsq8_rn(hi);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      slo = __fadd_rn(slo, __shfl_xor_sync(0xffffffffu, slo, o));
      shi = __fadd_rn(shi, __shfl_xor_sync(0xffffffffu, shi, o));
    }
    const float rn = rms_inv_rn(__fadd_rn(slo, shi), kHD, p.eps);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      lo[k] = norm_rn(lo[k], rn, wlo[k]);
      hi[k] = norm_rn(hi[k], rn, whi[k]);
    }
  }
  if (rope) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float a = lo[k], b = hi[k];
      lo[k] = rope_first_rn(a, b, c[k], sv[k]);
      hi[k] = rope_second_rn(b, a, c[k], sv[k]);
    }
  }
}

// The group's query rows of an item as fp16 MMA operand rows (scaled into the
// log2 domain unless softcap). Rows >= R stay zero from the kernel start.
__device__ void prepare_qt_f16(const Params& p, const DItem& it, uint8_t* qt) {
  const int lane = threadIdx.x & 31, l8 = lane & 7, sub = lane >> 3;
  const int rows = p.S * p.G;
  const float qscale = p.softcap > 0.f ? p.scale : p.scale * kLog2e;
  const __half* q = reinterpret_cast<const __half*>(p.q);
  float wlo[8], whi[8];
  if (p.has_norm) {
    const __half* w = reinterpret_cast<const __half*>(p.qw);
    h8_to_f(*reinterpret_cast<const uint4*>(w + 8 * l8), wlo);
    h8_to_f(*reinterpret_cast<const uint4*>(w + 64 + 8 * l8), whi);
  }
#pragma unroll 1
  for (int r0 = 0; r0 < rows; r0 += 4) {
    const int r = min(r0 + sub, rows - 1);   // lanes past the last row redo it and do not store
    const int i = r / p.G, h = it.g * p.G + r % p.G;
    const __half* src = q + ((long long)(it.b * p.S + i) * p.N + h) * kHD;
    const uint4 xl = *reinterpret_cast<const uint4*>(src + 8 * l8);
    const uint4 xh = *reinterpret_cast<const uint4*>(src + 64 + 8 * l8);
    uint4 cs, sn;
    if (p.has_rotary) {
      const long long cb = (long long)(it.past + it.off + i) * (kHD / 2) + 8 * l8;   // absolute position
      cs = *reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(p.cos_c) + cb);
      sn = *reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(p.sin_c) + cb);
    }
    float lo[8], hi[8], c[8], sv[8];
    h8_to_f(xl, lo);
    h8_to_f(xh, hi);
    if (p.has_rotary) {
      h8_to_f(cs, c);
      h8_to_f(sn, sv);
    }
    norm_rope8(p, lo, hi, wlo, whi, p.has_norm, p.has_rotary, c, sv);
    if (r0 + sub < rows) {
      *reinterpret_cast<uint4*>(qt + sw128_offset(r, l8)) = f_to_h8(lo, qscale);
      *reinterpret_cast<uint4*>(qt + kRowBox + sw128_offset(r, l8)) = f_to_h8(hi, qscale);
    }
  }
}

// Append the new rows of (b, g) that fall in the segment's keys to the
// present cache (K: norm, rotary; V: as given; fp16). Prompt padding rows
// (past the total length) go with the segment that holds the last tile. One
// pass handles four (row, K or V) pairs.
__device__ void append_rows_f16(const Params& p, const DItem& it) {
  const int lane = threadIdx.x & 31, l8 = lane & 7, sub = lane >> 3;
  float wlo[8], whi[8];
  if (p.has_norm) {
    const __half* w = reinterpret_cast<const __half*>(p.kw);
    h8_to_f(*reinterpret_cast<const uint4*>(w + 8 * l8), wlo);
    h8_to_f(*reinterpret_cast<const uint4*>(w + 64 + 8 * l8), whi);
  }
  const int n = 2 * p.S;   // pair x: row i = x / 2, K for even x, V for odd x
#pragma unroll 1
  for (int x0 = 0; x0 < n; x0 += 4) {
    const int x = min(x0 + sub, n - 1);
    const int i = x >> 1, j = it.past + i;
    const bool is_k = (x & 1) == 0;
    const bool mine = (x0 + sub < n) && (j < it.total ? (j >= it.j0 && j < it.jend) : it.last != 0);
    const long long src = ((long long)(it.b * p.S + i) * p.Nkv + it.g) * kHD;
    const __half* base = reinterpret_cast<const __half*>(is_k ? p.k : p.v) + src;
    const uint4 xl = *reinterpret_cast<const uint4*>(base + 8 * l8);
    const uint4 xh = *reinterpret_cast<const uint4*>(base + 64 + 8 * l8);
    uint4 cs, sn;
    const bool rope = is_k && p.has_rotary;
    if (rope) {
      const long long cb = (long long)(j + it.off) * (kHD / 2) + 8 * l8;   // absolute position
      cs = *reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(p.cos_c) + cb);
      sn = *reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(p.sin_c) + cb);
    }
    float lo[8], hi[8], c[8], sv[8];
    h8_to_f(xl, lo);
    h8_to_f(xh, hi);
    // K and V rows of a pass may sit in one 8-lane group's neighbours: every
    // lane takes part in the norm's shuffles; V rows ignore the result.
    float klo[8], khi[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      klo[k] = lo[k];
      khi[k] = hi[k];
    }
    norm_rope8(p, klo, khi, wlo, whi, p.has_norm, false, c, sv);
    if (is_k && p.has_norm) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        lo[k] = klo[k];
        hi[k] = khi[k];
      }
    }
    if (rope) {
      h8_to_f(cs, c);
      h8_to_f(sn, sv);
      norm_rope8(p, lo, hi, wlo, whi, false, true, c, sv);
    }
    if (mine) {
      __half* dst = reinterpret_cast<__half*>(is_k ? p.present_k : p.present_v) +
                    (((long long)it.b * p.Nkv + it.g) * p.C + j) * kHD;
      *reinterpret_cast<uint4*>(dst + 8 * l8) = f_to_h8(lo, 1.f);
      *reinterpret_cast<uint4*>(dst + 64 + 8 * l8) = f_to_h8(hi, 1.f);
    }
  }
}

// Output value of row r, dim d from (m, l, o): sink / smooth-softmax term, 1/l, fp16.
__device__ __forceinline__ void write_out_f16(const Params& p, int b, int g, int total, int r, int d, float m, float l,
                                          float o) {
  const int i = r / p.G, h = g * p.G + r % p.G;
  const long long oi = ((long long)(b * p.S + i) * p.N + h) * kHD + d;
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
  reinterpret_cast<__half*>(p.out)[oi] = __float2half_rn(val);
}

// The group's query rows of an item: q' = rotary(norm(q)) * scale (log2
// domain unless softcap) * K channel scale, times 2^-e with 2^e the power of
// two at or below the row's largest |q'|; hi = fp16(q' 2^-e) goes to MMA row
// r, lo = fp16(q' 2^-e - hi) to row r + R. Rows >= 2R stay zero.
__device__ void prepare_qt_i8(const Params& p, const DItem& it, int R, uint8_t* qt, float* qpow) {
  const int lane = threadIdx.x & 31, l8 = lane & 7, sub = lane >> 3;
  const int rows = p.S * p.G;
  const float qscale = p.softcap > 0.f ? p.scale : p.scale * kLog2e;
  const float* q = reinterpret_cast<const float*>(p.q);
  float wlo[8], whi[8], kslo[8], kshi[8];
  if (p.has_norm) {
    load8f(reinterpret_cast<const float*>(p.qw) + 8 * l8, wlo);
    load8f(reinterpret_cast<const float*>(p.qw) + 64 + 8 * l8, whi);
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    kslo[k] = channel_scale(p.k_scale, p.k_scale_n, it.g * kHD + 8 * l8 + k);
    kshi[k] = channel_scale(p.k_scale, p.k_scale_n, it.g * kHD + 64 + 8 * l8 + k);
  }
#pragma unroll 1
  for (int r0 = 0; r0 < rows; r0 += 4) {
    const int r = min(r0 + sub, rows - 1);   // lanes past the last row redo it and do not store
    const int i = r / p.G, h = it.g * p.G + r % p.G;
    const float* src = q + ((long long)(it.b * p.S + i) * p.N + h) * kHD;
    float lo[8], hi[8], c[8], sv[8];
    load8f(src + 8 * l8, lo);
    load8f(src + 64 + 8 * l8, hi);
    if (p.has_rotary) {
      const long long cb = (long long)(it.past + it.off + i) * (kHD / 2) + 8 * l8;   // absolute position
      load8f(reinterpret_cast<const float*>(p.cos_c) + cb, c);
      load8f(reinterpret_cast<const float*>(p.sin_c) + cb, sv);
    }
    norm_rope8(p, lo, hi, wlo, whi, p.has_norm, p.has_rotary, c, sv);
    float mx = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      lo[k] = lo[k] * qscale * kslo[k];
      hi[k] = hi[k] * qscale * kshi[k];
      mx = fmaxf(mx, fmaxf(fabsf(lo[k]), fabsf(hi[k])));
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    // 2^e <= mx < 2^(e+1) from the exponent bits (mx = 0 or subnormal: e = 0).
    const int ebits = (__float_as_int(mx) >> 23) & 0xff;
    const int e = ebits == 0 ? 0 : ebits - 127;
    const float down = __int_as_float((127 - e) << 23), up = __int_as_float((127 + e) << 23);
    float hl[8], hh[8], ll[8], lh[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float a = lo[k] * down, b = hi[k] * down;
      hl[k] = __half2float(__float2half_rn(a));
      hh[k] = __half2float(__float2half_rn(b));
      ll[k] = a - hl[k];
      lh[k] = b - hh[k];
    }
    if (r0 + sub < rows) {
      *reinterpret_cast<uint4*>(qt + sw128_offset(r, l8)) = f_to_h8(hl);
      *reinterpret_cast<uint4*>(qt + kRowBox + sw128_offset(r, l8)) = f_to_h8(hh);
      *reinterpret_cast<uint4*>(qt + sw128_offset(r + R, l8)) = f_to_h8(ll);
      *reinterpret_cast<uint4*>(qt + kRowBox + sw128_offset(r + R, l8)) = f_to_h8(lh);
      if (l8 == 0) qpow[r] = up;
    }
  }
}

// Eight int8 codes (clamp(rint(x / scale), -127, 127), IEEE division) as one 8-byte word.
__device__ __forceinline__ uint2 quant8(const float* x, const float* sc) {
  uint2 u;
  int8_t* b = reinterpret_cast<int8_t*>(&u);
#pragma unroll
  for (int k = 0; k < 8; ++k) b[k] = quant_i8(x[k], sc[k]);
  return u;
}

// Append the new rows of (b, g) that fall in the segment's keys to the
// present cache as int8 codes (K: norm, rotary, then k_scale; V: v_scale).
// Prompt padding rows (past the total length) go with the segment that holds
// the last tile. One pass handles four (row, K or V) pairs.
__device__ void append_rows_i8(const Params& p, const DItem& it) {
  const int lane = threadIdx.x & 31, l8 = lane & 7, sub = lane >> 3;
  float wlo[8], whi[8];
  if (p.has_norm) {
    load8f(reinterpret_cast<const float*>(p.kw) + 8 * l8, wlo);
    load8f(reinterpret_cast<const float*>(p.kw) + 64 + 8 * l8, whi);
  }
  const int n = 2 * p.S;   // pair x: row i = x / 2, K for even x, V for odd x
#pragma unroll 1
  for (int x0 = 0; x0 < n; x0 += 4) {
    const int x = min(x0 + sub, n - 1);
    const int i = x >> 1, j = it.past + i;
    const bool is_k = (x & 1) == 0;
    const bool mine = (x0 + sub < n) && (j < it.total ? (j >= it.j0 && j < it.jend) : it.last != 0);
    const float* base = reinterpret_cast<const float*>(is_k ? p.k : p.v) +
                        ((long long)(it.b * p.S + i) * p.Nkv + it.g) * kHD;
    float lo[8], hi[8], c[8], sv[8];
    load8f(base + 8 * l8, lo);
    load8f(base + 64 + 8 * l8, hi);
    const bool rope = is_k && p.has_rotary;
    if (rope) {
      const long long cb = (long long)(j + it.off) * (kHD / 2) + 8 * l8;   // absolute position
      load8f(reinterpret_cast<const float*>(p.cos_c) + cb, c);
      load8f(reinterpret_cast<const float*>(p.sin_c) + cb, sv);
    }
    // Every lane takes part in the norm's shuffles; V rows keep their values.
    float klo[8], khi[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      klo[k] = lo[k];
      khi[k] = hi[k];
    }
    norm_rope8(p, klo, khi, wlo, whi, p.has_norm, false, c, sv);
    if (is_k && p.has_norm) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        lo[k] = klo[k];
        hi[k] = khi[k];
      }
    }
    if (rope) norm_rope8(p, lo, hi, wlo, whi, false, true, c, sv);
    if (mine) {
      const float* scp = is_k ? p.k_scale : p.v_scale;
      const int nsc = is_k ? p.k_scale_n : p.v_scale_n;
      float slo[8], shi[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        slo[k] = channel_scale(scp, nsc, it.g * kHD + 8 * l8 + k);
        shi[k] = channel_scale(scp, nsc, it.g * kHD + 64 + 8 * l8 + k);
      }
      int8_t* dst = reinterpret_cast<int8_t*>(is_k ? p.present_k : p.present_v) +
                    (((long long)it.b * p.Nkv + it.g) * p.C + j) * kHD;
      *reinterpret_cast<uint2*>(dst + 8 * l8) = quant8(lo, slo);
      *reinterpret_cast<uint2*>(dst + 64 + 8 * l8) = quant8(hi, shi);
    }
  }
}

// One int8 tile (128 rows x 128 codes, 128-byte swizzle as TMA wrote it) as
// the fp16 operand tile (two 64-column boxes, 128-byte swizzle). Converter
// thread t takes row t. int8 -> fp16 without the conversion unit: the byte
// c+128 as the low mantissa bits of 1024.0 (fp16 0x6400) is 1152 + c exactly.
__device__ __forceinline__ void convert_tile(const uint8_t* src, uint8_t* dst, int t) {
  const __half2 bias = __floats2half2_rn(1152.f, 1152.f);
#pragma unroll
  for (int c = 0; c < 8; ++c) {   // 16-byte chunk c: codes 16c .. 16c+15
    const uint4 w = *reinterpret_cast<const uint4*>(src + sw128_offset(t, c));
    const uint32_t wv[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t p01 = __byte_perm(wv[k], 0x64646464u, 0x4140u);
      const uint32_t p23 = __byte_perm(wv[k], 0x64646464u, 0x4342u);
      const __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&p01), bias);
      const __half2 b2 = __hsub2(*reinterpret_cast<const __half2*>(&p23), bias);
      h[2 * k] = *reinterpret_cast<const uint32_t*>(&a);
      h[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    const int col = 16 * c, bx = col >> 6, ch = (col & 63) >> 3;
    *reinterpret_cast<uint4*>(dst + bx * kBox + sw128_offset(t, ch)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(dst + bx * kBox + sw128_offset(t, ch + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// Eight int8 codes (one 16-byte chunk, xor 0x80 applied by the caller's
// load) as eight fp16 values in four 32-bit words: the byte c + 128 as the low
// mantissa bits of 1024.0 (fp16 0x6400) is 1152 + c exactly.
__device__ __forceinline__ void codes_to_h8(uint32_t w0, uint32_t w1, uint32_t* h) {
  const __half2 bias = __floats2half2_rn(1152.f, 1152.f);
  const uint32_t wv[2] = {w0 ^ 0x80808080u, w1 ^ 0x80808080u};
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint32_t p01 = __byte_perm(wv[k], 0x64646464u, 0x4140u);
    const uint32_t p23 = __byte_perm(wv[k], 0x64646464u, 0x4342u);
    const __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&p01), bias);
    const __half2 b2 = __hsub2(*reinterpret_cast<const __half2*>(&p23), bias);
    h[2 * k] = *reinterpret_cast<const uint32_t*>(&a);
    h[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&b2);
  }
}

// One converter step: row t of the int8 K tile `ksrc` into fp16 pairs in 64
// tensor-memory columns of this thread's lane, and (when `vsrc` is not null)
// row t of the int8 V tile of the previous tile into the fp16 operand tile
// `vdst`. The loads of both rows are issued together, half a row at a time,
// so the two conversions overlap instead of running one after the other.
__device__ __forceinline__ void convert_kv_rows(const uint8_t* ksrc, const uint8_t* vsrc, uint8_t* vdst, int t,
                                                uint32_t taddr) {
#pragma unroll
  for (int hlf = 0; hlf < 2; ++hlf) {
    uint4 kw[4], vw[4];
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) kw[c4] = *reinterpret_cast<const uint4*>(ksrc + sw128_offset(t, 4 * hlf + c4));
    if (vsrc) {
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) vw[c4] = *reinterpret_cast<const uint4*>(vsrc + sw128_offset(t, 4 * hlf + c4));
    }
    uint32_t h[32];
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      codes_to_h8(kw[c4].x, kw[c4].y, h + 8 * c4);
      codes_to_h8(kw[c4].z, kw[c4].w, h + 8 * c4 + 4);
    }
    tmem_st32(taddr + 32 * hlf, h);
    if (vsrc) {
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {   // chunk c: codes 16c .. 16c+15 -> fp16 columns 16c ..
        uint32_t v[8];
        codes_to_h8(vw[c4].x, vw[c4].y, v);
        codes_to_h8(vw[c4].z, vw[c4].w, v + 4);
        const int col = 16 * (4 * hlf + c4), bx = col >> 6, ch = (col & 63) >> 3;
        *reinterpret_cast<uint4*>(vdst + bx * kBox + sw128_offset(t, ch)) = make_uint4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<uint4*>(vdst + bx * kBox + sw128_offset(t, ch + 1)) = make_uint4(v[4], v[5], v[6], v[7]);
      }
    }
  }
}

// Output value of row r, dim d from (m, l, o): sink / smooth-softmax term, 1/l, fp32.
__device__ __forceinline__ void write_out_i8(const Params& p, int b, int g, int total, int r, int d, float m, float l,
                                          float o) {
  const int i = r / p.G, h = g * p.G + r % p.G;
  const long long oi = ((long long)(b * p.S + i) * p.N + h) * kHD + d;
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
  reinterpret_cast<float*>(p.out)[oi] = val;
}

// ---------------------------------------------------------------- the kernel

// I8: int8 cache with fp32 queries (converter warps, hi / lo operand rows);
// otherwise fp16. R: query rows of a KV head, padded to a power of two.
// kPlain: no softcap and no bias (the tile loop has no code for them).
template <bool I8, int R, bool kPlain>
__global__ void __launch_bounds__(DCfg<I8>::kThreads, 1)
decode_tc_kernel(const Params p, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  constexpr int kNS = DCfg<I8>::kNS, kNSV = DCfg<I8>::kNSV, kThreads = DCfg<I8>::kThreads;
  extern __shared__ uint8_t smem_raw[];
  DSmem<I8>& sm =
      *reinterpret_cast<DSmem<I8>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // The preparer's first global loads overlap the set-up below.
  long long ntot = 0;
  if (warp == 2) ntot = count_units(p, blockIdx.x == 0);
  if (warp == 1) tmem_alloc(&sm.tmem, DCfg<I8>::kTmemCols);
  if (tid == 0) {
    // A K / V stage is released by an MMA commit (fp16) or by every
    // converter thread once it has read its row (int8).
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&sm.kfull[s], 1);
      mbar_init(&sm.kempty[s], I8 ? kConv : 1);
    }
    for (int s = 0; s < kNSV; ++s) {
      mbar_init(&sm.vfull[s], 1);
      mbar_init(&sm.vempty[s], I8 ? kConv : 1);
    }
    if constexpr (I8) {
      for (int s = 0; s < 2; ++s) {
        mbar_init(&sm.k16full[s], kConv);
        mbar_init(&sm.k16empty[s], 1);     // MMA commit after S
        mbar_init(&sm.v16full[s], kConv);
        mbar_init(&sm.v16empty[s], 1);     // MMA commit after P.V
      }
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.imap[s], 1);
      mbar_init(&sm.qready[s], 1);
      mbar_init(&sm.iready[s], 1);
      mbar_init(&sm.iempty[s], 2);  // MMA commit (Q^T reads done) + softmax release
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.s_free[s], kSoft / 32);   // one arrival per softmax warp
      mbar_init(&sm.p_full[s], kSoft / 32);
      mbar_init(&sm.p_free[s], 1);
    }
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    sm.last = 0;
    mbar_fence_init();
  }
  // Query / probability rows >= R are zero for the whole kernel.
  for (int x = tid; x < (int)(2 * 2 * kRowBox / 16); x += kThreads) {
    reinterpret_cast<uint4*>(&sm.qt[0][0])[x] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(&sm.pt[0][0])[x] = make_uint4(0, 0, 0, 0);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;

  if (warp == 2) {
    // ================================================================ preparer
    // With fewer tiles than CTAs only the first `ntot` CTAs work, so that
    // every working CTA's share is non-empty and the CTAs sharing a (b, g)
    // are consecutive.
    const long long nc = ntot < (long long)gridDim.x ? ntot : (long long)gridDim.x;
    long long t = 0, tend = 0;
    if ((long long)blockIdx.x < nc) {
      t = share_start(blockIdx.x, ntot, nc);
      tend = share_start(blockIdx.x + 1, ntot, nc);
    }
    int slot = 0;
    uint32_t iphase[2] = {0, 0};
    bool ok = true;
    while (true) {
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.iempty[slot], iphase[slot] ^ 1u, p.wait_budget)) || aborted(sm)) {
        ok = false;
        break;
      }
      DItem it;
      it.end = 1;
      while (t < tend) {
        map_segment(p, t, tend, ntot, nc, it);
        if (it.end != 2) break;
        t += it.ntiles;
        it.end = 1;
      }
      if (t >= tend) {
        if (lane == 0) {
          sm.item[slot].end = 1;
          mbar_arrive(&sm.imap[slot]);
          mbar_arrive(&sm.qready[slot]);
          mbar_arrive(&sm.iready[slot]);
        }
        break;
      }
      if (it.end) {   // unreachable: every t < ntot maps to a unit
        ok = false;
        break;
      }
      t += it.ntiles;
      // The TMA warp may stream the segment's cached tiles while the query
      // rows are prepared; tiles holding new rows wait for `iready`.
      if (lane == 0) {
        sm.item[slot] = it;
        mbar_arrive(&sm.imap[slot]);
      }
      if constexpr (I8)
        prepare_qt_i8(p, it, R, sm.qt[slot], sm.qpow[slot]);
      else
        prepare_qt_f16(p, it, sm.qt[slot]);
      fence_async_smem();   // query rows (shared) -> async proxy: the MMAs may start
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.qready[slot]);
      if constexpr (I8)
        append_rows_i8(p, it);
      else
        append_rows_f16(p, it);
      fence_async_all();  // appended rows (global) -> async proxy: the TMA may load their tile
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.iready[slot]);
      iphase[slot] ^= 1u;
      slot ^= 1;
    }
    if (!ok && lane == 0) set_abort(p, sm);
  } else if (warp == 0) {
    // ================================================================ TMA
    // K and V tiles have their own stages: K(u) is released as soon as
    // S(u) is done, V(u) after O += V P(u).
    int slot = 0, tau = 0, nk = 0, nv = 0;   // tiles begun; K and V fills issued
    uint32_t iphase[2] = {0, 0};
    bool ok = true, withheld = false;
    while (ok) {
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.imap[slot], iphase[slot], p.wait_budget))) {
        ok = false;
        break;
      }
      const DItem it = sm.item[slot];
      if (it.end) break;
      const int row0 = (it.b * p.Nkv + it.g) * p.C + it.j0;
      bool ready = false;
      for (int t = 0; t < it.ntiles; ++t, ++tau) {
        const int st = tau % kNS, sv = tau % kNSV;
        const uint32_t par = ((uint32_t)(tau / kNS) & 1u) ^ 1u, parv = ((uint32_t)(tau / kNSV) & 1u) ^ 1u;
        if (tau == p.withhold_tile) {   // testing: no copy of this tile, its waits expire
          withheld = true;
          ok = false;
          break;
        }
        if (!ready && it.j0 + (t + 1) * kKT > it.past) {   // the tile holds new rows
          if (!__all_sync(0xffffffffu, mbar_wait(&sm.iready[slot], iphase[slot], p.wait_budget))) {
            ok = false;
            break;
          }
          ready = true;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.kempty[st], par, p.wait_budget)) || aborted(sm)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          if constexpr (I8) {
            mbar_arrive_tx(&sm.kfull[st], kTile8);
            tma_load_2d(sm.k8[st], &tmk, 0, row0 + t * kKT, &sm.kfull[st]);
          } else {
            mbar_arrive_tx(&sm.kfull[st], kTile);
            tma_load_2d(sm.k[st], &tmk, 0, row0 + t * kKT, &sm.kfull[st]);
            tma_load_2d(sm.k[st] + kBox, &tmk, 64, row0 + t * kKT, &sm.kfull[st]);
          }
        }
        __syncwarp();
        ++nk;
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.vempty[sv], parv, p.wait_budget)) || aborted(sm)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          if constexpr (I8) {
            mbar_arrive_tx(&sm.vfull[sv], kTile8);
            tma_load_2d(sm.v8[sv], &tmv, 0, row0 + t * kKT, &sm.vfull[sv]);
          } else {
            mbar_arrive_tx(&sm.vfull[sv], kTile);
            tma_load_2d(sm.v[sv], &tmv, 0, row0 + t * kKT, &sm.vfull[sv]);
            tma_load_2d(sm.v[sv] + kBox, &tmv, 64, row0 + t * kKT, &sm.vfull[sv]);
          }
        }
        __syncwarp();
        ++nv;
      }
      iphase[slot] ^= 1u;
      slot ^= 1;
    }
    if (!ok && !withheld && lane == 0) set_abort(p, sm);
    // Drain: every fill this warp issued has landed before the CTA can exit
    // (older fills completed before their stage was refilled).
    for (int u = max(0, nk - kNS); u < nk; ++u) mbar_wait(&sm.kfull[u % kNS], (uint32_t)(u / kNS) & 1u, p.wait_budget);
    for (int u = max(0, nv - kNSV); u < nv; ++u) mbar_wait(&sm.vfull[u % kNSV], (uint32_t)(u / kNSV) & 1u, p.wait_budget);
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    int slot = 0, tau = 0;
    uint32_t iphase[2] = {0, 0};
    bool ok = true;
    // Shared-memory descriptors of every operand buffer, built once; a K step
    // adds its start-address offset (16-byte units) to the descriptor. V is
    // read from its TMA stage (fp16) or from its fp16 operand tile (int8), K
    // from its TMA stage (fp16) or from tensor memory (int8).
    constexpr int kVB = I8 ? 2 : kNSV;
    uint64_t dq[2], dp[2], dk[kNS], dv[kVB];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      dq[i] = desc_kmajor_sw128(smem_addr(sm.qt[i]));
      dp[i] = desc_kmajor_sw128(smem_addr(sm.pt[i]));
    }
    if constexpr (!I8) {
#pragma unroll
      for (int i = 0; i < kNS; ++i) dk[i] = desc_kmajor_sw128(smem_addr(sm.k[i]));
    }
#pragma unroll
    for (int i = 0; i < kVB; ++i) dv[i] = desc_mnmajor_sw128(smem_addr(sm.v[i]), kBox, 1024);
    auto issue_pv = [&](int u, bool acc) {
      const int pb = u & 1, vb = I8 ? pb : u % kNSV;
      const uint32_t vpar = I8 ? (uint32_t)(u >> 1) & 1u : (uint32_t)(u / kNSV) & 1u;
      uint64_t* vready = I8 ? &sm.v16full[vb] : &sm.vfull[vb];
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.p_full[pb], (uint32_t)(u >> 1) & 1u, p.wait_budget) &&
                                       mbar_wait(vready, vpar, p.wait_budget)))
        return false;
      if (elect_one()) {
        tc_fence_after();
        const uint64_t a0 = dv[vb], b0 = dp[pb];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_f16_ss(tmem + 32, a0 + (uint64_t)(ks * 128), b0 + (uint64_t)((ks >> 2) * 128 + (ks & 3) * 2), kIdO,
                     acc || ks > 0);
        mma_commit(&sm.p_free[pb]);
        mma_commit(I8 ? &sm.v16empty[vb] : &sm.vempty[vb]);
      }
      __syncwarp();
      return true;
    };
    while (ok) {
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.qready[slot], iphase[slot], p.wait_budget))) {
        ok = false;
        break;
      }
      const DItem it = sm.item[slot];
      if (it.end) break;
      for (int t = 0; t < it.ntiles && ok; ++t) {
        const int u = tau + t, sb = u & 1, kb = I8 ? u & 1 : u % kNS;
        const uint32_t kpar = I8 ? (uint32_t)(u >> 1) & 1u : (uint32_t)(u / kNS) & 1u;
        uint64_t* kready = I8 ? &sm.k16full[kb] : &sm.kfull[kb];
        if (!__all_sync(0xffffffffu, mbar_wait(kready, kpar, p.wait_budget) &&
                                         mbar_wait(&sm.s_free[sb], ((uint32_t)(u >> 1) & 1u) ^ 1u, p.wait_budget))) {
          ok = false;
          break;
        }
        if (elect_one()) {
          tc_fence_after();
          const uint64_t b0 = dq[slot];
          const uint32_t d = tmem + sb * 16;
          if constexpr (I8) {
            const uint32_t a0 = tmem + kKCol + kb * 64;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma_f16_ts(d, a0 + ks * 8, b0 + (uint64_t)((ks >> 2) * 128 + (ks & 3) * 2), kIdS, ks > 0);
          } else {
            const uint64_t a0 = dk[kb];
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma_f16_ss(d, a0 + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2),
                         b0 + (uint64_t)((ks >> 2) * 128 + (ks & 3) * 2), kIdS, ks > 0);
          }
          mma_commit(&sm.s_full[sb]);
          mma_commit(I8 ? &sm.k16empty[kb] : &sm.kempty[kb]);
        }
        __syncwarp();
        if (t > 0 && !issue_pv(u - 1, t - 1 > 0)) ok = false;
      }
      if (ok && it.ntiles > 0 && !issue_pv(tau + it.ntiles - 1, it.ntiles > 1)) ok = false;
      if (!ok) break;
      if (elect_one()) {
        mma_commit(&sm.o_full);
        mma_commit(&sm.iempty[slot]);
      }
      __syncwarp();
      tau += it.ntiles;
      iphase[slot] ^= 1u;
      slot ^= 1;
      if (__any_sync(0xffffffffu, aborted(sm))) ok = false;
    }
    if (!ok && lane == 0) set_abort(p, sm);
    if (elect_one()) {
      mma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, p.wait_budget);
    }
    __syncwarp();
  } else if (warp >= kConvWarp0) {   // int8 cache only (the fp16 form has no such warps)
    if constexpr (I8) {
      // ================================================================ converters
      // Row of the tile this thread converts = its tensor-memory lane.
      const int ct = (warp & 3) * 32 + lane;
      const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
      // K of tile u is converted before V of tile u - 1, so S(u) can be
      // issued while V(u - 1) is still being converted.
      auto convert_v = [&](int uv) {
        const int sv = uv % kNSV, vb = uv & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.vfull[sv], (uint32_t)(uv / kNSV) & 1u, p.wait_budget) &&
                                         mbar_wait(&sm.v16empty[vb], ((uint32_t)(uv >> 1) & 1u) ^ 1u, p.wait_budget)) ||
            aborted(sm))
          return false;
        convert_tile(sm.v8[sv], sm.v[vb], ct);
        fence_async_smem();
        mbar_arrive(&sm.v16full[vb]);
        mbar_arrive(&sm.vempty[sv]);
        return true;
      };
      int slot = 0, u = 0, uv = 0;   // tiles whose K / V are converted
      uint32_t iphase[2] = {0, 0};
      bool ok = true;
      while (ok) {
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.imap[slot], iphase[slot], p.wait_budget))) {
          ok = false;
          break;
        }
        const DItem it = sm.item[slot];
        if (it.end) break;
        for (int t = 0; t < it.ntiles; ++t, ++u) {
          // One step converts K(u) and V(u - 1) together (one set of waits,
          // one fence, interleaved loads).
          const int st = u % kNS, kb = u & 1;
          const bool with_v = uv < u;
          const int sv = uv % kNSV, vb = uv & 1;
          bool ready = mbar_wait(&sm.kfull[st], (uint32_t)(u / kNS) & 1u, p.wait_budget) &&
                       mbar_wait(&sm.k16empty[kb], ((uint32_t)(u >> 1) & 1u) ^ 1u, p.wait_budget);
          if (with_v)
            ready = ready && mbar_wait(&sm.vfull[sv], (uint32_t)(uv / kNSV) & 1u, p.wait_budget) &&
                    mbar_wait(&sm.v16empty[vb], ((uint32_t)(uv >> 1) & 1u) ^ 1u, p.wait_budget);
          if (!__all_sync(0xffffffffu, ready) || aborted(sm)) {
            ok = false;
            break;
          }
          convert_kv_rows(sm.k8[st], with_v ? sm.v8[sv] : nullptr, sm.v[vb], ct, tmem + lane_addr + kKCol + kb * 64);
          tmem_st_wait();
          tc_fence_before();
          if (with_v) fence_async_smem();
          mbar_arrive(&sm.k16full[kb]);
          mbar_arrive(&sm.kempty[st]);
          if (with_v) {
            mbar_arrive(&sm.v16full[vb]);
            mbar_arrive(&sm.vempty[sv]);
            ++uv;
          }
        }
        iphase[slot] ^= 1u;
        slot ^= 1;
      }
      while (ok && uv < u) {   // the last tile's V
        if (!convert_v(uv)) ok = false;
        ++uv;
      }
      if (!ok && lane == 0) set_abort(p, sm);
    }
  } else {
    // ================================================================ softmax
    // A warp leaves the loop only on a value reduced at a named barrier
    // (bar.red.or), so every softmax warp takes the same exit.
    const int quarter = warp & 3;
    const int kl = quarter * 32 + lane;           // tensor-memory lane: key of the tile, dim of O^T
    const int ws = warp - kSoftWarp0;             // softmax warp index 0..3
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const int rows = p.S * p.G;
    int slot = 0, tau = 0, icount = 0;
    uint32_t iphase[2] = {0, 0};
    while (true) {
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.qready[slot], iphase[slot], p.wait_budget)) && lane == 0) set_abort(p, sm);
      if (named_sync_or(aborted(sm))) break;   // one decision for every softmax warp
      const DItem it = sm.item[slot];
      if (it.end) break;
      const int b = it.b, g = it.g;
      int pos_r[R], ih_r[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int i = r < rows ? r / p.G : 0;
        pos_r[r] = it.past + i;
        ih_r[r] = r < rows ? i * p.N + g * p.G + r % p.G : -1;
      }
      float m_run[R], l_part[R], qp[R];   // qp: int8 cache, 2^e of each query row
#pragma unroll
      for (int r = 0; r < R; ++r) {
        m_run[r] = kNegBig;
        l_part[r] = 0.f;
        qp[r] = I8 && r < rows ? sm.qpow[slot][r] : 1.f;
      }
      // int8 cache: V channel scale of this thread's output dim (applied once to O).
      const float vsc = I8 ? channel_scale(p.v_scale, p.v_scale_n, g * kHD + kl) : 1.f;
      bool bad = false;
      for (int t = 0; t < it.ntiles; ++t) {
        const int u = tau + t, sb = u & 1, st = u % kNSV;
        const int jk = it.j0 + t * kKT + kl;      // this thread's key
        const bool key_ok = jk < it.jend;
        float s[R];
        bool grow_here = false;   // a visible score exceeds its row's reference by more than 2^kLazy
        bool got = __all_sync(0xffffffffu, mbar_wait(&sm.s_full[sb], (uint32_t)(u >> 1) & 1u, p.wait_budget));
        if (got) {
          tc_fence_after();
          uint32_t raw[16];
          tmem_ld16(tmem + lane_addr + sb * 16, raw);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.s_free[sb]);
          if constexpr (!I8) {
            // V rows past the key range may hold any bits: zero them (P is 0 there, 0 * NaN is not).
            // (int8 codes are finite.)
            if (!key_ok && !mbar_wait(&sm.vfull[st], (uint32_t)(u / kNSV) & 1u, p.wait_budget)) set_abort(p, sm);
            if (!key_ok && !aborted(sm)) {
#pragma unroll
              for (int bx = 0; bx < 2; ++bx)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                  *reinterpret_cast<uint4*>(sm.v[st] + bx * kBox + kl * 128 + c * 16) = make_uint4(0, 0, 0, 0);
            }
          }
#pragma unroll
          for (int r = 0; r < R; ++r) {
            float x = __uint_as_float(raw[r]);
            if constexpr (I8) x = (x + __uint_as_float(raw[r + R])) * qp[r];   // hi + lo rows
            bool vis = key_ok && ih_r[r] >= 0;
            if (p.causal) vis = vis && jk <= pos_r[r];
            if (p.window >= 0) vis = vis && jk >= pos_r[r] - p.window;
            if (!kPlain && p.softcap > 0.f) x = p.softcap * tanhf(x / p.softcap) * kLog2e;
            if (!kPlain && p.has_bias && vis) {
              const int i = ih_r[r] / p.N, h = ih_r[r] % p.N;
              const long long bi =
                  (((long long)(p.bias_bdim > 1 ? b : 0) * p.bias_ndim + (p.bias_ndim > 1 ? h : 0)) * p.S + i) *
                      p.bias_ld + jk + it.off;
              x += load_t(p.bias, bi, p.t_type) * kLog2e;
            }
            s[r] = vis ? x : -INFINITY;
            grow_here = grow_here || s[r] > m_run[r] + kLazy;
          }
        } else if (lane == 0) {
          set_abort(p, sm);
        }
        // One barrier tells every softmax thread whether any row needs a new
        // reference max (rare after an item's first tile).
        // The abort flag may be set by another warp role at any time, so the
        // softmax warps leave only on a value reduced at a barrier (the same
        // for all of them); the common case needs one barrier.
        const bool ab0 = aborted(sm);
        const bool any_grow = named_sync_or(grow_here || ab0);
        if (any_grow && named_sync_or(ab0)) {
          bad = true;
          break;
        }
        float mt[R];
        if (any_grow) {
#pragma unroll
          for (int r = 0; r < R; ++r) {
            float m = s[r];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) sm.red[sb][ws][r] = m;
          }
          named_sync();
#pragma unroll
          for (int r = 0; r < R; ++r)
            mt[r] = fmaxf(fmaxf(sm.red[sb][0][r], sm.red[sb][1][r]), fmaxf(sm.red[sb][2][r], sm.red[sb][3][r]));
        } else {
#pragma unroll
          for (int r = 0; r < R; ++r) mt[r] = m_run[r];
        }
        if (any_grow && t > 0) {
          // O^T must hold P.V up to tile t-1.
          const int pu = u - 1;
          if (__all_sync(0xffffffffu, mbar_wait(&sm.p_free[pu & 1], (uint32_t)(pu >> 1) & 1u, p.wait_budget))) {
            tc_fence_after();
            uint32_t o[16];
            tmem_ld16(tmem + lane_addr + 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int r = 0; r < R; ++r) {
              if (mt[r] > m_run[r] + kLazy) {
                const float f = ex2(m_run[r] - mt[r]);
                o[r] = __float_as_uint(__uint_as_float(o[r]) * f);
                if constexpr (I8) o[r + R] = __float_as_uint(__uint_as_float(o[r + R]) * f);
                l_part[r] *= f;
              }
            }
            tmem_st16(tmem + lane_addr + 32, o);
            tmem_st_wait();
          } else if (lane == 0) {
            set_abort(p, sm);
          }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (mt[r] > m_run[r] + kLazy) m_run[r] = mt[r];
        // P^T(u): its buffer is free once P.V(u-2) finished.
        if (__all_sync(0xffffffffu, mbar_wait(&sm.p_free[sb], ((uint32_t)(u >> 1) & 1u) ^ 1u, p.wait_budget))) {
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float pr = ex2(s[r] - m_run[r]);   // masked scores are -inf: 0
            l_part[r] += pr;
            const __half ph = __float2half_rn(pr);
            *reinterpret_cast<__half*>(sm.pt[sb] + sw_elem(r, kl, kRowBox)) = ph;
            if constexpr (I8)   // lo row
              *reinterpret_cast<__half*>(sm.pt[sb] + sw_elem(r + R, kl, kRowBox)) =
                  __float2half_rn(pr - __half2float(ph));
          }
        } else if (lane == 0) {
          set_abort(p, sm);
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[sb]);
      }
      if (bad) break;
      tau += it.ntiles;
      // ---- end of item: O^T row kl = dim kl of every query row
      const bool got = __all_sync(0xffffffffu, mbar_wait(&sm.o_full, (uint32_t)icount & 1u, p.wait_budget));
      uint32_t o[16];
      if (got) {
        tc_fence_after();
        tmem_ld16(tmem + lane_addr + 32, o);
        tmem_ld_wait();
        if constexpr (I8) {
#pragma unroll
          for (int r = 0; r < R; ++r)
            o[r] = __float_as_uint((__uint_as_float(o[r]) + __uint_as_float(o[r + R])) * vsc);
        }
      } else if (lane == 0) {
        set_abort(p, sm);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float l = l_part[r];
#pragma unroll
        for (int x = 16; x > 0; x >>= 1) l += __shfl_xor_sync(0xffffffffu, l, x);
        if (lane == 0) sm.redl[ws][r] = l;
      }
      if (named_sync_or(aborted(sm))) break;   // one decision for every softmax warp
      const int bg = b * p.Nkv + g;
      if (it.nsplit == 1) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (r >= rows) continue;
          const float l = sm.redl[0][r] + sm.redl[1][r] + sm.redl[2][r] + sm.redl[3][r];
          if constexpr (I8)
            write_out_i8(p, b, g, it.total, r, kl, m_run[r], l, __uint_as_float(o[r]));
          else
            write_out_f16(p, b, g, it.total, r, kl, m_run[r], l, __uint_as_float(o[r]));
        }
      } else {
        const long long pbase = (long long)it.slot * p.rows_pad;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (r >= rows) continue;
          p.part_o[(pbase + r) * kHD + kl] = __uint_as_float(o[r]);
          if (kl == 0) {
            p.part_ml[(pbase + r) * 2] = m_run[r];
            p.part_ml[(pbase + r) * 2 + 1] = sm.redl[0][r] + sm.redl[1][r] + sm.redl[2][r] + sm.redl[3][r];
          }
        }
        named_sync();
        if (tid == kSoftWarp0 * 32) {   // first softmax thread
          const unsigned ticket = ticket_acq_rel(&p.counters[bg]);
          sm.last = ticket == (unsigned)(it.nsplit - 1);
        }
        named_sync();
        if (sm.last) {
          // One pass over the splits (online merge); the loads of a split for
          // all rows are independent, so they are in flight together.
          float M[R], Ls[R], A[R];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            M[r] = kNegBig;
            Ls[r] = 0.f;
            A[r] = 0.f;
          }
          if constexpr (R > 4) {
            for (int s2 = 0; s2 < it.nsplit; ++s2) {
              const long long sb0 = (long long)(s2 == 0 ? it.slot0 : 2 * (it.cfirst + s2)) * p.rows_pad;
#pragma unroll
              for (int r = 0; r < R; ++r) {
                if (r >= rows) continue;
                const float m = __ldcg(&p.part_ml[(sb0 + r) * 2]);
                const float l = __ldcg(&p.part_ml[(sb0 + r) * 2 + 1]);
                const float ov = __ldcg(&p.part_o[(sb0 + r) * kHD + kl]);
                const float mn = fmaxf(M[r], m);
                const float fa = ex2(M[r] - mn), fb = ex2(m - mn);
                Ls[r] = Ls[r] * fa + l * fb;
                A[r] = A[r] * fa + ov * fb;
                M[r] = mn;
              }
            }
          } else {
            // Up to four rows: four splits per pass, their loads issued before any
            // is combined; more rows: one split per pass (register budget).
            constexpr int kMB = 4;
            for (int s0 = 0; s0 < it.nsplit; s0 += kMB) {
              float mv[kMB][R], lv[kMB][R], ovv[kMB][R];
#pragma unroll
              for (int k = 0; k < kMB; ++k) {
                const int s2 = min(s0 + k, it.nsplit - 1);   // a repeated split is not combined
                const long long sb0 = (long long)(s2 == 0 ? it.slot0 : 2 * (it.cfirst + s2)) * p.rows_pad;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                  if (r >= rows) continue;
                  mv[k][r] = __ldcg(&p.part_ml[(sb0 + r) * 2]);
                  lv[k][r] = __ldcg(&p.part_ml[(sb0 + r) * 2 + 1]);
                  ovv[k][r] = __ldcg(&p.part_o[(sb0 + r) * kHD + kl]);
                }
              }
#pragma unroll
              for (int k = 0; k < kMB; ++k) {
                if (s0 + k >= it.nsplit) break;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                  if (r >= rows) continue;
                  const float mn = fmaxf(M[r], mv[k][r]);
                  const float fa = ex2(M[r] - mn), fb = ex2(mv[k][r] - mn);
                  Ls[r] = Ls[r] * fa + lv[k][r] * fb;
                  A[r] = A[r] * fa + ovv[k][r] * fb;
                  M[r] = mn;
                }
              }
            }
          }
#pragma unroll
          for (int r = 0; r < R; ++r)
            if (r < rows) {
              if constexpr (I8)
                write_out_i8(p, b, g, it.total, r, kl, M[r], Ls[r], A[r]);
              else
                write_out_f16(p, b, g, it.total, r, kl, M[r], Ls[r], A[r]);
            }
          if (tid == kSoftWarp0 * 32) p.counters[bg] = 0;  // ready for the next call
        }
        named_sync();
        if (tid == kSoftWarp0 * 32) sm.last = 0;
      }
      named_sync();   // slot, reduction buffers and the ticket flag are free again
      if (tid == kSoftWarp0 * 32) mbar_arrive(&sm.iempty[slot]);
      iphase[slot] ^= 1u;
      slot ^= 1;
      ++icount;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, DCfg<I8>::kTmemCols);
}

// Per-device launch facts, looked up on the first launch on each device
// (racing first calls store the same values).
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
bool g_smem_set[2][10][kMaxDevices];

static_assert(sizeof(DSmem<false>) + 1024 <= 232448, "shared memory of one CTA");
static_assert(sizeof(DSmem<true>) + 1024 <= 232448, "shared memory of one CTA");

template <bool I8, int R, bool kPlain>
cudaError_t launch_rp(const Params& p, cudaStream_t st, const CUtensorMap& mk, const CUtensorMap& mv, int ri) {
  const int smem = (int)sizeof(DSmem<I8>) + 1024;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!g_smem_set[I8][ri][dev]) {
    e = cudaFuncSetAttribute(decode_tc_kernel<I8, R, kPlain>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    g_smem_set[I8][ri][dev] = true;
  }
  if (g_sm_count[dev] == 0) {
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    g_sm_count[dev] = sms;
  }
  const int sms = g_sm_count[dev];
  const int grid = sms < kTcDecodeMaxCtas ? sms : kTcDecodeMaxCtas;
  decode_tc_kernel<I8, R, kPlain><<<grid, DCfg<I8>::kThreads, smem, st>>>(p, mk, mv);
  return cudaGetLastError();
}

// Scores without softcap or bias take a kernel whose tile loop has no code
// for them.
template <bool I8, int R>
cudaError_t launch_r(const Params& p, cudaStream_t st, const CUtensorMap& mk, const CUtensorMap& mv, int ri) {
  if (p.softcap > 0.f || p.has_bias) return launch_rp<I8, R, false>(p, st, mk, mv, ri);
  return launch_rp<I8, R, true>(p, st, mk, mv, ri + 5);
}

}  // namespace

bool decode_tc_supported(const Params& p) {
  return p.t_type == kF16 && p.cache_type == kF16 && p.H == kHD && p.S * p.G <= kNR;
}

bool decode_tc_i8_supported(const Params& p) {
  return p.t_type == kF32 && p.cache_type == kI8 && p.H == kHD && 2 * p.S * p.G <= kNR;
}

cudaError_t prepare_decode_tc(const Params& p, TmaMaps* maps) {
  const long long krows = (long long)p.B * p.Nkv * p.C;
  cudaError_t e = encode_fp16_2d_sw128(&maps->m[0], p.present_k, (uint64_t)krows, kHD, kHD * 2, 64, kKT);
  if (e != cudaSuccess) return e;
  return encode_fp16_2d_sw128(&maps->m[1], p.present_v, (uint64_t)krows, kHD, kHD * 2, 64, kKT);
}

cudaError_t prepare_decode_tc_i8(const Params& p, TmaMaps* maps) {
  const long long krows = (long long)p.B * p.Nkv * p.C;
  cudaError_t e = encode_u8_2d_sw128(&maps->m[0], p.present_k, (uint64_t)krows, kHD, kHD, kHD, kKT);
  if (e != cudaSuccess) return e;
  return encode_u8_2d_sw128(&maps->m[1], p.present_v, (uint64_t)krows, kHD, kHD, kHD, kKT);
}

cudaError_t launch_decode_tc(const Params& p, cudaStream_t st, const TmaMaps& maps) {
  const CUtensorMap& mk = maps.m[0];
  const CUtensorMap& mv = maps.m[1];
  switch (p.rows_pad) {
    case 1: return launch_r<false, 1>(p, st, mk, mv, 0);
    case 2: return launch_r<false, 2>(p, st, mk, mv, 1);
    case 4: return launch_r<false, 4>(p, st, mk, mv, 2);
    case 8: return launch_r<false, 8>(p, st, mk, mv, 3);
    case 16: return launch_r<false, 16>(p, st, mk, mv, 4);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_tc_i8(const Params& p, cudaStream_t st, const TmaMaps& maps) {
  const CUtensorMap& mk = maps.m[0];
  const CUtensorMap& mv = maps.m[1];
  switch (p.rows_pad) {
    case 1: return launch_r<true, 1>(p, st, mk, mv, 0);
    case 2: return launch_r<true, 2>(p, st, mk, mv, 1);
    case 4: return launch_r<true, 4>(p, st, mk, mv, 2);
    case 8: return launch_r<true, 8>(p, st, mk, mv, 3);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gqa
