// CUDA-core flash prefill for GroupQueryAttention: float32 Q/K/V (including
// an int8 or 4-bit cache read back through its scales) and head sizes the
// tensor-core kernel does not take. Reads the prepared queries the pre-pass left in the
// workspace and the present cache after the append.
//
// com.microsoft.GroupQueryAttention, section Implementation variants
// (qkv_present_flash_cluster / past_kv_flash_prefill / new_kv_past_flash_prefill
// / quant_int8_flash_prefill / quant_int4_flash_prefill: online-softmax
// prefill over the cache as stored,
// causal bound right-aligned at the live length, window floor, softcap, bias
// and head sink) and sections Inputs / Attributes.
//
// CTA (row block, KV head g, batch b) takes 16 consecutive rows of the
// (position, grouped head) row list of its KV head, so every K/V tile staged
// in shared memory serves all grouped heads. Scores: one key per lane.
// P.V: each lane owns dims lane, lane+32, ... with the probabilities
// broadcast by warp shuffles.
#include "common.cuh"

namespace gqa {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRows = kWarps * kRowsPerWarp;
constexpr int kTile = 32;
constexpr int kMaxH = 256;

template <typename T, typename CacheT>
__global__ void __launch_bounds__(kWarps * 32)
prefill_simt_kernel(const Params p) {
  extern __shared__ float smem[];
  const int H = p.H, HP = H + 1;          // padded row stride: conflict-free column reads
  float* qs = smem;                        // [kRows][H]
  float* ks = qs + kRows * H;              // [kTile][HP]
  float* vs = ks + kTile * HP;             // [kTile][HP]

  const int rb = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int total = p.seqlens[b] + 1;
  const int past = batch_past(p, total);
  if (past < 0) {
    if (rb == 0 && g == 0 && tid == 0) flag_status(p, GQA_DEVICE_BAD_SEQLEN_BIT);
    return;
  }
  if (p.has_rotary && past + p.S > p.rotary_rows) return;  // flagged by the pre-pass
  const int nrows = p.S * p.G;
  const int r0 = rb * kRows;
  const int live_i = p.mode == kPrompt ? min(p.S, total) : p.S;  // rows i >= live_i are padding

  // Stage the prepared query rows (fp32, layout [B][N_kv][S*G][H]).
  const float* qp = reinterpret_cast<const float*>(p.qprep) + ((long long)(b * p.Nkv + g) * nrows) * H;
  for (int x = tid; x < kRows * H; x += kWarps * 32) {
    const int r = r0 + x / H;
    qs[x] = r < nrows ? qp[(long long)r * H + x % H] : 0.f;
  }
  // Key range of the block in cache rows: [kmin, kmax). Cache row j holds
  // absolute position off + j (off = 0 except for a sliding-window cache).
  const BatchRows br = batch_rows(p, total, past);
  const int off = br.off, past_row = past - off;
  const int i_lo = r0 / p.G;
  const int i_hi = min((min(r0 + kRows, nrows) - 1) / p.G, live_i - 1);
  int kmin = 0, kmax = br.live;
  if (p.causal) kmax = min(br.live, past_row + i_hi + 1);
  if (p.window >= 0) kmin = max(0, past_row + i_lo - p.window);

  const float qscale = p.softcap > 0.f ? p.scale : p.scale * kLog2e;
  float m[kRowsPerWarp], l[kRowsPerWarp], o[kRowsPerWarp][kMaxH / 32];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    m[rr] = kNegBig;
    l[rr] = 0.f;
#pragma unroll
    for (int e = 0; e < kMaxH / 32; ++e) o[rr][e] = 0.f;
  }
  // CacheT = uint8_t: 4-bit cache, H/2 bytes per row (+8-biased nibbles, even coordinate low).
  constexpr bool i4 = std::is_same<CacheT, uint8_t>::value;
  constexpr bool i8 = std::is_same<CacheT, int8_t>::value;
  const long long row_elems = i4 ? H / 2 : H;
  // Attention reads the present cache, or the new rows in T when a prompt's
  // cache has another float dtype (kv_separate: [B][N_kv][S][H], S rows).
  const void* ksrc = p.kv_separate ? p.kv_sep_k : p.present_k;
  const void* vsrc = p.kv_separate ? p.kv_sep_v : p.present_v;
  const long long rows = p.kv_separate ? p.S : p.C;
  const CacheT* kb = reinterpret_cast<const CacheT*>(ksrc) + ((long long)b * p.Nkv + g) * rows * row_elems;
  const CacheT* vb = reinterpret_cast<const CacheT*>(vsrc) + ((long long)b * p.Nkv + g) * rows * row_elems;

  for (int t0 = kmin; t0 < kmax; t0 += kTile) {
    __syncthreads();
    for (int x = tid; x < kTile * H; x += kWarps * 32) {
      const int j = x / H, d = x % H;
      float kv = 0.f, vv = 0.f;
      if (t0 + j < kmax) {
        const long long idx = (long long)(t0 + j) * H + d;
        if constexpr (i4) {
          const long long bi = (long long)(t0 + j) * (H / 2) + (d >> 1);
          const int sh = (d & 1) * 4;
          const int kc = (int)((reinterpret_cast<const uint8_t*>(kb)[bi] >> sh) & 15) - 8;
          const int vc = (int)((reinterpret_cast<const uint8_t*>(vb)[bi] >> sh) & 15) - 8;
          kv = (float)kc * channel_scale(p.k_scale, p.k_scale_n, g * H + d);
          vv = (float)vc * channel_scale(p.v_scale, p.v_scale_n, g * H + d);
        } else if (i8) {
          kv = (float)reinterpret_cast<const int8_t*>(kb)[idx] * channel_scale(p.k_scale, p.k_scale_n, g * H + d);
          vv = (float)reinterpret_cast<const int8_t*>(vb)[idx] * channel_scale(p.v_scale, p.v_scale_n, g * H + d);
        } else if (sizeof(CacheT) == 2) {
          kv = __half2float(reinterpret_cast<const __half*>(kb)[idx]);
          vv = __half2float(reinterpret_cast<const __half*>(vb)[idx]);
        } else {
          kv = reinterpret_cast<const float*>(kb)[idx];
          vv = reinterpret_cast<const float*>(vb)[idx];
        }
      }
      ks[j * HP + d] = kv;
      vs[j * HP + d] = vv;
    }
    __syncthreads();
    const int j = t0 + lane;  // this lane's key
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const int rl = warp * kRowsPerWarp + rr, r = r0 + rl;
      if (r >= nrows) continue;                     // warp-uniform
      const int i = r / p.G, h = g * p.G + r % p.G, pos = past_row + i;   // position in cache rows
      if (i >= live_i) continue;
      float s = 0.f;
      for (int d = 0; d < H; ++d) s += qs[rl * H + d] * ks[lane * HP + d];
      s *= qscale;
      bool vis = j < kmax;
      if (p.causal) vis = vis && j <= pos;
      if (p.window >= 0) vis = vis && j >= pos - p.window;
      if (p.softcap > 0.f) s = p.softcap * tanhf(s / p.softcap) * kLog2e;
      if (p.has_bias && vis) {
        const long long bi = (((long long)(p.bias_bdim > 1 ? b : 0) * p.bias_ndim + (p.bias_ndim > 1 ? h : 0)) *
                                  p.S + i) * p.bias_ld + j + off;
        s += load_t(p.bias, bi, p.t_type) * kLog2e;
      }
      s = vis ? s : kNegBig;
      float mt = s;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      const float mn = fmaxf(m[rr], mt);
      const float f = ex2(m[rr] - mn);
      m[rr] = mn;
      const float pj = vis ? ex2(s - mn) : 0.f;
      float ps = pj;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l[rr] = l[rr] * f + ps;
#pragma unroll
      for (int e = 0; e < kMaxH / 32; ++e) o[rr][e] *= f;
      for (int jj = 0; jj < kTile; ++jj) {
        const float pb = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
        for (int e = 0; e < kMaxH / 32; ++e) {
          const int d = lane + 32 * e;
          if (d < H) o[rr][e] += pb * vs[jj * HP + d];
        }
      }
    }
  }

  // Epilogue: out = o / (l + sink term), cast to T; padding rows get 0.
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int r = r0 + warp * kRowsPerWarp + rr;
    if (r >= nrows) continue;
    const int i = r / p.G, h = g * p.G + r % p.G;
    float mf = m[rr], extra = 0.f;
    if (p.has_sink || p.smooth) {
      const float sg = (p.has_sink ? load_t(p.sink, h, p.t_type) : 0.f) * kLog2e;
      mf = fmaxf(m[rr], sg);
      extra = ex2(sg - mf);
    }
    const float f = ex2(m[rr] - mf);
    const float den = l[rr] * f + extra;
    const bool pad = i >= live_i;
#pragma unroll
    for (int e = 0; e < kMaxH / 32; ++e) {
      const int d = lane + 32 * e;
      if (d >= H) continue;
      const float val = (pad || den <= 0.f) ? 0.f : o[rr][e] * f / den;
      const long long oi = ((long long)(b * p.S + i) * p.N + h) * H + d;
      if (sizeof(T) == 2) reinterpret_cast<__half*>(p.out)[oi] = __float2half_rn(val);
      else reinterpret_cast<float*>(p.out)[oi] = val;
    }
  }
}

}  // namespace

bool prefill_simt_supported(const Params& p) { return p.H <= kMaxH && p.H % 16 == 0; }

cudaError_t launch_prefill_simt(const Params& p, cudaStream_t st) {
  const int nrows = p.S * p.G;
  dim3 grid((nrows + kRows - 1) / kRows, p.Nkv, p.B), block(kWarps * 32);
  const size_t smem = (size_t)(kRows * p.H + 2 * kTile * (p.H + 1)) * sizeof(float);
  cudaError_t e;
  // With kv_separate the rows attention reads have the query dtype.
  const int src = p.kv_separate ? p.t_type : p.cache_type;
  if (p.t_type == kF16) {
    e = cudaFuncSetAttribute(prefill_simt_kernel<__half, __half>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_simt_kernel<__half, __half><<<grid, block, smem, st>>>(p);
  } else if (src == kI8) {
    e = cudaFuncSetAttribute(prefill_simt_kernel<float, int8_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_simt_kernel<float, int8_t><<<grid, block, smem, st>>>(p);
  } else if (src == kI4) {
    e = cudaFuncSetAttribute(prefill_simt_kernel<float, uint8_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_simt_kernel<float, uint8_t><<<grid, block, smem, st>>>(p);
  } else {
    e = cudaFuncSetAttribute(prefill_simt_kernel<float, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_simt_kernel<float, float><<<grid, block, smem, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace gqa
