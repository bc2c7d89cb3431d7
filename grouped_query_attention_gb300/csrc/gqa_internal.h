// Internal interface between the host entry points (gqa_api.cu) and the
// kernel translation units. Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gqa {

enum CacheMode : int { kPrompt = 0, kShared = 1, kCopy = 2 };
enum ElemType : int { kF32 = 1, kF16 = 2, kI8 = 3, kI4 = 4 };  // kI4: two +8-biased nibbles per byte

// Everything a kernel needs about one gqa_forward call. Passed by value as a
// kernel parameter (well under the 32 KB parameter limit).
struct Params {
  // ---- sizes
  int B, S, N, Nkv, G, H;
  int C;          // present capacity (sequence axis of present_key/value)
  int past_cap;   // sequence axis of past_key/value (copy mode), else 0
  int total_len;  // total_sequence_length (host scalar)
  int mode;       // CacheMode
  int t_type;     // ElemType of query/key/value/output (kF32 | kF16)
  int cache_type; // ElemType of the cache (kF32 | kF16 | kI8 | kI4)
  int kv_separate; // 1: a prompt's float cache of another dtype than T; attention reads kv_sep_k/v
  int window_cache; // 1: sliding_window_cache with a past cache (window-shift update, see batch_rows)
  int k_quant, v_quant;  // gqa_quant values
  // ---- attributes (resolved)
  int causal;
  int window;            // local_window_size (-1 = none)
  float scale;           // resolved score scale
  float softcap;         // 0 = none
  float eps;             // qk_norm_epsilon
  int has_norm, has_rotary, has_bias, has_sink, smooth;
  int bias_bdim, bias_ndim;  // leading dims of attention_bias (1 or B, 1 or N)
  int bias_ld;               // last dim of attention_bias (total_sequence_length)
  int rotary_rows;           // rows of cos/sin caches
  int k_scale_n, v_scale_n;  // 1 or N_kv*H
  // ---- tensors (device)
  const void* q;
  const void* k;
  const void* v;
  const void* past_k;
  const void* past_v;
  void* present_k;
  void* present_v;
  const int* seqlens;
  const void* cos_c;
  const void* sin_c;
  const void* bias;
  const void* sink;
  const float* k_scale;
  const float* v_scale;
  const void* qw;
  const void* kw;
  void* out;
  // ---- workspace (device)
  unsigned int* status;  // OR of GQA_DEVICE_* bits
  void* qprep;           // prepared queries, layout [B][N_kv][S*G][H]
  int qprep_type;        // ElemType of qprep
  int q_in_prefill;      // 1: the tensor-core prefill loads raw query rows and applies norm / rotary
                         // itself (no qprep; the pre-pass appends K/V only)
  float* bias_stage;     // bias * log2(e) as fp32 rows of bias_stage_ld floats ([bdim*S] rows) for the
  int bias_stage_ld;     // tensor-core prefill's TMA bias staging (16-byte row stride), else null
  void* kv_sep_k;        // kv_separate: new K/V rows in T as attention reads them, [B][N_kv][S][H]
  void* kv_sep_v;
  float* part_o;         // decode partial outputs [B*N_kv][max_splits][R][H]
                         // (tensor-core decode: [max_splits][R][H], one slot per CTA segment)
  float* part_ml;        // decode partial (m, l)   [B*N_kv][max_splits][R][2] (same note)
  unsigned int* counters;  // decode merge tickets  [B*N_kv]
  int split_len;         // keys per decode split (tensor-core decode: keys per balanced unit)
  int max_splits;        // grid extent of the split axis (tensor-core decode: partial slots)
  int rows_pad;          // R: decode rows per (b, g) rounded to a power of two
  // ---- bounded waits of the tensor-core kernels (gqa_set_wait_limit)
  long long wait_budget; // clock cycles each pipeline wait may take before the CTA gives up
  int withhold_tile;     // >= 0: the TMA warp stops before its copy of this key tile (tests the timeout path)
};

// Batch-level data check shared by all kernels: returns past_b (rows already
// cached) or -1 if seqlens_k[b] is inconsistent with the shapes.
__host__ __device__ inline int batch_past(const Params& p, int total) {
  if (total < 1 || total > p.total_len || (total > p.C && !p.window_cache)) return -1;
  if (p.mode == kPrompt) return total <= p.S ? 0 : -1;
  int past = total - p.S;
  if (past < 0) return -1;
  if (p.mode == kCopy && past > p.past_cap && !p.window_cache) return -1;
  return past;
}

// Cache rows of one batch entry. Without a window cache, row r holds absolute
// position r: the new rows start at row past and rows [0, total) are live.
// With a window cache (sliding_window_cache = 1 and a past cache) the past
// buffer holds the most recent n_old = min(past, L) rows (L its capacity);
// the present keeps the last keep = live - S of them at rows 0 .. keep-1 and
// the new rows follow, live = min(n_old + S, C); row r holds absolute position
// off + r, off = total - live.
struct BatchRows {
  int keep;  // cache row of the first new row
  int live;  // live cache rows after the update
  int off;   // absolute position of cache row 0
  int n_old; // live rows of the past buffer before the update
};

__host__ __device__ inline BatchRows batch_rows(const Params& p, int total, int past) {
  BatchRows r;
  if (p.window_cache) {
    const int L = p.mode == kShared ? p.C : p.past_cap;
    r.n_old = past < L ? past : L;
    r.live = r.n_old + p.S < p.C ? r.n_old + p.S : p.C;
    r.keep = r.live - p.S;
    r.off = total - r.live;
  } else {
    r.n_old = past;
    r.keep = past;
    r.live = total;
    r.off = 0;
  }
  return r;
}

// Launch order of the flash prefills, whose CTAs are (query block of 256
// rows, KV head (b, g)) pairs. Without a past cache (prompt) a block's key
// range depends only on its query block, and a grid that runs
// query-block-major (x = KV head, y = query block from the last) starts the
// longest blocks of every KV head first and leaves the short ones for the
// tail. With a past the lengths also depend on seqlens_k (device data): the
// grid runs KV-head-major (x = query block from the last, y = KV head),
// longest first within a head. Each kernel states when it takes the first.
__host__ __device__ inline bool prefill_prompt_qb_major(const Params& p) {
  return p.mode == kPrompt && (p.S * p.G + 255) / 256 <= 65535;
}

// Size of the fixed scratch array behind gqa_forward_noalloc (16 MiB).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
// Device address of that array on the current device (looked up once per device).
cudaError_t noalloc_scratch(void** ptr);

// Launchers (return the launch's cudaError_t).
cudaError_t launch_copy_past(const Params& p, cudaStream_t st);
cudaError_t launch_window_shift(const Params& p, cudaStream_t st);
cudaError_t launch_prepass(const Params& p, cudaStream_t st);
cudaError_t launch_decode(const Params& p, cudaStream_t st);
// TMA tensor maps of a tensor-core launch, encoded on the host before the
// launch (kept out of the launch itself so nothing but the launch sits
// between a caller's timing events).
cudaError_t launch_bias_stage(const Params& p, cudaStream_t st);
// Whether the tensor-core prefill stages the bias (shared by all heads, G >= 8) by TMA.
bool prefill_tc_bias_staged(const Params& p);

struct TmaMaps {
  CUtensorMap m[5];
};
cudaError_t prepare_decode_tc(const Params& p, TmaMaps* maps);
cudaError_t launch_decode_tc(const Params& p, cudaStream_t st, const TmaMaps& maps);
// Tensor-core decode for an int8 cache with fp32 queries (head size 128, <= 8 rows).
bool decode_tc_i8_supported(const Params& p);
cudaError_t prepare_decode_tc_i8(const Params& p, TmaMaps* maps);
cudaError_t launch_decode_tc_i8(const Params& p, cudaStream_t st, const TmaMaps& maps);
// The tensor-core decode runs min(SM count, kTcDecodeMaxCtas) persistent CTAs
// and keeps two partial slots per CTA.
constexpr int kTcDecodeMaxCtas = 256;
constexpr int kTcDecodeTile = 128;
bool decode_tc_supported(const Params& p);
cudaError_t launch_prefill_simt(const Params& p, cudaStream_t st);
cudaError_t prepare_prefill_tc(const Params& p, TmaMaps* maps);
cudaError_t launch_prefill_tc(const Params& p, cudaStream_t st, const TmaMaps& maps);
bool prefill_tc_supported(const Params& p);
// Tensor-core prefill over an int8 / 4-bit cache with fp32 Q/K/V (hi/lo fp16 split).
bool prefill_tcq_supported(const Params& p);
cudaError_t prepare_prefill_tcq(const Params& p, TmaMaps* maps);
cudaError_t launch_prefill_tcq(const Params& p, cudaStream_t st, const TmaMaps& maps);
bool decode_supported(const Params& p);
bool prepass_supported(const Params& p);
bool prefill_simt_supported(const Params& p);

}  // namespace gqa
