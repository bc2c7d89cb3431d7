// Host side of the C ABI declared in include/gqa.h: argument checks, the
// workspace plan and the launch sequence of one forward call.
//
// Launch sequence (all on the caller's stream, nothing allocated):
//   decode regime (S * G <= 8, head size 64/128): [copy of live past rows in
//     copy mode] -> one fused split-KV decode launch (append + attention +
//     merge);
//   prefill regime: [copy] -> pre-pass (append K/V; prepared queries into the
//     workspace for the CUDA-core prefill, the tensor-core prefill prepares
//     its own) -> [bias staging] -> flash prefill.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/gqa.h"
#include "gqa_internal.h"

struct gqa_handle {
  gqa_attrs attrs;
  long long wait_budget;    // bound of each pipeline wait of the tensor-core kernels (clock cycles)
  int withhold_tile;        // >= 0: testing the timeout path (see gqa_set_wait_limit)
  // per-launch profiling (gqa_profile_begin / gqa_profile_end)
  bool profiling;
  std::vector<cudaEvent_t> events;  // 2 per launch
  std::vector<int> kinds;
  int used;
};

namespace {

thread_local std::string g_last_error;

gqa_status fail(gqa_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
gqa_status fail(gqa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

constexpr size_t kAlign = 256;
constexpr long long kDefaultWaitBudget = 4000000000LL;   // clock cycles, about 2 s at the maximum SM clock
constexpr long long kDecodeTargetCtas = 152LL * 16;  // GB300: 152 SMs, ~16 split CTAs per SM

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool present(const gqa_tensor& t) { return t.data != nullptr; }

bool shape_is(const gqa_tensor& t, int ndim, const int64_t* s) {
  if (t.ndim != ndim) return false;
  for (int i = 0; i < ndim; ++i)
    if (t.shape[i] != s[i]) return false;
  return true;
}

std::string shape_str(const gqa_tensor& t) {
  std::string r = "(";
  for (int i = 0; i < t.ndim && i < 4; ++i) {
    if (i) r += ",";
    r += std::to_string((long long)t.shape[i]);
  }
  return r + ")";
}

struct Plan {
  gqa::Params P;
  bool decode;
  bool tensor_core;  // prefill on a tcgen05 kernel (head size 128)
  bool tcq;          // ... the one over an int8 / 4-bit cache with fp32 Q/K/V
  bool tc_decode;    // decode on a tcgen05 kernel (fp16 cache <= 16 rows, or int8 cache with fp32 <= 8 rows; H=128)
  bool tc_i8;        // ... the int8-cache one
  size_t hdr_bytes, qprep_bytes, kvsep_bytes, bias_bytes, part_bytes, total_bytes;
  bool bias_staged;  // tensor-core prefill with the bias staged by a small kernel and copied by TMA
  size_t part_rows;  // decode partial rows (part_o holds part_rows x H floats, part_ml part_rows x 2)
};

gqa_status check_aligned(const gqa_tensor& t, const char* name) {
  if (present(t) && (reinterpret_cast<uintptr_t>(t.data) & 15u) != 0)
    return fail(GQA_ERR_INVALID_ARGUMENT, "%s: data pointer is not 16-byte aligned", name);
  return GQA_OK;
}

gqa_status plan_call(const gqa_handle* hd, const gqa_inputs* in, const gqa_outputs* out, Plan* pl) {
  if (!hd || !in || !out || !pl) return fail(GQA_ERR_INVALID_ARGUMENT, "NULL handle, inputs or outputs");
  const gqa_attrs& a = hd->attrs;
  gqa::Params& P = pl->P;
  memset(&P, 0, sizeof(P));

  // ---- query / key / value (section Inputs)
  const gqa_tensor& q = in->query;
  if (!present(q)) return fail(GQA_ERR_INVALID_ARGUMENT, "query is required");
  if (q.dtype == GQA_BF16) return fail(GQA_ERR_UNSUPPORTED, "bfloat16 is not implemented");
  if (q.dtype != GQA_F32 && q.dtype != GQA_F16)
    return fail(GQA_ERR_INVALID_ARGUMENT, "query dtype must be float32 or float16");
  if (q.ndim != 3) return fail(GQA_ERR_INVALID_ARGUMENT, "query must be rank 3 (B, S, N*H)");
  if (!present(in->key) || !present(in->value))
    return fail(GQA_ERR_UNSUPPORTED, "packed QKV (key/value absent) is not implemented");
  const long long B = q.shape[0], S = q.shape[1], hidden = q.shape[2];
  const int N = a.num_heads, Nkv = a.kv_num_heads;
  if (B < 1 || S < 1 || hidden < 1) return fail(GQA_ERR_INVALID_ARGUMENT, "empty query %s", shape_str(q).c_str());
  if (hidden % N != 0) return fail(GQA_ERR_INVALID_ARGUMENT, "query hidden size %lld is not a multiple of num_heads %d", hidden, N);
  const long long H = hidden / N;
  const int G = N / Nkv;
  const int64_t kv_shape[3] = {B, S, Nkv * H};
  for (const gqa_tensor* t : {&in->key, &in->value}) {
    if (t->dtype != q.dtype) return fail(GQA_ERR_INVALID_ARGUMENT, "key/value dtype must match query");
    if (!shape_is(*t, 3, kv_shape))
      return fail(GQA_ERR_INVALID_ARGUMENT, "key/value must be (B, S, kv_num_heads*head_size) = (%lld,%lld,%lld), got %s",
                  B, S, Nkv * H, shape_str(*t).c_str());
  }
  if (H % 16 != 0 || H < 16 || H > 256)
    return fail(GQA_ERR_UNSUPPORTED, "head_size %lld: supported head sizes are multiples of 16 in [16, 256]", H);

  // ---- cache dtypes (section Type constraints / Description)
  const bool kq = a.k_quant_type != GQA_QUANT_NONE, vq = a.v_quant_type != GQA_QUANT_NONE;
  if (kq != vq) return fail(GQA_ERR_UNSUPPORTED, "quantising only one of the K/V caches is not implemented");
  const gqa_tensor& pk = out->present_key;
  const gqa_tensor& pv = out->present_value;
  if (!present(pk) || !present(pv)) return fail(GQA_ERR_INVALID_ARGUMENT, "present_key and present_value are required");
  int cache_dt = q.dtype;
  bool i4 = false;   // 4-bit cache: uint8 rows of head_size/2 bytes, two +8-biased nibbles each
  if (kq) {
    if (q.dtype != GQA_F32) return fail(GQA_ERR_INVALID_ARGUMENT, "a quantised cache requires float32 query/key/value/output");
    if (a.kv_cache_bit_width != 8 && a.kv_cache_bit_width != 4)
      return fail(GQA_ERR_INVALID_ARGUMENT, "kv_cache_bit_width must be 8 or 4");
    i4 = a.kv_cache_bit_width == 4;
    cache_dt = i4 ? GQA_U8 : GQA_I8;
  }
  // A prompt (no past) may write its float cache as float16 or float32 whatever
  // the query dtype (section Description); an existing cache has the query dtype.
  const bool separate = !kq && pk.dtype != q.dtype && (pk.dtype == GQA_F32 || pk.dtype == GQA_F16) &&
                        pv.dtype == pk.dtype;
  if (separate) {
    if (present(in->past_key) || present(in->past_value))
      return fail(GQA_ERR_INVALID_ARGUMENT, "past_key/past_value must have the query dtype");
    cache_dt = pk.dtype;
  }
  if (pk.dtype != cache_dt || pv.dtype != cache_dt)
    return fail(GQA_ERR_INVALID_ARGUMENT, "present cache dtype must be %s",
                i4 ? "uint8 (packed 4-bit codes)" : kq ? "int8" : "float16 or float32 (one dtype for K and V)");
  const long long row_w = i4 ? H / 2 : H;   // cache elements per row
  if (pk.ndim != 4 || pk.shape[0] != B || pk.shape[1] != Nkv || pk.shape[3] != row_w)
    return fail(GQA_ERR_INVALID_ARGUMENT, "present_key must be (B, kv_num_heads, C, %s), got %s",
                i4 ? "head_size/2" : "head_size", shape_str(pk).c_str());
  if (!shape_is(pv, 4, pk.shape))
    return fail(GQA_ERR_INVALID_ARGUMENT, "present_value shape must equal present_key shape");
  const long long C = pk.shape[2];

  // ---- past / cache mode
  const bool has_pk = present(in->past_key), has_pv = present(in->past_value);
  if (has_pk != has_pv) return fail(GQA_ERR_INVALID_ARGUMENT, "past_key and past_value come together");
  int mode = gqa::kPrompt;
  long long past_cap = 0;
  if (has_pk && i4) return fail(GQA_ERR_UNSUPPORTED, "a 4-bit cache is prompt-only: past_key/past_value are not accepted");
  if (has_pk) {
    const gqa_tensor& qk = in->past_key;
    const gqa_tensor& qv = in->past_value;
    if (qk.dtype != cache_dt || qv.dtype != cache_dt) return fail(GQA_ERR_INVALID_ARGUMENT, "past cache dtype must equal the present cache dtype");
    if (qk.ndim != 4 || qk.shape[0] != B || qk.shape[1] != Nkv || qk.shape[3] != H ||
        !shape_is(qv, 4, qk.shape))
      return fail(GQA_ERR_INVALID_ARGUMENT, "past_key/past_value must both be (B, kv_num_heads, L, head_size)");
    const bool sk = qk.data == pk.data, sv = qv.data == pv.data;
    if (sk != sv) return fail(GQA_ERR_INVALID_ARGUMENT, "past/present must be shared for both K and V or for neither");
    past_cap = qk.shape[2];
    if (sk) {
      if (past_cap != C) return fail(GQA_ERR_INVALID_ARGUMENT, "a shared past/present buffer must have one capacity");
      mode = gqa::kShared;
    } else {
      if (C != past_cap + S && !a.sliding_window_cache)
        return fail(GQA_ERR_INVALID_ARGUMENT, "present length must be past length + S when not shared");
      mode = gqa::kCopy;
    }
    if (a.sliding_window_cache && (C < S + a.local_window_size || past_cap < a.local_window_size))
      return fail(GQA_ERR_INVALID_ARGUMENT,
                  "a window cache needs capacity >= S + local_window_size (%lld < %lld) and a past of >= %d rows", C,
                  S + a.local_window_size, a.local_window_size);
    if (!a.causal) return fail(GQA_ERR_UNSUPPORTED, "bidirectional attention over a past cache is not implemented");
  } else if (C < S) {
    return fail(GQA_ERR_INVALID_ARGUMENT, "present capacity %lld is smaller than sequence_length %lld", C, S);
  }

  // ---- seqlens_k, total_sequence_length
  const int64_t b1[1] = {B};
  if (!present(in->seqlens_k) || in->seqlens_k.dtype != GQA_I32 || !shape_is(in->seqlens_k, 1, b1))
    return fail(GQA_ERR_INVALID_ARGUMENT, "seqlens_k must be int32 of shape (B)");
  const long long T = in->total_sequence_length;
  if (T < 1) return fail(GQA_ERR_INVALID_ARGUMENT, "total_sequence_length must be >= 1");
  if (mode == gqa::kPrompt && T > S)
    return fail(GQA_ERR_INVALID_ARGUMENT, "without a past cache total_sequence_length (%lld) cannot exceed S (%lld)", T, S);
  const bool window = a.sliding_window_cache == 1 && mode != gqa::kPrompt;   // window-shift update
  if (T > C && !window)
    return fail(GQA_ERR_INVALID_ARGUMENT, "total_sequence_length (%lld) exceeds the present capacity (%lld)", T, C);

  // ---- optional inputs
  const int tdt = q.dtype;
  if (a.do_rotary) {
    const gqa_tensor& cc = in->cos_cache;
    const gqa_tensor& sc = in->sin_cache;
    if (!present(cc) || !present(sc)) return fail(GQA_ERR_INVALID_ARGUMENT, "do_rotary needs cos_cache and sin_cache");
    if (cc.dtype != tdt || sc.dtype != tdt || cc.ndim != 2 || sc.ndim != 2 || cc.shape[1] != H / 2 ||
        sc.shape[0] != cc.shape[0] || sc.shape[1] != cc.shape[1])
      return fail(GQA_ERR_INVALID_ARGUMENT, "cos/sin_cache must be (max_sequence_length, head_size/2) of the query dtype");
    P.rotary_rows = (int)cc.shape[0];
    P.cos_c = cc.data;
    P.sin_c = sc.data;
    P.has_rotary = 1;
  }
  if (present(in->attention_bias)) {
    const gqa_tensor& t = in->attention_bias;
    if (t.dtype != tdt || t.ndim != 4 || !(t.shape[0] == 1 || t.shape[0] == B) || !(t.shape[1] == 1 || t.shape[1] == N) ||
        t.shape[2] != S || t.shape[3] != T)
      return fail(GQA_ERR_INVALID_ARGUMENT, "attention_bias must be (B or 1, num_heads or 1, S, total_sequence_length), got %s",
                  shape_str(t).c_str());
    P.has_bias = 1;
    P.bias = t.data;
    P.bias_bdim = (int)t.shape[0];
    P.bias_ndim = (int)t.shape[1];
    P.bias_ld = (int)t.shape[3];
  }
  if (present(in->head_sink)) {
    const int64_t n1[1] = {N};
    if (in->head_sink.dtype != tdt || !shape_is(in->head_sink, 1, n1))
      return fail(GQA_ERR_INVALID_ARGUMENT, "head_sink must be (num_heads) of the query dtype");
    P.has_sink = 1;
    P.sink = in->head_sink.data;
  }
  const bool qn = present(in->q_norm_weight), kn = present(in->k_norm_weight);
  if (qn != kn) return fail(GQA_ERR_INVALID_ARGUMENT, "q_norm_weight and k_norm_weight must be given together");
  if (qn) {
    const int64_t h1[1] = {H};
    if (in->q_norm_weight.dtype != tdt || in->k_norm_weight.dtype != tdt || !shape_is(in->q_norm_weight, 1, h1) ||
        !shape_is(in->k_norm_weight, 1, h1))
      return fail(GQA_ERR_INVALID_ARGUMENT, "q/k_norm_weight must be (head_size) of the query dtype");
    P.has_norm = 1;
    P.qw = in->q_norm_weight.data;
    P.kw = in->k_norm_weight.data;
  }
  if (kq) {
    for (const gqa_tensor* t : {&in->k_scale, &in->v_scale}) {
      const int qt = t == &in->k_scale ? a.k_quant_type : a.v_quant_type;
      const long long want = qt == GQA_QUANT_PER_TENSOR ? 1 : Nkv * H;
      const int64_t w1[1] = {want};
      if (!present(*t) || t->dtype != GQA_F32 || !shape_is(*t, 1, w1))
        return fail(GQA_ERR_INVALID_ARGUMENT, "k/v_scale must be float32 of length %lld for this quant type", want);
    }
    P.k_scale = static_cast<const float*>(in->k_scale.data);
    P.v_scale = static_cast<const float*>(in->v_scale.data);
    P.k_scale_n = (int)in->k_scale.shape[0];
    P.v_scale_n = (int)in->v_scale.shape[0];
  }
  const int64_t oshape[3] = {B, S, hidden};
  if (!present(out->output) || out->output.dtype != tdt || !shape_is(out->output, 3, oshape))
    return fail(GQA_ERR_INVALID_ARGUMENT, "output must be (B, S, num_heads*head_size) of the query dtype");

  const gqa_tensor* all[] = {&in->query, &in->key, &in->value, &in->past_key, &in->past_value, &in->seqlens_k,
                             &in->cos_cache, &in->sin_cache, &in->attention_bias, &in->head_sink, &in->k_scale,
                             &in->v_scale, &in->q_norm_weight, &in->k_norm_weight, &out->output, &out->present_key,
                             &out->present_value};
  const char* names[] = {"query", "key", "value", "past_key", "past_value", "seqlens_k", "cos_cache", "sin_cache",
                         "attention_bias", "head_sink", "k_scale", "v_scale", "q_norm_weight", "k_norm_weight",
                         "output", "present_key", "present_value"};
  for (int i = 0; i < 17; ++i) {
    gqa_status s = check_aligned(*all[i], names[i]);
    if (s != GQA_OK) return s;
  }
  const long long big = 1LL << 31;
  if (B * S * hidden >= big * 8 || B * Nkv * C * H >= big * 8 || C >= big)
    return fail(GQA_ERR_UNSUPPORTED, "tensor too large");

  // ---- parameter block
  P.B = (int)B; P.S = (int)S; P.N = N; P.Nkv = Nkv; P.G = G; P.H = (int)H;
  P.C = (int)C; P.past_cap = (int)past_cap; P.total_len = (int)T; P.mode = mode;
  P.t_type = tdt == GQA_F16 ? gqa::kF16 : gqa::kF32;
  P.cache_type = i4 ? gqa::kI4 : kq ? gqa::kI8 : cache_dt == GQA_F16 ? gqa::kF16 : gqa::kF32;
  P.kv_separate = separate ? 1 : 0;
  P.window_cache = window ? 1 : 0;
  P.k_quant = a.k_quant_type; P.v_quant = a.v_quant_type;
  P.causal = a.causal ? 1 : 0;
  P.window = a.local_window_size;
  P.scale = a.scale != 0.f ? a.scale : 1.0f / sqrtf((float)H);
  P.softcap = a.softcap;
  P.eps = a.qk_norm_epsilon;
  P.smooth = a.smooth_softmax == 1 ? 1 : 0;
  P.q = q.data; P.k = in->key.data; P.v = in->value.data;
  P.past_k = in->past_key.data; P.past_v = in->past_value.data;
  P.present_k = pk.data; P.present_v = pv.data;
  P.seqlens = static_cast<const int*>(in->seqlens_k.data);
  P.out = out->output.data;
  P.wait_budget = hd->wait_budget;
  P.withhold_tile = hd->withhold_tile;

  // ---- regime and workspace plan
  // A 4-bit cache is built by a prompt and always takes the prefill kernels, as
  // does a prompt whose float cache has another dtype than the query.
  // A window cache takes the tensor-core decode kernels (which work in cache
  // rows with an absolute offset) or else the pre-pass and the CUDA-core prefill.
  pl->decode = !i4 && !separate &&
               (window ? (gqa::decode_tc_supported(P) || gqa::decode_tc_i8_supported(P))
                       : (gqa::decode_supported(P) || (S * G <= 16 && gqa::decode_tc_supported(P))));
  pl->tc_i8 = pl->decode && gqa::decode_tc_i8_supported(P);
  pl->tc_decode = pl->decode && (gqa::decode_tc_supported(P) || pl->tc_i8);
  pl->tensor_core = false;
  pl->tcq = false;
  pl->hdr_bytes = align_up(sizeof(unsigned int) * (1 + (size_t)B * Nkv));  // status, tickets
  pl->qprep_bytes = 0;
  pl->kvsep_bytes = 0;
  pl->bias_bytes = 0;
  pl->bias_staged = false;
  pl->part_bytes = 0;
  pl->part_rows = 0;
  if (pl->decode) {
    int rp = 1;
    while (rp < S * G) rp <<= 1;
    P.rows_pad = rp;
    size_t nb;
    if (pl->tc_decode) {
      // Balanced decomposition: every CTA takes an equal share of the 128-key
      // tiles of all (b, g) ranges; at most its first and last segment are
      // shared with another CTA and need a partial slot.
      P.split_len = gqa::kTcDecodeTile;
      P.max_splits = 2 * gqa::kTcDecodeMaxCtas;
      nb = (size_t)P.max_splits * rp;
    } else {
      long long L = 64;
      const long long work = B * Nkv * T;
      while (L < 4096 && work / L > kDecodeTargetCtas) L <<= 1;
      P.split_len = (int)L;
      P.max_splits = (int)((T + L - 1) / L);
      nb = (size_t)B * Nkv * P.max_splits * rp;
    }
    pl->part_rows = nb;
    pl->part_bytes = align_up(nb * H * sizeof(float)) + align_up(nb * 2 * sizeof(float));
  } else {
    if (!gqa::prefill_simt_supported(P) || !gqa::prepass_supported(P))
      return fail(GQA_ERR_UNSUPPORTED, "no prefill kernel for head_size %lld", H);
    pl->tcq = !window && gqa::prefill_tcq_supported(P);
    pl->tensor_core = !window && (gqa::prefill_tc_supported(P) || pl->tcq);
    // The tensor-core prefill loads the raw query rows of a tile (when the
    // group size divides its 128 rows) and applies norm / rotary itself;
    // otherwise the pre-pass prepares fp16 queries for it, and fp32 ones for
    // the CUDA-core prefill.
    P.q_in_prefill = pl->tensor_core && 128 % G == 0 ? 1 : 0;
    P.qprep_type = pl->tensor_core ? gqa::kF16 : gqa::kF32;
    pl->qprep_bytes = P.q_in_prefill ? 0 : align_up((size_t)B * S * N * H * (pl->tensor_core ? 2 : 4));
    if (separate) pl->kvsep_bytes = 2 * align_up((size_t)B * Nkv * S * H * (tdt == GQA_F16 ? 2 : 4));
    if (pl->tensor_core && !pl->tcq && gqa::prefill_tc_bias_staged(P)) {
      pl->bias_staged = true;
      P.bias_stage_ld = (int)((P.bias_ld + 3) & ~3);   // 16-byte rows for the tensor copies
      pl->bias_bytes = align_up((size_t)P.bias_bdim * S * P.bias_stage_ld * sizeof(float));
    }
  }
  pl->total_bytes = pl->hdr_bytes + pl->qprep_bytes + pl->kvsep_bytes + pl->bias_bytes + pl->part_bytes;
  return GQA_OK;
}

void bind_workspace(Plan* pl, void* ws) {
  char* w = static_cast<char*>(ws);
  gqa::Params& P = pl->P;
  P.status = reinterpret_cast<unsigned int*>(w);
  P.counters = P.status + 1;
  char* cur = w + pl->hdr_bytes;
  if (pl->qprep_bytes) {
    P.qprep = cur;
    cur += pl->qprep_bytes;
  }
  if (pl->kvsep_bytes) {
    P.kv_sep_k = cur;
    P.kv_sep_v = cur + pl->kvsep_bytes / 2;
    cur += pl->kvsep_bytes;
  }
  if (pl->bias_bytes) {
    P.bias_stage = reinterpret_cast<float*>(cur);
    cur += pl->bias_bytes;
  }
  if (pl->part_bytes) {
    P.part_o = reinterpret_cast<float*>(cur);
    P.part_ml = reinterpret_cast<float*>(cur + align_up(pl->part_rows * P.H * sizeof(float)));
  }
}

gqa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(GQA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Launch through `fn`, bracketed by an event pair when the handle is profiling.
template <typename F>
cudaError_t timed_launch(gqa_handle* h, int kind, cudaStream_t st, F fn) {
  const bool rec = h->profiling && h->used < (int)h->kinds.size();
  if (rec) cudaEventRecord(h->events[2 * h->used], st);
  cudaError_t e = fn();
  if (rec) {
    cudaEventRecord(h->events[2 * h->used + 1], st);
    h->kinds[h->used++] = kind;
  }
  return e;
}

// The decode launch a plan selected.
cudaError_t launch_decode_any(const Plan& pl, cudaStream_t st, const gqa::TmaMaps& maps) {
  if (!pl.tc_decode) return gqa::launch_decode(pl.P, st);
  return pl.tc_i8 ? gqa::launch_decode_tc_i8(pl.P, st, maps) : gqa::launch_decode_tc(pl.P, st, maps);
}

}  // namespace

extern "C" {

void gqa_attrs_default(gqa_attrs* a) {
  if (!a) return;
  memset(a, 0, sizeof(*a));
  a->causal = 1;
  a->do_rotary = 0;
  a->local_window_size = -1;
  a->scale = 0.f;
  a->softcap = 0.f;
  a->qk_norm_epsilon = 1e-6f;
  a->smooth_softmax = -1;
  a->k_quant_type = GQA_QUANT_NONE;
  a->v_quant_type = GQA_QUANT_NONE;
  a->kv_cache_bit_width = 8;
  a->sliding_window_cache = 0;
}

gqa_status gqa_create(const gqa_attrs* a, gqa_handle** out) {
  if (!a || !out) return fail(GQA_ERR_INVALID_ARGUMENT, "NULL attrs or handle pointer");
  *out = nullptr;
  if (a->num_heads < 1 || a->kv_num_heads < 1) return fail(GQA_ERR_INVALID_ARGUMENT, "num_heads and kv_num_heads must be positive");
  if (a->num_heads % a->kv_num_heads != 0)
    return fail(GQA_ERR_INVALID_ARGUMENT, "num_heads (%d) must be a multiple of kv_num_heads (%d)", a->num_heads, a->kv_num_heads);
  if (a->causal != 0 && a->causal != 1) return fail(GQA_ERR_INVALID_ARGUMENT, "causal must be 0 or 1");
  if (a->local_window_size < -1) return fail(GQA_ERR_INVALID_ARGUMENT, "local_window_size must be >= -1");
  if (a->causal == 0 && a->local_window_size != -1)
    return fail(GQA_ERR_INVALID_ARGUMENT, "causal=0 requires local_window_size=-1");
  if (!std::isfinite(a->scale) || !std::isfinite(a->softcap) || !std::isfinite(a->qk_norm_epsilon) || a->softcap < 0.f ||
      a->qk_norm_epsilon < 0.f)
    return fail(GQA_ERR_INVALID_ARGUMENT, "scale/softcap/qk_norm_epsilon must be finite, softcap and epsilon >= 0");
  for (int qt : {a->k_quant_type, a->v_quant_type})
    if (qt < GQA_QUANT_NONE || qt > GQA_QUANT_PER_CHANNEL) return fail(GQA_ERR_INVALID_ARGUMENT, "unknown quant type %d", qt);
  if (a->sliding_window_cache != 0 && a->sliding_window_cache != 1)
    return fail(GQA_ERR_INVALID_ARGUMENT, "sliding_window_cache must be 0 or 1");
  if (a->sliding_window_cache == 1 && (a->causal != 1 || a->local_window_size <= 0))
    return fail(GQA_ERR_INVALID_ARGUMENT, "sliding_window_cache needs causal attention and local_window_size > 0");
  if (a->k_quant_type != GQA_QUANT_NONE && a->kv_cache_bit_width != 8 && a->kv_cache_bit_width != 4)
    return fail(GQA_ERR_INVALID_ARGUMENT, "kv_cache_bit_width must be 8 or 4");
  gqa_handle* h = new (std::nothrow) gqa_handle;
  if (!h) return fail(GQA_ERR_INVALID_ARGUMENT, "out of host memory");
  h->attrs = *a;
  h->wait_budget = kDefaultWaitBudget;
  h->withhold_tile = -1;
  h->profiling = false;
  h->used = 0;
  *out = h;
  return GQA_OK;
}

gqa_status gqa_workspace_size(const gqa_handle* h, const gqa_inputs* in, const gqa_outputs* out, size_t* bytes) {
  if (!bytes) return fail(GQA_ERR_INVALID_ARGUMENT, "NULL bytes pointer");
  Plan pl;
  gqa_status s = plan_call(h, in, out, &pl);
  if (s != GQA_OK) return s;
  *bytes = pl.total_bytes;
  return GQA_OK;
}

gqa_status gqa_describe_plan(const gqa_handle* h, const gqa_inputs* in, const gqa_outputs* out,
                             gqa_plan_info* info) {
  if (!info) return fail(GQA_ERR_INVALID_ARGUMENT, "NULL info pointer");
  Plan pl;
  gqa_status s = plan_call(h, in, out, &pl);
  if (s != GQA_OK) return s;
  info->regime = pl.decode ? GQA_REGIME_DECODE : GQA_REGIME_PREFILL;
  info->launches = (pl.P.mode == gqa::kCopy || pl.P.window_cache ? 1 : 0) + (pl.decode ? 1 : 2) + (pl.bias_staged ? 1 : 0);
  info->split_len = pl.decode ? pl.P.split_len : 0;
  info->max_splits = pl.decode ? pl.P.max_splits : 0;
  info->workspace_bytes = pl.total_bytes;
  return GQA_OK;
}

gqa_status gqa_forward(gqa_handle* h, const gqa_inputs* in, const gqa_outputs* out, void* ws, size_t ws_bytes,
                       void* stream) {
  Plan pl;
  gqa_status s = plan_call(h, in, out, &pl);
  if (s != GQA_OK) return s;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0)
    return fail(GQA_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
  if (ws_bytes < pl.total_bytes)
    return fail(GQA_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, pl.total_bytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bind_workspace(&pl, ws);
  // The header (status word, merge tickets) is cleared by every call: the
  // caller may reuse the workspace for anything between calls, and a call
  // that timed out leaves tickets behind.
  cudaError_t eh = cudaMemsetAsync(ws, 0, pl.hdr_bytes, st);
  if (eh != cudaSuccess) return cuda_fail(eh, "workspace header clear");
  const gqa::Params& P = pl.P;
  cudaError_t e = cudaSuccess;
  gqa::TmaMaps maps;   // host work of the tensor-core launches, done before the first launch
  if (pl.decode && pl.tc_decode)
    e = pl.tc_i8 ? gqa::prepare_decode_tc_i8(P, &maps) : gqa::prepare_decode_tc(P, &maps);
  else if (!pl.decode && pl.tensor_core)
    e = pl.tcq ? gqa::prepare_prefill_tcq(P, &maps) : gqa::prepare_prefill_tc(P, &maps);
  if (e != cudaSuccess) return cuda_fail(e, "TMA tensor maps");
  if (P.window_cache) {
    e = timed_launch(h, GQA_KERNEL_WINDOW_SHIFT, st, [&] { return gqa::launch_window_shift(P, st); });
    if (e != cudaSuccess) return cuda_fail(e, "window shift of the cache");
  } else if (P.mode == gqa::kCopy) {
    e = timed_launch(h, GQA_KERNEL_COPY_PAST, st, [&] { return gqa::launch_copy_past(P, st); });
    if (e != cudaSuccess) return cuda_fail(e, "copy of past rows");
  }
  if (pl.decode) {
    e = timed_launch(h, pl.tc_decode ? GQA_KERNEL_DECODE_TENSOR_CORE : GQA_KERNEL_DECODE, st,
                     [&] { return launch_decode_any(pl, st, maps); });
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  } else {
    e = timed_launch(h, GQA_KERNEL_PREPASS, st, [&] { return gqa::launch_prepass(P, st); });
    if (e != cudaSuccess) return cuda_fail(e, "pre-pass launch");
    if (pl.bias_staged) {
      e = timed_launch(h, GQA_KERNEL_BIAS_STAGE, st, [&] { return gqa::launch_bias_stage(P, st); });
      if (e != cudaSuccess) return cuda_fail(e, "bias staging launch");
    }
    if (pl.tensor_core)
      e = timed_launch(h, GQA_KERNEL_PREFILL_TENSOR_CORE, st, [&] {
        return pl.tcq ? gqa::launch_prefill_tcq(P, st, maps) : gqa::launch_prefill_tc(P, st, maps);
      });
    else
      e = timed_launch(h, GQA_KERNEL_PREFILL_CUDA_CORE, st, [&] { return gqa::launch_prefill_simt(P, st); });
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  }
  return GQA_OK;
}

gqa_status gqa_forward_noalloc(gqa_handle* h, const gqa_inputs* in, const gqa_outputs* out, void* stream) {
  Plan pl;
  gqa_status s = plan_call(h, in, out, &pl);
  if (s != GQA_OK) return s;
  if (!pl.decode)
    return fail(GQA_ERR_UNSUPPORTED,
                "gqa_forward_noalloc runs the decode regime only (gqa_describe_plan reports the regime)");
  if (pl.total_bytes > gqa::kNoAllocScratchBytes)
    return fail(GQA_ERR_WORKSPACE, "call needs %zu bytes of scratch; the fixed scratch holds %zu (use gqa_forward)",
                pl.total_bytes, gqa::kNoAllocScratchBytes);
  void* scratch = nullptr;
  cudaError_t e = gqa::noalloc_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "address of the fixed scratch");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bind_workspace(&pl, scratch);
  e = cudaMemsetAsync(scratch, 0, pl.hdr_bytes, st);  // status word and merge tickets start at zero
  if (e != cudaSuccess) return cuda_fail(e, "scratch header clear");
  const gqa::Params& P = pl.P;
  gqa::TmaMaps maps;
  if (pl.tc_decode &&
      (e = pl.tc_i8 ? gqa::prepare_decode_tc_i8(P, &maps) : gqa::prepare_decode_tc(P, &maps)) != cudaSuccess)
    return cuda_fail(e, "TMA tensor maps");
  if (P.window_cache) {
    e = timed_launch(h, GQA_KERNEL_WINDOW_SHIFT, st, [&] { return gqa::launch_window_shift(P, st); });
    if (e != cudaSuccess) return cuda_fail(e, "window shift of the cache");
  } else if (P.mode == gqa::kCopy) {
    e = timed_launch(h, GQA_KERNEL_COPY_PAST, st, [&] { return gqa::launch_copy_past(P, st); });
    if (e != cudaSuccess) return cuda_fail(e, "copy of past rows");
  }
  e = timed_launch(h, pl.tc_decode ? GQA_KERNEL_DECODE_TENSOR_CORE : GQA_KERNEL_DECODE, st,
                   [&] { return launch_decode_any(pl, st, maps); });
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return GQA_OK;
}

gqa_status gqa_set_wait_limit(gqa_handle* h, int64_t cycles, int32_t withhold_copy) {
  if (!h) return fail(GQA_ERR_INVALID_ARGUMENT, "NULL handle");
  if (cycles < 0 || (cycles > 0 && cycles < 1000))
    return fail(GQA_ERR_INVALID_ARGUMENT, "wait limit must be 0 (default) or at least 1000 cycles");
  if (withhold_copy < -1) return fail(GQA_ERR_INVALID_ARGUMENT, "withhold_copy must be -1 (off) or a tile index");
  h->wait_budget = cycles == 0 ? kDefaultWaitBudget : (long long)cycles;
  h->withhold_tile = withhold_copy;
  return GQA_OK;
}

gqa_status gqa_read_device_status(gqa_handle* h, void* ws, void* stream, uint32_t* status) {
  if (!h || !ws || !status) return fail(GQA_ERR_INVALID_ARGUMENT, "NULL handle, workspace or status pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned int v = 0;
  e = cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  e = cudaMemsetAsync(ws, 0, sizeof(v), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "status clear");
  *status = v;
  if (v) return fail(GQA_ERR_DEVICE_STATUS, "device status 0x%x", v);
  return GQA_OK;
}

gqa_status gqa_profile_begin(gqa_handle* h, int32_t max_launches) {
  if (!h || max_launches < 1) return fail(GQA_ERR_INVALID_ARGUMENT, "NULL handle or max_launches < 1");
  if (h->profiling) return fail(GQA_ERR_INVALID_ARGUMENT, "profiling already on");
  h->events.assign(2 * (size_t)max_launches, nullptr);
  for (auto& ev : h->events) {
    cudaError_t e = cudaEventCreate(&ev);
    if (e != cudaSuccess) {
      for (auto& x : h->events)
        if (x) cudaEventDestroy(x);
      h->events.clear();
      return cuda_fail(e, "event creation");
    }
  }
  h->kinds.assign((size_t)max_launches, 0);
  h->used = 0;
  h->profiling = true;
  return GQA_OK;
}

gqa_status gqa_profile_end(gqa_handle* h, int32_t* kinds, float* ms, int32_t capacity, int32_t* count) {
  if (!h || !count || (capacity > 0 && (!kinds || !ms))) return fail(GQA_ERR_INVALID_ARGUMENT, "NULL argument");
  if (!h->profiling) return fail(GQA_ERR_INVALID_ARGUMENT, "profiling is not on");
  gqa_status st = GQA_OK;
  cudaError_t e = h->used > 0 ? cudaEventSynchronize(h->events[2 * h->used - 1]) : cudaSuccess;
  if (e != cudaSuccess) st = cuda_fail(e, "event synchronize");
  for (int i = 0; st == GQA_OK && i < h->used && i < capacity; ++i) {
    float t = 0.f;
    e = cudaEventElapsedTime(&t, h->events[2 * i], h->events[2 * i + 1]);
    if (e != cudaSuccess) {
      st = cuda_fail(e, "event elapsed time");
      break;
    }
    kinds[i] = h->kinds[i];
    ms[i] = t;
  }
  *count = h->used;
  for (auto& ev : h->events) cudaEventDestroy(ev);
  h->events.clear();
  h->kinds.clear();
  h->used = 0;
  h->profiling = false;
  return st;
}

void gqa_destroy(gqa_handle* h) {
  if (!h) return;
  for (auto& ev : h->events) cudaEventDestroy(ev);
  delete h;
}

const char* gqa_status_string(gqa_status s) {
  switch (s) {
    case GQA_OK: return "GQA_OK";
    case GQA_ERR_INVALID_ARGUMENT: return "GQA_ERR_INVALID_ARGUMENT";
    case GQA_ERR_UNSUPPORTED: return "GQA_ERR_UNSUPPORTED";
    case GQA_ERR_CUDA: return "GQA_ERR_CUDA";
    case GQA_ERR_DEVICE_STATUS: return "GQA_ERR_DEVICE_STATUS";
    case GQA_ERR_WORKSPACE: return "GQA_ERR_WORKSPACE";
  }
  return "GQA_ERR_UNKNOWN";
}

const char* gqa_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
