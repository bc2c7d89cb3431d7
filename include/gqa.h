/*
 * gqa.h -- C ABI of the GB300 (sm_103a) GroupQueryAttention forward pass.
 *
 * The operation is com.microsoft.GroupQueryAttention as its README states it
 * (sections Description, Inputs, Outputs, Attributes, Type constraints):
 * grouped-query attention over BSH query/key/value and a BNSH key/value cache,
 * with optional paired Q/K RMS normalisation, NeoX rotary embedding, causal
 * and local-window masks, additive attention bias, softcap, head sink /
 * smooth softmax, an int8 (per-tensor or per-channel) or, for prompts, a
 * packed 4-bit quantised cache, a sliding-window (window-shift) cache, and a
 * prompt's float cache in the other float dtype.
 *
 * Conventions for every entry point:
 *   - All tensors are dense, row-major (C-contiguous) and live in device
 *     memory of the current CUDA device, except where a field says "host".
 *     Pointers must be 16-byte aligned.
 *   - The caller owns every buffer and the stream. No entry point allocates
 *     device memory; scratch space is the caller's workspace
 *     (gqa_workspace_size).
 *   - Work is enqueued asynchronously on the given stream (a cudaStream_t
 *     passed as void*; NULL is the legacy default stream).
 *   - Failures return a gqa_status; gqa_last_error() gives a one-line reason
 *     (per calling thread). Nothing is launched when a check fails.
 */
#ifndef GQA_GB300_H
#define GQA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GQA_API __attribute__((visibility("default")))
#else
#define GQA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gqa_status {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARGUMENT = 1, /* shapes, dtypes, attributes or pointers break the contract */
  GQA_ERR_UNSUPPORTED = 2,      /* allowed by the operator but not implemented here */
  GQA_ERR_CUDA = 3,             /* a CUDA runtime/driver call or a launch failed */
  GQA_ERR_DEVICE_STATUS = 4,    /* a kernel flagged bad data (see gqa_read_device_status) */
  GQA_ERR_WORKSPACE = 5         /* workspace NULL, misaligned or smaller than required */
} gqa_status;

/* Element types (section Type constraints: T in {float32, float16},
 * T_CACHE in {float32, float16, uint8, int8}, T_KV_SCALE float32, M int32).
 * GQA_BF16 exists only so that such a tensor is rejected as UNSUPPORTED. */
typedef enum gqa_dtype {
  GQA_DTYPE_NONE = 0,
  GQA_F32 = 1,
  GQA_F16 = 2,
  GQA_I8 = 3,
  GQA_U8 = 4,
  GQA_I32 = 5,
  GQA_BF16 = 6
} gqa_dtype;

/* k_quant_type / v_quant_type (section Attributes). */
typedef enum gqa_quant {
  GQA_QUANT_NONE = 0,
  GQA_QUANT_PER_TENSOR = 1,
  GQA_QUANT_PER_CHANNEL = 2
} gqa_quant;

/* One tensor: data == NULL means "input absent". shape[0..ndim-1] are used. */
typedef struct gqa_tensor {
  void* data;
  int32_t dtype; /* gqa_dtype */
  int32_t ndim;
  int64_t shape[4];
} gqa_tensor;

/* Attributes, section Attributes of the operator page; gqa_attrs_default()
 * fills the page's defaults (num_heads / kv_num_heads have none). */
typedef struct gqa_attrs {
  int32_t num_heads;            /* N, query heads */
  int32_t kv_num_heads;         /* N_kv, key/value heads; N % N_kv == 0 */
  int32_t causal;               /* 1 (default) causal; 0 bidirectional (needs local_window_size == -1) */
  int32_t do_rotary;            /* 0 (default) or 1: NeoX rotary on Q and on K before it is cached */
  int32_t local_window_size;    /* -1 (default) disables; W >= 0: key j visible from p iff p-W <= j <= p */
  float scale;                  /* 0 (default) selects 1/sqrt(head_size) */
  float softcap;                /* 0 (default) disables; c > 0: score -> c*tanh(score/c) before the bias */
  float qk_norm_epsilon;        /* 1e-6 (default) */
  int32_t smooth_softmax;       /* -1 (default); 1 adds exp(0 - max) to the denominator when no head_sink */
  int32_t k_quant_type;         /* gqa_quant; NONE (default) */
  int32_t v_quant_type;         /* gqa_quant; NONE (default) */
  int32_t kv_cache_bit_width;   /* 8: int8 cache; 4: packed 4-bit cache (prompt only); ignored when not quantised */
  int32_t sliding_window_cache; /* 0 (default); 1: past/present are window buffers (see gqa_outputs) */
} gqa_attrs;

/* Inputs, section Inputs of the operator page (same names, same shapes):
 *   query          T      (B, S, N*H)
 *   key, value     T      (B, S, N_kv*H)            -- kv_sequence_length == S
 *   past_key/value T_CACHE (B, N_kv, L, H) or absent. L is the capacity when
 *                  past and present are one buffer (past.data == present.data),
 *                  else the past length (copy mode). Absent for a 4-bit cache.
 *   seqlens_k      int32  (B): total length of batch b minus one (device)
 *   cos/sin_cache  T      (R, H/2), R > largest position; required iff do_rotary
 *   attention_bias T      (B or 1, N or 1, S, total_sequence_length) or absent
 *   head_sink      T      (N) or absent
 *   k/v_scale      float32 (1) for PER_TENSOR or (N_kv*H) for PER_CHANNEL
 *   q/k_norm_weight T     (H), both or neither
 * total_sequence_length is a HOST scalar: the largest seqlens_k[b] + 1. */
typedef struct gqa_inputs {
  gqa_tensor query, key, value;
  gqa_tensor past_key, past_value;
  gqa_tensor seqlens_k;
  gqa_tensor cos_cache, sin_cache;
  gqa_tensor attention_bias;
  gqa_tensor head_sink;
  gqa_tensor k_scale, v_scale;
  gqa_tensor q_norm_weight, k_norm_weight;
  int32_t total_sequence_length;
} gqa_inputs;

/* Outputs, section Outputs: output T (B, S, N*H); present_key/value T_CACHE
 * (B, N_kv, C, H). Shared buffer: present.data == past.data and C == L.
 * Copy mode: C == L + S. No past: C >= S (a capacity buffer).
 * sliding_window_cache == 1 with a past cache (section Attributes): the past
 * buffer (capacity L) holds the most recent n_old = min(past_b, L) rows of
 * the sequence, oldest first; the present keeps the last n_new - S of them at
 * rows 0 .. n_new-S-1 (older rows are evicted from the front) and appends the
 * S new rows after them, n_new = min(n_old + S, C); row r holds absolute
 * position total_b - n_new + r (masks and bias columns use it; rotary uses
 * the absolute position). Needs causal = 1, local_window_size W > 0,
 * C >= S + W and, for a separate past, L >= W; C need not equal L + S and
 * total_sequence_length may exceed C. Without a past the flag changes nothing.
 * 4-bit cache (kv_cache_bit_width == 4, section Inputs past_key / present_key):
 * GQA_U8 of shape (B, N_kv, C, H/2); byte k of a row holds code(2k) + 8 in
 * its low nibble and code(2k+1) + 8 in its high nibble, code =
 * clamp(rint(x / scale), -7, 7) with the fp32 division of the int8 code. */
typedef struct gqa_outputs {
  gqa_tensor output;
  gqa_tensor present_key, present_value;
} gqa_outputs;

typedef struct gqa_handle gqa_handle;

/* Fill *attrs with the defaults of section Attributes. */
GQA_API void gqa_attrs_default(gqa_attrs* attrs);

/* Create a handle holding a copy of the attributes (host memory only).
 * Returns INVALID_ARGUMENT for a NULL pointer, non-positive head counts,
 * num_heads % kv_num_heads != 0, causal == 0 with local_window_size != -1,
 * local_window_size < -1, softcap < 0, a non-finite scale or epsilon, or a
 * quant type outside gqa_quant, or a quantised cache whose kv_cache_bit_width
 * is neither 8 nor 4, or sliding_window_cache not 0 / 1, or 1 without causal
 * attention and local_window_size > 0. */
GQA_API gqa_status gqa_create(const gqa_attrs* attrs, gqa_handle** out);

/* Bytes of device workspace gqa_forward needs for these shapes (host-only;
 * makes no CUDA call). Runs every host-side check of gqa_forward, so it is
 * also the way to validate a call without a GPU. */
GQA_API gqa_status gqa_workspace_size(const gqa_handle* handle, const gqa_inputs* in,
                              const gqa_outputs* out, size_t* bytes);

/* Forward pass (whole operator) on `stream`:
 *   1. append the S new K/V rows of every (batch, KV head) at positions
 *      past_b .. past_b+S-1 of the present cache, past_b = seqlens_k[b]+1-S
 *      with a past cache and 0 without (K: RMS norm, then rotary at the
 *      absolute position, then cast, int8-quantise or pack 4-bit codes;
 *      V: the same store without norm or rotary);
 *      in copy mode the live past rows 0 .. past_b-1 are copied first;
 *   2. output[b, i, h] = softmax over the visible cache rows of
 *      scale * q_h . k (softcapped, plus bias), with query head h reading KV
 *      head h / (N/N_kv), the head-sink logit in the denominator, times V.
 * Operator page sections Description, Inputs, Outputs, Attributes and
 * Implementation variants (share_append / new_kv_past / quant_int8 decode and
 * flash prefill: append first, then attend over the cache as stored, with
 * causal bounds right-aligned at the live length from seqlens_k).
 * Present rows that are not appended (or copied) keep their bytes. Output
 * rows i >= total_b of a prompt without past (padding) are written as 0.
 * workspace: device buffer of at least gqa_workspace_size bytes, 256-byte
 * aligned, owned by the caller, not used concurrently by another call. Its
 * contents need not survive between calls: every call first clears the
 * workspace header (status word and split-merge tickets) on `stream`, so the
 * caller may use the buffer for anything else in between.
 * Host-side checks as in gqa_workspace_size. Data errors found on the device
 * (seqlens_k[b]+1 outside [S or 1, min(C, total_sequence_length)], a rotary
 * position beyond the cos/sin rows) skip that batch entry without any write
 * out of bounds and set a bit of the workspace's status word, which then
 * describes this call until the next call on the same workspace clears it. */
GQA_API gqa_status gqa_forward(gqa_handle* handle, const gqa_inputs* in, const gqa_outputs* out,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Forward pass without any workspace, for callers that cannot allocate device
 * memory: a plugin inside a host runtime that hands it only its input and output
 * buffers and exposes no allocator, or code on a latency-critical path where
 * cudaMalloc / cudaFree (which may synchronise the device) are not acceptable.
 * The operator's pages have no counterpart: this is a deployment variant of
 * gqa_forward's decode regime, with the same inputs, outputs and results.
 *   - Scratch (status word, merge tickets, split partials) comes from one
 *     fixed array of 16 MiB compiled into the library; every GPU that loads
 *     the library holds it until the process exits. Nothing is allocated:
 *     no cudaMalloc, cudaFree or allocating library routine is called.
 *   - Only the decode regime (gqa_describe_plan reports GQA_REGIME_DECODE);
 *     other calls return GQA_ERR_UNSUPPORTED. A call that needs more than
 *     16 MiB of scratch returns GQA_ERR_WORKSPACE with the size it needs.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call shares the one array and it keeps the last call's contents;
 *     each call clears the status word and tickets on its stream first. Calls
 *     that overlap on the GPU (other streams, threads or handles) race and give
 *     wrong results: serialise them.
 *   - Data errors found on the device skip that batch entry as in gqa_forward,
 *     but are not reported: no entry point reads this status word. */
GQA_API gqa_status gqa_forward_noalloc(gqa_handle* handle, const gqa_inputs* in, const gqa_outputs* out,
                                       void* stream);

/* Bound of the pipeline waits of the tensor-core kernels, for callers that
 * want a data-dependent stall reported sooner, and a switch to test the
 * timeout path (no counterpart on the operator's pages).
 *   cycles: every barrier wait of a tensor-core CTA gives up after this many
 *     SM clock cycles (0 restores the default, 4e9 cycles, about 2 s at the
 *     maximum clock; otherwise at least 1000). A CTA whose wait gives up sets
 *     GQA_DEVICE_TIMEOUT, stops its pipeline, waits for its own copies and
 *     MMAs in flight, frees its tensor memory and returns; the call's outputs
 *     are then undefined. The next call on the handle and workspace is
 *     unaffected (each call clears the workspace header).
 *   withhold_copy: -1 (default) off; k >= 0 makes the TMA warp of every
 *     tensor-core CTA stop before the copy of its k-th key tile (in the
 *     prefill over an int8 / 4-bit cache: the converter warps before its
 *     conversion), so the waits for that tile expire: a test of the timeout
 *     path that faults nothing.
 * Applies to the following gqa_forward / gqa_forward_noalloc calls on the
 * handle. Host-only; INVALID_ARGUMENT for a NULL handle or a value out of range. */
GQA_API gqa_status gqa_set_wait_limit(gqa_handle* handle, int64_t cycles, int32_t withhold_copy);

/* Synchronise `stream`, read and clear the status word that the kernels of
 * the most recent gqa_forward call on `workspace` set (each call clears it
 * first). *status receives the OR of GQA_DEVICE_* bits (0 = no data error).
 * Returns DEVICE_STATUS if it is non-zero, CUDA on a runtime failure. */
#define GQA_DEVICE_BAD_SEQLEN 1u  /* seqlens_k out of range for the cache / total length / S */
#define GQA_DEVICE_BAD_ROTARY 2u  /* a rotary position is not covered by cos/sin_cache rows */
#define GQA_DEVICE_TIMEOUT 4u     /* a bounded pipeline wait gave up (kernel returned early) */
GQA_API gqa_status gqa_read_device_status(gqa_handle* handle, void* workspace, void* stream, uint32_t* status);

/* Host-only description of how gqa_forward would run a call: the regime
 * (GQA_REGIME_DECODE: one fused split-KV launch; GQA_REGIME_PREFILL: pre-pass
 * then flash prefill), the number of kernel launches per call, the decode
 * split length / split count (0 for prefill) and the workspace bytes. Same
 * checks and status codes as gqa_workspace_size.
 * Decode regime: up to 8 query rows per KV head (S * num_heads / kv_num_heads)
 * with head size 64 or 128 on the CUDA-core kernel (split_len = keys per
 * split, max_splits = splits per (batch, KV head)), or, for fp16 inputs and
 * cache with head size 128, up to 16 rows on the tensor-core kernel
 * (split_len = 128 keys per work unit, max_splits = partial-result slots). */
#define GQA_REGIME_DECODE 1
#define GQA_REGIME_PREFILL 2
typedef struct gqa_plan_info {
  int32_t regime;
  int32_t launches;
  int32_t split_len;
  int32_t max_splits;
  uint64_t workspace_bytes;
} gqa_plan_info;
GQA_API gqa_status gqa_describe_plan(const gqa_handle* handle, const gqa_inputs* in, const gqa_outputs* out,
                                     gqa_plan_info* info);

/* Per-launch timing for measurement tools. gqa_profile_begin creates
 * 2*max_launches CUDA events (host-side driver objects, no device memory);
 * while profiling is on, every gqa_forward / gqa_forward_noalloc call on this
 * handle records an event pair around each kernel it launches (up to
 * max_launches launches in total). gqa_profile_end synchronises the events,
 * writes up to `capacity` (kind, milliseconds) pairs in launch order, sets
 * *count to the number of launches recorded, releases the events and turns
 * profiling off. Kinds: */
#define GQA_KERNEL_COPY_PAST 1
#define GQA_KERNEL_PREPASS 2
#define GQA_KERNEL_DECODE 3
#define GQA_KERNEL_PREFILL_CUDA_CORE 4
#define GQA_KERNEL_PREFILL_TENSOR_CORE 5
#define GQA_KERNEL_DECODE_TENSOR_CORE 6
#define GQA_KERNEL_WINDOW_SHIFT 7
#define GQA_KERNEL_BIAS_STAGE 8
GQA_API gqa_status gqa_profile_begin(gqa_handle* handle, int32_t max_launches);
GQA_API gqa_status gqa_profile_end(gqa_handle* handle, int32_t* kinds, float* ms, int32_t capacity, int32_t* count);

/* Release the handle (host memory only). NULL is a no-op. */
GQA_API void gqa_destroy(gqa_handle* handle);

/* Static name of a status code. */
GQA_API const char* gqa_status_string(gqa_status status);

/* One-line reason of the last non-OK status returned on this thread. */
GQA_API const char* gqa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_GB300_H */
