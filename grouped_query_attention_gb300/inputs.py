"""Seeded synthetic inputs for the GroupQueryAttention forward pass.

This module only draws random tensors and builds the rotary cos/sin tables
that the operator takes as inputs; it holds none of the operator's
arithmetic. The same host arrays feed the CUDA library (after a copy to the
device) and the CPU oracle used by the tests and the benchmark.

Every tensor comes from its own numpy generator seeded with
``(seed, tensor_index)``, the index being the tensor's place in the
operator's input list (com.microsoft.GroupQueryAttention, section Inputs).
Normal draws are fp32 then rounded to the tensor dtype (round to nearest).
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

# Input order of the operator (section Inputs); the index seeds each tensor.
INPUT_ORDER = ["query", "key", "value", "past_key", "past_value", "seqlens_k",
               "total_sequence_length", "cos_cache", "sin_cache", "attention_bias",
               "head_sink", "k_scale", "v_scale", "q_norm_weight", "k_norm_weight"]
_PRESENT_INDEX = 100  # initial (sentinel) contents of separate present buffers

NP_DTYPE = {"f32": np.float32, "f16": np.float16}


@dataclass(frozen=True)
class CaseSpec:
    """Shape, dtype and feature recipe of one synthetic call.

    mode: "prompt" (no past; present is a capacity buffer C >= S),
          "shared" (past and present are one capacity buffer C, updated in place),
          "copy"   (separate past of length past_len and present of length
                    past_len + S).
    seqlens_k: explicit tuple of B values (total length minus one), or empty
          when seqlens_range is given.
    seqlens_range: (lo, hi) inclusive range of seqlens_k drawn uniformly per batch.
    """
    name: str
    dtype: str
    B: int
    S: int
    N: int
    Nkv: int
    H: int
    capacity: int
    mode: str = "prompt"
    past_len: int = 0
    seqlens_k: tuple = ()
    seqlens_range: tuple | None = None
    causal: int = 1
    rotary_theta: float | None = None
    rotary_rows: int | None = None
    qk_norm: bool = False
    qk_norm_epsilon: float = 1e-6
    local_window_size: int = -1
    softcap: float = 0.0
    head_sink: bool = False
    smooth_softmax: int = -1
    bias: tuple | None = None          # (batch_dim, head_dim, std): dims are B or 1, N or 1
    scale: float = 0.0
    quant: str = "NONE"                # NONE | PER_TENSOR | PER_CHANNEL (quantised cache)
    bits: int = 8                      # 8: int8 codes; 4: two 4-bit codes per byte (prompt only)
    cache_dtype: str | None = None     # float cache dtype of a prompt ("f16" / "f32"); None: the query dtype
    sliding_window_cache: int = 0      # 1: past/present are window buffers (evict from the front)
    scale_range: tuple = (0.005, 0.02)
    extra: dict = field(default_factory=dict)

    def with_(self, **kw) -> "CaseSpec":
        return replace(self, **kw)


def _rng(seed: int, name: str) -> np.random.Generator:
    idx = INPUT_ORDER.index(name) if name in INPUT_ORDER else _PRESENT_INDEX + len(name)
    return np.random.default_rng([int(seed), idx])


def _normal(rng, shape, dtype, std=1.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x.astype(dtype)


def _int8_uniform(rng, shape):
    return rng.integers(-127, 128, size=shape, dtype=np.int16).astype(np.int8)


def rotary_tables(rows: int, head_size: int, theta: float, dtype) -> tuple[np.ndarray, np.ndarray]:
    """cos/sin caches of shape (rows, head_size/2): angle p * theta^(-2d/head_size), fp64 then cast."""
    d = np.arange(head_size // 2, dtype=np.float64)
    inv = theta ** (-2.0 * d / head_size)
    ang = np.arange(rows, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(dtype), np.sin(ang).astype(dtype)


def draw_seqlens(spec: CaseSpec, seed: int) -> np.ndarray:
    if spec.seqlens_range is not None:
        lo, hi = spec.seqlens_range
        return _rng(seed, "seqlens_k").integers(lo, hi + 1, size=spec.B).astype(np.int32)
    return np.asarray(spec.seqlens_k, dtype=np.int32)


def generate(spec: CaseSpec, seed: int = 0) -> dict:
    """Host arrays for one call: dict(inputs, attrs, present_key, present_value, share_buffer, spec)."""
    T = NP_DTYPE[spec.dtype]
    B, S, N, Nkv, H = spec.B, spec.S, spec.N, spec.Nkv, spec.H
    quant = spec.quant != "NONE"
    int4 = quant and spec.bits == 4
    cache_dtype = (np.uint8 if int4 else np.int8) if quant else NP_DTYPE[spec.cache_dtype or spec.dtype]
    seqlens = draw_seqlens(spec, seed)
    if seqlens.shape != (B,):
        raise ValueError("seqlens_k must give one value per batch")
    total_len = int(seqlens.max()) + 1

    inp = {}
    inp["query"] = _normal(_rng(seed, "query"), (B, S, N * H), T)
    inp["key"] = _normal(_rng(seed, "key"), (B, S, Nkv * H), T)
    inp["value"] = _normal(_rng(seed, "value"), (B, S, Nkv * H), T)
    inp["seqlens_k"] = seqlens
    inp["total_sequence_length"] = np.array([total_len], dtype=np.int32)

    def cache(name, length):
        rng = _rng(seed, name)
        if int4:   # packed bytes: any bit pattern is a valid pair of codes
            return rng.integers(0, 256, size=(B, Nkv, length, H // 2), dtype=np.int16).astype(np.uint8)
        shape = (B, Nkv, length, H)
        return _int8_uniform(rng, shape) if quant else _normal(rng, shape, cache_dtype)

    share = spec.mode == "shared"
    if spec.mode == "shared":
        inp["past_key"] = cache("past_key", spec.capacity)
        inp["past_value"] = cache("past_value", spec.capacity)
        present_k = present_v = None
    elif spec.mode == "copy":
        inp["past_key"] = cache("past_key", spec.past_len)
        inp["past_value"] = cache("past_value", spec.past_len)
        present_k = cache("present_key_init", spec.past_len + S)
        present_v = cache("present_value_init", spec.past_len + S)
    elif spec.mode == "prompt":
        present_k = cache("present_key_init", spec.capacity)
        present_v = cache("present_value_init", spec.capacity)
    else:
        raise ValueError(spec.mode)

    if spec.rotary_theta is not None:
        rows = spec.rotary_rows or max(spec.capacity, total_len)
        inp["cos_cache"], inp["sin_cache"] = rotary_tables(rows, H, spec.rotary_theta, T)
    if spec.bias is not None:
        bdim, ndim, std = spec.bias
        inp["attention_bias"] = _normal(_rng(seed, "attention_bias"), (bdim, ndim, S, total_len), T, std)
    if spec.head_sink:
        inp["head_sink"] = _normal(_rng(seed, "head_sink"), (N,), T)
    if quant:
        n = 1 if spec.quant == "PER_TENSOR" else Nkv * H
        lo, hi = spec.scale_range
        inp["k_scale"] = _rng(seed, "k_scale").uniform(lo, hi, size=n).astype(np.float32)
        inp["v_scale"] = _rng(seed, "v_scale").uniform(lo, hi, size=n).astype(np.float32)
    if spec.qk_norm:
        inp["q_norm_weight"] = (1.0 + 0.1 * _rng(seed, "q_norm_weight").standard_normal(H)).astype(T)
        inp["k_norm_weight"] = (1.0 + 0.1 * _rng(seed, "k_norm_weight").standard_normal(H)).astype(T)

    attrs = dict(num_heads=N, kv_num_heads=Nkv, causal=spec.causal,
                 do_rotary=1 if spec.rotary_theta is not None else 0,
                 local_window_size=spec.local_window_size, scale=spec.scale, softcap=spec.softcap,
                 qk_norm_epsilon=spec.qk_norm_epsilon, smooth_softmax=spec.smooth_softmax,
                 k_quant_type=spec.quant, v_quant_type=spec.quant, kv_cache_bit_width=spec.bits,
                 sliding_window_cache=spec.sliding_window_cache)
    return dict(inputs=inp, attrs=attrs, present_key=present_k, present_value=present_v,
                share_buffer=share, spec=spec)


# The synthetic workloads (sizes and distributions of the operator's use
# cases): a tiny fp32 prompt, fp16 decode over a shared cache, fp16 causal
# prefill with Q/K RMS norm and rotary, fp16 chunked prefill with window,
# softcap, head sink, bias and rotary, fp32 decode over an int8 cache, an
# fp16 bidirectional prompt that writes an fp32 cache, fp16 decode over a
# sliding-window cache (4096 rows, window 4000), and fp32 prompts that
# build an int8 or a 4-bit cache (the quantised-cache prefill variants of
# section Implementation variants).
WORKLOADS = {
    "prompt_f32_b1_s16": CaseSpec(
        name="prompt_f32_b1_s16", dtype="f32", B=1, S=16, N=4, Nkv=2, H=32, capacity=16,
        mode="prompt", seqlens_k=(15,)),
    "decode_f16_b16_c8192": CaseSpec(
        name="decode_f16_b16_c8192", dtype="f16", B=16, S=1, N=32, Nkv=8, H=128, capacity=8192,
        mode="shared", seqlens_range=(1024, 8191), rotary_theta=1e4, rotary_rows=8192),
    "prefill_f16_b4_s4096": CaseSpec(
        name="prefill_f16_b4_s4096", dtype="f16", B=4, S=4096, N=32, Nkv=8, H=128, capacity=8192,
        mode="prompt", seqlens_k=(4095, 4095, 4095, 4095), rotary_theta=1e4, rotary_rows=8192,
        qk_norm=True),
    "chunked_prefill_f16_b8_s512": CaseSpec(
        name="chunked_prefill_f16_b8_s512", dtype="f16", B=8, S=512, N=64, Nkv=8, H=128,
        capacity=8192, mode="shared", seqlens_range=(2048 + 511, 6144 + 511), rotary_theta=1e6,
        rotary_rows=8192, local_window_size=4096, softcap=50.0, head_sink=True, bias=(1, 1, 0.5)),
    "decode_int8_f32_b32_c16384": CaseSpec(
        name="decode_int8_f32_b32_c16384", dtype="f32", B=32, S=1, N=32, Nkv=8, H=128,
        capacity=16384, mode="shared", seqlens_range=(4096, 16383), quant="PER_CHANNEL"),
    "prompt_bidirectional_f16_cache_f32_b4_s2048": CaseSpec(
        name="prompt_bidirectional_f16_cache_f32_b4_s2048", dtype="f16", B=4, S=2048, N=32, Nkv=8, H=128,
        capacity=2048, mode="prompt", seqlens_k=(2047, 2047, 2047, 2047), causal=0, cache_dtype="f32"),
    "decode_window_f16_b16_c4096": CaseSpec(
        name="decode_window_f16_b16_c4096", dtype="f16", B=16, S=1, N=32, Nkv=8, H=128, capacity=4096,
        mode="shared", seqlens_range=(6000, 12000), rotary_theta=1e4, local_window_size=4000,
        sliding_window_cache=1),
    "prefill_int8_f32_b2_s2048": CaseSpec(
        name="prefill_int8_f32_b2_s2048", dtype="f32", B=2, S=2048, N=32, Nkv=8, H=128, capacity=2048,
        mode="prompt", seqlens_k=(2047, 2047), quant="PER_CHANNEL"),
    "prefill_int4_f32_b2_s2048": CaseSpec(
        name="prefill_int4_f32_b2_s2048", dtype="f32", B=2, S=2048, N=32, Nkv=8, H=128, capacity=2048,
        mode="prompt", seqlens_k=(2047, 2047), quant="PER_TENSOR", bits=4, scale_range=(0.3, 0.5)),
}
WORKLOAD_ORDER = list(WORKLOADS)
