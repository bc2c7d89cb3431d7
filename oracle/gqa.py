"""fp64 reference semantics of com.microsoft.GroupQueryAttention (forward).

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product
path may import this module.

Notation: B batch, S new rows (``sequence_length`` = ``kv_sequence_length``),
N = ``num_heads``, N_kv = ``kv_num_heads``, G = N / N_kv, H = head size,
C = capacity of the present cache (its sequence axis), total_b =
seqlens_k[b] + 1, past_b = rows already cached for batch b, p = past_b + i the
absolute position of new row i.

Readings where the page is silent (each has a switch here; the defaults are
the readings the library implements):
  * query head h reads KV head h // G (consecutive query heads share a KV head);
  * local window: key j is visible from position p iff p - W <= j <= p;
  * softcap c * tanh(s / c) is applied to the scaled score, then the bias is added;
  * the head sink (or 0 under smooth_softmax=1 without a sink) is one extra
    logit that enters only the softmax denominator;
  * int8 code = clamp(round_half_even(fp32(x) / fp32(scale)), -127, 127),
    the division done in IEEE fp32, dequantised as code * scale;
  * int4 (kv_cache_bit_width = 4) code = clamp(round_half_even(fp32(x) /
    fp32(scale)), -7, 7), stored as the nibble code + 8, two per byte with
    the even coordinate in the low nibble; only prompts (no past cache);
  * a prompt (no past cache) may store its float cache as float16 or float32
    whatever the query dtype; attention then reads the new K/V rows as they
    would be stored in the query dtype (computed from Q/K/V directly, the
    cache written separately), so the output does not depend on that choice;
  * sliding_window_cache = 1 with a past cache: the past buffer holds the
    most recent n_old = min(past_b, L) rows of the sequence (L its capacity),
    oldest first; the present keeps the last n_new - S of them at rows
    0 .. n_new-S-1 (evicted from the front, compacted) and appends the S new
    rows after them, n_new = min(n_old + S, C); cache row r then holds
    absolute position total_b - n_new + r, which masks, bias columns and
    rotary use. Requires causal attention, local_window_size W > 0,
    C >= S + W and L >= W, so every key a query can see is kept. Without a
    past cache the flag changes nothing;
  * RMS norm y = x / sqrt(mean(x^2) + eps) * w, weight used as given;
  * the K rows stored in the cache are computed in fp32 in one fixed order
    (rms_norm_fp32, rotary_neox_fp32) and then cast or quantised, so that the
    stored bytes are reproducible; attention reads those stored values. The
    fp64 functions define the mathematics and pin the fp32 recipe within its
    rounding-error bound (the pages fix no evaluation order);
  * padding rows of a prompt (i >= total_b, no past) produce a zero output row;
    their K/V rows are still appended.
"""

from __future__ import annotations

import numpy as np

DEFAULT_ATTRS = dict(
    num_heads=None,
    kv_num_heads=None,
    causal=1,
    do_rotary=0,
    local_window_size=-1,
    scale=0.0,
    softcap=0.0,
    qk_norm_epsilon=1e-6,
    smooth_softmax=-1,
    k_quant_type="NONE",
    v_quant_type="NONE",
    kv_cache_bit_width=8,
    sliding_window_cache=0,
)


def rms_norm(x: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """Per-head RMS normalisation over the last (head) axis, in fp64.

    com.microsoft.GroupQueryAttention, section Inputs (q_norm_weight,
    k_norm_weight: "per-head RMS-normalization weight of shape (head_size)")
    and section Attributes (qk_norm_epsilon).
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + float(eps)) * w


def rotary_neox(x: np.ndarray, cos_row: np.ndarray, sin_row: np.ndarray) -> np.ndarray:
    """Non-interleaved (NeoX half-split) rotary embedding over the last axis.

    Dimension d < H/2 is paired with d + H/2 and the pair is rotated by the
    angle whose cosine/sine are ``cos_row[d]`` / ``sin_row[d]``.
    com.microsoft.GroupQueryAttention, section Inputs (cos_cache, sin_cache of
    shape (max_sequence_length, head_size / 2)) and section Description
    ("interleaved rotary ... not implemented"); the half-split layout is the
    one com.microsoft.SparseAttention, section Attributes (rotary_interleaved)
    calls NeoX.
    """
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(cos_row, dtype=np.float64)
    s = np.asarray(sin_row, dtype=np.float64)
    half = x.shape[-1] // 2
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def _sum_squares_fp32(x32: np.ndarray) -> np.ndarray:
    """Sum of squares over the last axis in the fp32 order of the stored-row recipe.

    Every square is rounded to fp32; the squares of each group of four
    consecutive coordinates are added left to right; the H/4 group sums are
    then added as a pairwise tree (neighbours first: (g0+g1), (g2+g3), ...,
    then the pairs of pairs, ...), the group sums padded with zeros to a power
    of two. Each addition is one fp32 rounding.
    """
    sq = x32 * x32
    g = sq[..., 0::4]
    for k in (1, 2, 3):
        g = g + sq[..., k::4]
    n = g.shape[-1]
    width = 1
    while width < n:
        width *= 2
    if width > n:
        g = np.concatenate([g, np.zeros(g.shape[:-1] + (width - n,), np.float32)], axis=-1)
    while g.shape[-1] > 1:
        g = g[..., 0::2] + g[..., 1::2]
    return g[..., 0]


def rms_norm_fp32(x: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """RMS normalisation of the rows that are stored in the cache, in fp32.

    Same function as rms_norm (section Inputs, q_norm_weight / k_norm_weight;
    section Attributes, qk_norm_epsilon), evaluated in one fixed fp32 order so
    that the stored bytes are reproducible: ss = _sum_squares_fp32(x);
    ms = ss / H; r = 1 / sqrt(ms + eps) (IEEE division and square root, each
    rounded); y = (x * r) * w as two rounded products. The pages fix no
    evaluation order; this one (groups of four coordinates, then a pairwise
    tree) is the reading the library follows.
    """
    x32 = np.asarray(x, dtype=np.float32)
    w32 = np.asarray(weight, dtype=np.float32)
    H = x32.shape[-1]
    ms = _sum_squares_fp32(x32) / np.float32(H)
    r = np.float32(1.0) / np.sqrt(ms + np.float32(eps))
    return (x32 * r[..., None]) * w32


def rotary_neox_fp32(x: np.ndarray, cos_row: np.ndarray, sin_row: np.ndarray) -> np.ndarray:
    """NeoX rotary of stored rows in fp32: every product rounded, then one add or subtract.

    Same function as rotary_neox (section Inputs, cos_cache / sin_cache) in a
    fixed fp32 order: y[d] = fl(x[d] c) - fl(x[d+H/2] s) and y[d+H/2] =
    fl(x[d+H/2] c) + fl(x[d] s), each result rounded once (no fused
    multiply-add), with c, s the table entries converted exactly to fp32.
    """
    x32 = np.asarray(x, dtype=np.float32)
    c = np.asarray(cos_row, dtype=np.float32)
    s = np.asarray(sin_row, dtype=np.float32)
    half = x32.shape[-1] // 2
    x1, x2 = x32[..., :half], x32[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softcap_scores(s: np.ndarray, softcap: float) -> np.ndarray:
    """Soft-capping of attention scores: c * tanh(s / c) when c > 0.

    com.microsoft.GroupQueryAttention, section Attributes (softcap: "positive
    softcap applied to attention scores; the default 0 disables soft-capping").
    """
    if softcap > 0.0:
        return softcap * np.tanh(s / softcap)
    return s


def _scale_vector(scale: np.ndarray, quant_type: str, g: int, head_size: int) -> np.ndarray:
    """Scales of KV head g: one value (PER_TENSOR) or the channels g*H .. g*H+H-1 (PER_CHANNEL).

    com.microsoft.GroupQueryAttention, section Inputs (k_scale / v_scale: "one
    value for PER_TENSOR, or kv_num_heads * head_size values for PER_CHANNEL").
    """
    scale = np.asarray(scale, dtype=np.float32).reshape(-1)
    if quant_type == "PER_TENSOR":
        return np.full(head_size, scale[0], dtype=np.float32)
    if quant_type == "PER_CHANNEL":
        return scale[g * head_size:(g + 1) * head_size]
    raise ValueError(f"not a quantised cache: {quant_type}")


def quantize_int8(x: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Symmetric int8 code of fp32 values: clamp(rint(fp32(x) / scale), -127, 127).

    The division is IEEE fp32 (numpy float32 / float32) and the rounding is
    to nearest, ties to even. com.microsoft.GroupQueryAttention, section
    Inputs (k_scale, v_scale are float32) and section Attributes
    (k_quant_type / v_quant_type, kv_cache_bit_width = 8).
    """
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    t = x32 / np.asarray(scale, dtype=np.float32)
    return np.clip(np.rint(t), -127, 127).astype(np.int8)


def dequantize_int8(q: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Value of an int8 code: code * scale (exact in fp64).

    com.microsoft.GroupQueryAttention, section Implementation variants
    (quant_int8_decode_splitk: attention reads the appended int8 rows).
    """
    return np.asarray(q, dtype=np.float64) * np.asarray(scale, dtype=np.float64)


def quantize_int4(x: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Symmetric 4-bit code of fp32 values: clamp(rint(fp32(x) / scale), -7, 7) (int8 array).

    Same rounding as the int8 code (IEEE fp32 division, ties to even) with the
    symmetric 4-bit range. com.microsoft.GroupQueryAttention, section
    Attributes (kv_cache_bit_width = 4) and section Implementation variants
    (quant_int4_flash_prefill builds a 4-bit cache).
    """
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    t = x32 / np.asarray(scale, dtype=np.float32)
    return np.clip(np.rint(t), -7, 7).astype(np.int8)


def pack_int4(codes: np.ndarray) -> np.ndarray:
    """Codes (..., H) in [-8, 7] as bytes (..., H/2): nibble = code + 8, coordinate
    2k in the low nibble of byte k and 2k+1 in the high nibble.

    com.microsoft.GroupQueryAttention, section Attributes (kv_cache_bit_width:
    "four-bit values are packed two per uint8 element").
    """
    n = (np.asarray(codes, dtype=np.int16) + 8).astype(np.uint8)
    return (n[..., 0::2] | (n[..., 1::2] << 4)).astype(np.uint8)


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """Inverse of pack_int4: bytes (..., H/2) to codes (..., H) in [-8, 7]."""
    b = np.asarray(packed, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.int8)
    out[..., 0::2] = (b & 0x0F).astype(np.int16) - 8
    out[..., 1::2] = (b >> 4).astype(np.int16) - 8
    return out


def _store(x64: np.ndarray, cache_dtype, quant_type: str, scale, g: int, head_size: int,
           bits: int = 8) -> np.ndarray:
    """Value written into the present cache for one new row (round to nearest, or an int8 / packed int4 code)."""
    if quant_type != "NONE":
        sv = _scale_vector(scale, quant_type, g, head_size)
        if bits == 4:
            return pack_int4(quantize_int4(x64, sv))
        return quantize_int8(x64, sv)
    return np.asarray(x64, dtype=np.float64).astype(cache_dtype)


def _load(rows: np.ndarray, quant_type: str, scale, g: int, head_size: int, bits: int = 8) -> np.ndarray:
    """fp64 values of cached rows as attention reads them (dequantised if quantised)."""
    if quant_type != "NONE":
        sv = _scale_vector(scale, quant_type, g, head_size)
        codes = unpack_int4(rows) if bits == 4 else rows
        return dequantize_int8(codes, sv)
    return np.asarray(rows, dtype=np.float64)


def gqa_forward(inputs: dict, attrs: dict, present_key: np.ndarray | None = None,
                present_value: np.ndarray | None = None, share_buffer: bool = False,
                sample=None, window_inclusive: bool = True, bias_after_softcap: bool = True,
                head_of_group: str = "block") -> dict:
    """Forward pass of GroupQueryAttention; returns the output and present caches.

    inputs: numpy arrays keyed by the operator's input names (query, key,
      value, past_key, past_value, seqlens_k, total_sequence_length,
      cos_cache, sin_cache, attention_bias, head_sink, k_scale, v_scale,
      q_norm_weight, k_norm_weight); absent optional inputs are None/missing.
    attrs: the operator's attributes (DEFAULT_ATTRS holds the defaults).
    present_key / present_value: initial contents of the present buffers
      (rows that the operator does not write keep these bytes). With
      share_buffer=True they are ignored and the past buffers are updated in
      place, as when past and present are one allocation.
    sample: None for every output row, or an iterable of (b, h, i) triples;
      only those output rows are computed (the others stay 0). The caches
      are always updated in full.
    Returns output (dtype of query), output_f64, present_key/value, and the
    fp64 values of the appended rows before the storage cast
    (appended_key_f64 / appended_value_f64, (B, N_kv, S, H); the stored K
    rows come from the fp32 recipe instead) with their cache rows
    (appended_pos, (B, S)).

    com.microsoft.GroupQueryAttention: section Description (grouped-query
    attention over BSH Q/K/V and BNSH caches), sections Inputs / Outputs /
    Attributes, and section Implementation variants (share_append: new rows
    are appended at the live length and every causal bound is the live
    length from seqlens_k, right-aligned; quant_int8_decode_splitk: int8 rows
    are appended first and attention reads the cache as stored).
    """
    a = dict(DEFAULT_ATTRS)
    a.update(attrs)
    q_in = np.asarray(inputs["query"])
    k_in = np.asarray(inputs["key"])
    v_in = np.asarray(inputs["value"])
    out_dtype = q_in.dtype
    B, S, hidden_q = q_in.shape
    N, Nkv = int(a["num_heads"]), int(a["kv_num_heads"])
    if N % Nkv != 0:
        raise ValueError("num_heads must be a multiple of kv_num_heads")
    H = hidden_q // N
    G = N // Nkv
    if k_in.shape != (B, S, Nkv * H) or v_in.shape != (B, S, Nkv * H):
        raise ValueError("key/value must be (batch, sequence_length, kv_num_heads*head_size)")

    past_k = inputs.get("past_key")
    past_v = inputs.get("past_value")
    has_past = past_k is not None
    if share_buffer:
        if not has_past:
            raise ValueError("a shared buffer needs past_key/past_value")
        pk = np.array(past_k, copy=True)
        pv = np.array(past_v, copy=True)
    else:
        pk = np.array(present_key, copy=True)
        pv = np.array(present_value, copy=True)
    C = pk.shape[2]

    seqlens = np.asarray(inputs["seqlens_k"], dtype=np.int64).reshape(-1)
    total_len = int(np.asarray(inputs["total_sequence_length"]).reshape(-1)[0])
    kq, vq = a["k_quant_type"], a["v_quant_type"]
    # A prompt's float cache may have another float dtype than the query
    # (section Description: direct Q/K/V may store its generated cache as
    # float16 or float32); an existing cache has the query dtype.
    separate = kq == "NONE" and pk.dtype != out_dtype
    if separate and (has_past or pk.dtype not in (np.float16, np.float32)):
        raise ValueError("a float cache of another dtype than the query is only written by a prompt")
    attn_k = np.zeros((B, Nkv, C, H), dtype=out_dtype) if separate else pk
    attn_v = np.zeros((B, Nkv, C, H), dtype=out_dtype) if separate else pv
    bits = int(a["kv_cache_bit_width"])
    if kq != "NONE" and bits == 4 and has_past:
        raise ValueError("a 4-bit cache is built by a prompt (no past cache)")
    k_scale, v_scale = inputs.get("k_scale"), inputs.get("v_scale")
    qw, kw = inputs.get("q_norm_weight"), inputs.get("k_norm_weight")
    if (qw is None) != (kw is None):
        raise ValueError("q_norm_weight and k_norm_weight come together")
    eps = float(a["qk_norm_epsilon"])
    rotary = int(a["do_rotary"]) == 1
    cos_c = np.asarray(inputs["cos_cache"], dtype=np.float64) if rotary else None
    sin_c = np.asarray(inputs["sin_cache"], dtype=np.float64) if rotary else None
    causal = int(a["causal"]) == 1
    W = int(a["local_window_size"])
    scale = float(a["scale"]) if float(a["scale"]) != 0.0 else 1.0 / np.sqrt(H)
    softcap = float(a["softcap"])
    bias = None if inputs.get("attention_bias") is None else np.asarray(inputs["attention_bias"])
    sink = inputs.get("head_sink")
    smooth = int(a["smooth_softmax"]) == 1
    # Window-shift cache (section Attributes, sliding_window_cache; section
    # Implementation variants, window_shift: compact the surviving rows, append
    # the chunk, enforce the window floor and the causal bound).
    window_cache = int(a["sliding_window_cache"]) == 1
    if window_cache:
        if not causal or W <= 0:
            raise ValueError("sliding_window_cache needs causal attention and local_window_size > 0")
        if has_past and (C < S + W or np.asarray(past_k).shape[2] < W):
            raise ValueError("a window cache needs capacity >= S + local_window_size and a past of >= W rows")

    wanted = None
    if sample is not None:
        wanted = {}
        for (b, h, i) in sample:
            wanted.setdefault((int(b), int(h)), set()).add(int(i))

    out = np.zeros((B, S, N * H), dtype=np.float64)
    new_k = np.zeros((B, Nkv, S, H))
    new_v = np.zeros((B, Nkv, S, H))
    new_pos = np.zeros((B, S), dtype=np.int64)
    for b in range(B):
        total_b = int(seqlens[b]) + 1
        past_b = total_b - S if has_past else 0
        win = window_cache and has_past
        if win:
            if total_b < S or total_b > total_len:
                raise ValueError(f"batch {b}: seqlens_k inconsistent with the cache")
            n_old = min(past_b, np.asarray(past_k).shape[2])
            n_live = min(n_old + S, C)            # cache rows after the update
            keep = n_live - S                     # past rows that survive, most recent first kept
        else:
            if total_b < 1 or total_b > total_len or past_b < 0 or past_b + S > C or total_b > C:
                raise ValueError(f"batch {b}: seqlens_k inconsistent with the cache")
            n_live, keep = total_b, past_b
        off = total_b - n_live                    # absolute position of cache row 0
        pos = past_b + np.arange(S)               # absolute positions of the new rows
        rows_new = keep + np.arange(S)            # their cache rows

        # Cache update. Copy mode keeps the live past rows; a window cache keeps
        # the most recent `keep` of them at the front; then the S new rows are
        # appended at rows keep .. keep+S-1 (K: norm, then rotary at the
        # absolute position, then cast or int8 code; V: cast or int8 code).
        if win:
            pk[b, :, :keep] = np.asarray(past_k)[b, :, n_old - keep:n_old]
            pv[b, :, :keep] = np.asarray(past_v)[b, :, n_old - keep:n_old]
        elif has_past and not share_buffer:
            pk[b, :, :past_b] = np.asarray(past_k)[b, :, :past_b]
            pv[b, :, :past_b] = np.asarray(past_v)[b, :, :past_b]
        for g in range(Nkv):
            kr = k_in[b, :, g * H:(g + 1) * H].astype(np.float64)
            vr = v_in[b, :, g * H:(g + 1) * H].astype(np.float64)
            # The stored K row is the fp32 recipe (rms_norm_fp32, rotary_neox_fp32);
            # the fp64 row is kept beside it for the cross-check of that recipe.
            k32 = k_in[b, :, g * H:(g + 1) * H].astype(np.float32)
            if kw is not None:
                kr = rms_norm(kr, kw, eps)
                k32 = rms_norm_fp32(k32, kw, eps)
            if rotary:
                kr = rotary_neox(kr, cos_c[pos], sin_c[pos])
                k32 = rotary_neox_fp32(k32, inputs["cos_cache"][pos], inputs["sin_cache"][pos])
            pk[b, g, rows_new] = _store(k32, pk.dtype, kq, k_scale, g, H, bits)
            pv[b, g, rows_new] = _store(vr, pv.dtype, vq, v_scale, g, H, bits)
            if separate:   # the rows attention reads: the query dtype
                attn_k[b, g, rows_new] = k32.astype(out_dtype)
                attn_v[b, g, rows_new] = vr.astype(out_dtype)
            new_k[b, g], new_v[b, g] = kr, vr
        new_pos[b] = rows_new

        # Attention of every live query row over cache rows 0 .. n_live-1 as stored.
        live_rows = S if has_past else min(S, total_b)
        j = off + np.arange(n_live)               # absolute positions of cache rows 0 .. n_live-1
        for h in range(N):
            if wanted is not None and (b, h) not in wanted:
                continue
            rows = np.arange(live_rows)
            if wanted is not None:
                rows = np.array(sorted(i for i in wanted[(b, h)] if i < live_rows), dtype=np.int64)
                if rows.size == 0:
                    continue
            g = h // G if head_of_group == "block" else h % Nkv
            kd = _load(attn_k[b, g, :n_live], kq, k_scale, g, H, bits)
            vd = _load(attn_v[b, g, :n_live], vq, v_scale, g, H, bits)
            qr = q_in[b, rows, h * H:(h + 1) * H].astype(np.float64)
            if qw is not None:
                qr = rms_norm(qr, qw, eps)
            if rotary:
                qr = rotary_neox(qr, cos_c[pos[rows]], sin_c[pos[rows]])
            s = scale * (qr @ kd.T)                      # (rows, n_live)
            if bias_after_softcap:
                s = softcap_scores(s, softcap)
            if bias is not None:
                bb = bias[b if bias.shape[0] > 1 else 0, h if bias.shape[1] > 1 else 0]
                s = s + bb[rows][:, j].astype(np.float64)
            if not bias_after_softcap:
                s = softcap_scores(s, softcap)
            p = pos[rows][:, None]
            vis = np.ones_like(s, dtype=bool)
            if causal:
                vis &= j[None, :] <= p
            if W >= 0:
                vis &= (j[None, :] >= p - W) if window_inclusive else (j[None, :] > p - W)
            if sink is not None:
                sigma = float(np.asarray(sink, dtype=np.float64)[h])
            elif smooth:
                sigma = 0.0
            else:
                sigma = -np.inf
            smax = np.where(vis, s, -np.inf).max(axis=1)
            m = np.maximum(smax, sigma)
            ok = np.isfinite(m)                      # a row with no visible key and no sink
            m_safe = np.where(ok, m, 0.0)
            e = np.where(vis, np.exp(np.where(vis, s, 0.0) - m_safe[:, None]), 0.0)
            den = e.sum(axis=1) + (np.exp(sigma - m_safe) if np.isfinite(sigma) else 0.0)
            o = (e @ vd) / np.where(ok, den, 1.0)[:, None]
            out[b, rows, h * H:(h + 1) * H] = np.where(ok[:, None], o, 0.0)
    return dict(output=out.astype(out_dtype), output_f64=out, present_key=pk, present_value=pv,
                appended_key_f64=new_k, appended_value_f64=new_v, appended_pos=new_pos)
