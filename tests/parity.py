"""GPU-vs-oracle parity helpers (tests only).

Tolerances: output |gpu - ref| <= atol + rtol * |ref| with (2e-3, 1e-2) for
float16 and (1e-4, 1e-4) for float32 output, ref being the oracle's fp64
value. Present caches: bit-exact, except appended K rows that went through
RMS norm / rotary, whose stored value must be the fp16 rounding of a value
within the fp32 compute error (8 fp32 ulps of the row's largest value) of the
oracle's fp64 value (fp16; where rotary cancels a value into the fp16
subnormal range that error spans more than one fp16 ulp), within 4 fp32 ulps
of the row scale (fp32), or, for int8 and 4-bit codes, either integer when
x/scale lies within 1e-3 of a half-integer.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from grouped_query_attention_gb300 import GroupQueryAttention

TOL = {np.float16: (2e-3, 1e-2), np.float32: (1e-4, 1e-4)}


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_gpu(case, op=None, repeat=1):
    """Run the case through the C ABI; returns host arrays and the device status."""
    inp, at = case["inputs"], case["attrs"]
    if op is None:
        op = GroupQueryAttention(**at)
    dev = {k: to_dev(v) for k, v in inp.items() if v is not None and k != "total_sequence_length"}
    if case["share_buffer"]:
        pk, pv = dev["past_key"], dev["past_value"]
    else:
        pk, pv = to_dev(case["present_key"]), to_dev(case["present_value"])
    opt = {k: dev[k] for k in ("past_key", "past_value", "cos_cache", "sin_cache", "attention_bias",
                               "head_sink", "k_scale", "v_scale", "q_norm_weight", "k_norm_weight") if k in dev}
    out = None
    for _ in range(repeat):
        out = op(dev["query"], dev["key"], dev["value"], dev["seqlens_k"], int(inp["total_sequence_length"][0]),
                 pk, pv, **opt)
    torch.cuda.synchronize()
    status = op.device_status()
    return dict(output=out.cpu().numpy(), present_key=pk.cpu().numpy(), present_value=pv.cpu().numpy(),
                status=status, op=op)


def run_oracle(case, sample=None):
    return oracle.gqa_forward(case["inputs"], case["attrs"], case["present_key"], case["present_value"],
                              case["share_buffer"], sample=sample)


def valid_rows(case):
    """(b, i) pairs whose output is defined (prompt padding rows excluded)."""
    inp = case["inputs"]
    B, S = inp["query"].shape[:2]
    has_past = inp.get("past_key") is not None
    ok = np.ones((B, S), dtype=bool)
    if not has_past:
        for b in range(B):
            ok[b, int(inp["seqlens_k"][b]) + 1:] = False
    return ok


def check_output(case, gpu, ref, sample=None):
    T = case["inputs"]["query"].dtype.type
    atol, rtol = TOL[T]
    B, S, NH = ref["output_f64"].shape
    N = case["attrs"]["num_heads"]
    H = NH // N
    got = gpu["output"].astype(np.float64).reshape(B, S, N, H)
    want = ref["output_f64"].reshape(B, S, N, H)
    if sample is None:
        ok = valid_rows(case)
        err = np.abs(got - want) - (atol + rtol * np.abs(want))
        bad = err[ok] > 0
        assert not bad.any(), (f"{int(bad.sum())} output values out of tolerance; max abs diff "
                               f"{np.abs(got - want)[ok].max():.3e}")
        pad = ~ok
        assert np.all(got[pad] == 0), "padding rows must be zero"
    else:
        for (b, h, i) in sample:
            g_, w_ = got[b, i, h], want[b, i, h]
            assert np.all(np.abs(g_ - w_) <= atol + rtol * np.abs(w_)), \
                f"row (b={b}, h={h}, i={i}): max diff {np.abs(g_ - w_).max():.3e}"
    return float(np.abs(got - want).max()) if sample is None else None


def _allowed_k_mismatch(case, ref, b, g, pos, gpu_row, ref_row):
    """Whether a differing appended K row is still a correct rounding of the oracle's fp64 row."""
    inp = case["inputs"]
    s_idx = np.where(ref["appended_pos"][b] == pos)[0]
    if s_idx.size == 0:
        return False
    x = ref["appended_key_f64"][b, g, s_idx[0]]
    if gpu_row.dtype == np.float16:
        # The kernel computes in fp32 (error <= eps32 below, relative to the row scale: rotary can
        # cancel down to values whose fp16 ulp is that small) and rounds once to fp16; the stored
        # value must be the fp16 rounding of some value within eps32 of the exact one.
        y = gpu_row.astype(np.float64)
        r = ref_row.astype(np.float64)
        eps32 = 8 * 2.0 ** -24 * np.abs(x).max()
        ulp = np.maximum(np.spacing(np.abs(gpu_row)).astype(np.float64), np.spacing(np.abs(ref_row)).astype(np.float64))
        ok = (y == r) | (np.abs(y - x) <= 0.5 * ulp + eps32)
        return bool(ok.all())
    if gpu_row.dtype == np.float32:
        y = gpu_row.astype(np.float64)
        bound = 4 * 2.0 ** -24 * (np.abs(x).max() + np.abs(x))
        return bool(np.all(np.abs(y - x) <= bound))
    if gpu_row.dtype in (np.int8, np.uint8):
        qt = case["attrs"]["k_quant_type"]
        H = x.shape[0]
        sc = np.asarray(inp["k_scale"], np.float32).reshape(-1)
        sc = np.full(H, sc[0], np.float32) if qt == "PER_TENSOR" else sc[g * H:(g + 1) * H]
        t = x.astype(np.float32) / sc
        if gpu_row.dtype == np.uint8:     # packed 4-bit codes: compare the codes
            gpu_row, ref_row = oracle.unpack_int4(gpu_row), oracle.unpack_int4(ref_row)
        diff = gpu_row.astype(np.int32) - ref_row.astype(np.int32)
        near_tie = np.abs(np.abs(t - np.trunc(t)) - 0.5) < 1e-3
        return bool(np.all((diff == 0) | ((np.abs(diff) == 1) & near_tie)))
    return False


def check_caches(case, gpu, ref):
    """Bit-exact caches (appended-K rounding rule aside); returns the number of tolerated K mismatches."""
    at = case["attrs"]
    k_processed = bool(at.get("do_rotary")) or case["inputs"].get("q_norm_weight") is not None
    tolerated = 0
    for name in ("present_key", "present_value"):
        g_, r_ = gpu[name], ref[name]
        assert g_.shape == r_.shape and g_.dtype == r_.dtype
        neq = np.any(g_.reshape(g_.shape[:3] + (-1,)).view(np.uint8) != r_.reshape(r_.shape[:3] + (-1,)).view(np.uint8),
                     axis=-1) if g_.dtype != np.int8 else np.any(g_ != r_, axis=-1)
        if not neq.any():
            continue
        assert name == "present_key" and k_processed, f"{name}: {int(neq.sum())} rows differ"
        for (b, g, pos) in zip(*np.nonzero(neq)):
            if not _allowed_k_mismatch(case, ref, b, g, pos, g_[b, g, pos], r_[b, g, pos]):
                gr, rr = g_[b, g, pos], r_[b, g, pos]
                cols = np.nonzero(gr != rr)[0][:4]
                s_idx = np.where(ref["appended_pos"][b] == pos)[0]
                x = ref["appended_key_f64"][b, g, s_idx[0]][cols] if s_idx.size else None
                raise AssertionError(f"{name}[{b},{g},{pos}] differs beyond the rounding rule: cols {cols}, "
                                     f"gpu {gr[cols]}, oracle {rr[cols]}, fp64 {x}")
            tolerated += 1
    return tolerated


def sample_rows(case, n, seed=0):
    """n random defined (b, h, i) output rows plus the last row of every batch (the decode row)."""
    inp = case["inputs"]
    B, S = inp["query"].shape[:2]
    N = case["attrs"]["num_heads"]
    ok = valid_rows(case)
    rng = np.random.default_rng(seed)
    out = set()
    for b in range(B):
        live = np.nonzero(ok[b])[0]
        out.add((b, int(rng.integers(N)), int(live[-1])))
    while len(out) < n + B:
        b = int(rng.integers(B))
        live = np.nonzero(ok[b])[0]
        out.add((b, int(rng.integers(N)), int(live[rng.integers(live.size)])))
    return sorted(out)
