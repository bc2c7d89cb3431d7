"""GPU-vs-oracle parity helpers (tests only).

Tolerances: output |gpu - ref| <= atol + rtol * |ref| with (2e-3, 1e-2) for
float16 and (1e-4, 1e-4) for float32 output, ref being the oracle's fp64
value. Present caches: byte for byte, every row, int8 and 4-bit codes
included (appended K rows follow the oracle's fp32 recipe of the stored rows).
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


def check_caches(case, gpu, ref):
    """Present caches byte for byte: copied and untouched rows keep their input bytes, appended V
    rows are the cast / code of the input, appended K rows the cast / code of the fp32 recipe."""
    for name in ("present_key", "present_value"):
        g_, r_ = gpu[name], ref[name]
        assert g_.shape == r_.shape and g_.dtype == r_.dtype
        neq = np.any(g_.reshape(g_.shape[:3] + (-1,)).view(np.uint8) != r_.reshape(r_.shape[:3] + (-1,)).view(np.uint8),
                     axis=-1)
        if neq.any():
            b, g, pos = (int(v) for v in np.argwhere(neq)[0])
            gr, rr = g_[b, g, pos], r_[b, g, pos]
            cols = np.nonzero(gr.view(np.uint8) != rr.view(np.uint8))[0][:4]
            raise AssertionError(f"{name}: {int(neq.sum())} rows differ, first [{b},{g},{pos}] bytes {cols}: "
                                 f"gpu {gr.view(np.uint8)[cols]}, oracle {rr.view(np.uint8)[cols]}")


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
