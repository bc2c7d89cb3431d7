"""The benchmark's work accounting (CPU): visible (query, key) pairs, live K/V
bytes and the window-shift bytes, each against a brute-force count."""

import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from grouped_query_attention_gb300.inputs import WORKLOADS, CaseSpec, generate  # noqa: E402


def _brute_pairs(case):
    inp, at = case["inputs"], case["attrs"]
    B, S = inp["query"].shape[:2]
    N, Nkv, W = at["num_heads"], at["kv_num_heads"], at["local_window_size"]
    has_past = inp.get("past_key") is not None
    pairs = 0
    rows = 0
    for b in range(B):
        total = int(inp["seqlens_k"][b]) + 1
        past = total - S if has_past else 0
        live = S if has_past else min(S, total)
        for i in range(live):
            p = past + i
            for j in range(total):
                if at["causal"] and j > p:
                    continue
                if W >= 0 and j < p - W:
                    continue
                pairs += N
        kstart = max(0, past - W) if W >= 0 else 0
        rows += (total - kstart) * Nkv
    return pairs, rows


@pytest.mark.parametrize("kw", [
    dict(mode="prompt", S=7, capacity=9, seqlens_k=(6, 3)),
    dict(mode="prompt", S=7, capacity=7, seqlens_k=(6, 2), causal=0),
    dict(mode="shared", S=3, capacity=20, seqlens_k=(10, 19), local_window_size=4),
    dict(mode="copy", S=2, past_len=9, capacity=11, seqlens_k=(5, 10), local_window_size=0),
])
def test_visible_pairs_and_rows_match_brute_force(kw):
    spec = CaseSpec(name="acc", dtype="f32", B=2, N=4, Nkv=2, H=16, **kw)
    case = generate(spec, seed=3)
    assert bench.visible_pairs(case) == _brute_pairs(case)


def test_workload_units():
    """The published units of the headline workloads: live K/V bytes for decode,
    4*H flops per visible pair for prefill."""
    case = generate(WORKLOADS["prefill_f16_b4_s4096"], seed=0)
    w = bench.work(case)
    assert w["kind"] == "prefill" and abs(w["flops"] - 4 * 128 * 32 * 4 * 4096 * 4097 / 2) < 1
    case = generate(WORKLOADS["decode_f16_b16_c8192"], seed=0)
    w = bench.work(case)
    totals = case["inputs"]["seqlens_k"].astype(np.int64) + 1
    assert w["kind"] == "decode" and w["kv_bytes"] == int(totals.sum()) * 8 * 128 * 2 * 2


def test_window_shift_bytes():
    """Kept rows move (read + write, K and V) unless they are already at the front."""
    spec = CaseSpec(name="w", dtype="f16", B=3, S=1, N=4, Nkv=2, H=16, capacity=10, mode="shared",
                    seqlens_k=(3, 10, 25), local_window_size=5, sliding_window_cache=1)
    case = generate(spec, seed=1)
    # batch 0: past 3, kept 3 already at the front: nothing moves; batch 1: past 10 = C, the
    # 9 newest rows move by one; batch 2: past 25 -> n_old 10, the 9 newest rows move by one
    assert bench.window_shift_bytes(case) == 2 * 2 * (9 + 9) * 2 * 16 * 2
