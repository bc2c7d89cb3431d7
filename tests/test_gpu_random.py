"""GPU parity over random configurations: modes, regimes, masks, softcap, bias,
sinks, quantised caches, sliding-window caches and prompt cache dtypes drawn
at random (seeded), each compared in full with the fp64 oracle."""

import numpy as np
import pytest

from grouped_query_attention_gb300.inputs import CaseSpec, generate
from tests.parity import check_caches, check_output, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def random_spec(rng) -> CaseSpec:
    dtype = str(rng.choice(["f16", "f32"]))
    H = int(rng.choice([64, 128, 128, 128, 256]))
    Nkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8]))
    B = int(rng.integers(1, 4))
    mode = str(rng.choice(["prompt", "shared", "shared", "copy"]))
    S = int(rng.integers(1, 5)) if rng.random() < 0.5 else int(rng.integers(8, 81))
    kw = dict(name="rand", dtype=dtype, B=B, S=S, N=G * Nkv, Nkv=Nkv, H=H, mode=mode, seqlens_range=None)
    causal = 1 if mode != "prompt" else int(rng.random() < 0.8)
    kw["causal"] = causal
    window = int(rng.integers(0, 300)) if causal and rng.random() < 0.4 else -1
    kw["local_window_size"] = window
    win_cache = mode != "prompt" and window > 0 and rng.random() < 0.5
    if mode == "prompt":
        cap = S + int(rng.integers(0, 9))
        kw.update(capacity=cap, seqlens_k=tuple(int(x) for x in rng.integers(0, S, B)))
    elif mode == "shared":
        cap = S + int(rng.integers(50, 600))
        if win_cache:
            cap = max(cap, S + window)
            hi = 3 * cap
        else:
            hi = cap
        kw.update(capacity=cap, seqlens_k=tuple(int(x) for x in rng.integers(S - 1, hi, B)))
    else:
        past = int(rng.integers(10, 400))
        if win_cache:
            past = max(past, window)
            kw.update(capacity=past + S, past_len=past,
                      seqlens_k=tuple(int(x) for x in rng.integers(S - 1, 3 * (past + S), B)))
        else:
            kw.update(capacity=past + S, past_len=past, seqlens_k=tuple(int(x) for x in rng.integers(S - 1, past + S, B)))
    kw["sliding_window_cache"] = int(win_cache)
    if rng.random() < 0.5:
        kw["rotary_theta"] = float(rng.choice([1e4, 1e6]))
    if rng.random() < 0.3:
        kw["qk_norm"] = True
    if rng.random() < 0.3:
        kw["softcap"] = float(rng.choice([1.0, 20.0, 50.0]))
    if rng.random() < 0.3:
        kw["bias"] = (int(rng.choice([1, B])), int(rng.choice([1, G * Nkv])), float(rng.choice([0.5, 2.0])))
    if rng.random() < 0.25:
        kw["head_sink"] = True
    elif rng.random() < 0.2:
        kw["smooth_softmax"] = 1
    if dtype == "f32" and rng.random() < 0.4:
        kw.update(quant=str(rng.choice(["PER_TENSOR", "PER_CHANNEL"])), scale_range=(0.01, 0.05))
        if mode == "prompt" and rng.random() < 0.5:
            kw.update(bits=4, scale_range=(0.15, 0.4))
    elif mode == "prompt" and rng.random() < 0.3:
        kw["cache_dtype"] = "f32" if dtype == "f16" else "f16"
    return CaseSpec(**kw)


@pytest.mark.parametrize("seed", range(24))
def test_random_config_parity(seed):
    spec = random_spec(np.random.default_rng(5000 + seed))
    case = generate(spec, seed=seed)
    gpu = run_gpu(case)
    assert gpu["status"] == 0, f"device status {gpu['status']:#x} for {spec}"
    ref = run_oracle(case)
    check_output(case, gpu, ref)
    check_caches(case, gpu, ref)
