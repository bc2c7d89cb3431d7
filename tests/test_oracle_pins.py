"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against a closed form, an invariant, a library
routine (torch SDPA / rms_norm in fp64) or the pure-Python brute force, chosen
so that a plausible mistake (a dropped term, a wrong sign or index, a
transposed operand, an off-by-one mask) fails at least one of them.
CPU only.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from grouped_query_attention_gb300.inputs import CaseSpec, generate, rotary_tables
from tests._brute import brute_forward


def run(case, **kw):
    return oracle.gqa_forward(case["inputs"], case["attrs"], case["present_key"],
                              case["present_value"], case["share_buffer"], **kw)


def tiny(**kw):
    base = dict(name="t", dtype="f32", B=2, S=3, N=4, Nkv=2, H=8, capacity=8, mode="prompt",
                seqlens_k=(2, 2))
    base.update(kw)
    return CaseSpec(**base)


# ---------------------------------------------------------------- brute force (whole pipeline)

BRUTE_CASES = {
    "prompt": tiny(),
    "prompt_padding": tiny(seqlens_k=(2, 1)),
    "shared_rotary_norm": tiny(mode="shared", S=2, capacity=9, seqlens_k=(5, 8), rotary_theta=1e4,
                               qk_norm=True),
    "copy_mode": tiny(mode="copy", S=2, past_len=5, seqlens_k=(6, 3), rotary_theta=100.0),
    "window_softcap_bias_sink": tiny(mode="shared", S=3, capacity=10, seqlens_k=(7, 9),
                                     local_window_size=2, softcap=0.7, bias=(2, 4, 0.5),
                                     head_sink=True, rotary_theta=1e3),
    "bias_broadcast_smooth": tiny(mode="shared", S=2, capacity=7, seqlens_k=(4, 6),
                                  bias=(1, 4, 1.0), smooth_softmax=1),
    "int8_per_channel": tiny(mode="shared", S=1, capacity=6, seqlens_k=(3, 5), quant="PER_CHANNEL",
                             scale_range=(0.01, 0.03)),
    "int8_per_tensor_norm_rotary": tiny(mode="shared", S=2, capacity=7, seqlens_k=(3, 6),
                                        quant="PER_TENSOR", qk_norm=True, rotary_theta=1e4,
                                        scale_range=(0.02, 0.03)),
    "f16_mha": tiny(dtype="f16", N=2, Nkv=2, mode="shared", S=2, capacity=6, seqlens_k=(3, 5)),
    "bidirectional": tiny(causal=0, seqlens_k=(2, 2)),
    "explicit_scale_g4": tiny(N=8, Nkv=2, scale=0.3, mode="shared", S=1, capacity=5, seqlens_k=(2, 4)),
    "f16_prompt_f32_cache_rotary": tiny(dtype="f16", S=4, capacity=6, seqlens_k=(3, 2), cache_dtype="f32",
                                        rotary_theta=1e4, qk_norm=True),
    "f32_prompt_f16_cache_bidirectional": tiny(S=4, capacity=5, seqlens_k=(3, 3), cache_dtype="f16", causal=0),
    "int4_per_channel_prompt": tiny(S=4, capacity=6, seqlens_k=(3, 2), quant="PER_CHANNEL", bits=4,
                                    scale_range=(0.15, 0.4)),
    "int4_per_tensor_norm_rotary": tiny(S=3, capacity=5, seqlens_k=(2, 2), quant="PER_TENSOR", bits=4,
                                        qk_norm=True, rotary_theta=1e4, scale_range=(0.2, 0.3)),
}


@pytest.mark.parametrize("name", sorted(BRUTE_CASES))
def test_brute_force_matches(name):
    case = generate(BRUTE_CASES[name], seed=7)
    res = run(case)
    out_b, pk_b, pv_b = brute_forward(case["inputs"], case["attrs"], case["present_key"],
                                      case["present_value"], case["share_buffer"])
    np.testing.assert_allclose(res["output_f64"], out_b, rtol=1e-11, atol=1e-12)
    for got, want in ((res["present_key"], pk_b), (res["present_value"], pv_b)):
        assert got.dtype == want.dtype
        assert np.array_equal(got, want)      # every cache byte, appended K rows included


def test_brute_force_catches_planted_mistakes():
    """A wrong rotary sign or a missing scale in the oracle would be caught by the brute force."""
    case = generate(BRUTE_CASES["shared_rotary_norm"], seed=3)
    out_b, _, _ = brute_forward(case["inputs"], case["attrs"], case["present_key"],
                                case["present_value"], case["share_buffer"])
    bad = dict(case["inputs"])
    bad["sin_cache"] = -bad["sin_cache"]                       # planted: rotation the wrong way
    res = oracle.gqa_forward(bad, case["attrs"], None, None, True)
    assert np.abs(res["output_f64"] - out_b).max() > 1e-3
    res2 = oracle.gqa_forward(case["inputs"], dict(case["attrs"], scale=0.5), None, None, True)
    assert np.abs(res2["output_f64"] - out_b).max() > 1e-3      # planted: wrong score scale


# ---------------------------------------------------------------- library routine: SDPA in fp64

def _sdpa_reference(case):
    """torch SDPA (fp64, CPU) over the cache rows with an explicit mask; no softcap/sink/norm/rotary."""
    inp, at = case["inputs"], case["attrs"]
    res = run(case)
    pk = res["present_key"].astype(np.float64)
    pv = res["present_value"].astype(np.float64)
    N, Nkv = at["num_heads"], at["kv_num_heads"]
    B, S, hq = inp["query"].shape
    H = hq // N
    G = N // Nkv
    out = np.zeros((B, S, N * H))
    has_past = inp.get("past_key") is not None
    for b in range(B):
        total = int(inp["seqlens_k"][b]) + 1
        past = total - S if has_past else 0
        q = torch.tensor(inp["query"][b].astype(np.float64).reshape(S, N, H).transpose(1, 0, 2))
        k = torch.tensor(pk[b, :, :total]).repeat_interleave(G, dim=0)
        v = torch.tensor(pv[b, :, :total]).repeat_interleave(G, dim=0)
        pos = past + torch.arange(S)[:, None]
        j = torch.arange(total)[None, :]
        vis = torch.ones(S, total, dtype=torch.bool)
        if at["causal"]:
            vis &= j <= pos
        if at["local_window_size"] >= 0:
            vis &= j >= pos - at["local_window_size"]
        mask = torch.zeros(N, S, total, dtype=torch.float64)
        mask = mask.masked_fill(~vis, float("-inf"))
        if inp.get("attention_bias") is not None:
            bias = torch.tensor(inp["attention_bias"].astype(np.float64))
            bias = bias[b if bias.shape[0] > 1 else 0][:, :, :total]
            mask = mask + bias.expand(N, S, total)
        scale = at["scale"] or 1.0 / math.sqrt(H)
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
        out[b] = o.transpose(0, 1).reshape(S, N * H).numpy()
        if not has_past:
            out[b, total:] = 0.0
    return res["output_f64"], out


@pytest.mark.parametrize("spec", [
    tiny(B=2, S=5, N=6, Nkv=3, H=16, capacity=5, seqlens_k=(4, 4)),
    tiny(mode="shared", B=3, S=4, N=8, Nkv=2, H=16, capacity=20, seqlens_k=(9, 19, 3)),
    tiny(mode="shared", B=2, S=3, N=4, Nkv=1, H=8, capacity=12, seqlens_k=(10, 6),
         local_window_size=3, bias=(2, 1, 0.7)),
    tiny(mode="shared", B=2, S=1, N=4, Nkv=2, H=8, capacity=12, seqlens_k=(11, 0)),
    tiny(mode="copy", B=2, S=2, N=4, Nkv=2, H=8, past_len=6, seqlens_k=(7, 4), bias=(1, 4, 1.0)),
    tiny(causal=0, B=1, S=6, capacity=6, seqlens_k=(5,)),
])
def test_matches_torch_sdpa_fp64(spec):
    got, want = _sdpa_reference(generate(spec, seed=11))
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_gqa_equals_mha_on_repeated_kv():
    """GQA with N/N_kv = G equals MHA on K/V heads repeated G times (head h reads KV head h // G)."""
    spec = tiny(mode="shared", B=2, S=2, N=6, Nkv=2, H=8, capacity=9, seqlens_k=(4, 8))
    case = generate(spec, seed=5)
    res = run(case)
    G = 3
    inp = dict(case["inputs"])
    B, S = 2, 2
    for name in ("key", "value"):
        x = inp[name].reshape(B, S, 2, 8)
        inp[name] = np.repeat(x, G, axis=2).reshape(B, S, 6 * 8)
    for name in ("past_key", "past_value"):
        inp[name] = np.repeat(inp[name], G, axis=1)
    mha = oracle.gqa_forward(inp, dict(case["attrs"], kv_num_heads=6), None, None, True)
    np.testing.assert_allclose(res["output_f64"], mha["output_f64"], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- closed forms of the softmax

def _equal_score_case(n_keys_live, sink=None, smooth=-1, window=-1, S=1):
    """Shared cache where every K row is the same unit vector a*e0 and V rows are distinct."""
    spec = tiny(mode="shared", B=1, S=S, N=2, Nkv=1, H=4, capacity=n_keys_live + 2,
                seqlens_k=(n_keys_live - 1,), local_window_size=window, smooth_softmax=smooth,
                head_sink=sink is not None)
    case = generate(spec, seed=1)
    inp = case["inputs"]
    a = 1.5
    inp["key"][:] = 0.0
    inp["key"][..., 0] = a
    inp["past_key"][:] = 0.0
    inp["past_key"][..., 0] = a
    inp["query"][:] = 0.0
    inp["query"].reshape(1, S, 2, 4)[..., 0] = a
    if sink is not None:
        inp["head_sink"][:] = sink
    return case, 0.5 * a * a          # score = scale * a^2 with scale = 1/sqrt(4)


def test_constant_v_returns_v():
    case, _ = _equal_score_case(6)
    inp = case["inputs"]
    inp["past_value"][:] = 0.25
    inp["value"][:] = 0.25
    # random (not equal) keys: the output must still be the constant
    inp["past_key"][:] = np.random.default_rng(0).standard_normal(inp["past_key"].shape)
    res = run(case)
    np.testing.assert_allclose(res["output_f64"], 0.25, rtol=1e-14)


def test_constant_v_with_sink_closed_form():
    n = 5
    for sink in (-1.0, 0.3, 2.0):
        case, s = _equal_score_case(n, sink=sink)
        inp = case["inputs"]
        inp["past_value"][:] = 0.5
        inp["value"][:] = 0.5
        res = run(case)
        sig = float(np.float32(sink))                       # the sink as stored (fp32)
        want = 0.5 * n * math.exp(s) / (n * math.exp(s) + math.exp(sig))
        np.testing.assert_allclose(res["output_f64"], want, rtol=1e-13)


def test_equal_scores_average_v_rows():
    """Equal scores over the n live keys give the plain mean of their V rows (no sink)."""
    n = 7
    case, _ = _equal_score_case(n)
    res = run(case)
    pv = res["present_value"].astype(np.float64)
    want = pv[0, 0, :n].mean(axis=0)
    for h in range(2):
        np.testing.assert_allclose(res["output_f64"][0, 0, h * 4:(h + 1) * 4], want, rtol=1e-13)


def test_window_reading_inclusive():
    """W=1: position p sees keys p-1 and p (left window plus self); W=0 sees only itself."""
    n = 6
    case, _ = _equal_score_case(n, window=1)
    res = run(case)
    pv = res["present_value"].astype(np.float64)
    want = (pv[0, 0, n - 2] + pv[0, 0, n - 1]) / 2
    np.testing.assert_allclose(res["output_f64"][0, 0, :4], want, rtol=1e-13)
    case0, _ = _equal_score_case(n, window=0)
    res0 = run(case0)
    np.testing.assert_allclose(res0["output_f64"][0, 0, :4],
                               res0["present_value"][0, 0, n - 1].astype(np.float64), rtol=1e-13)


def test_single_visible_key_first_prompt_row():
    spec = tiny(B=1, S=4, N=2, Nkv=1, H=8, capacity=4, seqlens_k=(3,))
    case = generate(spec, seed=2)
    res = run(case)
    v0 = case["inputs"]["value"][0, 0, :8].astype(np.float64)
    np.testing.assert_allclose(res["output_f64"][0, 0, :8], v0, rtol=1e-14)
    np.testing.assert_allclose(res["output_f64"][0, 0, 8:], v0, rtol=1e-14)


def test_sink_minus_inf_is_plain_softmax_and_smooth_equals_zero_sink():
    spec = tiny(mode="shared", S=2, capacity=9, seqlens_k=(5, 8), head_sink=True)
    case = generate(spec, seed=4)
    plain = oracle.gqa_forward({k: v for k, v in case["inputs"].items() if k != "head_sink"},
                               case["attrs"], None, None, True)
    inp = dict(case["inputs"])
    inp["head_sink"] = np.full_like(inp["head_sink"], -np.inf)
    res = oracle.gqa_forward(inp, case["attrs"], None, None, True)
    np.testing.assert_allclose(res["output_f64"], plain["output_f64"], rtol=1e-14)
    inp["head_sink"] = np.zeros_like(inp["head_sink"])
    zero_sink = oracle.gqa_forward(inp, case["attrs"], None, None, True)
    smooth = oracle.gqa_forward({k: v for k, v in case["inputs"].items() if k != "head_sink"},
                                dict(case["attrs"], smooth_softmax=1), None, None, True)
    np.testing.assert_allclose(smooth["output_f64"], zero_sink["output_f64"], rtol=1e-14)
    assert np.abs(smooth["output_f64"] - plain["output_f64"]).max() > 1e-3


def test_softcap_limits_and_bias_shift_invariance():
    spec = tiny(mode="shared", S=2, capacity=9, seqlens_k=(5, 8), bias=(2, 4, 1.0))
    case = generate(spec, seed=6)
    base = run(case)
    huge = oracle.gqa_forward(case["inputs"], dict(case["attrs"], softcap=1e9), None, None, True)
    np.testing.assert_allclose(huge["output_f64"], base["output_f64"], rtol=1e-9, atol=1e-12)
    inp = dict(case["inputs"])
    inp["attention_bias"] = (inp["attention_bias"].astype(np.float64) + 3.0).astype(np.float32)
    shifted = oracle.gqa_forward(inp, case["attrs"], None, None, True)
    np.testing.assert_allclose(shifted["output_f64"], base["output_f64"], rtol=1e-6, atol=1e-7)


def test_softcap_closed_form_two_keys():
    """Two keys with scores s0, s1: weights are softmax(c*tanh(s/c)) (then the bias)."""
    spec = tiny(mode="shared", B=1, S=1, N=1, Nkv=1, H=2, capacity=2, seqlens_k=(1,), softcap=0.8,
                bias=(1, 1, 1.0))
    case = generate(spec, seed=8)
    inp = case["inputs"]
    inp["query"][0, 0] = [1.0, 0.0]
    inp["past_key"][0, 0, 0] = [2.0, 0.0]
    inp["key"][0, 0] = [-1.0, 0.0]
    inp["past_value"][0, 0, 0] = [1.0, 0.0]
    inp["value"][0, 0] = [0.0, 1.0]
    inp["attention_bias"][:] = [[[[0.25, -0.5]]]]
    res = run(case)
    sc = 1 / math.sqrt(2)
    l0 = 0.8 * math.tanh(2.0 * sc / 0.8) + 0.25
    l1 = 0.8 * math.tanh(-1.0 * sc / 0.8) - 0.5
    w0 = 1 / (1 + math.exp(l1 - l0))
    np.testing.assert_allclose(res["output_f64"][0, 0], [w0, 1 - w0], rtol=1e-13)


def test_bias_broadcast_matches_expanded():
    spec = tiny(mode="shared", B=2, S=2, N=4, Nkv=2, capacity=8, seqlens_k=(5, 7), bias=(1, 1, 1.0))
    case = generate(spec, seed=9)
    res = run(case)
    inp = dict(case["inputs"])
    inp["attention_bias"] = np.broadcast_to(inp["attention_bias"], (2, 4) + inp["attention_bias"].shape[2:]).copy()
    full = oracle.gqa_forward(inp, case["attrs"], None, None, True)
    np.testing.assert_array_equal(res["output_f64"], full["output_f64"])


# ---------------------------------------------------------------- RMS norm and rotary

def test_rms_norm_closed_form_and_torch():
    x = np.array([3.0, 4.0])
    w = np.array([2.0, 0.5])
    got = oracle.rms_norm(x, w, 0.0)
    r = 1.0 / math.sqrt((9 + 16) / 2)
    np.testing.assert_allclose(got, [3 * r * 2, 4 * r * 0.5], rtol=1e-15)
    xs = np.random.default_rng(1).standard_normal((5, 64))
    ws = np.random.default_rng(2).standard_normal(64)
    t = torch.nn.functional.rms_norm(torch.tensor(xs), (64,), torch.tensor(ws), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rms_norm(xs, ws, 1e-6), t, rtol=1e-13)
    c = np.full(16, -0.1)
    np.testing.assert_allclose(oracle.rms_norm(c, np.ones(16), 1e-6),
                               -1.0 / math.sqrt(1 + 1e-6 / 0.01), rtol=1e-14)


def test_rotary_is_complex_rotation():
    H = 16
    rng = np.random.default_rng(3)
    x = rng.standard_normal(H)
    ang = rng.uniform(-3, 3, H // 2)
    got = oracle.rotary_neox(x, np.cos(ang), np.sin(ang))
    z = (x[:H // 2] + 1j * x[H // 2:]) * np.exp(1j * ang)
    np.testing.assert_allclose(got, np.concatenate([z.real, z.imag]), rtol=1e-14, atol=1e-15)


def test_rotary_norm_identity_composition_relative():
    H = 32
    cos, sin = rotary_tables(64, H, 1e4, np.float64)
    rng = np.random.default_rng(4)
    x, y = rng.standard_normal(H), rng.standard_normal(H)
    np.testing.assert_array_equal(oracle.rotary_neox(x, cos[0], sin[0]), x)         # p = 0
    r = oracle.rotary_neox(x, cos[17], sin[17])
    pair = lambda v: v[:H // 2] ** 2 + v[H // 2:] ** 2
    np.testing.assert_allclose(pair(r), pair(x), rtol=1e-13)                          # per-pair norm
    twice = oracle.rotary_neox(oracle.rotary_neox(x, cos[5], sin[5]), cos[12], sin[12])
    np.testing.assert_allclose(twice, r, rtol=1e-12, atol=1e-13)                        # 5 + 12 = 17
    d1 = oracle.rotary_neox(x, cos[20], sin[20]) @ oracle.rotary_neox(y, cos[13], sin[13])
    d2 = oracle.rotary_neox(x, cos[9], sin[9]) @ oracle.rotary_neox(y, cos[2], sin[2])
    np.testing.assert_allclose(d1, d2, rtol=1e-12)                                       # relative position


def test_rotary_position_is_absolute_in_cache():
    """New row i of a chunk over a past of length past_b is rotated at position past_b + i."""
    spec = tiny(mode="shared", B=1, S=2, N=2, Nkv=1, H=8, capacity=10, seqlens_k=(6,), rotary_theta=50.0)
    case = generate(spec, seed=12)
    res = run(case)
    inp = case["inputs"]
    for i in range(2):
        p = 5 + i
        k = inp["key"][0, i].astype(np.float64)
        half = 4
        stored = res["present_key"][0, 0, p].astype(np.float64)

        def rotated(q):
            z = (k[:half] + 1j * k[half:]) * (inp["cos_cache"][q].astype(np.float64)
                                              + 1j * inp["sin_cache"][q].astype(np.float64))
            return np.concatenate([z.real, z.imag])
        # the stored fp32 row (fp32 recipe: rounded products, then one add) is within a few fp32
        # rounding errors of the exact rotation at position p, and far from the neighbours' rotations
        bound = 3 * 2.0 ** -24 * (np.abs(k) + np.abs(np.roll(k, half)))
        assert np.all(np.abs(stored - rotated(p)) <= bound)
        for q in (p - 1, p + 1):
            assert np.abs(stored - rotated(q)).max() > 1e-3


# ---------------------------------------------------------------- int8 quantisation

def test_int8_round_trip_error_bound_saturation_ties():
    scale = np.float32(0.0125)
    codes = np.arange(-127, 128)
    vals = (codes * np.float64(scale)).astype(np.float32)
    assert np.array_equal(oracle.quantize_int8(vals, scale), codes.astype(np.int8))
    x = np.random.default_rng(5).uniform(-1.5, 1.5, 4096).astype(np.float32)
    q = oracle.quantize_int8(x, scale)
    assert np.all(np.abs(x - oracle.dequantize_int8(q, scale)) <= scale / 2 * (1 + 1e-6))
    assert oracle.quantize_int8(np.float32(100.0), scale) == 127
    assert oracle.quantize_int8(np.float32(-100.0), scale) == -127
    s1 = np.float32(1.0)
    assert list(oracle.quantize_int8(np.array([2.5, 3.5, -2.5, 0.5], np.float32), s1)) == [2, 4, -2, 0]


def test_int8_per_channel_scale_index():
    """PER_CHANNEL channel of KV head g, dim d is g*H + d."""
    spec = tiny(mode="shared", B=1, S=1, N=4, Nkv=2, H=8, capacity=3, seqlens_k=(1,), quant="PER_CHANNEL")
    case = generate(spec, seed=13)
    inp = case["inputs"]
    inp["k_scale"][:] = np.arange(1, 17, dtype=np.float32) / 64
    inp["key"][0, 0] = np.arange(1, 17, dtype=np.float32) / 64 * 3
    res = run(case)
    assert np.all(res["present_key"][0, :, 1] == 3)


# ---------------------------------------------------------------- int4 quantisation and packing

def test_int4_pack_layout_worked_example():
    """+8-biased nibbles, even head coordinate low (com.microsoft.GroupQueryAttention, section Inputs)."""
    codes = np.array([-7, 7, 0, 1, -8, 3], dtype=np.int8)
    # byte 0: low nibble -7+8 = 0x1, high 7+8 = 0xF; byte 1: 0x8 | 0x9 << 4; byte 2: 0x0 | 0xB << 4
    assert list(oracle.pack_int4(codes)) == [0xF1, 0x98, 0xB0]
    every = np.arange(256, dtype=np.uint8)
    assert np.array_equal(oracle.pack_int4(oracle.unpack_int4(every)), every)
    u = oracle.unpack_int4(every)
    assert u.min() == -8 and u.max() == 7 and list(u[:4]) == [-8, -8, -7, -8]


def test_int4_round_trip_error_bound_saturation_ties():
    scale = np.float32(0.25)
    codes = np.arange(-7, 8)
    vals = (codes * np.float64(scale)).astype(np.float32)
    assert np.array_equal(oracle.quantize_int4(vals, scale), codes.astype(np.int8))
    x = np.random.default_rng(6).uniform(-1.75, 1.75, 4096).astype(np.float32)
    q = oracle.quantize_int4(x, scale)
    assert np.all(np.abs(x - q * np.float64(scale)) <= scale / 2 * (1 + 1e-6))
    assert oracle.quantize_int4(np.float32(9.0), scale) == 7
    assert oracle.quantize_int4(np.float32(-9.0), scale) == -7      # symmetric: never -8
    s1 = np.float32(1.0)
    assert list(oracle.quantize_int4(np.array([2.5, 3.5, -2.5, 0.5, 6.5], np.float32), s1)) == [2, 4, -2, 0, 6]


def test_int4_prompt_cache_bytes_and_rejects_past():
    """A prompt writes packed codes of K/V into present rows [0, S); a past cache is rejected."""
    spec = tiny(B=1, S=2, N=2, Nkv=1, H=4, capacity=3, seqlens_k=(1,), quant="PER_TENSOR", bits=4)
    case = generate(spec, seed=21)
    inp = case["inputs"]
    inp["k_scale"][:] = 0.5
    inp["key"][0] = np.array([[1.0, -1.0, 3.5, -3.5], [0.25, 0.75, 9.0, -0.2]], np.float32)
    res = run(case)
    # codes [2,-2,7,-7] -> nibbles [10,6,15,1]; [0,2,7,0] -> nibbles [8,10,15,8] (0.25/0.5 ties to 0)
    assert list(res["present_key"][0, 0, 0]) == [10 | 6 << 4, 15 | 1 << 4]
    assert list(res["present_key"][0, 0, 1]) == [8 | 10 << 4, 15 | 8 << 4]
    assert np.array_equal(res["present_key"][0, 0, 2], case["present_key"][0, 0, 2])
    shared = generate(tiny(mode="shared", S=1, capacity=4, seqlens_k=(2, 3), quant="PER_TENSOR", bits=4),
                      seed=21)
    with pytest.raises(ValueError):
        run(shared)


# ---------------------------------------------------------------- prompt cache dtype

@pytest.mark.parametrize("dtype,cache", [("f16", "f32"), ("f32", "f16")])
def test_prompt_cache_dtype_does_not_change_the_output(dtype, cache):
    """A prompt's float cache may be float16 or float32 whatever the query dtype
    (com.microsoft.GroupQueryAttention, section Description): attention is computed
    from Q/K/V and the cache is written separately, so the output is the same as with
    a cache of the query dtype and the cache holds the rows rounded to its own dtype."""
    base = tiny(dtype=dtype, S=5, capacity=7, seqlens_k=(4, 2), rotary_theta=1e4, qk_norm=True)
    same = run(generate(base, seed=31))
    case = generate(base.with_(cache_dtype=cache), seed=31)
    other = run(case)
    assert np.array_equal(other["output_f64"], same["output_f64"])
    want = np.float32 if cache == "f32" else np.float16
    assert other["present_key"].dtype == want
    # the same fp32 row is stored in both caches: the fp32 cache's rows round to the fp16 cache's rows
    wide, narrow = (other, same) if cache == "f32" else (same, other)
    for name in ("present_key", "present_value"):
        np.testing.assert_array_equal(wide[name][:, :, :5].astype(np.float16), narrow[name][:, :, :5])
    # and each is within the fp32 recipe's rounding error of the fp64 row, rounded to its dtype
    x64 = other["appended_key_f64"]
    got = other["present_key"][:, :, :5].astype(np.float64)
    ulp = np.spacing(np.abs(x64).astype(want)).astype(np.float64)
    assert np.all(np.abs(got - x64) <= ulp + 1e-6 * np.abs(x64).max())
    np.testing.assert_array_equal(other["present_key"][:, :, 5:], case["present_key"][:, :, 5:])


def test_float_cache_of_another_dtype_with_a_past_is_rejected():
    case = generate(tiny(dtype="f16", mode="shared", S=1, capacity=4, seqlens_k=(1, 2)), seed=32)
    case["inputs"]["past_key"] = case["inputs"]["past_key"].astype(np.float32)
    case["inputs"]["past_value"] = case["inputs"]["past_value"].astype(np.float32)
    with pytest.raises(ValueError):
        run(case)


# ---------------------------------------------------------------- sliding-window cache

def _window_pair(S, W, L, C, totals, seed, share=True, rotary=True, bias=True):
    """The same call twice: over a full-history cache (no eviction) and over a
    window buffer holding the most recent rows of the same history."""
    big = max(totals) + 4
    spec = tiny(mode="shared", S=S, capacity=big, seqlens_k=tuple(t - 1 for t in totals), local_window_size=W,
                rotary_theta=1e4 if rotary else None, rotary_rows=big, bias=(2, 1, 0.5) if bias else None)
    full = generate(spec, seed=seed)
    inp = dict(full["inputs"])
    B, Nkv, H = 2, 2, 8
    dt = inp["past_key"].dtype
    win_k = np.zeros((B, Nkv, L, H), dt) + 7
    win_v = np.zeros((B, Nkv, L, H), dt) - 7
    for b, t in enumerate(totals):
        past = t - S
        n_old = min(past, L)
        win_k[b, :, :n_old] = inp["past_key"][b, :, past - n_old:past]
        win_v[b, :, :n_old] = inp["past_value"][b, :, past - n_old:past]
    attrs = dict(full["attrs"], sliding_window_cache=1)
    if share:
        inp_w = dict(inp, past_key=win_k, past_value=win_v)
        res_w = oracle.gqa_forward(inp_w, attrs, None, None, True)
    else:
        inp_w = dict(inp, past_key=win_k, past_value=win_v)
        pres_k = np.zeros((B, Nkv, C, H), dt) + 3
        pres_v = np.zeros((B, Nkv, C, H), dt) - 3
        res_w = oracle.gqa_forward(inp_w, attrs, pres_k, pres_v, False)
    res_full = oracle.gqa_forward(inp, full["attrs"], None, None, True)
    return res_full, res_w


@pytest.mark.parametrize("S,W,L,C,totals,share", [
    (1, 3, 4, 4, (9, 3), True),        # decode: full buffer evicts one row; short history no eviction
    (2, 2, 5, 5, (12, 6), True),       # chunk of two rows
    (3, 2, 4, 6, (10, 4), False),      # separate past (4 rows) and present (6 rows)
])
def test_window_cache_equals_full_history(S, W, L, C, totals, share):
    """Evicting keys that no query can see (window W, capacity >= S + W) changes
    nothing: the output equals attention over the full history, and the window
    buffer holds the most recent rows of the full cache, oldest first
    (com.microsoft.GroupQueryAttention, section Attributes, sliding_window_cache)."""
    full, win = _window_pair(S, W, L, C if not share else L, totals, seed=41, share=share)
    np.testing.assert_allclose(win["output_f64"], full["output_f64"], rtol=1e-12, atol=1e-14)
    cap = win["present_key"].shape[2]
    for b, t in enumerate(totals):
        n_live = min(min(t - S, L) + S, cap)
        np.testing.assert_array_equal(win["present_key"][b, :, :n_live], full["present_key"][b, :, t - n_live:t])
        np.testing.assert_array_equal(win["present_value"][b, :, :n_live], full["present_value"][b, :, t - n_live:t])


def test_window_cache_flag_without_past_changes_nothing():
    spec = tiny(S=4, capacity=6, seqlens_k=(3, 2), local_window_size=2)
    case = generate(spec, seed=42)
    a = run(case)
    b = oracle.gqa_forward(case["inputs"], dict(case["attrs"], sliding_window_cache=1), case["present_key"],
                           case["present_value"])
    assert np.array_equal(a["output_f64"], b["output_f64"])
    assert np.array_equal(a["present_key"], b["present_key"])


def test_window_cache_rejects_bad_settings():
    case = generate(tiny(mode="shared", S=1, capacity=4, seqlens_k=(5, 2), local_window_size=3), seed=43)
    for over in (dict(local_window_size=-1), dict(local_window_size=0), dict(local_window_size=4),
                 dict(causal=0, local_window_size=-1)):
        with pytest.raises(ValueError):
            oracle.gqa_forward(case["inputs"], dict(case["attrs"], sliding_window_cache=1, **over), None, None, True)


# ---------------------------------------------------------------- cache bookkeeping

def test_non_appended_rows_unchanged_shared_and_prompt():
    spec = tiny(mode="shared", B=3, S=2, capacity=12, seqlens_k=(3, 11, 6))
    case = generate(spec, seed=14)
    res = run(case)
    for name, src in (("present_key", "past_key"), ("present_value", "past_value")):
        before, after = case["inputs"][src], res[name]
        for b, sl in enumerate(case["inputs"]["seqlens_k"]):
            total = int(sl) + 1
            rows = np.ones(12, bool)
            rows[total - 2:total] = False
            assert np.array_equal(before[b][:, rows], after[b][:, rows])
            assert not np.array_equal(before[b][:, ~rows], after[b][:, ~rows])
    spec = tiny(B=2, S=3, capacity=10, seqlens_k=(2, 1))
    case = generate(spec, seed=15)
    res = run(case)
    assert np.array_equal(case["present_key"][:, :, 3:], res["present_key"][:, :, 3:])
    np.testing.assert_array_equal(res["present_key"][:, :, :3].reshape(2, 2, 3, 8),
                                  case["inputs"]["key"].reshape(2, 3, 2, 8).transpose(0, 2, 1, 3))


def test_copy_mode_copies_live_past_only():
    spec = tiny(mode="copy", B=2, S=2, past_len=5, seqlens_k=(6, 3))
    case = generate(spec, seed=16)
    res = run(case)
    for b, total in enumerate((7, 4)):
        past = total - 2
        assert np.array_equal(res["present_key"][b, :, :past], case["inputs"]["past_key"][b, :, :past])
        assert np.array_equal(res["present_key"][b, :, total:], case["present_key"][b, :, total:])


def test_prompt_padding_rows_zero():
    spec = tiny(B=2, S=4, capacity=4, seqlens_k=(3, 1))
    case = generate(spec, seed=17)
    res = run(case)
    assert np.all(res["output"][1, 2:] == 0)
    assert np.any(res["output"][1, :2] != 0)


def test_output_dtype_and_pages_example_shapes():
    """Shapes of the usage example on the page (tests/golden/usage_example_shapes.json):
    query (2,1,16), key/value (2,1,8), shared past/present (2,1,8,8), num_heads 2, kv_num_heads 1."""
    import json
    import os
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "usage_example_shapes.json")))
    sh = gold["shapes"]
    spec = CaseSpec(name="js", dtype="f32", B=2, S=1, N=gold["attrs"]["num_heads"],
                    Nkv=gold["attrs"]["kv_num_heads"], H=8, capacity=8, mode="shared", seqlens_k=(4, 7))
    case = generate(spec, seed=18)
    for name in ("query", "key", "value", "past_key", "past_value", "seqlens_k", "total_sequence_length"):
        assert list(case["inputs"][name].shape) == sh[name], name
    res = run(case)
    assert list(res["output"].shape) == sh["query"] and res["output"].dtype == np.float32
    assert list(res["present_key"].shape) == sh["present_key"]
    assert list(res["present_value"].shape) == sh["present_value"]
    spec16 = spec.with_(dtype="f16")
    res16 = run(generate(spec16, seed=18))
    assert res16["output"].dtype == np.float16


def test_rejects_inconsistent_inputs():
    case = generate(tiny(mode="shared", S=2, capacity=6, seqlens_k=(0, 3)), seed=19)
    with pytest.raises(ValueError):
        run(case)      # total 1 < S = 2 with a past cache
    case = generate(tiny(N=3, Nkv=2, H=8, seqlens_k=(2, 2)).with_(N=4), seed=19)
    with pytest.raises(ValueError):
        oracle.gqa_forward(case["inputs"], dict(case["attrs"], num_heads=3), case["present_key"],
                           case["present_value"])


# ---------------------------------------------------------------- randomized sweep against the brute force

def _random_spec(rng):
    Nkv = int(rng.choice([1, 2]))
    G = int(rng.choice([1, 2, 3]))
    H = int(rng.choice([4, 8]))
    dtype = str(rng.choice(["f32", "f16"]))
    mode = str(rng.choice(["prompt", "shared", "copy"]))
    S = int(rng.integers(1, 4))
    B = int(rng.integers(1, 3))
    kw = dict(name="r", dtype=dtype, B=B, S=S, N=G * Nkv, Nkv=Nkv, H=H, mode=mode)
    if mode == "prompt":
        kw.update(capacity=S + int(rng.integers(0, 2)), seqlens_k=tuple(int(x) for x in rng.integers(0, S, B)))
    elif mode == "shared":
        cap = S + int(rng.integers(1, 5))
        kw.update(capacity=cap, seqlens_k=tuple(int(x) for x in rng.integers(S - 1, cap, B)))
    else:
        past = int(rng.integers(1, 5))
        kw.update(capacity=past + S, past_len=past, seqlens_k=tuple(int(x) for x in rng.integers(S - 1, past + S, B)))
    causal = int(rng.integers(0, 2)) if mode == "prompt" else 1
    kw["causal"] = causal
    if causal and rng.random() < 0.4:
        kw["local_window_size"] = int(rng.integers(0, 4))
    if rng.random() < 0.4:
        kw["rotary_theta"] = 1e4
    if rng.random() < 0.3:
        kw["qk_norm"] = True
    if rng.random() < 0.3:
        kw["softcap"] = float(rng.choice([0.5, 3.0]))
    if rng.random() < 0.3:
        kw["bias"] = (int(rng.choice([1, B])), int(rng.choice([1, G * Nkv])), 0.5)
    if rng.random() < 0.3:
        kw["head_sink"] = True
    elif rng.random() < 0.3:
        kw["smooth_softmax"] = 1
    if dtype == "f32" and mode != "copy" and rng.random() < 0.3:
        kw.update(quant=str(rng.choice(["PER_TENSOR", "PER_CHANNEL"])), scale_range=(0.02, 0.2))
        if mode == "prompt" and rng.random() < 0.5:
            kw["bits"] = 4
    return CaseSpec(**kw)


@pytest.mark.parametrize("seed", range(24))
def test_random_configs_match_brute_force(seed):
    """Random small configurations (modes, features, quantised caches, dtypes) against the
    independently written brute force: outputs to 1e-11 relative, caches byte for byte."""
    spec = _random_spec(np.random.default_rng(1000 + seed))
    case = generate(spec, seed=seed)
    res = run(case)
    out_b, pk_b, pv_b = brute_forward(case["inputs"], case["attrs"], case["present_key"], case["present_value"],
                                      case["share_buffer"])
    np.testing.assert_allclose(res["output_f64"], out_b, rtol=1e-11, atol=1e-12)
    for got, want in ((res["present_key"], pk_b), (res["present_value"], pv_b)):
        assert got.dtype == want.dtype and np.array_equal(got, want)
