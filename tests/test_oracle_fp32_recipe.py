"""Pins of the oracle's fp32 recipe for the K rows stored in the cache.

The operator page fixes what a stored K row is (section Inputs: RMS norm with
q_norm_weight / k_norm_weight and qk_norm_epsilon, then rotary with
cos_cache / sin_cache; section Implementation variants: the appended row is
what attention reads) but not the fp32 evaluation order. The oracle computes
those rows in one fixed order (oracle.rms_norm_fp32, oracle.rotary_neox_fp32)
so that cache bytes can be compared exactly. These CPU tests pin that recipe:

* bit for bit against a scalar restatement written independently
  (tests/_brute.py: recursive pairwise tree, every operation rounded through
  numpy's fp32 scalar), for head sizes whose group count is and is not a
  power of two;
* against the fp64 definition within the rounding-error bound that the
  recipe's operation count gives (derived below), on random rows and on rows
  where rotary cancels most of a value;
* the evaluation order is observable: a plain left-to-right sum of squares
  gives other bytes on some rows, so the first pin really checks the order;
* planted mistakes (a dropped group, a wrong rotary sign, a missing epsilon)
  break the error bound;
* after the cast to fp16 every stored value is the fp16 rounding of a value
  within that bound of the exact one, and int8 codes differ from the codes of
  the exact value only where the exact value lies within the bound of a
  rounding tie.
"""

import numpy as np
import pytest

import oracle
from grouped_query_attention_gb300.inputs import rotary_tables
from tests._brute import f32, norm32, rope32

U = 2.0 ** -24       # unit roundoff of fp32


def _rows(rng, n, H, dtype=np.float32):
    return rng.standard_normal((n, H)).astype(dtype)


def _weights(rng, H, dtype=np.float32):
    return (1.0 + 0.1 * rng.standard_normal(H)).astype(dtype)


def _tree_depth(H):
    groups = H // 4
    depth = 0
    while (1 << depth) < groups:
        depth += 1
    return depth


def _norm_rel_bound(H):
    """Relative error bound of each value of rms_norm_fp32.

    ss: every square rounded once, then at most 3 + depth additions on the
    path of any term; all terms are positive, so |ss32 - ss| <= (4 + depth) u ss.
    ms = ss / H and v = ms + eps add one rounding each; sqrt halves the
    relative error and adds one rounding; 1 / sqrt adds one; (x * r) * w adds
    two. Total <= (4 + depth + 2) / 2 + 1 + 1 + 2 = 7 + depth / 2 roundings,
    doubled here to cover the second-order terms generously.
    """
    return (14 + _tree_depth(H)) * U


@pytest.mark.parametrize("H", [16, 32, 48, 64, 80, 128, 192, 256])
@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_recipe_matches_scalar_restatement(H, dtype):
    rng = np.random.default_rng(H)
    x = _rows(rng, 24, H, dtype)
    x[0] *= dtype(1e-3)                      # small row: eps matters
    x[1, :] = x[1, 0]                        # constant row
    w = _weights(rng, H, dtype)
    cos, sin = rotary_tables(64, H, 1e4, dtype)
    pos = rng.integers(0, 64, size=24)
    got_n = oracle.rms_norm_fp32(x, w, 1e-6)
    got_r = oracle.rotary_neox_fp32(got_n, cos[pos], sin[pos])
    got_rot_only = oracle.rotary_neox_fp32(x, cos[pos], sin[pos])
    for i in range(24):
        row = [float(v) for v in x[i]]
        n = norm32(row, w, 1e-6)
        assert np.array_equal(got_n[i], np.array(n, np.float32)), i
        assert np.array_equal(got_r[i], np.array(rope32(n, cos[pos[i]], sin[pos[i]]), np.float32)), i
        assert np.array_equal(got_rot_only[i], np.array(rope32(row, cos[pos[i]], sin[pos[i]]), np.float32)), i


def _exact_and_bound(x, w, cos_row, sin_row, eps):
    """fp64 norm + rotary of fp32 rows and the recipe's absolute error bound per value."""
    H = x.shape[-1]
    half = H // 2
    n64 = oracle.rms_norm(x.astype(np.float64), w.astype(np.float64), eps)
    y64 = oracle.rotary_neox(n64, cos_row, sin_row)
    en = _norm_rel_bound(H)
    c, s = np.asarray(cos_row, np.float64), np.asarray(sin_row, np.float64)
    a, b = n64[..., :half], n64[..., half:]
    terms = np.concatenate([np.abs(a * c) + np.abs(b * s), np.abs(b * c) + np.abs(a * s)], axis=-1)
    # rotary: operands carry the norm error, each product one rounding, the add one more
    bound = (en + 2 * U) * (1 + 4 * U) * terms + U * np.abs(y64)
    return y64, bound


@pytest.mark.parametrize("H", [32, 64, 128, 256])
def test_recipe_within_error_bound_of_fp64(H):
    rng = np.random.default_rng(100 + H)
    x = _rows(rng, 400, H)
    w = _weights(rng, H)
    cos, sin = rotary_tables(4096, H, 1e4, np.float32)
    pos = rng.integers(0, 4096, size=400)
    # rows where rotary cancels most of the first value: x[d] c ~ x[d+H/2] s
    for i in range(0, 400, 4):
        d = int(rng.integers(0, H // 2))
        c, s = float(cos[pos[i], d]), float(sin[pos[i], d])
        if abs(s) > 1e-3:
            x[i, d + H // 2] = np.float32(x[i, d] * c / s * (1 + 1e-6))
    y32 = oracle.rotary_neox_fp32(oracle.rms_norm_fp32(x, w, 1e-6), cos[pos], sin[pos]).astype(np.float64)
    y64, bound = _exact_and_bound(x, w, cos[pos], sin[pos], 1e-6)
    err = np.abs(y32 - y64)
    assert np.all(err <= bound), f"max err / bound {np.max(err / bound):.3f}"
    # norm alone: relative bound
    n32 = oracle.rms_norm_fp32(x, w, 1e-6).astype(np.float64)
    n64 = oracle.rms_norm(x.astype(np.float64), w.astype(np.float64), 1e-6)
    assert np.all(np.abs(n32 - n64) <= _norm_rel_bound(H) * np.abs(n64))


def test_recipe_order_is_observable():
    """A left-to-right fp32 sum of squares gives other bytes on some rows, so the bit-for-bit
    pin above distinguishes the recipe's order from a plausible other one."""
    rng = np.random.default_rng(7)
    H = 128
    x = _rows(rng, 2000, H)
    w = np.ones(H, np.float32)
    got = oracle.rms_norm_fp32(x, w, 1e-6)
    differs = 0
    for i in range(2000):
        ss = 0.0
        for v in x[i]:
            ss = f32(ss + f32(float(v) * float(v)))
        r = f32(1.0 / f32(np.sqrt(np.float32(f32(ss / H) + np.float32(1e-6)))))
        seq = np.array([f32(f32(float(v) * r) * 1.0) for v in x[i]], np.float32)
        differs += int(not np.array_equal(seq, got[i]))
    assert differs > 0


def test_planted_mistakes_break_the_bound():
    rng = np.random.default_rng(8)
    H = 128
    x = _rows(rng, 50, H)
    w = _weights(rng, H)
    cos, sin = rotary_tables(256, H, 1e4, np.float32)
    pos = rng.integers(1, 256, size=50)
    y64, bound = _exact_and_bound(x, w, cos[pos], sin[pos], 1e-6)

    def over(y):
        return np.any(np.abs(y.astype(np.float64) - y64) > bound)

    ss_bad = np.sum(x[:, 4:] * x[:, 4:], axis=-1, dtype=np.float32)      # one group left out of the sum
    r_bad = np.float32(1.0) / np.sqrt(ss_bad / np.float32(H) + np.float32(1e-6))
    n_bad = (x * r_bad[:, None]) * w
    assert over(oracle.rotary_neox_fp32(n_bad, cos[pos], sin[pos]))
    assert over(oracle.rotary_neox_fp32(oracle.rms_norm_fp32(x, w, 1e-6), cos[pos], -sin[pos]))   # wrong sign
    small = x * np.float32(1e-3)
    ys, bs = _exact_and_bound(small, w, cos[pos], sin[pos], 1e-6)
    no_eps = oracle.rotary_neox_fp32(oracle.rms_norm_fp32(small, w, 0.0), cos[pos], sin[pos])
    assert np.any(np.abs(no_eps.astype(np.float64) - ys) > bs)                                     # eps dropped


def test_stored_fp16_and_int8_values_are_roundings_within_the_bound():
    rng = np.random.default_rng(9)
    H = 128
    x = _rows(rng, 3000, H)
    w = _weights(rng, H)
    cos, sin = rotary_tables(8192, H, 1e4, np.float32)
    pos = rng.integers(0, 8192, size=3000)
    y32 = oracle.rotary_neox_fp32(oracle.rms_norm_fp32(x, w, 1e-6), cos[pos], sin[pos])
    y64, bound = _exact_and_bound(x, w, cos[pos], sin[pos], 1e-6)
    # fp16: the stored value is the rounding of some value within the bound of the exact one
    h = y32.astype(np.float16).astype(np.float64)
    lo = (y64 - bound).astype(np.float16).astype(np.float64)
    hi = (y64 + bound).astype(np.float16).astype(np.float64)
    assert np.all((h >= np.minimum(lo, hi)) & (h <= np.maximum(lo, hi)))
    # most values agree with the exact value's rounding; the others are one fp16 step away
    h64 = y64.astype(np.float16).astype(np.float64)
    assert np.mean(h == h64) > 0.999
    step = np.spacing(np.abs(y64).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(h - h64) <= step)
    # int8 codes (per-channel scales): differ only next to a tie of the exact value
    sc = rng.uniform(0.005, 0.02, size=H).astype(np.float32)
    q32 = oracle.quantize_int8(y32, sc).astype(np.int32)
    t64 = y64 / sc.astype(np.float64)
    q64 = np.clip(np.rint(t64), -127, 127).astype(np.int32)
    near_tie = np.abs(np.abs(t64 - np.floor(t64)) - 0.5) <= bound / sc + 2 * U * np.abs(t64)
    assert np.all((q32 == q64) | ((np.abs(q32 - q64) == 1) & near_tie))
