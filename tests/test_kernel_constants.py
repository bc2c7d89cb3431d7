"""Constants compiled into the CUDA kernels, checked on the CPU against the
functions they approximate (no GPU needed)."""

import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "grouped_query_attention_gb300",
                   "csrc", "prefill_tc.cu")


def _tanh_coefficients():
    text = open(SRC).read()
    c = [1.0]
    for k in range(1, 3):
        m = re.search(rf"constexpr float kTanhP{k} = ([-+0-9.eE]+)f;", text)
        assert m, f"kTanhP{k} not found"
        c.append(float(m.group(1)))
    return np.array(c, dtype=np.float32)


def test_softcap_polynomial_matches_tanh():
    """tanh(u) = u P(u^2) on |u| <= 1/8 (P of degree 2 in u^2): within 1e-8 relative in
    fp64, within 2 fp32 ulps when evaluated in fp32 Horner with fused multiply-adds."""
    c = _tanh_coefficients()
    u = np.linspace(-0.125, 0.125, 200001)
    u = u[u != 0]
    t = np.tanh(u)
    p64 = np.polyval(c.astype(np.float64)[::-1], u * u) * u
    assert np.max(np.abs(p64 - t) / np.abs(t)) < 1e-8
    u32 = u.astype(np.float32)
    z = (u32.astype(np.float64) ** 2).astype(np.float32)
    q = np.full_like(z, c[2])
    for k in (1, 0):   # fma: one rounding per step
        q = (q.astype(np.float64) * z + c[k]).astype(np.float32)
    p32 = (q.astype(np.float64) * u32).astype(np.float32)
    ref = np.tanh(u32.astype(np.float64))
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(p32 - ref) / ulp) < 2.0


def test_softcap_polynomial_is_odd_and_saturating_elsewhere():
    """The polynomial is used only for |u| <= 1/8; at the switch it still tracks tanh
    and its coefficients alternate in sign like tanh's series (-1/3, 2/15, ...)."""
    c = _tanh_coefficients()
    assert np.all(np.sign(c[1:]) == np.array([-1, 1]))
    assert abs(c[1] + 1 / 3) < 1e-4 and abs(c[2] - 2 / 15) < 5e-3
    u = np.float64(0.125)
    assert abs(np.polyval(c.astype(np.float64)[::-1], u * u) * u - np.tanh(u)) < 1e-8


def test_softcap_folded_coefficients_keep_the_accuracy():
    """The kernel evaluates x Q(x^2) on the raw product x with C_n = w P_n k^(2n)
    (k = scale / c, w = scale log2 e) rounded to fp32; at the workloads' scales this
    stays within 4 fp32 ulps of c tanh(x k) log2(e) over the polynomial's range."""
    c = _tanh_coefficients().astype(np.float32)
    for scale, cap in ((1 / np.sqrt(128), 50.0), (1 / np.sqrt(128), 20.0), (1 / np.sqrt(64), 30.0)):
        k = np.float32(scale / cap)
        w = np.float32(np.float32(scale) * np.float32(1.4426950408889634))
        k2 = np.float32(k * k)
        C, pw = [], np.float32(1.0)
        for n in range(3):
            C.append(np.float32(np.float32(w * c[n]) * pw))
            pw = np.float32(pw * k2)
        xmax = 0.125 / float(k)
        x = np.linspace(-xmax, xmax, 100001).astype(np.float32)
        x = x[x != 0]
        y = (x.astype(np.float64) ** 2).astype(np.float32)
        q = np.full_like(y, C[2])
        for n in (1, 0):
            q = (q.astype(np.float64) * y + C[n]).astype(np.float32)
        got = (x.astype(np.float64) * q).astype(np.float32).astype(np.float64)
        want = cap * np.tanh(x.astype(np.float64) * scale / cap) * 1.4426950408889634
        ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
        assert np.max(np.abs(got - want) / ulp) < 4.0
