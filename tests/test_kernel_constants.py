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
    for k in range(1, 6):
        m = re.search(rf"constexpr float kTanhP{k} = ([-+0-9.eE]+)f;", text)
        assert m, f"kTanhP{k} not found"
        c.append(float(m.group(1)))
    return np.array(c, dtype=np.float32)


def test_softcap_polynomial_matches_tanh():
    """tanh(u) = u P(u^2) on |u| <= 1/2: within 1e-8 relative in fp64, within 2 fp32 ulps
    when evaluated as the kernel does (fp32 Horner with fused multiply-adds)."""
    c = _tanh_coefficients()
    u = np.linspace(-0.5, 0.5, 200001)
    u = u[u != 0]
    t = np.tanh(u)
    p64 = np.polyval(c.astype(np.float64)[::-1], u * u) * u
    assert np.max(np.abs(p64 - t) / np.abs(t)) < 1e-8
    u32 = u.astype(np.float32)
    z = (u32.astype(np.float64) ** 2).astype(np.float32)
    q = np.full_like(z, c[5])
    for k in (4, 3, 2, 1, 0):   # fma: one rounding per step
        q = (q.astype(np.float64) * z + c[k]).astype(np.float32)
    p32 = (q.astype(np.float64) * u32).astype(np.float32)
    ref = np.tanh(u32.astype(np.float64))
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(p32 - ref) / ulp) < 2.0


def test_softcap_polynomial_is_odd_and_saturating_elsewhere():
    """The polynomial is used only for |u| <= 1/2; just past it, it still tracks tanh
    (no blow-up at the switch) and its coefficients alternate in sign like tanh's series."""
    c = _tanh_coefficients()
    assert np.all(np.sign(c[1:]) == np.array([-1, 1, -1, 1, -1]))
    u = np.float64(0.5)
    assert abs(np.polyval(c.astype(np.float64)[::-1], u * u) * u - np.tanh(u)) < 1e-8
