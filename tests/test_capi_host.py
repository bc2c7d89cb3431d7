"""The C-ABI library on the host: it loads, exports every symbol include/gqa.h
declares, and its host-side checks return the documented status codes.
No CUDA call is made (gqa_create / gqa_workspace_size are host-only), so this
runs without a GPU; device pointers are fake aligned addresses."""

import ctypes
import os
import re

import pytest

from grouped_query_attention_gb300 import capi
from grouped_query_attention_gb300.inputs import WORKLOADS, CaseSpec

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    if not os.path.exists(capi.LIB_PATH):
        from grouped_query_attention_gb300 import build
        build.build()
    return capi.load_library()


def test_exports_every_declared_symbol():
    header = open(os.path.join(ROOT, "include", "gqa.h")).read()
    declared = set(re.findall(r"GQA_API\s+[\w\s\*]+?\b(gqa_\w+)\s*\(", header))
    assert declared == set(capi.EXPORTS)
    lib = ctypes.CDLL(capi.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings():
    for code, name in enumerate(["GQA_OK", "GQA_ERR_INVALID_ARGUMENT", "GQA_ERR_UNSUPPORTED", "GQA_ERR_CUDA",
                                 "GQA_ERR_DEVICE_STATUS", "GQA_ERR_WORKSPACE"]):
        assert capi.gqa_status_string(code) == name


def test_attrs_defaults_match_page():
    a = capi.gqa_attrs_default()
    assert (a.causal, a.do_rotary, a.local_window_size, a.scale, a.softcap, a.smooth_softmax,
            a.k_quant_type, a.v_quant_type, a.sliding_window_cache) == (1, 0, -1, 0.0, 0.0, -1, 0, 0, 0)
    assert abs(a.qk_norm_epsilon - 1e-6) < 1e-12


@pytest.mark.parametrize("kw,status", [
    (dict(num_heads=6, kv_num_heads=4), capi.GQA_ERR_INVALID_ARGUMENT),
    (dict(num_heads=0, kv_num_heads=1), capi.GQA_ERR_INVALID_ARGUMENT),
    (dict(num_heads=4, kv_num_heads=2, causal=0, local_window_size=8), capi.GQA_ERR_INVALID_ARGUMENT),
    (dict(num_heads=4, kv_num_heads=2, local_window_size=-2), capi.GQA_ERR_INVALID_ARGUMENT),
    (dict(num_heads=4, kv_num_heads=2, softcap=-1.0), capi.GQA_ERR_INVALID_ARGUMENT),
    (dict(num_heads=4, kv_num_heads=2, k_quant_type=7), capi.GQA_ERR_INVALID_ARGUMENT),
    (dict(num_heads=4, kv_num_heads=2, sliding_window_cache=1), capi.GQA_ERR_INVALID_ARGUMENT),   # no window
    (dict(num_heads=4, kv_num_heads=2, sliding_window_cache=1, local_window_size=0), capi.GQA_ERR_INVALID_ARGUMENT),
    (dict(num_heads=4, kv_num_heads=2, sliding_window_cache=2, local_window_size=8), capi.GQA_ERR_INVALID_ARGUMENT),
    (dict(num_heads=4, kv_num_heads=2, k_quant_type=2, v_quant_type=2, kv_cache_bit_width=5),
     capi.GQA_ERR_INVALID_ARGUMENT),
])
def test_create_rejects(kw, status):
    with pytest.raises(capi.GqaError) as e:
        capi.gqa_create(capi.make_attrs(**kw))
    assert e.value.status == status


class FakeCall:
    """Descriptors of a call with fake 256-byte-aligned device addresses."""

    def __init__(self, dtype="f16", B=2, S=1, N=8, Nkv=2, H=128, C=64, mode="shared", **feat):
        self.next = 0x10000
        t = capi.GQA_F16 if dtype == "f16" else capi.GQA_F32
        bits = feat.get("bits", 8)
        cache_t = (capi.GQA_U8 if bits == 4 else capi.GQA_I8) if feat.get("quant") else t
        row = H // 2 if feat.get("quant") and bits == 4 else H
        self.inp = capi.GqaInputs()
        self.out = capi.GqaOutputs()
        self.inp.query = self.t(t, (B, S, N * H))
        self.inp.key = self.t(t, (B, S, Nkv * H))
        self.inp.value = self.t(t, (B, S, Nkv * H))
        self.inp.seqlens_k = self.t(capi.GQA_I32, (B,))
        self.inp.total_sequence_length = C if mode != "prompt" else S
        self.out.output = self.t(t, (B, S, N * H))
        self.out.present_key = self.t(cache_t, (B, Nkv, C, row))
        self.out.present_value = self.t(cache_t, (B, Nkv, C, row))
        if mode == "shared":
            self.inp.past_key = self.out.present_key
            self.inp.past_value = self.out.present_value
        if feat.get("quant"):
            n = 1 if feat["quant"] == "PER_TENSOR" else Nkv * H
            self.inp.k_scale = self.t(capi.GQA_F32, (n,))
            self.inp.v_scale = self.t(capi.GQA_F32, (n,))
        self.attrs = dict(num_heads=N, kv_num_heads=Nkv)
        if feat.get("quant"):
            self.attrs.update(k_quant_type=feat["quant"], v_quant_type=feat["quant"], kv_cache_bit_width=bits)

    def t(self, dtype, shape):
        self.next += 1 << 24
        return capi.describe(self.next, dtype, shape)

    def size(self, **attr_over):
        h = capi.gqa_create(capi.make_attrs(**{**self.attrs, **attr_over}))
        try:
            return capi.gqa_workspace_size(h, self.inp, self.out)
        finally:
            capi.gqa_destroy(h)


def _expect(call, status, **attr_over):
    with pytest.raises(capi.GqaError) as e:
        call.size(**attr_over)
    assert e.value.status == status, capi.gqa_last_error()


def test_valid_calls_have_a_workspace():
    for dtype in ("f16", "f32"):
        for S in (1, 64):
            assert FakeCall(dtype=dtype, S=S).size() > 0
    assert FakeCall(dtype="f32", quant="PER_CHANNEL").size() > 0


def test_workloads_validate():
    for name, sp in WORKLOADS.items():
        c = FakeCall(dtype=sp.dtype, B=sp.B, S=sp.S, N=sp.N, Nkv=sp.Nkv, H=sp.H, C=sp.capacity,
                     mode=sp.mode, quant=sp.quant if sp.quant != "NONE" else None, bits=sp.bits)
        if sp.sliding_window_cache:
            c.attrs.update(sliding_window_cache=1, local_window_size=sp.local_window_size)
        if sp.cache_dtype not in (None, sp.dtype):
            ct = capi.GQA_F32 if sp.cache_dtype == "f32" else capi.GQA_F16
            c.out.present_key = c.t(ct, (sp.B, sp.Nkv, sp.capacity, sp.H))
            c.out.present_value = c.t(ct, (sp.B, sp.Nkv, sp.capacity, sp.H))
        assert c.size() > 0, name


def test_shape_and_dtype_errors():
    c = FakeCall()
    c.inp.key = c.t(capi.GQA_F16, (2, 1, 3 * 128))                       # wrong KV hidden size
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)
    c = FakeCall()
    c.inp.key = capi.GqaTensor()                                          # packed QKV
    _expect(c, capi.GQA_ERR_UNSUPPORTED)
    c = FakeCall()
    c.inp.query = c.t(capi.GQA_BF16, (2, 1, 8 * 128))                     # bfloat16
    _expect(c, capi.GQA_ERR_UNSUPPORTED)
    c = FakeCall(dtype="f16", quant="PER_CHANNEL")                        # int8 cache needs fp32 Q/K/V
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)
    c = FakeCall(dtype="f32", quant="PER_CHANNEL")
    c.inp.k_scale = c.t(capi.GQA_F32, (7,))                               # scale length not 1 / N_kv*H
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)
    c = FakeCall()
    c.out.present_key = c.t(capi.GQA_F32, (2, 2, 64, 128))                # past of another dtype than query
    c.out.present_value = c.t(capi.GQA_F32, (2, 2, 64, 128))
    c.inp.past_key, c.inp.past_value = c.out.present_key, c.out.present_value
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)
    c = FakeCall(mode="prompt", S=4, C=64)
    c.out.present_key = c.t(capi.GQA_F32, (2, 2, 64, 128))                # K and V caches of two dtypes
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)
    c = FakeCall(H=40, N=8)                                               # head size not a multiple of 16
    _expect(c, capi.GQA_ERR_UNSUPPORTED)


def test_cache_mode_errors():
    c = FakeCall()
    c.inp.past_value = c.t(capi.GQA_F16, (2, 2, 64, 128))                 # K shared, V not
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)
    c = FakeCall(mode="copy")
    c.inp.past_key = c.t(capi.GQA_F16, (2, 2, 60, 128))                   # present != past + S
    c.inp.past_value = c.t(capi.GQA_F16, (2, 2, 60, 128))
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)
    c = FakeCall(mode="prompt", S=8, C=4)                                 # capacity < S
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)
    c = FakeCall()
    _expect(c, capi.GQA_ERR_UNSUPPORTED, causal=0)                         # bidirectional with a past


def test_optional_input_errors():
    c = FakeCall()
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT, do_rotary=1)                # rotary without cos/sin
    c = FakeCall()
    c.inp.cos_cache = c.t(capi.GQA_F16, (64, 32))                         # width != H/2
    c.inp.sin_cache = c.t(capi.GQA_F16, (64, 32))
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT, do_rotary=1)
    c = FakeCall()
    c.inp.q_norm_weight = c.t(capi.GQA_F16, (128,))                       # only one norm weight
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)
    c = FakeCall()
    c.inp.head_sink = c.t(capi.GQA_F16, (3,))                             # sink length != N
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)
    c = FakeCall()
    c.inp.attention_bias = c.t(capi.GQA_F16, (2, 3, 1, 64))               # head dim not 1 or N
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)
    c = FakeCall()
    c.inp.attention_bias = c.t(capi.GQA_F16, (1, 1, 1, 64))               # broadcast dims: fine
    assert c.size() > 0


def test_prompt_cache_of_another_float_dtype():
    """A prompt may write an fp32 cache for fp16 Q/K/V and the reverse; it takes the prefill regime
    and a workspace copy of the new rows in the query dtype."""
    for dtype, cache in (("f16", capi.GQA_F32), ("f32", capi.GQA_F16)):
        for S in (1, 40):
            c = FakeCall(dtype=dtype, mode="prompt", S=S, C=64)
            base = c.size()
            c.out.present_key = c.t(cache, (2, 2, 64, 128))
            c.out.present_value = c.t(cache, (2, 2, 64, 128))
            h = capi.gqa_create(capi.make_attrs(**c.attrs))
            try:
                info = capi.gqa_describe_plan(h, c.inp, c.out)
                assert info.regime == capi.GQA_REGIME_PREFILL
                esize = 2 if dtype == "f16" else 4
                assert info.workspace_bytes >= 2 * 2 * 2 * S * 128 * esize
                if S == 40:
                    assert info.workspace_bytes > base
            finally:
                capi.gqa_destroy(h)


def test_int4_cache_checks():
    """A 4-bit cache: uint8 rows of H/2 bytes, fp32 Q/K/V, prompt only, always the prefill regime."""
    c = FakeCall(dtype="f32", S=1, C=8, mode="prompt", quant="PER_CHANNEL", bits=4)
    assert c.size() > 0
    h = capi.gqa_create(capi.make_attrs(**c.attrs))
    try:
        assert capi.gqa_describe_plan(h, c.inp, c.out).regime == capi.GQA_REGIME_PREFILL
    finally:
        capi.gqa_destroy(h)
    c = FakeCall(dtype="f32", S=1, C=8, mode="shared", quant="PER_TENSOR", bits=4)   # a past cache
    _expect(c, capi.GQA_ERR_UNSUPPORTED)
    c = FakeCall(dtype="f32", S=4, C=8, mode="prompt", quant="PER_CHANNEL", bits=4)
    c.out.present_key = c.t(capi.GQA_U8, (2, 2, 8, 128))                 # row of H bytes, not H/2
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)
    c = FakeCall(dtype="f32", S=4, C=8, mode="prompt", quant="PER_CHANNEL", bits=4)
    c.out.present_key = c.t(capi.GQA_I8, (2, 2, 8, 64))                  # int8 dtype for a 4-bit cache
    c.out.present_value = c.t(capi.GQA_I8, (2, 2, 8, 64))
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)
    c = FakeCall(dtype="f32", S=4, C=8, mode="prompt", quant="PER_CHANNEL")
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT, kv_cache_bit_width=4)     # int8 buffers, 4-bit attribute


def test_window_cache_checks():
    """sliding_window_cache: capacity >= S + W (and a separate past of >= W rows); the
    present need not be past + S; total_sequence_length may exceed the capacity;
    the window-shift launch comes first, then the tensor-core decode (fp16, H=128,
    S*G <= 16) or the pre-pass and the CUDA-core prefill."""
    w = dict(sliding_window_cache=1, local_window_size=16)
    for S, regime, launches in ((1, capi.GQA_REGIME_DECODE, 2), (8, capi.GQA_REGIME_PREFILL, 3)):
        c = FakeCall(S=S, C=64)
        c.inp.total_sequence_length = 1000
        assert c.size(**w) > 0
        h = capi.gqa_create(capi.make_attrs(**{**c.attrs, **w}))
        try:
            info = capi.gqa_describe_plan(h, c.inp, c.out)
            assert info.regime == regime and info.launches == launches
        finally:
            capi.gqa_destroy(h)
    c = FakeCall(S=1, C=64)
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT, sliding_window_cache=1, local_window_size=64)   # C < S + W
    c = FakeCall(S=2, C=40, mode="copy")
    c.inp.past_key = c.t(capi.GQA_F16, (2, 2, 40, 128))                   # present = past, not past + S
    c.inp.past_value = c.t(capi.GQA_F16, (2, 2, 40, 128))
    assert c.size(**w) > 0
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)                               # without the window flag
    c.inp.past_key = c.t(capi.GQA_F16, (2, 2, 8, 128))                    # past shorter than the window
    c.inp.past_value = c.t(capi.GQA_F16, (2, 2, 8, 128))
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT, **w)


def test_total_length_beyond_capacity_rejected():
    c = FakeCall(C=64)
    c.inp.total_sequence_length = 65
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)


def test_plan_regimes():
    h = capi.gqa_create(capi.make_attrs(num_heads=8, kv_num_heads=2))
    try:
        c = FakeCall(S=1)
        info = capi.gqa_describe_plan(h, c.inp, c.out)
        assert info.regime == capi.GQA_REGIME_DECODE and info.launches == 1 and info.split_len >= 64
        c = FakeCall(S=64, C=128)
        info = capi.gqa_describe_plan(h, c.inp, c.out)
        assert info.regime == capi.GQA_REGIME_PREFILL and info.launches == 2
        assert info.workspace_bytes == capi.gqa_workspace_size(h, c.inp, c.out)
    finally:
        capi.gqa_destroy(h)


def test_misaligned_pointer_rejected():
    c = FakeCall()
    c.inp.query.data = c.inp.query.data + 2
    _expect(c, capi.GQA_ERR_INVALID_ARGUMENT)


def test_c_abi_from_plain_c(tmp_path):
    """include/gqa.h compiles as C11 and the library links and answers host-only calls from C."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(capi.LIB_PATH)
    exe = str(tmp_path / "host_check")
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi", "host_check.c"), "-L", libdir, "-lgqa_gb300",
           "-Wl,-rpath," + libdir, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert "c abi host check: ok" in r.stdout


def test_bias_staging_plan():
    """A bias shared by all heads with G >= 8 on the tensor-core prefill adds the bias-staging
    launch and its workspace (rows of a 16-byte multiple); per-head bias or G < 8 does not."""
    def plan(N, ndim, T=130):
        c = FakeCall(S=64, C=256, N=N, Nkv=2)
        c.inp.total_sequence_length = T
        c.inp.attention_bias = c.t(capi.GQA_F16, (1, ndim, 64, T))
        h = capi.gqa_create(capi.make_attrs(**c.attrs))
        try:
            return capi.gqa_describe_plan(h, c.inp, c.out)
        finally:
            capi.gqa_destroy(h)
    staged, per_head, small_group = plan(16, 1), plan(16, 16), plan(8, 1)
    assert staged.launches == 3 and per_head.launches == 2 and small_group.launches == 2
    # staged bias: 64 rows x ceil(130 / 4) * 4 floats, 256-byte aligned
    extra = staged.workspace_bytes - per_head.workspace_bytes
    assert extra >= 64 * 132 * 4 and extra < 64 * 132 * 4 + 256


def test_binding_constants_match_header():
    """The ctypes binding's enum values and kernel kinds are the header's."""
    header = open(os.path.join(ROOT, "include", "gqa.h")).read()
    kinds = {int(v): k for k, v in re.findall(r"#define GQA_KERNEL_(\w+) (\d+)", header)}
    assert {k: v.lower() for k, v in kinds.items()} == {k: v for k, v in capi.KERNEL_KINDS.items()}
    dt = dict(re.findall(r"(GQA_(?:DTYPE_NONE|F32|F16|I8|U8|I32|BF16)) = (\d+)", header))
    for name, value in dt.items():
        assert getattr(capi, name) == int(value), name
    reg = dict(re.findall(r"#define (GQA_REGIME_\w+) (\d+)", header))
    for name, value in reg.items():
        assert getattr(capi, name) == int(value), name


def test_set_wait_limit_argument_checks():
    """gqa_set_wait_limit: 0 (default) or >= 1000 cycles, withhold_copy >= -1, a handle."""
    lib = capi.load_library()
    h = capi.gqa_create(capi.make_attrs(4, 2))
    try:
        assert lib.gqa_set_wait_limit(None, 0, -1) == capi.GQA_ERR_INVALID_ARGUMENT
        assert lib.gqa_set_wait_limit(h, 999, -1) == capi.GQA_ERR_INVALID_ARGUMENT
        assert lib.gqa_set_wait_limit(h, -5, -1) == capi.GQA_ERR_INVALID_ARGUMENT
        assert lib.gqa_set_wait_limit(h, 2_000_000, -2) == capi.GQA_ERR_INVALID_ARGUMENT
        assert lib.gqa_set_wait_limit(h, 2_000_000, 0) == capi.GQA_OK
        assert lib.gqa_set_wait_limit(h, 0, -1) == capi.GQA_OK
    finally:
        capi.gqa_destroy(h)


def test_call_reuses_descriptors_while_tensors_stay(monkeypatch):
    """The binding rebuilds the C descriptors (and asks the workspace size again) only when a
    tensor's address, shape, dtype or layout, the total length or the set of inputs changes;
    every call passes the descriptors of the tensors it was given."""
    import torch

    import grouped_query_attention_gb300 as G

    sizes, seen = [], []
    monkeypatch.setattr(capi, "gqa_workspace_size", lambda h, i, o: sizes.append(1) or 256)
    monkeypatch.setattr(capi, "gqa_forward", lambda h, i, o, ws, n, st: seen.append(
        (i.query.data, i.query.shape[2], i.cos_cache.data, o.output.data, i.total_sequence_length)))
    op = G.GroupQueryAttention(num_heads=4, kv_num_heads=2)
    base = torch.zeros(256)
    q = base[:128].view(1, 1, 128)
    k, v = torch.zeros(1, 1, 64), torch.zeros(1, 1, 64)
    pk, pv = torch.zeros(1, 2, 8, 32), torch.zeros(1, 2, 8, 32)
    call = dict(query=q, key=k, value=v, seqlens_k=torch.zeros(1, dtype=torch.int32), total_sequence_length=1,
                present_key=pk, present_value=pv, output=torch.empty(1, 1, 128), past_key=pk, past_value=pv,
                workspace=torch.empty(256, dtype=torch.uint8), stream=0)
    op(**call)
    op(**call)
    assert len(sizes) == 1 and len(seen) == 2 and seen[0] == seen[1]
    q2 = torch.zeros(1, 1, 128)
    op(**dict(call, query=q2))                                  # another address
    assert len(sizes) == 2 and seen[-1][0] == q2.data_ptr()
    op(**dict(call, total_sequence_length=2))                   # another total length
    assert len(sizes) == 3 and seen[-1][4] == 2
    cos = torch.zeros(8, 16)
    op(**dict(call, cos_cache=cos, sin_cache=cos))              # another set of inputs
    assert len(sizes) == 4 and seen[-1][2] == cos.data_ptr()
    op(**call)
    assert len(sizes) == 5 and seen[-1] == seen[0]
    strided = base.as_strided((1, 1, 128), (256, 256, 2))      # same address, shape and dtype, not contiguous
    with pytest.raises(ValueError):
        op(**dict(call, query=strided))
