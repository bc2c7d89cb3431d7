"""GPU tests of buffer ownership: the caller's workspace, and nothing written
outside the output, present and workspace buffers.

* One handle and one workspace serve calls of different shapes and regimes in
  a row (decode with many (batch, KV head) merge tickets, decode with few, a
  prefill, then the large decode again); each call is checked against the
  oracle.
* The workspace is overwritten with 0xFF bytes between two calls (a caller
  that reuses its scratch arena for other work); the second call is still
  oracle-exact and reports no device error.
* Guard regions stand in for a memory checker: output, present caches and
  workspace each sit inside a larger buffer whose bytes before and after them
  hold a sentinel, for every regime (tensor-core and CUDA-core decode, plain
  and staged-bias chunked prefill on the tensor cores, the CUDA-core prefill
  with an int8 cache, a sliding-window cache). Every sentinel byte must be
  unchanged afterwards (section Outputs: present rows other than the appended
  ones keep their values; nothing else is the operator's to write).
"""

import numpy as np
import pytest
import torch

from grouped_query_attention_gb300 import GroupQueryAttention
from grouped_query_attention_gb300.inputs import CaseSpec, generate
from tests.parity import check_caches, check_output, run_oracle

pytestmark = pytest.mark.gpu

GUARD = 4096      # sentinel bytes on each side (a multiple of 256 keeps every view aligned)
SENTINEL = 0xA5

_OPTIONAL = ("past_key", "past_value", "cos_cache", "sin_cache", "attention_bias", "head_sink", "k_scale",
             "v_scale", "q_norm_weight", "k_norm_weight")


def _guarded(arr: np.ndarray):
    """A device copy of `arr` placed inside a sentinel-filled uint8 buffer: (buffer, view)."""
    arr = np.ascontiguousarray(arr)
    nbytes = arr.nbytes
    buf = torch.full((2 * GUARD + nbytes,), SENTINEL, dtype=torch.uint8, device="cuda")
    src = torch.from_numpy(arr.view(np.uint8).reshape(-1)).cuda()
    buf[GUARD:GUARD + nbytes].copy_(src)
    view = buf[GUARD:GUARD + nbytes].view(torch.from_numpy(arr[:0].copy()).dtype).view(arr.shape)
    return buf, view


def _guards_intact(buf: torch.Tensor) -> bool:
    head, tail = buf[:GUARD], buf[-GUARD:]
    return bool((head == SENTINEL).all().item()) and bool((tail == SENTINEL).all().item())


def _dev(case):
    return {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in case["inputs"].items()
            if v is not None and k != "total_sequence_length"}


def _call(op, case, dev, pk, pv, out, workspace=None):
    inp = case["inputs"]
    opt = {k: dev[k] for k in _OPTIONAL if k in dev}
    if case["share_buffer"]:
        opt["past_key"], opt["past_value"] = pk, pv
    op(dev["query"], dev["key"], dev["value"], dev["seqlens_k"], int(inp["total_sequence_length"][0]), pk, pv,
       output=out, workspace=workspace, **opt)


def _caches(case):
    if case["share_buffer"]:
        return case["inputs"]["past_key"], case["inputs"]["past_value"]
    return case["present_key"], case["present_value"]


def _check_against_oracle(case, out, pk, pv, op):
    torch.cuda.synchronize()
    status = op.device_status()
    assert status == 0, f"device status {status:#x}"
    gpu = dict(output=out.cpu().numpy(), present_key=pk.cpu().numpy(), present_value=pv.cpu().numpy())
    ref = run_oracle(case)
    check_output(case, gpu, ref)
    check_caches(case, gpu, ref)


ATTRS_SPEC = dict(dtype="f16", N=32, Nkv=8, H=128, rotary_theta=1e4, qk_norm=True)


def _shape_sequence():
    """Decode (B*N_kv = 128 tickets), decode (8 tickets), prefill, decode (128 tickets) on one handle."""
    return [
        CaseSpec(name="ws_decode_b16", B=16, S=1, capacity=1500, mode="shared", seqlens_range=(300, 1499),
                 **ATTRS_SPEC),
        CaseSpec(name="ws_decode_b1", B=1, S=1, capacity=3000, mode="shared", seqlens_range=(2000, 2999),
                 **ATTRS_SPEC),
        CaseSpec(name="ws_prefill", B=2, S=100, capacity=700, mode="shared", seqlens_range=(150, 699),
                 **ATTRS_SPEC),
        CaseSpec(name="ws_decode_b16_again", B=16, S=1, capacity=1500, mode="shared", seqlens_range=(300, 1499),
                 **ATTRS_SPEC),
    ]


def test_workspace_reused_across_shapes_and_regimes():
    specs = _shape_sequence()
    cases = [generate(sp, seed=70 + i) for i, sp in enumerate(specs)]
    op = GroupQueryAttention(**cases[0]["attrs"])
    # one workspace large enough for every call, reused as is
    need = 0
    prepared = []
    for case in cases:
        assert case["attrs"] == cases[0]["attrs"]
        dev = _dev(case)
        k0, v0 = _caches(case)
        pk = torch.from_numpy(np.ascontiguousarray(k0)).cuda()
        pv = torch.from_numpy(np.ascontiguousarray(v0)).cuda()
        out = torch.empty_like(dev["query"])
        opt = {k: dev[k] for k in _OPTIONAL if k in dev}
        if case["share_buffer"]:
            opt["past_key"], opt["past_value"] = pk, pv
        need = max(need, op.workspace_size(query=dev["query"], key=dev["key"], value=dev["value"],
                                           seqlens_k=dev["seqlens_k"],
                                           total_sequence_length=int(case["inputs"]["total_sequence_length"][0]),
                                           present_key=pk, present_value=pv, output=out, **opt))
        prepared.append((case, dev, pk, pv, out))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for case, dev, pk, pv, out in prepared:
        _call(op, case, dev, pk, pv, out, workspace=ws)
        _check_against_oracle(case, out, pk, pv, op)
    op.close()


@pytest.mark.parametrize("name", ["decode_tc", "decode_i8_tc", "decode_cuda_core", "prefill_tc"])
def test_workspace_overwritten_between_calls(name):
    specs = {
        "decode_tc": CaseSpec(name="ow_decode", B=16, S=1, capacity=2000, mode="shared",
                              seqlens_range=(500, 1999), **ATTRS_SPEC),
        "decode_i8_tc": CaseSpec(name="ow_i8", dtype="f32", B=8, S=1, N=32, Nkv=8, H=128, capacity=2000,
                                 mode="shared", seqlens_range=(500, 1999), quant="PER_CHANNEL"),
        "decode_cuda_core": CaseSpec(name="ow_f32", dtype="f32", B=8, S=1, N=16, Nkv=8, H=64, capacity=3000,
                                     mode="shared", seqlens_range=(500, 2999)),
        "prefill_tc": CaseSpec(name="ow_prefill", B=2, S=64, capacity=700, mode="shared",
                               seqlens_range=(150, 699), **ATTRS_SPEC),
    }
    case = generate(specs[name], seed=80)
    op = GroupQueryAttention(**case["attrs"])
    dev = _dev(case)
    k0, v0 = _caches(case)
    pk = torch.from_numpy(np.ascontiguousarray(k0)).cuda()
    pv = torch.from_numpy(np.ascontiguousarray(v0)).cuda()
    out = torch.empty_like(dev["query"])
    _call(op, case, dev, pk, pv, out)
    ws = op.last_workspace
    torch.cuda.synchronize()
    ws.fill_(0xFF)                       # the caller used its scratch for something else
    out.fill_(0)
    _call(op, case, dev, pk, pv, out, workspace=ws)   # appending the same rows again is idempotent
    _check_against_oracle(case, out, pk, pv, op)
    op.close()


GUARD_CASES = {
    "decode_tc_rotary_norm": CaseSpec(name="g_dec", dtype="f16", B=4, S=1, N=32, Nkv=8, H=128, capacity=1200,
                                      mode="shared", seqlens_range=(100, 1199), rotary_theta=1e4, qk_norm=True),
    "decode_i8_tc_copy": CaseSpec(name="g_i8", dtype="f32", B=3, S=2, N=8, Nkv=2, H=128, mode="copy",
                                  capacity=602, past_len=600, seqlens_range=(50, 590), quant="PER_CHANNEL"),
    "decode_cuda_core_f32": CaseSpec(name="g_f32", dtype="f32", B=3, S=2, N=8, Nkv=2, H=64, capacity=900,
                                     mode="shared", seqlens_range=(10, 899), softcap=20.0, bias=(3, 8, 0.5)),
    "prefill_tc_prompt": CaseSpec(name="g_pf", dtype="f16", B=2, S=300, N=16, Nkv=2, H=128, capacity=320,
                                  mode="prompt", seqlens_k=(299, 150), rotary_theta=1e4, qk_norm=True),
    "prefill_tc_staged_bias": CaseSpec(name="g_chunk", dtype="f16", B=2, S=70, N=16, Nkv=2, H=128, capacity=800,
                                       mode="shared", seqlens_range=(70, 799), local_window_size=90, softcap=30.0,
                                       bias=(1, 1, 0.5), head_sink=True, rotary_theta=1e4),
    "prefill_cuda_core_int8": CaseSpec(name="g_pf_i8", dtype="f32", B=2, S=40, N=8, Nkv=2, H=128, capacity=900,
                                       mode="shared", seqlens_range=(40, 899), quant="PER_TENSOR",
                                       scale_range=(0.02, 0.04), qk_norm=True, rotary_theta=1e4),
    "window_cache_decode": CaseSpec(name="g_win", dtype="f16", B=3, S=1, N=16, Nkv=2, H=128, capacity=300,
                                    mode="shared", seqlens_range=(250, 900), local_window_size=200,
                                    sliding_window_cache=1, rotary_theta=1e4),
    "window_cache_chunk_copy": CaseSpec(name="g_win_copy", dtype="f32", B=3, S=5, N=4, Nkv=2, H=128, mode="copy",
                                        capacity=155, past_len=150, seqlens_range=(10, 700), local_window_size=100,
                                        sliding_window_cache=1),
}


@pytest.mark.parametrize("name", sorted(GUARD_CASES))
def test_guard_regions_untouched(name):
    case = generate(GUARD_CASES[name], seed=90)
    op = GroupQueryAttention(**case["attrs"])
    dev = _dev(case)
    k0, v0 = _caches(case)
    kbuf, pk = _guarded(k0)
    vbuf, pv = _guarded(v0)
    obuf, out = _guarded(np.zeros(case["inputs"]["query"].shape, case["inputs"]["query"].dtype))
    opt = {k: dev[k] for k in _OPTIONAL if k in dev}
    if case["share_buffer"]:
        opt["past_key"], opt["past_value"] = pk, pv
    need = op.workspace_size(query=dev["query"], key=dev["key"], value=dev["value"], seqlens_k=dev["seqlens_k"],
                             total_sequence_length=int(case["inputs"]["total_sequence_length"][0]),
                             present_key=pk, present_value=pv, output=out, **opt)
    wbuf, ws = _guarded(np.zeros(need, np.uint8))
    _call(op, case, dev, pk, pv, out, workspace=ws)
    _check_against_oracle(case, out, pk, pv, op)
    for label, buf in (("output", obuf), ("present_key", kbuf), ("present_value", vbuf), ("workspace", wbuf)):
        assert _guards_intact(buf), f"{label}: bytes outside the buffer were written"
    op.close()
