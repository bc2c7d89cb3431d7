"""gqa_forward_noalloc: the decode entry point for callers that cannot allocate
device memory (a plugin handed only its input and output buffers, or a
latency-critical path that must not call cudaMalloc). It takes its scratch from
a fixed array inside the library instead of a caller workspace.

Checked through the C ABI against gqa_forward on two calls in a row with
different shapes (so the shared scratch's tickets and partials are reused),
within the fp16 output tolerance of the parity tests, and with identical caches.
"""

import numpy as np
import pytest
import torch

from grouped_query_attention_gb300 import GroupQueryAttention, capi
from grouped_query_attention_gb300.inputs import CaseSpec, generate

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


def _device_case(case):
    inp = case["inputs"]
    dev = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in inp.items()
           if v is not None and k != "total_sequence_length"}
    opt = {k: dev[k] for k in ("past_key", "past_value", "cos_cache", "sin_cache") if k in dev}
    return dev, opt


def _run(case, noalloc: bool):
    inp = case["inputs"]
    dev, opt = _device_case(case)
    op = GroupQueryAttention(**case["attrs"])
    out = torch.empty_like(dev["query"])
    pk, pv = dev["past_key"], dev["past_value"]          # shared past/present buffer
    stream = torch.cuda.current_stream().cuda_stream
    if noalloc:
        ins, outs = op._structs(dev["query"], dev["key"], dev["value"], dev["seqlens_k"],
                                int(inp["total_sequence_length"][0]), pk, pv, out, **opt)
        capi.gqa_forward_noalloc(op.handle, ins, outs, stream)
    else:
        op(dev["query"], dev["key"], dev["value"], dev["seqlens_k"], int(inp["total_sequence_length"][0]),
           pk, pv, output=out, **opt)
    torch.cuda.synchronize()
    res = out.cpu().numpy().astype(np.float64), pk.cpu().numpy(), pv.cpu().numpy()
    op.close()
    return res


@pytest.mark.parametrize("call", [0, 1])
def test_noalloc_matches_forward_two_calls(call):
    specs = [
        CaseSpec(name="na0", dtype="f16", B=4, S=1, N=32, Nkv=8, H=128, capacity=4096, mode="shared",
                 seqlens_range=(500, 4095), rotary_theta=1e4),
        CaseSpec(name="na1", dtype="f16", B=3, S=2, N=8, Nkv=2, H=64, capacity=1500, mode="shared",
                 seqlens_range=(2, 1499)),
    ]
    for i, sp in enumerate(specs):           # two calls in a row on the shared scratch
        case = generate(sp, seed=40 + 10 * call + i)
        want, pk_w, pv_w = _run(case, noalloc=False)
        got, pk_g, pv_g = _run(case, noalloc=True)
        assert np.all(np.abs(got - want) <= ATOL + RTOL * np.abs(want)), sp.name
        assert np.array_equal(pk_g, pk_w) and np.array_equal(pv_g, pv_w), sp.name


def test_noalloc_rejects_prefill_regime():
    sp = CaseSpec(name="na_pf", dtype="f16", B=1, S=64, N=8, Nkv=2, H=128, capacity=64, mode="prompt",
                  seqlens_k=(63,))
    case = generate(sp, seed=3)
    inp = case["inputs"]
    dev, opt = _device_case(case)
    op = GroupQueryAttention(**case["attrs"])
    pk = torch.from_numpy(case["present_key"]).cuda()
    pv = torch.from_numpy(case["present_value"]).cuda()
    ins, outs = op._structs(dev["query"], dev["key"], dev["value"], dev["seqlens_k"],
                            int(inp["total_sequence_length"][0]), pk, pv, torch.empty_like(dev["query"]), **opt)
    with pytest.raises(capi.GqaError) as e:
        capi.gqa_forward_noalloc(op.handle, ins, outs, torch.cuda.current_stream().cuda_stream)
    assert e.value.status == capi.GQA_ERR_UNSUPPORTED
