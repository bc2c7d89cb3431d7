"""Bounded waits of the tensor-core kernels, made to expire without any fault.

With gqa_set_wait_limit(handle, 2e6 cycles, withhold_copy=0) the TMA warp of
every tensor-core CTA stops before the copy of its first key tile (the
converter warps before its conversion, in the prefill over an int8 cache), so
the waits for that tile run out (about 1 ms each at the maximum clock). The call
must return, the status word must report GQA_DEVICE_TIMEOUT, and an ordinary
call right after, on the same handle and workspace, must match the oracle:
tensor memory was freed and the merge tickets left behind are cleared by the
next call. Covers the fp16 and the int8-cache decode kernels, the fp16 prefill
kernel with and without the staged bias and the prefill over an int8 cache.
"""

import time

import numpy as np
import pytest
import torch

from grouped_query_attention_gb300 import GroupQueryAttention, capi
from grouped_query_attention_gb300.inputs import CaseSpec, generate
from tests.parity import check_caches, check_output, run_oracle

pytestmark = pytest.mark.gpu

CASES = {
    "decode_tc": (CaseSpec(name="to_dec", dtype="f16", B=2, S=1, N=8, Nkv=2, H=128, capacity=600, mode="shared",
                           seqlens_range=(200, 590), rotary_theta=1e4), "decode_tensor_core"),
    "decode_tc_i8": (CaseSpec(name="to_i8", dtype="f32", B=2, S=1, N=8, Nkv=2, H=128, capacity=600, mode="shared",
                              seqlens_range=(200, 590), quant="PER_CHANNEL"), "decode_tensor_core"),
    "prefill_tc": (CaseSpec(name="to_pf", dtype="f16", B=1, S=200, N=8, Nkv=2, H=128, capacity=256, mode="prompt",
                            seqlens_k=(199,), rotary_theta=1e4, qk_norm=True), "prefill_tensor_core"),
    "prefill_tc_int8_fp32": (CaseSpec(name="to_pq", dtype="f32", B=1, S=200, N=8, Nkv=2, H=128, capacity=256,
                                      mode="prompt", seqlens_k=(199,), quant="PER_CHANNEL"), "prefill_tensor_core"),
    "prefill_tc_staged_bias": (CaseSpec(name="to_ch", dtype="f16", B=1, S=64, N=16, Nkv=2, H=128, capacity=600,
                                        mode="shared", seqlens_range=(300, 590), softcap=30.0, bias=(1, 1, 0.5),
                                        rotary_theta=1e4), "prefill_tensor_core"),
}

_OPTIONAL = ("past_key", "past_value", "cos_cache", "sin_cache", "attention_bias", "head_sink", "k_scale",
             "v_scale", "q_norm_weight", "k_norm_weight")


@pytest.mark.parametrize("name", sorted(CASES))
def test_expired_wait_reports_timeout_then_next_call_is_exact(name):
    spec, kind = CASES[name]
    case = generate(spec, seed=60)
    inp = case["inputs"]
    dev = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in inp.items()
           if v is not None and k != "total_sequence_length"}
    if case["share_buffer"]:
        pk, pv = dev["past_key"], dev["past_value"]
    else:
        pk = torch.from_numpy(case["present_key"]).cuda()
        pv = torch.from_numpy(case["present_value"]).cuda()
    opt = {k: dev[k] for k in _OPTIONAL if k in dev}
    out = torch.empty_like(dev["query"])
    op = GroupQueryAttention(**case["attrs"])

    def call():
        op(dev["query"], dev["key"], dev["value"], dev["seqlens_k"], int(inp["total_sequence_length"][0]),
           pk, pv, output=out, **opt)

    capi.gqa_set_wait_limit(op.handle, 2_000_000, 0)
    capi.gqa_profile_begin(op.handle, 8)
    t0 = time.perf_counter()
    call()
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    kinds = [k for k, _ in capi.gqa_profile_end(op.handle)]
    assert kind in kinds, f"{name}: expected a {kind} launch, got {kinds}"
    status = op.device_status()
    assert status & capi.GQA_DEVICE_TIMEOUT, f"{name}: status {status:#x}"
    assert elapsed < 5.0

    capi.gqa_set_wait_limit(op.handle, 0, -1)     # ordinary call on the same handle and workspace
    out.fill_(0)
    call()
    torch.cuda.synchronize()
    assert op.device_status() == 0
    gpu = dict(output=out.cpu().numpy(), present_key=pk.cpu().numpy(), present_value=pv.cpu().numpy())
    ref = run_oracle(case)
    check_output(case, gpu, ref)
    check_caches(case, gpu, ref)
    op.close()
