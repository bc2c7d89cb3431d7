"""GPU parity: the CUDA library (through the C ABI) against the fp64 oracle.

Tiny sweeps cover every feature and cache mode, several splits / tiles and a
ragged tail in both regimes (fused split-KV decode for up to 8 query rows per
KV head, or 16 on the tensor-core decode; pre-pass + flash prefill
otherwise). The five workloads run at full size with the
launch configuration the benchmark uses; their outputs are checked on
sampled rows the oracle computes one by one (for the prefill workloads every
row of one whole KV-head group and the last 64 positions of every head) and
their caches in full, byte for byte.
"""

import numpy as np
import pytest

from grouped_query_attention_gb300.inputs import WORKLOADS, CaseSpec, generate
from tests.parity import check_caches, check_output, run_gpu, run_oracle, sample_rows, valid_rows

pytestmark = pytest.mark.gpu


def spec(**kw):
    base = dict(name="c", dtype="f16", B=3, S=1, N=8, Nkv=2, H=128, capacity=800, mode="shared",
                seqlens_range=(100, 700))
    base.update(kw)
    return CaseSpec(**base)


DECODE = {
    "f16_h128_g4_rotary": spec(rotary_theta=1e4),
    "f16_h64_g8_all_features": spec(H=64, N=16, Nkv=2, local_window_size=37, softcap=30.0, bias=(3, 16, 0.5),
                                    head_sink=True, qk_norm=True, rotary_theta=1e4),
    "f32_h128_g2_s2_smooth": spec(dtype="f32", N=4, Nkv=2, S=2, smooth_softmax=1, bias=(1, 4, 1.0)),
    "i8_per_channel_h128_g4": spec(dtype="f32", quant="PER_CHANNEL"),
    "i8_per_tensor_h64_s2_copy_norm_rotary": spec(dtype="f32", H=64, N=2, Nkv=2, S=2, mode="copy", past_len=600,
                                                  seqlens_range=(50, 590), quant="PER_TENSOR", qk_norm=True,
                                                  rotary_theta=1e4, scale_range=(0.02, 0.04)),
    "f16_g8_copy": spec(N=8, Nkv=1, mode="copy", past_len=500, seqlens_range=(1, 500)),
    "f16_prompt_s2_padding": spec(S=2, mode="prompt", capacity=4, seqlens_k=(0, 1, 1), seqlens_range=None,
                                  rotary_theta=1e4),
    "f32_g1_bias_shared": spec(dtype="f32", N=2, Nkv=2, bias=(1, 1, 0.5), seqlens_range=(0, 300)),
    "f16_long_many_splits": spec(B=2, capacity=6000, seqlens_range=(3000, 5999)),
    # degenerate windows and groups: a window of 0 keys besides self, one KV head for 64 query heads
    "f16_window0_decode": spec(local_window_size=0, rotary_theta=1e4),
    "f32_window1_g1_decode": spec(dtype="f32", N=2, Nkv=2, local_window_size=1, seqlens_range=(0, 300)),
    "f16_g64_decode_shape_prefill": spec(N=64, Nkv=1, seqlens_range=(100, 700), rotary_theta=1e4),
    # sliding-window cache: rows evicted from the front, compacted in place, new rows appended
    "f16_window_cache_decode": spec(S=1, capacity=300, seqlens_range=(250, 900), local_window_size=200,
                                    sliding_window_cache=1, rotary_theta=1e4),
    "i8_window_cache_decode": spec(dtype="f32", quant="PER_CHANNEL", capacity=200, seqlens_range=(100, 700),
                                   local_window_size=150, sliding_window_cache=1),
    "f32_window_cache_chunk_copy": spec(dtype="f32", S=5, mode="copy", past_len=150, seqlens_range=(10, 700),
                                        local_window_size=100, sliding_window_cache=1, bias=(3, 1, 0.5),
                                        softcap=20.0),
    "f16_window_cache_tc_all_features": spec(S=2, N=16, Nkv=2, capacity=300, seqlens_range=(200, 900),
                                             local_window_size=250, sliding_window_cache=1, bias=(3, 1, 0.5),
                                             softcap=30.0, rotary_theta=1e4, qk_norm=True, head_sink=True),
    "f16_window_cache_copy_decode": spec(S=1, mode="copy", past_len=300, seqlens_range=(100, 900),
                                         local_window_size=250, sliding_window_cache=1, rotary_theta=1e4),
    "f16_window_cache_g8_chunk": spec(S=16, N=16, Nkv=2, capacity=400, seqlens_range=(16, 1500),
                                      local_window_size=300, sliding_window_cache=1, qk_norm=True,
                                      rotary_theta=1e4, head_sink=True),
    "f16_window_zero": spec(local_window_size=0),
    "f32_bidirectional_prompt": spec(dtype="f32", mode="prompt", capacity=1, S=1, N=4, Nkv=1, causal=0,
                                     seqlens_k=(0, 0, 0), seqlens_range=None),
    # tensor-core decode (fp16, head size 128): 16 query rows per KV head, every feature
    "f16_tc_r16_all_features": spec(N=16, Nkv=2, S=2, capacity=1200, seqlens_range=(1, 1100),
                                    local_window_size=300, softcap=20.0, bias=(3, 16, 0.5), head_sink=True,
                                    qk_norm=True, rotary_theta=1e4),
    "f16_tc_r16_smooth_short": spec(N=16, Nkv=1, S=1, capacity=300, seqlens_range=(0, 299), smooth_softmax=1),
    # one (b, g) spread over every CTA: a merge of one partial per CTA
    "f16_tc_one_head_long": spec(B=1, N=8, Nkv=1, capacity=40000, seqlens_range=(39000, 39990), rotary_theta=1e4),
    # fewer tiles than CTAs (only the first CTAs work)
    "f16_tc_few_tiles": spec(B=2, N=4, Nkv=2, capacity=200, seqlens_range=(0, 150)),
    # new rows straddling a 128-key tile boundary (keys 1022..1025), S*G = 16
    "f16_tc_s4_straddle": spec(S=4, N=16, Nkv=4, capacity=1100, seqlens_k=(1025, 130, 3), seqlens_range=None,
                               rotary_theta=1e4, qk_norm=True),
    # tensor-core decode for int8 caches with fp32 queries (head size 128, up to 8 rows per KV head)
    "i8_tc_per_tensor_s2_copy_norm_rotary": spec(dtype="f32", N=8, Nkv=2, S=2, mode="copy", past_len=600,
                                                  seqlens_range=(50, 590), quant="PER_TENSOR", qk_norm=True,
                                                  rotary_theta=1e4, scale_range=(0.02, 0.04)),
    "i8_tc_all_features": spec(dtype="f32", N=8, Nkv=4, quant="PER_CHANNEL", seqlens_range=(1, 700),
                               local_window_size=200, softcap=30.0, bias=(3, 8, 0.5), head_sink=True, qk_norm=True,
                               rotary_theta=1e4),
    "i8_tc_one_head_long": spec(dtype="f32", B=1, N=8, Nkv=1, capacity=20000, seqlens_range=(19000, 19990),
                                quant="PER_CHANNEL"),
}

PREFILL = {
    "f32_prompt_tiny": WORKLOADS["prompt_f32_b1_s16"],
    "f32_prompt_padding_h64_g4": spec(dtype="f32", H=64, N=8, Nkv=2, S=37, mode="prompt", capacity=40,
                                      seqlens_k=(20, 36, 0), seqlens_range=None),
    "f32_chunk_all_features": spec(dtype="f32", S=9, N=8, Nkv=2, local_window_size=50, softcap=20.0,
                                   bias=(3, 8, 0.5), head_sink=True, qk_norm=True, rotary_theta=1e4),
    "i8_per_channel_prefill": spec(dtype="f32", S=17, quant="PER_CHANNEL"),
    "i8_per_tensor_prefill_all_features": spec(dtype="f32", S=40, N=8, Nkv=2, quant="PER_TENSOR",
                                               scale_range=(0.02, 0.04), local_window_size=60, softcap=20.0,
                                               bias=(3, 8, 0.5), head_sink=True, qk_norm=True, rotary_theta=1e4),
    "i8_per_channel_prompt_h64_g8": spec(dtype="f32", H=64, N=16, Nkv=2, S=70, mode="prompt", capacity=80,
                                         seqlens_k=(69, 33, 1), seqlens_range=None, quant="PER_CHANNEL"),
    "f16_h256_g2": spec(H=256, N=4, Nkv=2, S=20, capacity=500, seqlens_range=(20, 480)),
    # head sizes whose group count (H/4) is not a power of two: the generic pre-pass pads the
    # norm's pairwise tree with zero groups; H = 192 in fp32 spreads a row over two lane blocks
    "f16_h48_norm_rotary_generic_prepass": spec(H=48, N=4, Nkv=2, S=9, capacity=300, seqlens_range=(9, 290),
                                                qk_norm=True, rotary_theta=1e4),
    "f32_h80_norm_rotary_i8": spec(dtype="f32", H=80, N=4, Nkv=2, S=6, capacity=300, seqlens_range=(6, 290),
                                   qk_norm=True, rotary_theta=1e4, quant="PER_CHANNEL", scale_range=(0.01, 0.03)),
    "f32_h192_norm_rotary": spec(dtype="f32", H=192, N=4, Nkv=2, S=7, capacity=300, seqlens_range=(7, 290),
                                 qk_norm=True, rotary_theta=1e4),
    "f16_h128_g8_s65": spec(N=16, Nkv=2, S=65, seqlens_range=(65, 700), rotary_theta=1e4, qk_norm=True),
    "f16_copy_s12": spec(S=12, N=8, Nkv=2, mode="copy", past_len=300, seqlens_range=(11, 311)),
    "f32_bidirectional_prompt_s33": spec(dtype="f32", N=4, Nkv=2, S=33, mode="prompt", capacity=33, causal=0,
                                         seqlens_k=(32, 20, 5), seqlens_range=None),
    "f16_h32_smooth_window": spec(H=32, N=4, Nkv=1, S=24, local_window_size=5, smooth_softmax=1),
    # tensor-core path (fp16, head size 128): ragged key tiles, query-tile tails, every feature
    "f16_tc_all_features": spec(S=40, N=16, Nkv=2, local_window_size=100, softcap=30.0, bias=(3, 16, 0.5),
                                head_sink=True, qk_norm=True, rotary_theta=1e4, seqlens_range=(40, 700)),
    "f16_tc_prompt_padding_bias": spec(S=150, N=8, Nkv=2, mode="prompt", capacity=160, seqlens_k=(149, 70, 3),
                                       seqlens_range=None, bias=(1, 1, 1.0)),
    "f16_tc_bidirectional": spec(S=130, N=4, Nkv=2, mode="prompt", capacity=130, causal=0,
                                 seqlens_k=(129, 100, 7), seqlens_range=None),
    "f16_tc_smooth_multi_block": spec(B=2, S=300, N=8, Nkv=2, capacity=2500, seqlens_range=(300, 2400),
                                      smooth_softmax=1, rotary_theta=1e4),
    "f16_tc_window0": spec(S=40, N=16, Nkv=2, local_window_size=0, seqlens_range=(40, 700)),
    "f16_tc_single_key_prompt": spec(S=1, N=8, Nkv=1, mode="prompt", capacity=1, seqlens_k=(0, 0, 0),
                                     seqlens_range=None, rotary_theta=1e4, qk_norm=True),
    # bias shared by all heads with G >= 8: staged through shared memory by the TMA warp
    "f16_tc_staged_bias_softcap_window": spec(S=70, N=16, Nkv=2, local_window_size=90, softcap=30.0,
                                              bias=(3, 1, 0.5), head_sink=True, rotary_theta=1e4,
                                              seqlens_range=(70, 700)),
    "f16_tc_bias_g6_prompt_padding": spec(S=150, N=12, Nkv=2, mode="prompt", capacity=160,
                                          seqlens_k=(149, 70, 3), seqlens_range=None, bias=(1, 1, 1.0)),
    "f16_tc_staged_bias_g8_prompt_padding": spec(S=150, N=16, Nkv=2, mode="prompt", capacity=160,
                                                 seqlens_k=(149, 70, 3), seqlens_range=None, bias=(1, 1, 1.0)),
    # bias of large spread: the reference max rises inside a tile (second half) and across tiles
    "f16_tc_staged_bias_large_spread": spec(S=64, N=16, Nkv=2, softcap=30.0, bias=(1, 1, 8.0),
                                            seqlens_range=(64, 600)),
    "f16_tc_per_head_bias_large_spread": spec(S=40, N=4, Nkv=2, bias=(3, 4, 8.0), seqlens_range=(40, 500)),
    # softcap small against the scores: the exp2 / reciprocal form instead of the polynomial
    "f16_tc_small_softcap": spec(S=40, N=16, Nkv=2, softcap=1.0, seqlens_range=(40, 700), rotary_theta=1e4),
    "f16_tc_staged_bias_small_softcap": spec(S=64, N=16, Nkv=2, softcap=2.0, bias=(1, 1, 0.5),
                                             local_window_size=200, seqlens_range=(64, 600)),
    # a prompt's float cache of the other float dtype (attention reads the new rows in the query dtype)
    "f16_prompt_f32_cache_tc_rotary_norm": spec(S=150, N=8, Nkv=2, mode="prompt", capacity=160,
                                                seqlens_k=(149, 70, 3), seqlens_range=None, cache_dtype="f32",
                                                rotary_theta=1e4, qk_norm=True),
    "f16_prompt_f32_cache_bidirectional_h64": spec(H=64, N=4, Nkv=2, S=33, mode="prompt", capacity=33, causal=0,
                                                   seqlens_k=(32, 20, 5), seqlens_range=None, cache_dtype="f32"),
    "f16_prompt_f32_cache_h256_generic_prepass": spec(H=256, N=4, Nkv=2, S=20, mode="prompt", capacity=24,
                                                      seqlens_k=(19, 19, 10), seqlens_range=None, cache_dtype="f32"),
    "f32_prompt_f16_cache_s1": spec(dtype="f32", S=1, mode="prompt", capacity=2, seqlens_k=(0, 0, 0),
                                    seqlens_range=None, cache_dtype="f16"),
    "f32_prompt_f16_cache_all_features": spec(dtype="f32", N=8, Nkv=2, S=37, mode="prompt", capacity=40,
                                              seqlens_k=(36, 20, 0), seqlens_range=None, cache_dtype="f16",
                                              local_window_size=7, softcap=20.0, head_sink=True,
                                              bias=(3, 8, 0.5)),
    # 4-bit prompt cache (fp32 Q/K/V): packed nibbles written by the pre-pass, unpacked by the prefill
    "i4_per_channel_prompt_padding": spec(dtype="f32", S=37, N=8, Nkv=2, mode="prompt", capacity=40,
                                          seqlens_k=(36, 20, 0), seqlens_range=None, quant="PER_CHANNEL", bits=4,
                                          scale_range=(0.15, 0.4)),
    "i4_per_tensor_h64_norm_rotary": spec(dtype="f32", H=64, N=8, Nkv=2, S=50, mode="prompt", capacity=64,
                                          seqlens_k=(49, 49, 30), seqlens_range=None, quant="PER_TENSOR", bits=4,
                                          qk_norm=True, rotary_theta=1e4, scale_range=(0.2, 0.3)),
    "i4_s1_prompt": spec(dtype="f32", S=1, mode="prompt", capacity=2, seqlens_k=(0, 0, 0), seqlens_range=None,
                         quant="PER_CHANNEL", bits=4),
    "i4_bidirectional_softcap_sink": spec(dtype="f32", N=4, Nkv=2, S=33, mode="prompt", capacity=33, causal=0,
                                          seqlens_k=(32, 20, 5), seqlens_range=None, quant="PER_TENSOR", bits=4,
                                          softcap=20.0, head_sink=True, scale_range=(0.2, 0.3)),
    # tensor-core prefill over int8 / 4-bit caches with fp32 Q/K/V (hi/lo fp16 split): several
    # query-tile pairs and key tiles, ragged tails, group sizes 1 and 8, every feature
    "i8_tcq_multi_tile_g8_norm_rotary": spec(dtype="f32", B=2, S=300, N=16, Nkv=2, capacity=2500,
                                             seqlens_range=(300, 2400), quant="PER_CHANNEL", qk_norm=True,
                                             rotary_theta=1e4, scale_range=(0.01, 0.05)),
    "i4_tcq_bidirectional_g1_prompt_padding": spec(dtype="f32", S=150, N=2, Nkv=2, mode="prompt", capacity=160,
                                                   seqlens_k=(149, 70, 3), seqlens_range=None, causal=0,
                                                   quant="PER_TENSOR", bits=4, scale_range=(0.2, 0.3)),
    "i8_tcq_copy_smooth_window": spec(dtype="f32", S=12, N=8, Nkv=2, mode="copy", past_len=300,
                                      seqlens_range=(11, 311), local_window_size=100, smooth_softmax=1,
                                      quant="PER_TENSOR", scale_range=(0.01, 0.03)),
    "i8_tcq_bias_large_spread_softcap": spec(dtype="f32", S=64, N=16, Nkv=2, softcap=30.0, bias=(1, 1, 8.0),
                                             head_sink=True, seqlens_range=(64, 600), quant="PER_CHANNEL",
                                             scale_range=(0.01, 0.05)),
    "i8_tcq_per_head_bias_small_softcap": spec(dtype="f32", S=40, N=4, Nkv=2, softcap=1.0, bias=(3, 4, 2.0),
                                               seqlens_range=(40, 500), quant="PER_CHANNEL",
                                               scale_range=(0.01, 0.05)),
    "i4_tcq_prompt_g4_norm_rotary_window": spec(dtype="f32", B=2, S=700, N=16, Nkv=4, mode="prompt",
                                                capacity=700, seqlens_k=(699, 400), seqlens_range=None,
                                                quant="PER_CHANNEL", bits=4, qk_norm=True, rotary_theta=1e4,
                                                local_window_size=300, scale_range=(0.15, 0.4)),
    # group sizes 16 and 128: a query tile holds 8 and 1 positions (4-D copy boxes of 16 and 128 heads)
    "i8_tcq_g16_causal_norm_rotary": spec(dtype="f32", B=2, S=40, N=32, Nkv=2, capacity=700, seqlens_range=(40, 690),
                                          quant="PER_CHANNEL", qk_norm=True, rotary_theta=1e4,
                                          scale_range=(0.01, 0.05)),
    "i4_tcq_g128_prompt": spec(dtype="f32", B=2, S=20, N=128, Nkv=1, mode="prompt", capacity=24,
                               seqlens_k=(19, 7), seqlens_range=None, quant="PER_TENSOR", bits=4,
                               scale_range=(0.2, 0.3)),
    "i8_g3_simt_fallback": spec(dtype="f32", S=20, N=6, Nkv=2, quant="PER_CHANNEL", seqlens_range=(20, 500),
                                scale_range=(0.01, 0.05)),
    "i4_h256_window_generic_prepass": spec(dtype="f32", H=256, N=4, Nkv=2, S=20, mode="prompt", capacity=24,
                                           seqlens_k=(19, 19, 10), seqlens_range=None, quant="PER_CHANNEL", bits=4,
                                           local_window_size=5, scale_range=(0.1, 0.3)),
}


def _check(case, sample=None, repeat=1):
    gpu = run_gpu(case, repeat=repeat)
    assert gpu["status"] == 0, f"device status {gpu['status']:#x}"
    ref = run_oracle(case, sample=sample)
    check_output(case, gpu, ref, sample=sample)
    check_caches(case, gpu, ref)
    return gpu, ref


@pytest.mark.parametrize("name", sorted(DECODE))
def test_decode_parity(name):
    _check(generate(DECODE[name], seed=21))


@pytest.mark.parametrize("name", sorted(PREFILL))
def test_prefill_parity(name):
    _check(generate(PREFILL[name], seed=22))


def test_decode_idempotent_repeat():
    """Two calls in a row on a shared cache (the benchmark's loop) give the same result."""
    case = generate(DECODE["f16_h128_g4_rotary"], seed=23)
    _check(case, repeat=2)


def full_size_sample(case, n_random=48):
    """Output rows compared at full size: random rows and the last row of every batch entry;
    for a prefill (S > 1) also every row of the last KV-head group of the last batch entry
    (all its positions and heads: late key tiles, both query tiles of a CTA, lazy rescales
    across 4096 keys) and the last 64 positions of every head (the last query tiles)."""
    rows = set(sample_rows(case, n_random, seed=1))
    inp = case["inputs"]
    B, S = inp["query"].shape[:2]
    N, Nkv = case["attrs"]["num_heads"], case["attrs"]["kv_num_heads"]
    G = N // Nkv
    if S > 1:
        ok = valid_rows(case)
        b_last = B - 1
        for h in range((Nkv - 1) * G, N):
            rows.update((b_last, h, i) for i in np.nonzero(ok[b_last])[0])
        for b in range(B):
            live = np.nonzero(ok[b])[0]
            for h in range(N):
                rows.update((b, h, int(i)) for i in live[-64:])
    return sorted(rows)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_full_size(name):
    case = generate(WORKLOADS[name], seed=0)
    sample = None if name == "prompt_f32_b1_s16" else full_size_sample(case)
    _check(case, sample=sample)


def test_bad_seqlens_sets_device_status():
    """seqlens_k beyond the capacity: the batch entry is skipped and the status word says why."""
    case = generate(DECODE["f16_h128_g4_rotary"], seed=24)
    case["inputs"]["seqlens_k"] = case["inputs"]["seqlens_k"].copy()
    case["inputs"]["seqlens_k"][1] = 10_000          # beyond total_sequence_length and the capacity (800)
    gpu = run_gpu(case)
    assert gpu["status"] & 1
    # batch 1 is untouched
    assert np.array_equal(gpu["present_key"][1], case["inputs"]["past_key"][1])


@pytest.mark.parametrize("name", ["f16_tc_all_features", "i8_per_tensor_prefill_all_features"])
def test_bad_seqlens_prefill_skips_one_batch_entry(name):
    """A prefill with one batch entry's seqlens_k beyond the cache: that entry is skipped and flagged,
    the others match the oracle (outputs of every row, caches byte for byte), and the skipped
    entry's cache rows keep their bytes (tensor-core prefill, fp16 and over an int8 cache)."""
    case = generate(PREFILL[name], seed=25)
    good = case["inputs"]["seqlens_k"].copy()
    case["inputs"]["seqlens_k"] = good.copy()
    case["inputs"]["seqlens_k"][1] = 10_000   # beyond total_sequence_length and the capacity
    gpu = run_gpu(case)
    assert gpu["status"] & 1
    case["inputs"]["seqlens_k"] = good
    B, S = case["inputs"]["query"].shape[:2]
    N = case["attrs"]["num_heads"]
    ok = valid_rows(case)
    sample = [(b, h, i) for b in (0, 2) for h in range(N) for i in range(S) if ok[b, i]]
    ref = run_oracle(case, sample=sample)
    gpu["output"][1] = 0   # the skipped entry's output is undefined (uninitialised memory)
    check_output(case, gpu, ref, sample=sample)
    for nm in ("present_key", "present_value"):
        for b in (0, 2):
            assert np.array_equal(gpu[nm][b].view(np.uint8), ref[nm][b].view(np.uint8)), f"{nm}[{b}]"
        untouched = case["inputs"]["past_key" if nm == "present_key" else "past_value"][1]
        assert np.array_equal(gpu[nm][1].view(np.uint8), untouched.view(np.uint8)), f"{nm}[1] changed"
