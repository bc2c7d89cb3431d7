"""CPU oracle for the GroupQueryAttention forward pass.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package. The
CUDA library under ``grouped_query_attention_gb300/`` never imports, links or
calls anything here, and this package imports nothing from it.

The oracle is the plain definition of the operator written out in numpy with
fp64 arithmetic: no blocking, no online softmax, no split of the key axis.
Every function cites the passage of the operator's documentation page it
follows ("com.microsoft.GroupQueryAttention" README, sections Description,
Inputs, Outputs, Attributes, Type constraints, Implementation variants).

Pins: every function is checked in ``tests/test_oracle_pins.py`` against
closed forms, invariants, a pure-Python brute force and a library routine
(``torch.nn.functional.scaled_dot_product_attention`` in fp64). The fp32
recipe of the stored K rows (``rms_norm_fp32``, ``rotary_neox_fp32``) is
pinned in ``tests/test_oracle_fp32_recipe.py``: bit for bit against a scalar
restatement, and within its rounding-error bound of the fp64 definition. Readings that
the pages leave open (query-head to KV-head mapping, window bound, order of
softcap and bias, head-sink placement, int8 rounding, the 4-bit code range,
the row layout of a sliding-window cache) are fixed by explicit switches or
single documented choices; those readings are "parity unpinned" by the pages
themselves and are listed as such in the design notes. The 4-bit nibble
layout is pinned by the pages' description (+8 bias, even coordinate low) and
the sliding-window cache by equality with attention over the full history.
"""

from .gqa import (  # noqa: F401
    DEFAULT_ATTRS,
    dequantize_int8,
    gqa_forward,
    pack_int4,
    quantize_int4,
    quantize_int8,
    rms_norm,
    rms_norm_fp32,
    rotary_neox,
    rotary_neox_fp32,
    softcap_scores,
    unpack_int4,
)
