"""GB300-native GroupQueryAttention forward pass (com.microsoft.GroupQueryAttention).

The compute path is the CUDA library libgqa_gb300.so behind the C ABI of
include/gqa.h. This package adds argument marshalling for torch tensors:
``GroupQueryAttention`` keeps the handle and a workspace buffer obtained from
torch's allocator and calls ``gqa_forward`` on the current stream.
"""

from __future__ import annotations

import torch

from . import capi
from .capi import GqaError, GqaInputs, GqaOutputs, describe, make_attrs  # noqa: F401

_DTYPE_CODE = {torch.float32: capi.GQA_F32, torch.float16: capi.GQA_F16, torch.int8: capi.GQA_I8,
               torch.uint8: capi.GQA_U8, torch.int32: capi.GQA_I32, torch.bfloat16: capi.GQA_BF16}


def tensor_desc(t: torch.Tensor | None) -> capi.GqaTensor:
    """C descriptor of a contiguous CUDA tensor (or an absent input for None)."""
    if t is None:
        return capi.GqaTensor()
    if not t.is_contiguous():
        raise ValueError("tensors passed to the GQA library must be contiguous")
    if t.dtype not in _DTYPE_CODE:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return describe(t.data_ptr(), _DTYPE_CODE[t.dtype], tuple(t.shape))


def _tensor_key(t: torch.Tensor | None):
    """What a tensor's C descriptor depends on (None for an absent input)."""
    if t is None:
        return None
    return t.data_ptr(), t.shape, t.dtype, t.is_contiguous()


class GroupQueryAttention:
    """One operator instance: attributes fixed at construction (section Attributes)."""

    def __init__(self, num_heads: int, kv_num_heads: int, **attrs):
        capi.load_library()
        self.attrs = make_attrs(num_heads, kv_num_heads, **attrs)
        self.handle = capi.gqa_create(self.attrs)
        self._ws = None
        # The last call's descriptors and workspace size, reused while every tensor
        # keeps its address, shape, dtype and layout (a decode loop over fixed buffers).
        self._call_key = None
        self._call_structs = None

    def close(self) -> None:
        if getattr(self, "handle", None) is not None and self.handle.value:
            capi.gqa_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _structs(self, query, key, value, seqlens_k, total_sequence_length, present_key, present_value,
                 output, past_key=None, past_value=None, cos_cache=None, sin_cache=None,
                 attention_bias=None, head_sink=None, k_scale=None, v_scale=None,
                 q_norm_weight=None, k_norm_weight=None):
        inp = GqaInputs()
        named = dict(query=query, key=key, value=value, past_key=past_key, past_value=past_value,
                     seqlens_k=seqlens_k, cos_cache=cos_cache, sin_cache=sin_cache,
                     attention_bias=attention_bias, head_sink=head_sink, k_scale=k_scale, v_scale=v_scale,
                     q_norm_weight=q_norm_weight, k_norm_weight=k_norm_weight)
        for name, t in named.items():
            setattr(inp, name, tensor_desc(t))
        inp.total_sequence_length = int(total_sequence_length)
        out = GqaOutputs()
        out.output = tensor_desc(output)
        out.present_key = tensor_desc(present_key)
        out.present_value = tensor_desc(present_value)
        return inp, out

    def workspace_size(self, **tensors) -> int:
        inp, out = self._structs(**tensors)
        return capi.gqa_workspace_size(self.handle, inp, out)

    def plan(self, **tensors) -> capi.GqaPlanInfo:
        """Host-only: regime, kernel launches per call, split sizes and workspace bytes."""
        inp, out = self._structs(**tensors)
        return capi.gqa_describe_plan(self.handle, inp, out)

    def workspace(self, nbytes: int, device) -> torch.Tensor:
        if self._ws is None or self._ws.numel() < nbytes or self._ws.device != device:
            self._ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        return self._ws

    def __call__(self, query, key, value, seqlens_k, total_sequence_length, present_key, present_value,
                 output=None, workspace=None, stream=None, **optional):
        """Run the forward pass; returns ``output``. present_key/value are updated in place
        (pass past_key=present_key for a shared buffer, or a separate past for copy mode)."""
        if output is None:
            output = torch.empty_like(query)
        call_key = (int(total_sequence_length), tuple(optional),
                    *(_tensor_key(t) for t in (query, key, value, seqlens_k, present_key, present_value, output)),
                    *(_tensor_key(t) for t in optional.values()))
        if call_key != self._call_key:
            inp, out = self._structs(query, key, value, seqlens_k, total_sequence_length, present_key,
                                     present_value, output, **optional)
            nbytes = capi.gqa_workspace_size(self.handle, inp, out)
            self._call_key, self._call_structs = call_key, (inp, out, nbytes)
        inp, out, nbytes = self._call_structs
        ws = workspace if workspace is not None else self.workspace(nbytes, query.device)
        st = stream if stream is not None else torch.cuda.current_stream(query.device).cuda_stream
        capi.gqa_forward(self.handle, inp, out, ws.data_ptr(), ws.numel(), st)
        self.last_workspace = ws
        return output

    def device_status(self, stream=None) -> int:
        """Synchronise and return (then clear) the device status bits of the last workspace."""
        ws = self.last_workspace
        st = stream if stream is not None else torch.cuda.current_stream(ws.device).cuda_stream
        return capi.gqa_read_device_status(self.handle, ws.data_ptr(), st)
