"""ctypes binding of the C ABI in include/gqa.h: argument marshalling only.

The functions keep the C names (gqa_create, gqa_workspace_size, gqa_forward,
gqa_read_device_status, gqa_destroy, gqa_status_string, gqa_last_error).
Every step of the forward pass runs in the CUDA library; if the library is
not built this module raises instead of falling back to anything else.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgqa_gb300.so")

# gqa_status
GQA_OK, GQA_ERR_INVALID_ARGUMENT, GQA_ERR_UNSUPPORTED, GQA_ERR_CUDA, GQA_ERR_DEVICE_STATUS, GQA_ERR_WORKSPACE = range(6)
# gqa_dtype
GQA_DTYPE_NONE, GQA_F32, GQA_F16, GQA_I8, GQA_U8, GQA_I32, GQA_BF16 = range(7)
# gqa_quant
QUANT = {"NONE": 0, "PER_TENSOR": 1, "PER_CHANNEL": 2}
# device status bits
GQA_DEVICE_BAD_SEQLEN, GQA_DEVICE_BAD_ROTARY, GQA_DEVICE_TIMEOUT = 1, 2, 4

EXPORTS = ["gqa_attrs_default", "gqa_create", "gqa_workspace_size", "gqa_forward",
           "gqa_read_device_status", "gqa_describe_plan", "gqa_destroy", "gqa_status_string",
           "gqa_last_error", "gqa_forward_noalloc", "gqa_profile_begin", "gqa_profile_end",
           "gqa_set_wait_limit"]
KERNEL_KINDS = {1: "copy_past", 2: "prepass", 3: "decode", 4: "prefill_cuda_core", 5: "prefill_tensor_core",
                6: "decode_tensor_core", 7: "window_shift", 8: "bias_stage"}
GQA_REGIME_DECODE, GQA_REGIME_PREFILL = 1, 2


class GqaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4)]


class GqaAttrs(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int32), ("kv_num_heads", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("do_rotary", ctypes.c_int32), ("local_window_size", ctypes.c_int32), ("scale", ctypes.c_float),
                ("softcap", ctypes.c_float), ("qk_norm_epsilon", ctypes.c_float),
                ("smooth_softmax", ctypes.c_int32), ("k_quant_type", ctypes.c_int32),
                ("v_quant_type", ctypes.c_int32), ("kv_cache_bit_width", ctypes.c_int32),
                ("sliding_window_cache", ctypes.c_int32)]


INPUT_FIELDS = ["query", "key", "value", "past_key", "past_value", "seqlens_k", "cos_cache", "sin_cache",
                "attention_bias", "head_sink", "k_scale", "v_scale", "q_norm_weight", "k_norm_weight"]


class GqaInputs(ctypes.Structure):
    _fields_ = [(n, GqaTensor) for n in INPUT_FIELDS] + [("total_sequence_length", ctypes.c_int32)]


class GqaOutputs(ctypes.Structure):
    _fields_ = [("output", GqaTensor), ("present_key", GqaTensor), ("present_value", GqaTensor)]


class GqaPlanInfo(ctypes.Structure):
    _fields_ = [("regime", ctypes.c_int32), ("launches", ctypes.c_int32), ("split_len", ctypes.c_int32),
                ("max_splits", ctypes.c_int32), ("workspace_bytes", ctypes.c_uint64)]


class GqaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (built by grouped_query_attention_gb300.build)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"GQA CUDA library not built: {p} is missing "
                           "(run `python -m grouped_query_attention_gb300.build`)")
    lib = ctypes.CDLL(p)
    lib.gqa_attrs_default.argtypes = [ctypes.POINTER(GqaAttrs)]
    lib.gqa_attrs_default.restype = None
    lib.gqa_create.argtypes = [ctypes.POINTER(GqaAttrs), ctypes.POINTER(ctypes.c_void_p)]
    lib.gqa_create.restype = ctypes.c_int
    lib.gqa_workspace_size.argtypes = [ctypes.c_void_p, ctypes.POINTER(GqaInputs), ctypes.POINTER(GqaOutputs),
                                       ctypes.POINTER(ctypes.c_size_t)]
    lib.gqa_workspace_size.restype = ctypes.c_int
    lib.gqa_forward.argtypes = [ctypes.c_void_p, ctypes.POINTER(GqaInputs), ctypes.POINTER(GqaOutputs),
                                ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.gqa_forward.restype = ctypes.c_int
    lib.gqa_forward_noalloc.argtypes = [ctypes.c_void_p, ctypes.POINTER(GqaInputs), ctypes.POINTER(GqaOutputs),
                                        ctypes.c_void_p]
    lib.gqa_forward_noalloc.restype = ctypes.c_int
    lib.gqa_read_device_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.POINTER(ctypes.c_uint32)]
    lib.gqa_read_device_status.restype = ctypes.c_int
    lib.gqa_describe_plan.argtypes = [ctypes.c_void_p, ctypes.POINTER(GqaInputs), ctypes.POINTER(GqaOutputs),
                                      ctypes.POINTER(GqaPlanInfo)]
    lib.gqa_describe_plan.restype = ctypes.c_int
    lib.gqa_profile_begin.argtypes = [ctypes.c_void_p, ctypes.c_int32]
    lib.gqa_profile_begin.restype = ctypes.c_int
    lib.gqa_profile_end.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_float),
                                    ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
    lib.gqa_profile_end.restype = ctypes.c_int
    lib.gqa_set_wait_limit.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32]
    lib.gqa_set_wait_limit.restype = ctypes.c_int
    lib.gqa_destroy.argtypes = [ctypes.c_void_p]
    lib.gqa_destroy.restype = None
    lib.gqa_status_string.argtypes = [ctypes.c_int]
    lib.gqa_status_string.restype = ctypes.c_char_p
    lib.gqa_last_error.argtypes = []
    lib.gqa_last_error.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def _status_name(status: int) -> str:
    try:
        return load_library().gqa_status_string(status).decode()
    except Exception:
        return f"status {status}"


def _check(status: int) -> None:
    if status != GQA_OK:
        raise GqaError(status, gqa_last_error())


def gqa_attrs_default() -> GqaAttrs:
    a = GqaAttrs()
    load_library().gqa_attrs_default(ctypes.byref(a))
    return a


def gqa_create(attrs: GqaAttrs) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(load_library().gqa_create(ctypes.byref(attrs), ctypes.byref(h)))
    return h


def gqa_workspace_size(handle, inputs: GqaInputs, outputs: GqaOutputs) -> int:
    n = ctypes.c_size_t()
    _check(load_library().gqa_workspace_size(handle, ctypes.byref(inputs), ctypes.byref(outputs), ctypes.byref(n)))
    return n.value


def gqa_forward(handle, inputs: GqaInputs, outputs: GqaOutputs, workspace: int, workspace_bytes: int,
                stream: int) -> None:
    _check(load_library().gqa_forward(handle, ctypes.byref(inputs), ctypes.byref(outputs),
                                      ctypes.c_void_p(workspace), workspace_bytes, ctypes.c_void_p(stream)))


def gqa_forward_noalloc(handle, inputs: GqaInputs, outputs: GqaOutputs, stream: int) -> None:
    """Decode-regime forward pass with the library's fixed scratch instead of a workspace."""
    _check(load_library().gqa_forward_noalloc(handle, ctypes.byref(inputs), ctypes.byref(outputs),
                                              ctypes.c_void_p(stream)))


def gqa_read_device_status(handle, workspace: int, stream: int) -> int:
    v = ctypes.c_uint32()
    st = load_library().gqa_read_device_status(handle, ctypes.c_void_p(workspace), ctypes.c_void_p(stream),
                                               ctypes.byref(v))
    if st not in (GQA_OK, GQA_ERR_DEVICE_STATUS):
        _check(st)
    return v.value


def gqa_describe_plan(handle, inputs: GqaInputs, outputs: GqaOutputs) -> GqaPlanInfo:
    info = GqaPlanInfo()
    _check(load_library().gqa_describe_plan(handle, ctypes.byref(inputs), ctypes.byref(outputs),
                                            ctypes.byref(info)))
    return info


def gqa_profile_begin(handle, max_launches: int) -> None:
    _check(load_library().gqa_profile_begin(handle, int(max_launches)))


def gqa_profile_end(handle, capacity: int = 4096) -> list:
    """[(kernel kind name, milliseconds)] of the launches recorded since gqa_profile_begin."""
    kinds = (ctypes.c_int32 * capacity)()
    ms = (ctypes.c_float * capacity)()
    n = ctypes.c_int32()
    _check(load_library().gqa_profile_end(handle, kinds, ms, capacity, ctypes.byref(n)))
    return [(KERNEL_KINDS.get(kinds[i], str(kinds[i])), ms[i]) for i in range(min(n.value, capacity))]


def gqa_set_wait_limit(handle, cycles: int, withhold_copy: int = -1) -> None:
    """Bound of the tensor-core kernels' pipeline waits (0: default) and the timeout-path test switch."""
    _check(load_library().gqa_set_wait_limit(handle, int(cycles), int(withhold_copy)))


def gqa_destroy(handle) -> None:
    load_library().gqa_destroy(handle)


def gqa_status_string(status: int) -> str:
    return load_library().gqa_status_string(status).decode()


def gqa_last_error() -> str:
    return load_library().gqa_last_error().decode()


def make_attrs(num_heads: int, kv_num_heads: int, **kw) -> GqaAttrs:
    """gqa_attrs with the page's defaults, overridden by keyword (quant types by name)."""
    a = gqa_attrs_default()
    a.num_heads = int(num_heads)
    a.kv_num_heads = int(kv_num_heads)
    for k, v in kw.items():
        if k in ("k_quant_type", "v_quant_type") and isinstance(v, str):
            v = QUANT[v]
        if not hasattr(a, k):
            raise TypeError(f"unknown attribute {k}")
        setattr(a, k, v)
    return a


def describe(data_ptr: int, dtype_code: int, shape) -> GqaTensor:
    t = GqaTensor()
    t.data = data_ptr
    t.dtype = dtype_code
    t.ndim = len(shape)
    for i, s in enumerate(shape):
        t.shape[i] = int(s)
    return t
