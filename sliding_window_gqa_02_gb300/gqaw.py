"""ctypes binding of ``libgqaw.so`` (include/gqaw.h), with the same function names.

This module only marshals arguments: every step of the computation runs in the CUDA
kernels of the library.  If the library has not been built the first call raises;
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libgqaw.so")

GQAW_OK = 0
GQAW_EINVAL = 1
GQAW_EUNSUPPORTED = 2
GQAW_ECUDA = 3
GQAW_EWORKSPACE = 4
GQAW_EDEVICE = 5

GQAW_F32 = 0
GQAW_BF16 = 1

GQAW_I8 = 2
GQAW_E4M3 = 3
GQAW_DEV_BAD_SEQLEN = 1
GQAW_DEV_TIMEOUT = 2
GQAW_DEV_BAD_POSITION = 4
GQAW_DEV_QUERY_RANGE = 8
GQAW_DEV_INTERNAL = 16

STATUS_NAMES = {0: "GQAW_OK", 1: "GQAW_EINVAL", 2: "GQAW_EUNSUPPORTED", 3: "GQAW_ECUDA",
                4: "GQAW_EWORKSPACE", 5: "GQAW_EDEVICE"}

EXPORTED = ["gqaw_resident_len", "gqaw_rollback_exact", "gqaw_workspace_bytes", "gqaw_workspace_init",
            "gqa_windowed_step", "gqaw_attend", "gqaw_update_cache", "gqaw_device_status",
            "gqaw_last_error", "gqaw_launch_count", "gqaw_step_args_size", "gqa_windowed_step_noalloc"]

GQAW_NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024


class gqaw_step_args(ctypes.Structure):
    """Mirror of ``gqaw_step_args`` in include/gqaw.h (same field order and types)."""

    _fields_ = [
        ("batch_size", ctypes.c_int32),
        ("sequence_length", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("kv_num_heads", ctypes.c_int32),
        ("head_size", ctypes.c_int32),
        ("capacity", ctypes.c_int32),
        ("local_window_size", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("softcap", ctypes.c_float),
        ("total_sequence_length", ctypes.c_int32),
        ("split_keys", ctypes.c_int32),
        ("query", ctypes.c_void_p),
        ("key", ctypes.c_void_p),
        ("value", ctypes.c_void_p),
        ("past_key", ctypes.c_void_p),
        ("past_value", ctypes.c_void_p),
        ("present_key", ctypes.c_void_p),
        ("present_value", ctypes.c_void_p),
        ("seqlens_k", ctypes.c_void_p),
        ("attention_bias", ctypes.c_void_p),
        ("bias_stride_b", ctypes.c_int64),
        ("bias_stride_h", ctypes.c_int64),
        ("bias_stride_s", ctypes.c_int64),
        ("output", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("resident_len_out", ctypes.c_void_p),
        ("head_sink", ctypes.c_void_p),
        ("smooth_softmax", ctypes.c_int32),
        ("do_rotary", ctypes.c_int32),
        ("rotary_interleaved", ctypes.c_int32),
        ("rotary_dim", ctypes.c_int32),
        ("rotary_cache_len", ctypes.c_int32),
        ("cos_cache", ctypes.c_void_p),
        ("sin_cache", ctypes.c_void_p),
        ("position_ids", ctypes.c_void_p),
        ("cache_dtype", ctypes.c_int32),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
    ]


class GqawError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


_lib = None


def load(path: str = LIB_PATH):
    """Load the library (once).  Raises if it is missing: there is no CPU path."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libgqaw.so is not built (%s); run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(gqaw_step_args)
    lib.gqaw_resident_len.restype = ctypes.c_int64
    lib.gqaw_resident_len.argtypes = [ctypes.c_int64] * 3
    lib.gqaw_rollback_exact.restype = ctypes.c_int
    lib.gqaw_rollback_exact.argtypes = [ctypes.c_int64] * 4
    lib.gqaw_workspace_bytes.restype = ctypes.c_size_t
    lib.gqaw_workspace_bytes.argtypes = [P]
    lib.gqaw_workspace_init.restype = ctypes.c_int
    lib.gqaw_workspace_init.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    for name in ("gqa_windowed_step", "gqaw_attend", "gqaw_update_cache", "gqa_windowed_step_noalloc"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [P, ctypes.c_void_p]
    lib.gqaw_device_status.restype = ctypes.c_int
    lib.gqaw_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int,
                                       ctypes.c_void_p]
    lib.gqaw_last_error.restype = ctypes.c_char_p
    lib.gqaw_last_error.argtypes = []
    lib.gqaw_launch_count.restype = ctypes.c_uint64
    lib.gqaw_launch_count.argtypes = []
    lib.gqaw_step_args_size.restype = ctypes.c_size_t
    lib.gqaw_step_args_size.argtypes = []
    if lib.gqaw_step_args_size() != ctypes.sizeof(gqaw_step_args):
        raise RuntimeError("gqaw_step_args layout mismatch: library %d bytes, binding %d bytes"
                           % (lib.gqaw_step_args_size(), ctypes.sizeof(gqaw_step_args)))
    _lib = lib
    return lib


# ----------------------------------------------------------------- same-name wrappers


def gqaw_resident_len(T: int, C: int, W: int) -> int:
    return int(load().gqaw_resident_len(T, C, W))


def gqaw_rollback_exact(T: int, k: int, C: int, W: int) -> int:
    return int(load().gqaw_rollback_exact(T, k, C, W))


def gqaw_workspace_bytes(args: gqaw_step_args) -> int:
    return int(load().gqaw_workspace_bytes(ctypes.byref(args)))


def gqaw_workspace_init(workspace: int, nbytes: int, stream: int = 0) -> int:
    return int(load().gqaw_workspace_init(workspace, nbytes, stream))


def gqa_windowed_step(args: gqaw_step_args, stream: int = 0) -> int:
    return int(load().gqa_windowed_step(ctypes.byref(args), stream))


def gqa_windowed_step_noalloc(args: gqaw_step_args, stream: int = 0) -> int:
    """The step with its scratch taken from the library's static array (for callers
    that cannot allocate); ``args.workspace`` is ignored."""
    return int(load().gqa_windowed_step_noalloc(ctypes.byref(args), stream))


def gqaw_attend(args: gqaw_step_args, stream: int = 0) -> int:
    return int(load().gqaw_attend(ctypes.byref(args), stream))


def gqaw_update_cache(args: gqaw_step_args, stream: int = 0) -> int:
    return int(load().gqaw_update_cache(ctypes.byref(args), stream))


def gqaw_device_status(workspace: int, reset: bool = False, stream: int = 0):
    """Returns (status, flags)."""
    flags = ctypes.c_uint32(0)
    st = int(load().gqaw_device_status(workspace, ctypes.byref(flags), int(bool(reset)), stream))
    return st, int(flags.value)


def gqaw_last_error() -> str:
    return load().gqaw_last_error().decode()


def gqaw_launch_count() -> int:
    return int(load().gqaw_launch_count())


def check(status: int) -> None:
    if status != GQAW_OK:
        raise GqawError(status, gqaw_last_error())


# ----------------------------------------------------------------- torch marshalling


def _ptr(t):
    return None if t is None else int(t.data_ptr())


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.float32:
        return GQAW_F32
    if t.dtype == torch.bfloat16:
        return GQAW_BF16
    raise TypeError("query/key/value must be float32 or bfloat16, got %s" % t.dtype)


def _cache_code(cache, query) -> int:
    """0 when the caches hold the query's type; GQAW_I8 / GQAW_E4M3 for code caches."""
    import torch

    if cache.dtype == query.dtype:
        return 0
    if cache.dtype == torch.int8:
        return GQAW_I8
    if getattr(torch, "float8_e4m3fn", None) is not None and cache.dtype == torch.float8_e4m3fn:
        return GQAW_E4M3
    raise TypeError("caches must hold the query's type, int8 or float8_e4m3fn, got %s" % cache.dtype)


def make_args(query, key, value, past_key, past_value, present_key, present_value, seqlens_k,
              total_sequence_length: int, num_heads: int, kv_num_heads: int, local_window_size: int,
              output, workspace=None, scale: float = 0.0, softcap: float = 0.0, attention_bias=None,
              bias_strides=None, resident_len_out=None, split_keys: int = 0, head_sink=None,
              smooth_softmax: bool = False, cos_cache=None, sin_cache=None, position_ids=None,
              rotary_interleaved: bool = False, k_scale=None, v_scale=None) -> gqaw_step_args:
    """Fill a ``gqaw_step_args`` from CUDA tensors (shapes as in include/gqaw.h).

    ``attention_bias``: fp32 tensor whose last dimension is contiguous; its (b, h, s)
    strides are taken from the tensor (a size-1 dimension broadcasts with stride 0)
    unless ``bias_strides`` gives them in elements.  ``workspace``: a uint8 CUDA
    tensor, or None when only the size is wanted.  ``head_sink``: None or a contiguous
    fp32 (num_heads,) CUDA tensor of sink logits; ``smooth_softmax``: a sink of 0.
    ``cos_cache``/``sin_cache``: contiguous (max_pos, rd/2) CUDA tensors of the step's
    dtype; giving them turns on the rotary embedding (rd = twice their width);
    ``position_ids``: None or a contiguous int64 (B, S) CUDA tensor.  Caches of dtype
    int8 or float8_e4m3fn make a quantized cache; ``k_scale`` / ``v_scale`` are then
    one-element float32 CUDA tensors.
    """
    B, Nkv, C, D = past_key.shape
    S = query.shape[1]
    a = gqaw_step_args()
    a.batch_size, a.sequence_length = int(B), int(S)
    a.num_heads, a.kv_num_heads, a.head_size = int(num_heads), int(kv_num_heads), int(D)
    a.capacity, a.local_window_size = int(C), int(local_window_size)
    a.dtype = _dtype_code(query)
    a.cache_dtype = _cache_code(past_key, query)
    if a.cache_dtype:
        for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
            if t is None or str(t.dtype) != "torch.float32" or t.numel() != 1:
                raise ValueError("%s: a one-element float32 tensor is needed for a quantized cache" % name)
        a.k_scale, a.v_scale = _ptr(k_scale), _ptr(v_scale)
    a.scale, a.softcap = float(scale), float(softcap)
    a.total_sequence_length, a.split_keys = int(total_sequence_length), int(split_keys)
    a.query, a.key, a.value = _ptr(query), _ptr(key), _ptr(value)
    a.past_key, a.past_value = _ptr(past_key), _ptr(past_value)
    a.present_key, a.present_value = _ptr(present_key), _ptr(present_value)
    a.seqlens_k = _ptr(seqlens_k)
    if attention_bias is not None:
        if attention_bias.stride(-1) != 1:
            raise ValueError("attention_bias: last dimension must be contiguous")
        if bias_strides is None:
            bb, bh, bs, _ = attention_bias.shape
            st = attention_bias.stride()
            bias_strides = (0 if bb == 1 else st[0], 0 if bh == 1 else st[1], 0 if bs == 1 else st[2])
        a.attention_bias = _ptr(attention_bias)
        a.bias_stride_b, a.bias_stride_h, a.bias_stride_s = (int(x) for x in bias_strides)
    a.output = _ptr(output)
    if workspace is not None:
        a.workspace, a.workspace_bytes = _ptr(workspace), int(workspace.numel() * workspace.element_size())
    a.resident_len_out = _ptr(resident_len_out)
    if head_sink is not None:
        if str(head_sink.dtype) != "torch.float32" or tuple(head_sink.shape) != (int(num_heads),) \
                or not head_sink.is_contiguous():
            raise ValueError("head_sink: contiguous float32 tensor of shape (num_heads,)")
        a.head_sink = _ptr(head_sink)
    a.smooth_softmax = int(bool(smooth_softmax))
    if cos_cache is not None:
        if sin_cache is None or tuple(sin_cache.shape) != tuple(cos_cache.shape) or cos_cache.dim() != 2 \
                or not (cos_cache.is_contiguous() and sin_cache.is_contiguous()) \
                or cos_cache.dtype != query.dtype or sin_cache.dtype != query.dtype:
            raise ValueError("cos_cache/sin_cache: equal contiguous (max_pos, rd/2) tensors of the query's dtype")
        a.do_rotary, a.rotary_interleaved = 1, int(bool(rotary_interleaved))
        a.rotary_dim, a.rotary_cache_len = 2 * int(cos_cache.shape[1]), int(cos_cache.shape[0])
        a.cos_cache, a.sin_cache = _ptr(cos_cache), _ptr(sin_cache)
        if position_ids is not None:
            if str(position_ids.dtype) != "torch.int64" or tuple(position_ids.shape) != (int(B), int(S)) \
                    or not position_ids.is_contiguous():
                raise ValueError("position_ids: contiguous int64 tensor of shape (B, S)")
            a.position_ids = _ptr(position_ids)
    return a


def new_workspace(args: gqaw_step_args, device, stream: int = 0):
    """Allocate (torch) and zero-initialise a workspace large enough for ``args``."""
    import torch

    n = gqaw_workspace_bytes(args)
    if n == 0:
        check(GQAW_EINVAL)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    check(gqaw_workspace_init(int(ws.data_ptr()), n, stream))
    return ws
