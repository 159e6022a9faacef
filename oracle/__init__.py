"""Oracle for one windowed-KV-cache GroupQueryAttention step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library never
imports, links or calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``gqaw_oracle.c`` (plain C, fp64 accumulation).  This module
compiles it with gcc and marshals numpy arrays into it; it does no arithmetic of
the method itself except resolving the default scale ``1/sqrt(head_size)``
(mobius issue #111 "GQA In-Place KV Cache: Investigation Report", Part 1.3, the
``scale`` attribute).

Every function here cites the passage it follows inside ``gqaw_oracle.c``.
Functions without an independent pin: none (see ``tests/test_oracle_pins.py``),
except that the order "softcap first, bias after" is a reading of the pages and is
parity unpinned beyond that reading.
"""
from __future__ import annotations

import ctypes
import math
import os
import platform
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqaw_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_gqaw.%s.so" % platform.machine())

F32 = 0
BF16 = 1
I8 = 2      # quantized cache: int8 codes
E4M3 = 3    # quantized cache: fp8 e4m3 codes

_ERRORS = {
    1: "malformed sizes",
    2: "seqlens_k[b] + 1 - S < 0 for some item",
    3: "T_b > total_sequence_length for some item",
    4: "out of memory",
    5: "rotary position outside the cos/sin caches",
}


class _Args(ctypes.Structure):
    _fields_ = [
        ("batch_size", ctypes.c_int64),
        ("sequence_length", ctypes.c_int64),
        ("num_heads", ctypes.c_int64),
        ("kv_num_heads", ctypes.c_int64),
        ("head_size", ctypes.c_int64),
        ("capacity", ctypes.c_int64),
        ("local_window_size", ctypes.c_int64),
        ("scale", ctypes.c_double),
        ("softcap", ctypes.c_double),
        ("dtype", ctypes.c_int64),
        ("query", ctypes.c_void_p),
        ("key", ctypes.c_void_p),
        ("value", ctypes.c_void_p),
        ("past_key", ctypes.c_void_p),
        ("past_value", ctypes.c_void_p),
        ("present_key", ctypes.c_void_p),
        ("present_value", ctypes.c_void_p),
        ("seqlens_k", ctypes.c_void_p),
        ("total_sequence_length", ctypes.c_int64),
        ("attention_bias", ctypes.c_void_p),
        ("bias_stride_b", ctypes.c_int64),
        ("bias_stride_h", ctypes.c_int64),
        ("bias_stride_s", ctypes.c_int64),
        ("output", ctypes.c_void_p),
        ("output_f64", ctypes.c_void_p),
        ("resident_len", ctypes.c_void_p),
        ("s_begin", ctypes.c_int64),
        ("s_end", ctypes.c_int64),
        ("head_sink", ctypes.c_void_p),
        ("smooth_softmax", ctypes.c_int64),
        ("do_rotary", ctypes.c_int64),
        ("rotary_interleaved", ctypes.c_int64),
        ("rotary_dim", ctypes.c_int64),
        ("rotary_cache_len", ctypes.c_int64),
        ("cos_cache", ctypes.c_void_p),
        ("sin_cache", ctypes.c_void_p),
        ("position_ids", ctypes.c_void_p),
        ("cache_dtype", ctypes.c_int64),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
    ]


_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``liboracle_gqaw.so`` next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        # -ffp-contract=off: no fused multiply-add, so results do not depend on the host ISA.
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_resident_len.restype = ctypes.c_int64
        lib.oracle_resident_len.argtypes = [ctypes.c_int64] * 3
        lib.oracle_round_bf16.restype = ctypes.c_uint16
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_step.restype = ctypes.c_int
        lib.oracle_step.argtypes = [ctypes.POINTER(_Args)]
        lib.oracle_decode_e4m3.restype = ctypes.c_double
        lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_round_e4m3.restype = ctypes.c_uint8
        lib.oracle_round_e4m3.argtypes = [ctypes.c_float]
        lib.oracle_quantize.restype = ctypes.c_uint8
        lib.oracle_quantize.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_int64]
        _lib = lib
    return _lib


def resident_len(T: int, C: int, W: int) -> int:
    """L(T) of PR #32419 "Specify GroupQueryAttention windowed KV cache layout contract",
    Description (the resident-count formula)."""
    return int(_load().oracle_resident_len(int(T), int(C), int(W)))


def round_bf16(x: float) -> int:
    """bfloat16 bits nearest to ``x`` (ties to even), from fp64 in one rounding."""
    return int(_load().oracle_round_bf16(float(x)))


def decode_e4m3(code: int) -> float:
    """The value of an fp8 e4m3 code (OCP 8-bit floating point, E4M3FN)."""
    return float(_load().oracle_decode_e4m3(int(code) & 0xFF))


def round_e4m3(x: float) -> int:
    """The e4m3 code nearest to float32 x, ties to even, saturated to +-448."""
    return int(_load().oracle_round_e4m3(float(x)))


def quantize(x: float, scale: float, cache_dtype: int) -> int:
    """The quantized-cache code (a byte) of x: x / scale in float, rounded, saturated."""
    return int(_load().oracle_quantize(float(x), float(scale), int(cache_dtype)))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _elem_dtype(dtype: int):
    return np.float32 if dtype == F32 else np.uint16


def step(query, key, value, past_key, past_value, seqlens_k, total_sequence_length,
         num_heads, kv_num_heads, local_window_size, scale=0.0, softcap=0.0,
         attention_bias=None, bias_strides=None, dtype=F32, rows=None, head_sink=None, smooth_softmax=0,
         cos_cache=None, sin_cache=None, position_ids=None, rotary_interleaved=False,
         cache_dtype=None, k_scale=1.0, v_scale=1.0):
    """One windowed GQA step on host arrays.

    Arrays are numpy: float32 for ``dtype=F32``; uint16 bfloat16 bit patterns for
    ``dtype=BF16``.  Shapes: query (B,S,Nq*D); key/value (B,S,Nkv*D);
    past_key/past_value (B,Nkv,C,D); seqlens_k int32 (B,).  ``attention_bias`` is a
    float32 array indexed ``[b*sb + h*sh + s*ss + j]`` with ``bias_strides=(sb,sh,ss)``
    in elements (0 broadcasts); if ``bias_strides`` is None the bias must be a
    contiguous (B|1, Nq|1, S, total) array and its broadcast strides are derived.

    Returns dict(output, output_f64, present_key, present_value, resident_len).
    The present arrays start as copies of the past arrays; rows [0, L) are written.
    ``scale == 0`` selects 1/sqrt(head_size).  ``rows=(s0, s1)`` evaluates the attention
    only for new tokens s0 <= s < s1 (other output rows stay zero); ``rows=(0, 0)``
    gives the cache layout alone.  ``head_sink`` (float32 (Nq,)) adds a sink logit per
    head to the softmax denominator; ``smooth_softmax`` adds a sink of 0 to every head.
    ``cos_cache``/``sin_cache`` ((max_pos, rd/2) in the step's dtype) turn on the rotary
    embedding of the new query and key rows; ``position_ids`` (int64 (B, S)) overrides
    the positions P_b + s; ``rotary_interleaved`` pairs dimensions (2i, 2i+1).
    ``cache_dtype`` (I8 or E4M3) makes the caches quantized: past/present are uint8 code
    arrays and ``k_scale``/``v_scale`` their per-tensor scales.
    """
    lib = _load()
    et = _elem_dtype(dtype)
    query = np.ascontiguousarray(query, dtype=et)
    key = np.ascontiguousarray(key, dtype=et)
    value = np.ascontiguousarray(value, dtype=et)
    ct = np.uint8 if cache_dtype else et
    past_key = np.ascontiguousarray(past_key, dtype=ct)
    past_value = np.ascontiguousarray(past_value, dtype=ct)
    seqlens_k = np.ascontiguousarray(seqlens_k, dtype=np.int32)
    if head_sink is not None:
        head_sink = np.ascontiguousarray(head_sink, dtype=np.float32)
        if head_sink.shape != (num_heads,):
            raise ValueError("oracle.step: head_sink must be (num_heads,)")
    do_rotary = cos_cache is not None
    if do_rotary:
        cos_cache = np.ascontiguousarray(cos_cache, dtype=et)
        sin_cache = np.ascontiguousarray(sin_cache, dtype=et)
        if cos_cache.ndim != 2 or sin_cache.shape != cos_cache.shape:
            raise ValueError("oracle.step: cos_cache and sin_cache must be equal (max_pos, rd/2) arrays")
    B, Nkv, C, D = past_key.shape
    if do_rotary and position_ids is not None:
        position_ids = np.ascontiguousarray(position_ids, dtype=np.int64)
        if position_ids.shape != (B, query.shape[1]):
            raise ValueError("oracle.step: position_ids must be (B, S)")
    S = query.shape[1]
    if query.shape != (B, S, num_heads * D) or key.shape != (B, S, kv_num_heads * D):
        raise ValueError("oracle.step: shape mismatch")
    if Nkv != kv_num_heads or value.shape != key.shape or past_value.shape != past_key.shape:
        raise ValueError("oracle.step: shape mismatch")
    present_key = past_key.copy()
    present_value = past_value.copy()
    output = np.zeros((B, S, num_heads * D), dtype=et)
    output_f64 = np.zeros((B, S, num_heads * D), dtype=np.float64)
    resident = np.zeros((B,), dtype=np.int32)
    sb = sh = ss = 0
    if attention_bias is not None:
        attention_bias = np.ascontiguousarray(attention_bias, dtype=np.float32)
        if bias_strides is None:
            bb, bh, bs, bt = attention_bias.shape
            if bt != total_sequence_length or bs != S:
                raise ValueError("oracle.step: bias must be (B|1, Nq|1, S, total_sequence_length)")
            ss = bt
            sh = 0 if bh == 1 else bs * bt
            sb = 0 if bb == 1 else bh * bs * bt
        else:
            sb, sh, ss = (int(v) for v in bias_strides)
    a = _Args(
        batch_size=B, sequence_length=S, num_heads=num_heads, kv_num_heads=kv_num_heads,
        head_size=D, capacity=C, local_window_size=local_window_size,
        scale=float(scale) if scale else 1.0 / math.sqrt(D), softcap=float(softcap),
        dtype=dtype, query=_ptr(query), key=_ptr(key), value=_ptr(value),
        past_key=_ptr(past_key), past_value=_ptr(past_value),
        present_key=_ptr(present_key), present_value=_ptr(present_value),
        seqlens_k=_ptr(seqlens_k), total_sequence_length=int(total_sequence_length),
        attention_bias=_ptr(attention_bias), bias_stride_b=sb, bias_stride_h=sh,
        bias_stride_s=ss, output=_ptr(output), output_f64=_ptr(output_f64),
        resident_len=_ptr(resident),
        s_begin=0 if rows is None else int(rows[0]),
        s_end=S if rows is None else int(rows[1]),
        head_sink=_ptr(head_sink), smooth_softmax=int(bool(smooth_softmax)),
        do_rotary=int(do_rotary), rotary_interleaved=int(bool(rotary_interleaved)),
        rotary_dim=2 * cos_cache.shape[1] if do_rotary else 0,
        rotary_cache_len=cos_cache.shape[0] if do_rotary else 0,
        cos_cache=_ptr(cos_cache), sin_cache=_ptr(sin_cache),
        position_ids=_ptr(position_ids) if do_rotary else None,
        cache_dtype=int(cache_dtype or 0), k_scale=float(k_scale), v_scale=float(v_scale),
    )
    rc = lib.oracle_step(ctypes.byref(a))
    if rc != 0:
        raise ValueError("oracle.step: " + _ERRORS.get(rc, "error %d" % rc))
    return {
        "output": output,
        "output_f64": output_f64,
        "present_key": present_key,
        "present_value": present_value,
        "resident_len": resident,
    }
