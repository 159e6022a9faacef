"""Test helper: drive the oracle across several steps on one cache.

Holds the cache state between oracle calls (past := present after each step).  No
arithmetic of the method lives here.
"""
from __future__ import annotations

import numpy as np

import oracle


class OracleCache:
    def __init__(self, B, Nq, Nkv, D, C, W, dtype=oracle.F32, scale=0.0, softcap=0.0,
                 past_key=None, past_value=None, head_sink=None, smooth_softmax=False, cos_cache=None,
                 sin_cache=None, rotary_interleaved=False, cache_dtype=None, k_scale=1.0, v_scale=1.0):
        self.cache_dtype, self.k_scale, self.v_scale = cache_dtype, k_scale, v_scale
        self.head_sink, self.smooth_softmax = head_sink, smooth_softmax
        self.cos_cache, self.sin_cache, self.rotary_interleaved = cos_cache, sin_cache, rotary_interleaved
        self.B, self.Nq, self.Nkv, self.D, self.C, self.W = B, Nq, Nkv, D, C, W
        self.dtype, self.scale, self.softcap = dtype, scale, softcap
        et = np.uint8 if cache_dtype else (np.float32 if dtype == oracle.F32 else np.uint16)
        self.pk = np.zeros((B, Nkv, C, D), et) if past_key is None else np.array(past_key, et)
        self.pv = np.zeros((B, Nkv, C, D), et) if past_value is None else np.array(past_value, et)

    def step(self, q, k, v, seqlens, total=None, bias=None, bias_strides=None, position_ids=None):
        seqlens = np.asarray(seqlens, np.int32)
        if total is None:
            total = int(seqlens.max()) + 1
        r = oracle.step(q, k, v, self.pk, self.pv, seqlens, total, self.Nq, self.Nkv, self.W,
                        scale=self.scale, softcap=self.softcap, attention_bias=bias,
                        bias_strides=bias_strides, dtype=self.dtype, head_sink=self.head_sink,
                        smooth_softmax=self.smooth_softmax, cos_cache=self.cos_cache, sin_cache=self.sin_cache,
                        position_ids=position_ids, rotary_interleaved=self.rotary_interleaved,
                        cache_dtype=self.cache_dtype, k_scale=self.k_scale, v_scale=self.v_scale)
        self.pk, self.pv = r["present_key"], r["present_value"]
        return r
