"""Parity of the quantized KV cache with the oracle, on a GB300.

mobius issue #111 "GQA In-Place KV Cache: Investigation Report", Part 1.1, inputs k_scale
and v_scale: the caches hold int8 or fp8 e4m3 codes with one scale per tensor.  The
step's new rows are quantized on the device (x / scale in float, ties to even,
saturated) and must give the oracle's codes bit for bit; attention reads every key and
value as code * scale; outputs are held to the usual bf16 bar.  Scales are chosen so
that some codes saturate.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as wl
from test_gpu_parity import Pair

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


SCALES = {"i8": (0.02, 0.025), "e4m3": (0.01, 0.005)}


def _pair(sh, ct, seed, **kw):
    pk, pv = wl.code_cache(sh, seed, ct)
    ks, vs = SCALES[ct]
    return Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, softcap=sh.softcap, past_key=pk, past_value=pv,
                cache_dtype=ct, k_scale=ks, v_scale=vs, **kw)


@pytest.mark.parametrize("ct", ["i8", "e4m3"])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("heads", [(8, 2), (32, 8), (16, 1)])
def test_decode_and_multi_token(ct, D, heads):
    """1- and multi-token steps across compactions, a ragged batch with one item from an
    empty cache, every query-head block size."""
    Nq, Nkv = heads
    sh = wl.Shape("q8", B=3, Nq=Nq, Nkv=Nkv, D=D, W=40, C=48, dtype=wl.BF16)
    p = _pair(sh, ct, 51)
    T = np.array([0, 30, 90], np.int64)
    for t, S in enumerate([5, 1, 1, 3, 1]):
        q, k, v = wl.step_inputs(sh, S, 5100 + t)
        p.step(q, k, v, T + S - 1, phases=t == 4)
        T = T + S


@pytest.mark.parametrize("ct", ["i8", "e4m3"])
@pytest.mark.parametrize("split_keys", [0, 16])
@pytest.mark.parametrize("inplace", [True, False])
def test_softcap_bias_splits_buffers(ct, split_keys, inplace):
    """Softcap, an absolute-column bias, forced key splits and separate present buffers."""
    sh = wl.Shape("q8b", B=2, Nq=16, Nkv=4, D=128, W=100, C=107, dtype=wl.BF16, softcap=30.0)
    p = _pair(sh, ct, 52, split_keys=split_keys, inplace=inplace)
    T = np.array([10, 300], np.int64)
    for t, S in enumerate([4, 1, 8]):
        q, k, v = wl.step_inputs(sh, S, 5200 + t)
        total = int(T.max()) + S
        bias = wl.bias(sh.B, sh.Nq, S, total, 5200 + t, std=1.0)
        p.step(q, k, v, T + S - 1, total=total, bias=bias)
        T = T + S


@pytest.mark.parametrize("ct", ["i8", "e4m3"])
def test_rotary_and_sinks(ct):
    """The rotary embedding turns the keys before they are quantized (codes within one
    step of the oracle's); head_sink joins the softmax."""
    sh = wl.Shape("q8r", B=2, Nq=8, Nkv=2, D=128, W=60, C=64, dtype=wl.BF16)
    cos, sin = wl.rope_tables(1024, 64, wl.BF16)
    p = _pair(sh, ct, 53, cos_cache=cos, sin_cache=sin, head_sink=wl.head_sink(sh.Nq, 5300))
    T = np.array([0, 500], np.int64)
    for t, S in enumerate([3, 1, 1, 2]):
        q, k, v = wl.step_inputs(sh, S, 5310 + t)
        p.step(q, k, v, T + S - 1)
        T = T + S


@pytest.mark.parametrize("ct", ["i8", "e4m3"])
@pytest.mark.parametrize("heads,S", [((32, 8), 1), ((32, 8), 4), ((32, 8), 8), ((8, 8), 1), ((16, 2), 2), ((32, 1), 1)])
@pytest.mark.parametrize("split_keys", [0, 128])
def test_tensor_core_path(ct, heads, S, split_keys):
    """Head size 128 with S x group <= 32: the tensor-core kernel widens the code tiles to
    fp16 operands; every processed-row count (4, 8, 16, 32), a ragged batch with one
    item from an empty cache and a window crossing several 128-key tiles, key splits."""
    Nq, Nkv = heads
    sh = wl.Shape("q8t", B=3, Nq=Nq, Nkv=Nkv, D=128, W=300, C=310, dtype=wl.BF16)
    p = _pair(sh, ct, 55, split_keys=split_keys)
    T = np.array([0, 150, 2000], np.int64)
    for t in range(3):
        q, k, v = wl.step_inputs(sh, S, 5500 + 10 * S + t)
        p.step(q, k, v, T + S - 1)
        T = T + S


def test_long_context_decode_sampled():
    """The long-context shape (32/8 heads, head size 128, W 4096) on an int8 cache: the
    first step of a B=8 batch compared in full."""
    sh = wl.Shape("q8l", B=8, Nq=32, Nkv=8, D=128, W=4096, C=5120, dtype=wl.BF16)
    p = _pair(sh, "i8", 54)
    T = wl.lengths(sh.B, 4096, 20000, 54)
    for t in range(2):
        q, k, v = wl.step_inputs(sh, 1, 5400 + t)
        p.step(q, k, v, T)
        T = T + 1


@pytest.mark.parametrize("big,flagged", [(65280.0, False), (99840.0, True)])
def test_query_beyond_fp16_range_flagged(big, flagged):
    """On the tensor-core small-step path the query of a quantized cache becomes fp16: a
    finite bfloat16 element with no finite fp16 value (99840) sets GQAW_DEV_QUERY_RANGE;
    the largest bfloat16 below fp16's limit (65280) does not."""
    from gpu_driver import GpuCache
    from sliding_window_gqa_02_gb300 import gqaw

    sh = wl.Shape("q8f", B=2, Nq=8, Nkv=2, D=128, W=200, C=210, dtype=wl.BF16)
    pk, pv = wl.code_cache(sh, 56, "e4m3")
    ks, vs = SCALES["e4m3"]
    g = GpuCache(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv, cache_dtype="e4m3",
                 k_scale=ks, v_scale=vs)
    q, k, v = wl.step_inputs(sh, 1, 5600)
    q[1, 0, 5] = big
    rg = g.step(q, k, v, np.array([150, 160], np.int64))
    assert bool(rg["device_flags"] & gqaw.GQAW_DEV_QUERY_RANGE) == flagged
