"""Parity of the attention sinks (head_sink, smooth_softmax) with the oracle, on a GB300.

mobius issue #111 "GQA In-Place KV Cache: Investigation Report", Part 1.1 (optional
input head_sink) and Part 1.3 (attribute smooth_softmax): a sink is one more logit
per query head in the softmax denominator, with no value row.  Both kernels finish
a row by dividing by that denominator, so each is checked directly and through its
split-K merge; the bar is the one of the other parity tests.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_driver import GpuCache
from test_gpu_parity import Pair

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _sinks(mode, Nq, seed):
    """(head_sink, smooth_softmax) for a test mode."""
    if mode == "smooth":
        return None, True
    if mode == "both":  # head_sink wins over smooth_softmax
        return wl.head_sink(Nq, seed), True
    if mode == "large":  # sinks that dominate some heads, one far beyond fp32 exp range, one absent
        s = wl.head_sink(Nq, seed, mean=6.0, std=4.0)
        s[0] = 100.0
        s[1] = -float("inf")
        return s, False
    return wl.head_sink(Nq, seed), False


def _run(sh, pair, T, schedule, seed):
    for t, S in enumerate(schedule):
        q, k, v = wl.step_inputs(sh, S, seed + t)
        pair.step(q, k, v, T + S - 1)
        T = T + S
    return pair


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
@pytest.mark.parametrize("split_keys", [0, 16])
@pytest.mark.parametrize("mode", ["sink", "smooth", "both", "large"])
def test_decode_kernel_sinks(dtype, split_keys, mode):
    """FFMA kernel (head size 64): single- and multi-token steps across compactions,
    one item starting from an empty cache; split_keys=16 forces the ticket merge."""
    sh = wl.Shape("sink", B=3, Nq=8, Nkv=2, D=64, W=40, C=48, dtype=dtype)
    pk, pv = wl.cache(sh, 21)
    hs, smooth = _sinks(mode, sh.Nq, 2100)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, dtype, past_key=pk, past_value=pv, split_keys=split_keys,
             head_sink=hs, smooth_softmax=smooth)
    _run(sh, p, np.array([0, 30, 90], np.int64), [5, 1, 1, 3, 1], 2110)


@pytest.mark.parametrize("split_keys", [0, 128])
@pytest.mark.parametrize("mode", ["sink", "smooth", "large"])
@pytest.mark.parametrize("S", [9, 33])
def test_tensor_core_kernel_sinks(split_keys, mode, S):
    """tcgen05 kernel (bf16, head size 128, multi-token steps) with softcap and a
    bias; split_keys=128 forces the merge of key splits."""
    sh = wl.Shape("tcsink", B=2, Nq=16, Nkv=2, D=128, W=300, C=311, dtype=wl.BF16, softcap=20.0)
    pk, pv = wl.cache(sh, 22)
    hs, smooth = _sinks(mode, sh.Nq, 2200)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, softcap=sh.softcap, past_key=pk, past_value=pv,
             split_keys=split_keys, head_sink=hs, smooth_softmax=smooth)
    T = np.array([3, 400], np.int64)
    for t in range(2):
        q, k, v = wl.step_inputs(sh, S, 2210 + t)
        total = int(T.max()) + S
        bias = wl.bias(sh.B, sh.Nq, S, total, 2210 + t, std=1.0)
        p.step(q, k, v, T + S - 1, total=total, bias=bias)
        T = T + S


@pytest.mark.parametrize("dtype,D,S", [(wl.F32, 64, 1), (wl.BF16, 64, 3), (wl.BF16, 128, 9)])
def test_sink_special_values_bit_exact(dtype, D, S):
    """A sink of -inf is no sink, and smooth_softmax is a sink of 0: the outputs are
    bit-identical on the device (FFMA and tensor-core kernels)."""
    sh = wl.Shape("sinkeq", B=2, Nq=4, Nkv=1, D=D, W=20, C=24, dtype=dtype)
    pk, pv = wl.cache(sh, 23)
    q, k, v = wl.step_inputs(sh, S, 2300)
    seq = np.array([S + 10, S + 30], np.int64) - 1

    def out(**kw):
        g = GpuCache(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, dtype, past_key=pk.clone(), past_value=pv.clone(), **kw)
        return g.step(q, k, v, seq)["output"]

    assert torch.equal(out(), out(head_sink=torch.full((sh.Nq,), -float("inf"))))
    assert torch.equal(out(smooth_softmax=True), out(head_sink=torch.zeros(sh.Nq)))
    assert not torch.equal(out(), out(smooth_softmax=True))
