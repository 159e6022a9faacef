"""Parity of the small-step tensor-core kernel (keys as the MMA's M dimension) with the
oracle, on a GB300.

Steps whose S x group query rows per (item, kv head) number at most 32, with bf16
caches and head size 128, take this kernel: decode (S = 1) and short speculative
verify steps.  The cases cover every group size, row counts on both sides of the 16-row
padding, items whose window holds no cache row (the step's own rows only), windows
smaller than the step, softcap with an absolute-column bias, sinks, the rotary
embedding, forced stream-K splits (merged by the last contributor), separate present
buffers, and compaction steps.  The bar is the one of the other parity tests.
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


@pytest.mark.parametrize("heads,S", [((8, 8), 1), ((8, 2), 1), ((32, 8), 1), ((16, 1), 1), ((32, 1), 1),
                                     ((8, 4), 8), ((32, 8), 4), ((32, 8), 8), ((16, 2), 2), ((8, 1), 3),
                                     ((2, 2), 16)])
def test_group_sizes_and_rows(heads, S):
    """Group sizes 1..32 and S x g from 1 to 32; a ragged batch with one item from an
    empty cache, one item inside its first window, one item deep in the stream."""
    Nq, Nkv = heads
    sh = wl.Shape("sm", B=3, Nq=Nq, Nkv=Nkv, D=128, W=300, C=320, dtype=wl.BF16)
    pk, pv = wl.cache(sh, 41)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv)
    T = np.array([0, 150, 2000], np.int64)
    for t in range(3):
        q, k, v = wl.step_inputs(sh, S, 4100 + 10 * S + t)
        p.step(q, k, v, T + S - 1)
        T = T + S


@pytest.mark.parametrize("W,C", [(1, 1), (2, 3), (3, 9), (130, 140), (257, 300)])
def test_window_edges(W, C):
    """Windows of 1 key (no cache row is ever visible), windows narrower than the
    step, and windows that end one key into a new 128-key tile."""
    sh = wl.Shape("smw", B=2, Nq=8, Nkv=2, D=128, W=W, C=C, dtype=wl.BF16)
    pk, pv = wl.cache(sh, 42)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv)
    T = np.array([5, 700], np.int64)
    for t, S in enumerate([1, 4, 1, 2, 1]):
        q, k, v = wl.step_inputs(sh, S, 4200 + t)
        p.step(q, k, v, T + S - 1)
        T = T + S


@pytest.mark.parametrize("split_keys", [0, 1, 256])
@pytest.mark.parametrize("inplace", [True, False])
def test_softcap_bias_splits_buffers(split_keys, inplace):
    """Softcap 30 and an fp32 bias passed by stride (allocated at the maximum length),
    verify-shaped steps with rejected drafts, forced splits and separate present
    buffers."""
    sh = wl.Shape("smv", B=4, Nq=32, Nkv=8, D=128, W=1000, C=1007, dtype=wl.BF16, softcap=30.0)
    pk, pv = wl.cache(sh, 43)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, softcap=sh.softcap, past_key=pk, past_value=pv,
             inplace=inplace, split_keys=split_keys)
    T = np.array([10, 900, 1500, 3000], np.int64)
    TM = int(T.max()) + 40
    for t, S in enumerate([8, 4, 8]):
        q, k, v = wl.step_inputs(sh, S, 4300 + t)
        total = int(T.max()) + S
        bias = wl.bias(sh.B, sh.Nq, S, TM, 4300 + t)
        p.step(q, k, v, T + S - 1, total=total, bias=bias, bias_strides=(sh.Nq * S * TM, S * TM, TM))
        # in place, rejected drafts roll back by position alone; a separate present buffer
        # leaves rows past L(T) unspecified, so there every draft is accepted
        T = T + (wl.accepted(sh.B, S, 4300 + t) if inplace else S)


@pytest.mark.parametrize("mode", ["sink", "smooth", "large"])
@pytest.mark.parametrize("split_keys", [0, 128])
def test_sinks(mode, split_keys):
    """head_sink / smooth_softmax on this kernel, directly and through the split merge."""
    from test_gpu_sinks import _sinks

    sh = wl.Shape("sms", B=3, Nq=16, Nkv=4, D=128, W=400, C=410, dtype=wl.BF16)
    pk, pv = wl.cache(sh, 44)
    hs, smooth = _sinks(mode, sh.Nq, 4400)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv, split_keys=split_keys,
             head_sink=hs, smooth_softmax=smooth)
    T = np.array([0, 300, 900], np.int64)
    for t, S in enumerate([1, 4, 1]):
        q, k, v = wl.step_inputs(sh, S, 4410 + t)
        p.step(q, k, v, T + S - 1)
        T = T + S


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotary(interleaved):
    """The query map and the step's new keys are the turned rows of the workspace."""
    sh = wl.Shape("smr", B=2, Nq=32, Nkv=8, D=128, W=200, C=210, dtype=wl.BF16)
    pk, pv = wl.cache(sh, 45)
    cos, sin = wl.rope_tables(2048, 64, wl.BF16)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv, cos_cache=cos,
             sin_cache=sin, rotary_interleaved=interleaved)
    T = np.array([3, 500], np.int64)
    for t, S in enumerate([1, 4, 1, 1]):
        q, k, v = wl.step_inputs(sh, S, 4500 + t)
        p.step(q, k, v, T + S - 1, phases=t == 3)
        T = T + S


def test_slack_compactions_many_steps():
    """C = W + 8: a block is reclaimed every 9 steps; 30 decode steps on 8 items."""
    sh = wl.SHAPES["slack"]
    pk, pv = wl.cache(sh, 46)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv)
    T = wl.lengths(sh.B, 128, 160, 46)
    for t in range(30):
        q, k, v = wl.step_inputs(sh, 1, 4600 + t)
        p.step(q, k, v, T)
        T = T + 1


# ------------------------------------------------------------------ block compaction inside the attention pass


@pytest.mark.parametrize("S,split_keys", [(8, 0), (8, 128), (8, 256), (4, 128), (2, 128), (1, 128), (16, 384)])
def test_compaction_inside_attention_splits(S, split_keys):
    """C = W + S - 1 (a block of S rows reclaimed on every step once the cache is full):
    the kernel moves the surviving rows from its staged tiles and appends the new rows,
    and the host launches no cache-update kernel.  Forced splits put CTA range
    boundaries inside every unit -- rows stashed for the last contributor -- and the
    varying lengths give last tiles of fewer rows than the block (appends left to the
    last contributor).  Softcap and a bias as in the verify workload; 8 steps with
    accepted counts k ~ U{0..S}."""
    from sliding_window_gqa_02_gb300 import gqaw

    W, g = 300, min(4, 32 // S)  # S x g <= 32 query rows per unit
    sh = wl.Shape("cmp", B=4, Nq=4 * g, Nkv=4, D=128, W=W, C=W + S - 1, dtype=wl.BF16, softcap=30.0)
    pk, pv = wl.cache(sh, 43 + S)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, softcap=30.0, past_key=pk, past_value=pv,
             split_keys=split_keys)
    T = np.array([290, 299, 300, 1000], np.int64) + np.arange(4)
    TM = int(T.max()) + 8 * S + 8
    bias = wl.bias(sh.B, sh.Nq, S, TM, 43 + S)
    strides = (sh.Nq * S * TM, S * TM, TM)
    for t in range(8):
        q, k, v = wl.step_inputs(sh, S, 4300 + 10 * S + t)
        n0 = gqaw.gqaw_launch_count()
        p.step(q, k, v, T + S - 1, total=int(T.max()) + S, bias=bias, bias_strides=strides)
        assert gqaw.gqaw_launch_count() - n0 == 1  # the attention kernel alone
        T = T + wl.accepted(sh.B, S, 4300 + t)


@pytest.mark.parametrize("W,S", [(4, 4), (8, 8), (33, 1), (2, 2)])
def test_compaction_inside_attention_small_windows(W, S):
    """Windows of a few keys with C = W + S - 1 (every surviving row is inside the
    window, the new rows may outnumber them), and a block of 33 rows with S = 1 (larger
    than the rows a CTA may stash: the cache-update kernel takes it)."""
    sh = wl.Shape("cmpw", B=3, Nq=8, Nkv=2, D=128, W=W, C=W + S - 1 if W != 33 else 2 * W, dtype=wl.BF16)
    pk, pv = wl.cache(sh, 44)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv, split_keys=128)
    T = np.array([0, 7, 100], np.int64)
    for t in range(12):
        q, k, v = wl.step_inputs(sh, S, 4400 + t)
        p.step(q, k, v, T + S - 1)
        T = T + S


@pytest.mark.parametrize("split_keys", [0, 512])
def test_separate_present_long_context(split_keys):
    """Separate present buffers (mobius issue #111, Part 1.2, Mode A) on the long-context
    shape: the attention kernel writes the surviving rows of the window and the new rows,
    the cache-update kernel only the rows below the window (up to G - 1 = 1024 of them);
    items placed so that some steps reclaim a block.  Three decode steps, every item."""
    sh = wl.Shape("sepl", B=8, Nq=32, Nkv=8, D=128, W=4096, C=5120, dtype=wl.BF16)
    pk, pv = wl.cache(sh, 45)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv, inplace=False,
             split_keys=split_keys)
    G = sh.C - sh.W + 1
    T = wl.lengths(sh.B, 4096, 32768, 45)
    T[0], T[1], T[2] = sh.C + G, sh.C + 2 * G - 1, 4100  # reclaim at the first / second step; no block yet
    for t in range(3):
        q, k, v = wl.step_inputs(sh, 1, 4500 + t)
        p.step(q, k, v, T)
        T = T + 1
