"""Parity of the fused rotary embedding with the oracle, on a GB300.

mobius issue #111 "GQA In-Place KV Cache: Investigation Report", Part 1.1 (cos_cache,
sin_cache, position_ids) and Part 1.3 (do_rotary, rotary_interleaved): the new query
and key rows of a step are turned by the angles of their positions before attention
and before the keys enter the cache.  Outputs are held to the usual bar; the turned
key rows in the cache are floating-point results (fp32 turn on the device, fp64 in
the oracle, one rounding each), held to one spacing of the cache dtype plus 2^-21 of
the row scale; value rows and every row moved by compaction stay bit-exact.
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


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("rd", [64, 32, 12])
def test_decode_kernel_rotary(dtype, interleaved, rd):
    """FFMA kernel (head size 64): 1- and multi-token steps across compactions, a
    ragged batch with one item from an empty cache, full and partial rotary widths
    (rd = 12 does not split into 16-byte vectors for bf16 and for split fp32 pairs:
    the scalar rotary kernel); the last step goes through the two phase calls
    (attention, then cache update)."""
    sh = wl.Shape("rot", B=3, Nq=8, Nkv=2, D=64, W=40, C=48, dtype=dtype)
    pk, pv = wl.cache(sh, 31)
    cos, sin = wl.rope_tables(256, rd // 2, dtype)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, dtype, past_key=pk, past_value=pv, cos_cache=cos,
             sin_cache=sin, rotary_interleaved=interleaved)
    T = np.array([0, 30, 90], np.int64)
    for t, S in enumerate([5, 1, 1, 3, 1, 2]):
        q, k, v = wl.step_inputs(sh, S, 3100 + t)
        p.step(q, k, v, T + S - 1, phases=t == 5)
        T = T + S


@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("split_keys", [0, 128])
@pytest.mark.parametrize("S", [9, 33])
def test_tensor_core_kernel_rotary(interleaved, split_keys, S):
    """tcgen05 kernel (bf16, head size 128): the query and new-key tensor maps point at
    the turned rows; softcap, bias and forced key splits alongside."""
    sh = wl.Shape("tcrot", B=2, Nq=16, Nkv=2, D=128, W=300, C=311, dtype=wl.BF16, softcap=20.0)
    pk, pv = wl.cache(sh, 32)
    cos, sin = wl.rope_tables(1024, 64, wl.BF16)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, softcap=sh.softcap, past_key=pk, past_value=pv,
             split_keys=split_keys, cos_cache=cos, sin_cache=sin, rotary_interleaved=interleaved)
    T = np.array([3, 400], np.int64)
    for t in range(2):
        q, k, v = wl.step_inputs(sh, S, 3200 + t)
        total = int(T.max()) + S
        bias = wl.bias(sh.B, sh.Nq, S, total, 3200 + t, std=1.0)
        p.step(q, k, v, T + S - 1, total=total, bias=bias)
        T = T + S


@pytest.mark.parametrize("dtype,D,S", [(wl.F32, 64, 1), (wl.BF16, 64, 4), (wl.BF16, 128, 9)])
def test_position_ids(dtype, D, S):
    """Explicit position_ids (here positions far from the token counts, different per
    item) replace P_b + s on both kernels."""
    sh = wl.Shape("rotpos", B=2, Nq=4, Nkv=1, D=D, W=20, C=24, dtype=dtype)
    pk, pv = wl.cache(sh, 33)
    cos, sin = wl.rope_tables(4096, D // 2, dtype)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, dtype, past_key=pk, past_value=pv, cos_cache=cos,
             sin_cache=sin)
    T = np.array([10, 25], np.int64)
    for t in range(3):
        q, k, v = wl.step_inputs(sh, S, 3300 + t)
        ids = np.stack([1000 + T[0] + np.arange(S), 3000 - 7 * t + np.arange(S)]).astype(np.int64)
        p.step(q, k, v, T + S - 1, position_ids=ids)
        T = T + S


def test_bad_position_flagged_other_items_correct():
    """A position outside the cos/sin caches sets GQAW_DEV_BAD_POSITION; the other
    item's output and rows still match the oracle."""
    from gpu_driver import compare
    from oracle_driver import OracleCache
    from sliding_window_gqa_02_gb300 import gqaw

    sh = wl.Shape("rotbad", B=2, Nq=4, Nkv=1, D=64, W=20, C=24, dtype=wl.F32)
    cos, sin = wl.rope_tables(64, 32, wl.F32)
    q, k, v = wl.step_inputs(sh, 2, 3400)
    seq = np.array([5, 9], np.int64)
    ids = np.array([[4, 5], [63, 64]], np.int64)  # item 1's second token is past the last row
    g = GpuCache(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, cos_cache=cos, sin_cache=sin)
    rg = g.step(q, k, v, seq, position_ids=ids)
    assert rg["device_flags"] == gqaw.GQAW_DEV_BAD_POSITION
    o = OracleCache(1, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, cos_cache=wl.to_numpy(cos), sin_cache=wl.to_numpy(sin))
    ro = o.step(wl.to_numpy(q)[:1], wl.to_numpy(k)[:1], wl.to_numpy(v)[:1], seq[:1], total=10,
                position_ids=ids[:1])
    rg1 = {key: (val[:1] if key != "device_flags" else 0) for key, val in rg.items()}
    compare(rg1, ro, sh.dtype, turned_keys=True)


def test_rotary_off_is_plain_step():
    """cos/sin given with a zero angle everywhere (cos 1, sin 0) is the plain step,
    bit for bit: the turned copies equal the inputs."""
    sh = wl.Shape("rotid", B=2, Nq=8, Nkv=2, D=128, W=50, C=60, dtype=wl.BF16)
    pk, pv = wl.cache(sh, 35)
    ones = torch.ones((128, 64), dtype=torch.bfloat16)
    zeros = torch.zeros((128, 64), dtype=torch.bfloat16)
    q, k, v = wl.step_inputs(sh, 6, 3500)
    seq = np.array([20, 70], np.int64)
    outs = []
    for kw in ({}, dict(cos_cache=ones, sin_cache=zeros)):
        g = GpuCache(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk.clone(), past_value=pv.clone(),
                     **kw)
        outs.append(g.step(q, k, v, seq))
    assert torch.equal(outs[0]["output"], outs[1]["output"])
    assert np.array_equal(outs[0]["present_key"], outs[1]["present_key"])


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
def test_unaligned_tables(dtype):
    """cos/sin tables that are element-aligned but not 16-byte aligned take the
    scalar rotary kernel; results as before."""
    sh = wl.Shape("rotal", B=2, Nq=4, Nkv=2, D=64, W=20, C=24, dtype=dtype)
    cos, sin = wl.rope_tables(64, 32, dtype)
    flat_c = torch.empty(cos.numel() + 1, dtype=cos.dtype)
    flat_s = torch.empty(sin.numel() + 1, dtype=sin.dtype)
    flat_c[1:] = cos.reshape(-1)
    flat_s[1:] = sin.reshape(-1)
    p = Pair(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, dtype, cos_cache=cos, sin_cache=sin)
    # the device copies: same values at an odd element offset
    dc = flat_c.cuda()[1:].view(64, 32)
    ds = flat_s.cuda()[1:].view(64, 32)
    assert dc.data_ptr() % 16 != 0
    p.g.cos, p.g.sin = dc, ds
    T = np.array([0, 7], np.int64)
    for t, S in enumerate([3, 1]):
        q, k, v = wl.step_inputs(sh, S, 3600 + t)
        p.step(q, k, v, T + S - 1)
        T = T + S
