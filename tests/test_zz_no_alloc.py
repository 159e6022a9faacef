"""gqa_windowed_step_noalloc: the step for callers that cannot allocate device memory.

Such callers (a plugin whose host runtime owns all device memory, a serving loop that
allows no allocation after start-up) cannot hand the library a workspace, so this
entry point takes the split-K scratch from an array compiled into the library.  These
tests call it through the C ABI and check it against gqa_windowed_step on the same
inputs, for two calls in a row on each side.  The file is named to be collected last.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_driver import TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _pair_run(sh, B, S, lo, hi, seed, calls=2):
    from sliding_window_gqa_02_gb300 import gqaw

    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    pk, pv = wl.cache(sh, seed, B=B)
    ka, va = pk.to(dev), pv.to(dev)  # cache of the existing entry point
    kb, vb = pk.to(dev), pv.to(dev)  # cache of the no-allocation entry point
    T = wl.lengths(B, lo, hi, seed)
    for c in range(calls):
        q, k, v = (x.to(dev) for x in wl.step_inputs(sh, S, seed * 10 + c, B=B))
        seq = torch.tensor((T + S - 1).astype(np.int32), device=dev)
        total = int(T.max()) + S
        oa, ob = torch.empty_like(q), torch.full_like(q, float("nan"))
        ra = torch.zeros(B, dtype=torch.int32, device=dev)
        rb = torch.full((B,), -1, dtype=torch.int32, device=dev)
        a = gqaw.make_args(q, k, v, ka, va, ka, va, seq, total, sh.Nq, sh.Nkv, sh.W, oa, resident_len_out=ra)
        ws = gqaw.new_workspace(a, dev, stream)
        a = gqaw.make_args(q, k, v, ka, va, ka, va, seq, total, sh.Nq, sh.Nkv, sh.W, oa, workspace=ws,
                           resident_len_out=ra)
        b = gqaw.make_args(q, k, v, kb, vb, kb, vb, seq, total, sh.Nq, sh.Nkv, sh.W, ob, resident_len_out=rb)
        assert gqaw.gqaw_workspace_bytes(b) > 4096  # the split-K scratch is in use
        gqaw.check(gqaw.gqa_windowed_step(a, stream))
        gqaw.check(gqaw.gqa_windowed_step_noalloc(b, stream))
        torch.cuda.synchronize()
        ref = oa.float()
        err = (ob.float() - ref).abs().max().item() / ref.abs().max().item()
        assert err <= TOL[sh.dtype], err
        assert torch.equal(ra, rb)
        L = ra.cpu().numpy()
        for i in range(B):
            n = int(L[i])
            assert torch.equal(ka[i, :, :n], kb[i, :, :n])
            assert torch.equal(va[i, :, :n], vb[i, :, :n])
        T = T + S


def test_noalloc_matches_step_decode_small_slack():
    """B=8, bf16, W=128, C=136 decode: two calls in a row."""
    _pair_run(wl.SHAPES["slack"], 8, 1, 128, 160, seed=21)


def test_noalloc_matches_step_decode_long_window():
    """B=8 long-context decode (W=4096, C=5120): many key chunks, about 4 MB of scratch."""
    _pair_run(wl.SHAPES["longctx"], 8, 1, 4096, 32768, seed=22)


def test_noalloc_matches_step_multi_token():
    """fp32, 4-token steps crossing evictions (pages shape, B=1)."""
    _pair_run(wl.SHAPES["pages"], 1, 4, 500, 500, seed=23)


def test_noalloc_alternating_shapes():
    """Calls of different shapes in a row on one cache: single-token steps and 32-token
    chunks, with forced key splits so every call uses split-K tickets and partials.  A
    chunk's tickets lie where the single-token call before it left partial results (fp32
    pages shape: 8 units then 256), so each call must clear its own ticket region; the
    reference side gets a fresh workspace for every call."""
    from sliding_window_gqa_02_gb300 import gqaw

    sh = wl.SHAPES["pages"]
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    pk, pv = wl.cache(sh, 24, B=1)
    ka, va = pk.to(dev), pv.to(dev)
    kb, vb = pk.to(dev), pv.to(dev)
    T = 300
    for c, S in enumerate([1, 32, 1, 32, 32, 1]):
        q, k, v = (x.to(dev) for x in wl.step_inputs(sh, S, 2400 + c, B=1))
        seq = torch.tensor([T + S - 1], dtype=torch.int32, device=dev)
        oa, ob = torch.empty_like(q), torch.full_like(q, float("nan"))
        kw = dict(split_keys=32)
        a = gqaw.make_args(q, k, v, ka, va, ka, va, seq, T + S, sh.Nq, sh.Nkv, sh.W, oa, **kw)
        ws = gqaw.new_workspace(a, dev, stream)
        a = gqaw.make_args(q, k, v, ka, va, ka, va, seq, T + S, sh.Nq, sh.Nkv, sh.W, oa, workspace=ws, **kw)
        b = gqaw.make_args(q, k, v, kb, vb, kb, vb, seq, T + S, sh.Nq, sh.Nkv, sh.W, ob, **kw)
        gqaw.check(gqaw.gqa_windowed_step(a, stream))
        gqaw.check(gqaw.gqa_windowed_step_noalloc(b, stream))
        torch.cuda.synchronize()
        ref = oa.float()
        assert torch.isfinite(ob.float()).all(), "call %d (S=%d): rows left unwritten" % (c, S)
        err = (ob.float() - ref).abs().max().item() / ref.abs().max().item()
        assert err <= TOL[sh.dtype], (c, S, err)
        n = gqaw.gqaw_resident_len(T + S, sh.C, sh.W)
        assert torch.equal(ka[0, :, :n], kb[0, :, :n]) and torch.equal(va[0, :, :n], vb[0, :, :n])
        T += S


def test_noalloc_rejects_steps_needing_more_scratch():
    """A step whose split-K scratch exceeds the static array is refused on the host."""
    from sliding_window_gqa_02_gb300 import gqaw

    sh = wl.SHAPES["longctx"]
    a = gqaw.gqaw_step_args()
    # fp32, 4096 items x 512 tokens x 8 kv heads: one 4-byte ticket per attention unit
    # is already 64 MiB of scratch
    a.batch_size, a.sequence_length, a.num_heads, a.kv_num_heads = 4096, 512, sh.Nq, sh.Nkv
    a.head_size, a.capacity, a.local_window_size, a.dtype = sh.D, sh.C, sh.W, gqaw.GQAW_F32
    a.total_sequence_length = 40000
    assert gqaw.gqaw_workspace_bytes(a) > gqaw.GQAW_NOALLOC_SCRATCH_BYTES
    assert gqaw.gqa_windowed_step_noalloc(a, 0) == gqaw.GQAW_EWORKSPACE
    assert "static scratch" in gqaw.gqaw_last_error()
