"""Parity of the CUDA path with the oracle on the five workload configurations of the
pages, at their stated shapes and schedules.

PR #31142 "[CPU] Add windowed kv cache for GQA", Performance Results (512-, 2048- and
8192-token prompts fed in chunks, then decode) and Tests (many compactions at small
slack; chunked prefill); PR #32419 "Specify GroupQueryAttention windowed KV cache layout
contract", Description (C >= W + S - 1 for S-token verify steps; rollback of rejected
drafts is exact iff L(T - k) == L(T) - k).

The bar is the one of gpu_driver.compare: resident lengths and present rows [0, L)
bit-exact, outputs within 1e-5 (fp32) / 2e-2 (bf16) of the output scale.  Where the
oracle cannot evaluate every output of a full-size step in seconds, it evaluates sampled
items (and sampled query rows of long chunks) and the layout of every item.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_driver import GpuCache, compare
from test_gpu_parity import _shape_pair

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _layout_only(rg, lay, dtype, items=None):
    """Compare resident lengths and present rows of the given items, not outputs."""
    compare({**rg, "output": torch.zeros_like(rg["output"])}, {**lay, "output_f64": np.zeros_like(lay["output_f64"])},
            dtype, items=items)


def _item(rg, sl):
    return {k: (v[sl] if k != "device_flags" else v) for k, v in rg.items()}


# ------------------------------------------------------------------ pages-shaped decode (fp32, B=1)


@pytest.mark.parametrize("prompt", [2048, 8192])
def test_pages_long_prompt_chunks_then_decode(prompt):
    """B=1, 64/8 heads, D=64, fp32, W=128, C=384: a 2048- or 8192-token prompt fed as
    32-token chunked-prefill steps, then 256 single-token decode steps; every step
    against the oracle.  Chunks evict a 257-row block every eight or nine steps."""
    sh = wl.SHAPES["pages"]
    p = _shape_pair(sh)
    T = 0
    evictions = 0
    for c in range(prompt // 32):
        q, k, v = wl.step_inputs(sh, 32, 20000 + c)
        p.step(q, k, v, [T + 31])
        evictions += int(oracle.resident_len(T + 32, sh.C, sh.W) < oracle.resident_len(T, sh.C, sh.W) + 32)
        T += 32
    for t in range(256):
        q, k, v = wl.step_inputs(sh, 1, 30000 + t)
        p.step(q, k, v, [T])
        evictions += int(oracle.resident_len(T + 1, sh.C, sh.W) < oracle.resident_len(T, sh.C, sh.W) + 1)
        T += 1
    assert T == prompt + 256
    assert evictions >= (prompt + 256 - sh.C) // (sh.C - sh.W + 1)


# ------------------------------------------------------------------ small slack, many compactions


def test_slack_prefill_then_400_decode_steps():
    """B=8, 32/8 heads, D=128, bf16, W=128, C=136 (G=9): a 128-token prefill, then 400
    decode steps (T = 129..528); every step against the oracle.  The resident lengths the
    GPU reports show exactly 44 compactions per item, the count the pages give
    ("~44" for 400 decode steps at C = W + 8)."""
    sh = wl.SHAPES["slack"]
    p = _shape_pair(sh)
    q, k, v = wl.step_inputs(sh, 128, 40000)
    rg, _ = p.step(q, k, v, np.full(sh.B, 127, np.int64))
    L_prev = rg["resident_len"].astype(np.int64)
    assert np.all(L_prev == 128)
    events = np.zeros(sh.B, np.int64)
    T = np.full(sh.B, 128, np.int64)
    for t in range(400):
        q, k, v = wl.step_inputs(sh, 1, 40001 + t)
        rg, _ = p.step(q, k, v, T)
        L = rg["resident_len"].astype(np.int64)
        events += (L < L_prev + 1).astype(np.int64)  # a block of G rows was reclaimed
        L_prev = L
        T = T + 1
    assert np.all(events == 44), events


def test_slack_ragged_400_decode_steps():
    """The small-slack shape with per-item lengths ~ U[128, 160] (seeded caches), then
    400 decode steps; every step against the oracle, and each item's compaction count
    on the GPU equal to the number of eviction boundaries its positions cross."""
    sh = wl.SHAPES["slack"]
    pk, pv = wl.cache(sh, 41)
    p = _shape_pair(sh, past_key=pk, past_value=pv)
    T = wl.lengths(sh.B, 128, 160, 41)
    want = np.zeros(sh.B, np.int64)
    got = np.zeros(sh.B, np.int64)
    L_prev = np.array([oracle.resident_len(int(x), sh.C, sh.W) for x in T], np.int64)
    for t in range(400):
        q, k, v = wl.step_inputs(sh, 1, 41000 + t)
        rg, _ = p.step(q, k, v, T)
        L = rg["resident_len"].astype(np.int64)
        got += (L < L_prev + 1).astype(np.int64)
        want += np.array([int(oracle.resident_len(int(x) + 1, sh.C, sh.W) < oracle.resident_len(int(x), sh.C, sh.W) + 1)
                          for x in T], np.int64)
        L_prev = L
        T = T + 1
    assert np.array_equal(got, want) and np.all(got >= 43), (got, want)


# ------------------------------------------------------------------ speculative verify at full size


@pytest.mark.parametrize("S", [4, 8])
def test_verify_fullsize_steps_with_rollback(S):
    """B=16, 32/8 heads, D=128, bf16, W=4096, C=W+S-1, contexts ~6000, softcap 30, fp32
    bias ~ N(0, 0.5) allocated once at the maximum length and passed by stride: four
    S-token verify steps, accepted counts k_b ~ U{0..S} (the next step starts from the
    untouched buffer at T_b + k_b, rollbacks exact and inexact).  Every item's layout
    after every step; outputs of sampled items."""
    sh = wl.SHAPES["verify%d" % S]
    B, steps = sh.B, 4
    pk, pv = wl.cache(sh, 30 + S)
    T = np.full(B, 6000, np.int64) + wl.lengths(B, 0, 64, 30 + S)
    TM = int(T.max()) + steps * S + 8
    bias = wl.bias(B, sh.Nq, S, TM, 30 + S)
    strides = (sh.Nq * S * TM, S * TM, TM)
    g = GpuCache(B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, softcap=sh.softcap, past_key=pk, past_value=pv)
    opk, opv = wl.to_numpy(pk), wl.to_numpy(pv)
    exact = inexact = 0
    for t in range(steps):
        q, k, v = wl.step_inputs(sh, S, 31000 + 100 * S + t)
        seq = (T + S - 1).astype(np.int32)
        total = int(T.max()) + S
        rg = g.step(q, k, v, seq, total, bias, strides)
        nq, nk, nv = wl.to_numpy(q), wl.to_numpy(k), wl.to_numpy(v)
        lay = oracle.step(nq, nk, nv, opk, opv, seq, total, sh.Nq, sh.Nkv, sh.W, softcap=sh.softcap,
                          dtype=oracle.BF16, rows=(0, 0))
        _layout_only(rg, lay, sh.dtype)
        for b in (t % B, 7, 15):
            sl = slice(b, b + 1)
            ro = oracle.step(nq[sl], nk[sl], nv[sl], opk[sl], opv[sl], seq[sl], total, sh.Nq, sh.Nkv, sh.W,
                             softcap=sh.softcap, attention_bias=wl.to_numpy(bias[sl]).reshape(-1),
                             bias_strides=strides, dtype=oracle.BF16)
            compare(_item(rg, sl), ro, sh.dtype)
        opk, opv = lay["present_key"], lay["present_value"]
        acc = wl.accepted(B, S, 31000 + 100 * S + t)
        for b in range(B):
            ok = oracle.resident_len(int(T[b] + acc[b]), sh.C, sh.W) == \
                oracle.resident_len(int(T[b] + S), sh.C, sh.W) - (S - int(acc[b]))
            exact += int(ok)
            inexact += int(not ok)
        T = T + acc
    assert inexact > 0 and exact > 0, (exact, inexact)


# ------------------------------------------------------------------ large batch, long context, interleaved


def test_longctx_decode_interleaved_with_prefill_on_one_cache():
    """B=64, 32/8 heads, D=128, bf16, W=4096, C=5120, contexts U[4096, 32768]: decode
    steps on all 64 items interleaved with 512-token chunked-prefill calls on items 0-7,
    the prefill calls given pointers into the same cache (its first eight items).  Some
    items are placed so that a decode step reclaims their block.  Every item's layout
    after every call; outputs of sampled items (sampled query rows of the chunks)."""
    sh = wl.SHAPES["longctx"]
    B, S8, G = sh.B, 512, sh.C - sh.W + 1
    pk, pv = wl.cache(sh, 50)
    T = wl.lengths(B, 4096, 32768, 50)
    T[40:44] = sh.C + G * (1 + np.arange(4))        # reclaim on the first decode step
    T[44:48] = sh.C + G * (2 + np.arange(4)) - 1    # reclaim on the second one
    g64 = GpuCache(B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv)
    g8 = GpuCache(8, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype)
    g8.pk, g8.pv = g64.pk[:8], g64.pv[:8]  # views: the prefill call works on items 0-7 in place
    opk, opv = wl.to_numpy(pk), wl.to_numpy(pv)
    moved = 0
    for c, kind in enumerate(["decode", "prefill", "decode", "prefill", "decode"]):
        if kind == "decode":
            q, k, v = wl.step_inputs(sh, 1, 50000 + c)
            seq = T.astype(np.int32)
            total = int(T.max()) + 1
            rg = g64.step(q, k, v, seq, total)
            nq, nk, nv = wl.to_numpy(q), wl.to_numpy(k), wl.to_numpy(v)
            lay = oracle.step(nq, nk, nv, opk, opv, seq, total, sh.Nq, sh.Nkv, sh.W, dtype=oracle.BF16, rows=(0, 0))
            _layout_only(rg, lay, sh.dtype)
            for b in (0, 5, 40, 44, 63):
                sl = slice(b, b + 1)
                ro = oracle.step(nq[sl], nk[sl], nv[sl], opk[sl], opv[sl], seq[sl], total, sh.Nq, sh.Nkv, sh.W,
                                 dtype=oracle.BF16)
                compare(_item(rg, sl), ro, sh.dtype)
            moved += sum(int(oracle.resident_len(int(x) + 1, sh.C, sh.W) < oracle.resident_len(int(x), sh.C, sh.W) + 1)
                         for x in T)
            opk, opv = lay["present_key"], lay["present_value"]
            T = T + 1
        else:
            q, k, v = wl.step_inputs(sh, S8, 50000 + c, B=8)
            seq = (T[:8] + S8 - 1).astype(np.int32)
            total = int(T[:8].max()) + S8
            rg = g8.step(q, k, v, seq, total)
            nq, nk, nv = wl.to_numpy(q), wl.to_numpy(k), wl.to_numpy(v)
            lay = oracle.step(nq, nk, nv, opk[:8], opv[:8], seq, total, sh.Nq, sh.Nkv, sh.W, dtype=oracle.BF16,
                              rows=(0, 0))
            _layout_only(rg, lay, sh.dtype)
            for b in (2, 6):
                sl = slice(b, b + 1)
                for rows in ((0, 4), (254, 258), (508, 512)):
                    ro = oracle.step(nq[sl], nk[sl], nv[sl], opk[sl], opv[sl], seq[sl], total, sh.Nq, sh.Nkv, sh.W,
                                     dtype=oracle.BF16, rows=rows)
                    compare(_item(rg, sl), ro, sh.dtype, rows=rows)
            opk = opk.copy()
            opv = opv.copy()
            opk[:8], opv[:8] = lay["present_key"], lay["present_value"]
            T[:8] = T[:8] + S8
        # the items outside the call are untouched by it: all 64 against the oracle's state
        full = {"resident_len": np.array([oracle.resident_len(int(x), sh.C, sh.W) for x in T], np.int32),
                "present_key": opk, "present_value": opv, "output_f64": np.zeros((B, 1, 1))}
        got = {"resident_len": full["resident_len"], "present_key": wl.to_numpy(g64.pk.cpu()),
               "present_value": wl.to_numpy(g64.pv.cpu()), "device_flags": 0, "output": torch.zeros((B, 1, 1))}
        compare(got, full, sh.dtype)
    assert moved >= 8
