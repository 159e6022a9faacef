"""Parity of the CUDA path (through the C ABI) with the oracle, on a GB300.

Every step runs on both sides from the same seeded inputs; each side keeps its own
cache between steps.  The bar (see gpu_driver.compare): resident lengths and present
rows [0, L) bit-exact, outputs within 1e-5 (fp32) / 2e-2 (bf16) of the output scale.
Workload shapes follow the pages' configurations (workloads.py); the full-size cases
check sampled items with the oracle and every item's layout.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_driver import GpuCache, compare, oracle_dtype
from oracle_driver import OracleCache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


class Pair:
    """The same cache driven by the CUDA library and by the oracle."""

    def __init__(self, B, Nq, Nkv, D, C, W, dtype, scale=0.0, softcap=0.0, past_key=None, past_value=None,
                 inplace=True, split_keys=0, head_sink=None, smooth_softmax=False, cos_cache=None, sin_cache=None,
                 rotary_interleaved=False, cache_dtype=None, k_scale=1.0, v_scale=1.0):
        self.dtype = dtype
        self.cache_dtype = cache_dtype
        self.turned = cos_cache is not None
        self.g = GpuCache(B, Nq, Nkv, D, C, W, dtype, scale, softcap, past_key, past_value, inplace, split_keys,
                          head_sink, smooth_softmax, cos_cache, sin_cache, rotary_interleaved, cache_dtype, k_scale,
                          v_scale)
        self.o = OracleCache(B, Nq, Nkv, D, C, W, oracle_dtype(dtype), scale, softcap,
                             None if past_key is None else wl.to_numpy(past_key),
                             None if past_value is None else wl.to_numpy(past_value),
                             None if head_sink is None else wl.to_numpy(head_sink), smooth_softmax,
                             None if cos_cache is None else wl.to_numpy(cos_cache),
                             None if sin_cache is None else wl.to_numpy(sin_cache), rotary_interleaved,
                             {None: None, "i8": oracle.I8, "e4m3": oracle.E4M3}[cache_dtype], k_scale, v_scale)
        self.errs = []

    def step(self, q, k, v, seqlens, total=None, bias=None, bias_strides=None, phases=False, position_ids=None):
        rg = self.g.step(q, k, v, seqlens, total, bias, bias_strides, phases, position_ids)
        nb = None if bias is None else wl.to_numpy(bias).reshape(-1) if bias_strides else wl.to_numpy(bias)
        ro = self.o.step(wl.to_numpy(q), wl.to_numpy(k), wl.to_numpy(v), np.asarray(seqlens, np.int32), total,
                         nb, bias_strides, position_ids)
        self.errs.append(compare(rg, ro, self.dtype, turned_keys=self.turned, cache_dtype=self.cache_dtype))
        return rg, ro


def _shape_pair(sh, **kw):
    return Pair(sh.B if "B" not in kw else kw.pop("B"), sh.Nq, sh.Nkv, sh.D, kw.pop("C", sh.C), sh.W, sh.dtype,
                softcap=kw.pop("softcap", sh.softcap), **kw)


# ------------------------------------------------------------------ tiny contract


@pytest.mark.parametrize("inplace", [True, False])
@pytest.mark.parametrize("variant", ["uniform", "onehot", "zero_q"])
def test_tiny_contract_sequence(inplace, variant):
    """C=6, W=4, D=8: 8-token prefill (S > C), a 4-token step, 12 single steps (T up
    to 24), a 4-draft verify (T=28) accepting 2, and the next step from T=26."""
    sh = wl.SHAPES["tiny"]
    p = _shape_pair(sh, inplace=inplace)
    T = 0
    seed = 0
    for S in [8, 4] + [1] * 12 + [4]:
        seed += 1
        q, k, v = wl.step_inputs(sh, S, seed)
        if variant == "onehot":
            pos = torch.arange(T, T + S)
            v = torch.zeros(1, S, sh.D)
            v[0, torch.arange(S), pos % sh.D] = 1.0
        if variant == "zero_q":
            q = torch.zeros_like(q)
        p.step(q, k, v, [T + S - 1])
        T += S
    T -= 2  # 2 of the 4 drafts rejected: the buffer is reused untouched
    q, k, v = wl.step_inputs(sh, 1, 99)
    p.step(q, k, v, [T])
    assert max(p.errs) <= 1e-5


def test_tiny_exact_rollback_point():
    """Verify 20 -> 24 accepting 2 is exact (L(22) == L(24) - 2): resuming from the
    untouched buffer equals the accepted-only history, on the GPU."""
    sh = wl.SHAPES["tiny"]
    a = _shape_pair(sh)
    b = _shape_pair(sh)
    q, k, v = wl.step_inputs(sh, 24, 5)
    a.step(q[:, :20], k[:, :20], v[:, :20], [19])
    b.step(q[:, :20], k[:, :20], v[:, :20], [19])
    a.step(q[:, 20:24], k[:, 20:24], v[:, 20:24], [23])  # verify 4, accept 2
    b.step(q[:, 20:22], k[:, 20:22], v[:, 20:22], [21])  # accepted only
    q2, k2, v2 = wl.step_inputs(sh, 1, 6)
    ra, _ = a.step(q2, k2, v2, [22])
    rb, _ = b.step(q2, k2, v2, [22])
    assert torch.equal(ra["output"], rb["output"])
    n = int(ra["resident_len"][0])
    assert np.array_equal(ra["present_key"][:, :, :n], rb["present_key"][:, :, :n])


# ------------------------------------------------------------------ pages-shaped decode


def test_pages_decode_chunked_prompt():
    """B=1, 64/8 heads, D=64, fp32, W=128, C=384: a 512-token prompt in 32-token
    chunks, then 260 decode steps (crossing an eviction at T=642)."""
    sh = wl.SHAPES["pages"]
    p = _shape_pair(sh)
    T = 0
    for c in range(16):
        q, k, v = wl.step_inputs(sh, 32, 1000 + c)
        p.step(q, k, v, [T + 31])
        T += 32
    evictions = 0
    for t in range(260):
        q, k, v = wl.step_inputs(sh, 1, 2000 + t)
        rg, _ = p.step(q, k, v, [T])
        T += 1
        evictions += int(oracle.resident_len(T, sh.C, sh.W) < oracle.resident_len(T - 1, sh.C, sh.W) + 1)
    assert evictions == 1


# ------------------------------------------------------------------ small slack


def test_slack_decode_many_compactions():
    """B=8, 32/8 heads, D=128, bf16, W=128, C=136 (G=9): items seeded at ragged
    lengths in [128, 160], then 40 decode steps (every item compacts several times)."""
    sh = wl.SHAPES["slack"]
    pk, pv = wl.cache(sh, 3)
    p = _shape_pair(sh, past_key=pk, past_value=pv)
    T = wl.lengths(sh.B, 128, 160, 3)
    for t in range(40):
        q, k, v = wl.step_inputs(sh, 1, 3000 + t)
        p.step(q, k, v, T)  # seqlens_k = T_b - 1 + 1: one new token on a cache of T_b
        T = T + 1


@pytest.mark.parametrize("D", [16, 128])
def test_separate_present_many_items(D):
    """A separate present buffer registers every item each step; with 600 items the
    copy kernel keeps the first 512 plans in shared memory and computes the others per
    job.  Contexts cross the capacity (reclaiming and drifting items in one step); head
    size 16 runs the FFMA attention, 128 the small-step tensor-core kernel (which leaves
    only the rows below the window)."""
    sh = wl.Shape("many", B=600, Nq=2, Nkv=1, D=D, W=12, C=16, dtype=wl.BF16)
    pk, pv = wl.cache(sh, 61)
    p = _shape_pair(sh, past_key=pk, past_value=pv, inplace=False)
    T = wl.lengths(sh.B, 5, 60, 61)
    for t in range(3):
        q, k, v = wl.step_inputs(sh, 1, 6100 + t)
        p.step(q, k, v, T)
        T = T + 1


@pytest.mark.parametrize("inplace", [True, False])
def test_slack_chunked_prefill_from_drifted_point(inplace):
    """C = W + 8 with 32-token chunks: a chunk can compact below the history its own
    first query reads (the CPU stages these steps; here attention runs first)."""
    sh = wl.SHAPES["slack"]
    pk, pv = wl.cache(sh, 4)
    p = _shape_pair(sh, past_key=pk, past_value=pv, inplace=inplace)
    T = wl.lengths(sh.B, 128, 160, 4)
    hazards = 0
    for c in range(6):
        q, k, v = wl.step_inputs(sh, 32, 4000 + c)
        for b in range(sh.B):
            P = int(T[b])
            kept = oracle.resident_len(P + 32, sh.C, sh.W) - 32
            hazards += int(kept < min(P, sh.W - 1))
        p.step(q, k, v, T + 31)
        T = T + 32
    assert hazards > 0


# ------------------------------------------------------------------ speculative verify


@pytest.mark.parametrize("S", [4, 8])
def test_verify_rollback_softcap_bias_small(S):
    """Verify steps with accepted counts k_b ~ U{0..S}, softcap 30, fp32 bias
    ~ N(0, 0.5) allocated once at the maximum length and passed by stride; C = W+S-1
    (W reduced to 256 so the oracle runs every item)."""
    W, B, T0, steps = 256, 4, 400, 6
    sh = wl.SHAPES["verify%d" % S]
    C = W + S - 1
    pk, pv = wl.cache(sh, 5, B=B, capacity=C)
    p = Pair(B, sh.Nq, sh.Nkv, sh.D, C, W, sh.dtype, softcap=30.0, past_key=pk, past_value=pv)
    TM = T0 + steps * S + 8
    bias = wl.bias(B, sh.Nq, S, TM, 5)
    strides = (sh.Nq * S * TM, S * TM, TM)
    T = np.full(B, T0, np.int64) + wl.lengths(B, 0, 8, 5)
    inexact = 0
    for t in range(steps):
        q, k, v = wl.step_inputs(sh, S, 5000 + t, B=B)
        total = int(T.max()) + S
        p.step(q, k, v, T + S - 1, total=total, bias=bias, bias_strides=strides)
        acc = wl.accepted(B, S, 5000 + t)
        for b in range(B):
            inexact += int(oracle.resident_len(T[b] + acc[b], C, W) != oracle.resident_len(T[b] + S, C, W) - (S - acc[b]))
        T = T + acc
    assert inexact >= 0


def test_verify_fullsize_sampled():
    """The full verify workload (B=16, W=4096, C=W+7, S=8, T=6000, softcap, bias): one
    step on the GPU; outputs of sampled items against the oracle, layout of all."""
    sh = wl.SHAPES["verify8"]
    S = 8
    pk, pv = wl.cache(sh, 6)
    T = np.full(sh.B, 6000, np.int64) + wl.lengths(sh.B, 0, 64, 6)
    total = int(T.max()) + S
    bias = wl.bias(sh.B, sh.Nq, S, total, 6)
    q, k, v = wl.step_inputs(sh, S, 6000)
    g = GpuCache(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, softcap=30.0, past_key=pk, past_value=pv)
    rg = g.step(q, k, v, T + S - 1, total, bias)
    npk, npv = wl.to_numpy(pk), wl.to_numpy(pv)
    lay = oracle.step(wl.to_numpy(q), wl.to_numpy(k), wl.to_numpy(v), npk, npv, (T + S - 1).astype(np.int32), total,
                      sh.Nq, sh.Nkv, sh.W, softcap=30.0, dtype=oracle.BF16, rows=(0, 0))
    compare({**rg, "output": torch.zeros_like(rg["output"])}, {**lay, "output_f64": np.zeros_like(lay["output_f64"])},
            sh.dtype)
    for b in (0, 11):
        sl = slice(b, b + 1)
        ro = oracle.step(wl.to_numpy(q[sl]), wl.to_numpy(k[sl]), wl.to_numpy(v[sl]), npk[sl], npv[sl],
                         (T[sl] + S - 1).astype(np.int32), total, sh.Nq, sh.Nkv, sh.W, softcap=30.0,
                         attention_bias=wl.to_numpy(bias[sl]), dtype=oracle.BF16)
        sub = {k2: (v2[sl] if k2 != "device_flags" else v2) for k2, v2 in rg.items()}
        compare(sub, ro, sh.dtype)


# ------------------------------------------------------------------ large batch, long context


def _longctx_state(seed, evict_all=False):
    sh = wl.SHAPES["longctx"]
    pk, pv = wl.cache(sh, seed)
    T = wl.lengths(sh.B, 4096, 32768, seed)
    if evict_all:  # every item reclaims a block in this step: T_b + 1 = C + 1 + m*G
        G = sh.C - sh.W + 1
        T = sh.C + G * (T % 20)
    return sh, pk, pv, T


@pytest.mark.parametrize("evict_all", [False, True])
def test_longctx_decode_fullsize_sampled(evict_all):
    """B=64, 32/8 heads, D=128, bf16, W=4096, C=5120, contexts U[4096, 32768]: one
    decode step in the benchmark's launch configuration; sampled items against the
    oracle, every item's layout bit-exact (with evict_all every item moves 4095 rows)."""
    sh, pk, pv, T = _longctx_state(7, evict_all)
    q, k, v = wl.step_inputs(sh, 1, 7000)
    g = GpuCache(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv)
    rg = g.step(q, k, v, T)
    npk, npv = wl.to_numpy(pk), wl.to_numpy(pv)
    lay = oracle.step(wl.to_numpy(q), wl.to_numpy(k), wl.to_numpy(v), npk, npv, T.astype(np.int32), int(T.max()) + 1,
                      sh.Nq, sh.Nkv, sh.W, dtype=oracle.BF16, rows=(0, 0))
    compare({**rg, "output": torch.zeros_like(rg["output"])}, {**lay, "output_f64": np.zeros_like(lay["output_f64"])},
            sh.dtype)
    for b in (0, 31, 63):
        sl = slice(b, b + 1)
        ro = oracle.step(wl.to_numpy(q[sl]), wl.to_numpy(k[sl]), wl.to_numpy(v[sl]), npk[sl], npv[sl],
                         T[sl].astype(np.int32), int(T.max()) + 1, sh.Nq, sh.Nkv, sh.W, dtype=oracle.BF16)
        sub = {k2: (v2[sl] if k2 != "device_flags" else v2) for k2, v2 in rg.items()}
        compare(sub, ro, sh.dtype)


def test_longctx_chunked_prefill_sampled():
    """The 512-token chunked-prefill call on 8 items of the long-context workload;
    sampled query rows of two items against the oracle, layout of all 8."""
    sh = wl.SHAPES["longctx"]
    B, S = 8, 512
    pk, pv = wl.cache(sh, 8, B=B)
    T = wl.lengths(B, 4096, 32768, 8)
    q, k, v = wl.step_inputs(sh, S, 8000, B=B)
    g = GpuCache(B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv)
    rg = g.step(q, k, v, T + S - 1)
    npk, npv = wl.to_numpy(pk), wl.to_numpy(pv)
    total = int(T.max()) + S
    lay = oracle.step(wl.to_numpy(q), wl.to_numpy(k), wl.to_numpy(v), npk, npv, (T + S - 1).astype(np.int32), total,
                      sh.Nq, sh.Nkv, sh.W, dtype=oracle.BF16, rows=(0, 0))
    compare({**rg, "output": torch.zeros_like(rg["output"])}, {**lay, "output_f64": np.zeros_like(lay["output_f64"])},
            sh.dtype)
    for b in (2, 5):
        sl = slice(b, b + 1)
        for rows in ((0, 6), (253, 259), (506, 512)):
            ro = oracle.step(wl.to_numpy(q[sl]), wl.to_numpy(k[sl]), wl.to_numpy(v[sl]), npk[sl], npv[sl],
                             (T[sl] + S - 1).astype(np.int32), total, sh.Nq, sh.Nkv, sh.W, dtype=oracle.BF16,
                             rows=rows)
            sub = {k2: (v2[sl] if k2 != "device_flags" else v2) for k2, v2 in rg.items()}
            compare(sub, ro, sh.dtype, rows=rows)


# ------------------------------------------------------------------ shapes and edges


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
@pytest.mark.parametrize("D", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("heads", [(1, 1), (6, 2), (12, 1), (16, 2)])
def test_head_sizes_groups_ragged(dtype, D, heads):
    """Every supported head size and query-head grouping (group 1, 3, 12, 8), a ragged
    batch of 3, steps of 1, 3, 7 and 40 (> C) tokens, W=24, C=30."""
    Nq, Nkv = heads
    B, C, W = 3, 30, 24
    sh = wl.Shape("t", B=B, Nq=Nq, Nkv=Nkv, D=D, W=W, C=C, dtype=dtype)
    p = _shape_pair(sh)
    T = np.array([0, 5, 17], np.int64)
    seed = 100 * D + Nq
    for S in [40, 1, 3, 7, 1, 40, 3, 1]:
        seed += 1
        q, k, v = wl.step_inputs(sh, S, seed)
        p.step(q, k, v, T + S - 1)
        T = T + S


@pytest.mark.parametrize("C,W", [(1, 1), (2, 1), (5, 1), (8, 8), (9, 3)])
def test_window_edges(C, W):
    """W = 1 (self only), C = W (G = 1: a block of one row every step), first token."""
    sh = wl.Shape("e", B=2, Nq=4, Nkv=2, D=32, W=W, C=C, dtype=wl.F32)
    p = _shape_pair(sh)
    T = np.array([0, 3], np.int64)
    for i, S in enumerate([1, 2, 1, 5, 1, 1, 11, 1]):
        q, k, v = wl.step_inputs(sh, S, 700 + i)
        p.step(q, k, v, T + S - 1)
        T = T + S


def test_empty_batch_is_noop():
    from sliding_window_gqa_02_gb300 import gqaw

    dev = torch.device("cuda:0")
    z = torch.zeros((0, 1, 8), device=dev)
    c = torch.zeros((0, 1, 6, 8), device=dev)
    seq = torch.zeros(0, dtype=torch.int32, device=dev)
    a = gqaw.make_args(z, z, z, c, c, c, c, seq, 1, 1, 1, 4, z)
    assert gqaw.gqa_windowed_step(a, 0) == gqaw.GQAW_OK


@pytest.mark.parametrize("split_keys", [1, 32, 100, 4096])
def test_split_override(split_keys):
    """Forced split sizes (one tile per chunk, a non-multiple of the tile, no split)
    give the same parity."""
    sh = wl.SHAPES["slack"]
    pk, pv = wl.cache(sh, 9)
    p = _shape_pair(sh, past_key=pk, past_value=pv, split_keys=split_keys)
    T = wl.lengths(sh.B, 1, 300, 9)
    for t, S in enumerate([1, 1, 5, 1]):
        q, k, v = wl.step_inputs(sh, S, 9000 + t)
        p.step(q, k, v, T + S - 1)
        T = T + S


def test_phases_equal_one_call():
    """gqaw_attend followed by gqaw_update_cache equals gqa_windowed_step."""
    sh = wl.SHAPES["slack"]
    pk, pv = wl.cache(sh, 10)
    a = GpuCache(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv)
    b = GpuCache(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv)
    T = wl.lengths(sh.B, 128, 160, 10)
    for t in range(3):
        q, k, v = wl.step_inputs(sh, 1, 10000 + t)
        ra = a.step(q, k, v, T)
        rb = b.step(q, k, v, T, phases=True)
        assert torch.equal(ra["output"], rb["output"])
        assert np.array_equal(ra["present_key"], rb["present_key"])
        T = T + 1


def test_workspace_reused_across_shapes():
    """One workspace, sized for the largest step, serves steps of different shapes on
    one cache (single-token steps and 32-token chunks, forced key splits): a chunk's
    tickets lie where the single-token step before it left partial results, and the
    library clears them when the layout changes.  Checked against the oracle."""
    from sliding_window_gqa_02_gb300 import gqaw

    sh = wl.SHAPES["pages"]
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    pk, pv = wl.cache(sh, 25, B=1)
    o = OracleCache(1, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, oracle.F32, past_key=wl.to_numpy(pk),
                    past_value=wl.to_numpy(pv))
    gk, gv = pk.to(dev), pv.to(dev)
    T, shapes = 300, [1, 32, 1, 32, 32, 1]
    need = 0
    for S in shapes:  # the workspace is sized for the largest of the steps
        q0 = torch.empty((1, S, sh.Nq * sh.D), device=dev)
        a = gqaw.make_args(q0, q0[..., :sh.Nkv * sh.D], q0[..., :sh.Nkv * sh.D], gk, gv, gk, gv,
                           torch.zeros(1, dtype=torch.int32, device=dev), 2000, sh.Nq, sh.Nkv, sh.W, q0,
                           split_keys=32)
        need = max(need, gqaw.gqaw_workspace_bytes(a))
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    gqaw.check(gqaw.gqaw_workspace_init(int(ws.data_ptr()), need, stream))
    for c, S in enumerate(shapes):
        q, k, v = wl.step_inputs(sh, S, 2500 + c, B=1)
        dq, dk, dv = (x.to(dev) for x in (q, k, v))
        seq = torch.tensor([T + S - 1], dtype=torch.int32, device=dev)
        out = torch.full_like(dq, float("nan"))
        res = torch.full((1,), -1, dtype=torch.int32, device=dev)
        a = gqaw.make_args(dq, dk, dv, gk, gv, gk, gv, seq, T + S, sh.Nq, sh.Nkv, sh.W, out, workspace=ws,
                           resident_len_out=res, split_keys=32)
        gqaw.check(gqaw.gqa_windowed_step(a, stream))
        torch.cuda.synchronize()
        st, flags = gqaw.gqaw_device_status(int(ws.data_ptr()), stream=stream)
        ro = o.step(wl.to_numpy(q), wl.to_numpy(k), wl.to_numpy(v), np.array([T + S - 1], np.int32))
        rg = {"output": out.cpu(), "resident_len": res.cpu().numpy(), "present_key": wl.to_numpy(gk.cpu()),
              "present_value": wl.to_numpy(gv.cpu()), "device_flags": flags}
        compare(rg, ro, sh.dtype)
        T += S


def test_bias_broadcast_strides():
    """Bias shapes (1, Nq, S, total) and (B, 1, S, total): stride 0 broadcasts."""
    sh = wl.Shape("b", B=3, Nq=8, Nkv=2, D=64, W=16, C=20, dtype=wl.BF16, softcap=5.0)
    for bshape in [(1, 8), (3, 1)]:
        p = _shape_pair(sh)
        T = np.array([2, 9, 30], np.int64)
        for t, S in enumerate([3, 1, 6]):
            q, k, v = wl.step_inputs(sh, S, 1100 + t)
            total = int(T.max()) + S
            bias = wl.bias(bshape[0], bshape[1], S, total, 1100 + t, std=2.0)
            p.step(q, k, v, T + S - 1, total=total, bias=bias)
            T = T + S


def test_bad_seqlens_flagged_others_correct():
    """An item whose seqlens_k + 1 < S and one whose T > total_sequence_length set the
    device status bit; the other items are computed normally."""
    sh = wl.Shape("x", B=4, Nq=4, Nkv=1, D=64, W=8, C=10, dtype=wl.F32)
    g = GpuCache(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype)
    o = OracleCache(2, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W)
    S = 3
    q, k, v = wl.step_inputs(sh, S, 12)
    seq = np.array([5, 0, 11, 40], np.int64)  # item 1: P < 0; item 3: T = 41 > total
    rg = g.step(q, k, v, seq, total=13)
    assert rg["device_flags"] & 1
    good = [0, 2]
    ro = o.step(wl.to_numpy(q[good]), wl.to_numpy(k[good]), wl.to_numpy(v[good]), seq[good].astype(np.int32),
                total=13)
    sub = {kk: (vv[good] if kk != "device_flags" else 0) for kk, vv in rg.items()}
    compare(sub, ro, sh.dtype)


def test_positions_near_int32_max():
    """T close to INT32_MAX: 64-bit planning on the device keeps the layout."""
    sh = wl.SHAPES["tiny"]
    pk, pv = wl.cache(sh, 13)
    p = _shape_pair(sh, past_key=pk, past_value=pv)
    T = 2**31 - 40
    for t, S in enumerate([1, 4, 1, 8, 1]):
        q, k, v = wl.step_inputs(sh, S, 1300 + t)
        p.step(q, k, v, [T + S - 1], total=T + S)
        T += S


def test_multi_token_equals_single_tokens_gpu():
    """A 4-token step and four 1-token steps leave bit-identical present rows."""
    sh = wl.SHAPES["slack"]
    pk, pv = wl.cache(sh, 14)
    a = GpuCache(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv)
    b = GpuCache(sh.B, sh.Nq, sh.Nkv, sh.D, sh.C, sh.W, sh.dtype, past_key=pk, past_value=pv)
    T = wl.lengths(sh.B, 128, 160, 14)
    q, k, v = wl.step_inputs(sh, 4, 1400)
    ra = a.step(q, k, v, T + 3)
    for s in range(4):
        rb = b.step(q[:, s:s + 1], k[:, s:s + 1], v[:, s:s + 1], T + s)
        err = (rb["output"][:, 0].float() - ra["output"][:, s].float()).abs().max().item()
        assert err <= 2e-2 * ra["output"].float().abs().max().item()
    for i in range(sh.B):
        n = int(ra["resident_len"][i])
        assert np.array_equal(ra["present_key"][i, :, :n], rb["present_key"][i, :, :n])
        assert np.array_equal(ra["present_value"][i, :, :n], rb["present_value"][i, :, :n])


# ------------------------------------------------------------------ tensor-core path shapes


@pytest.mark.parametrize("heads", [(1, 1), (2, 1), (8, 1), (16, 2), (32, 1), (32, 8)])
@pytest.mark.parametrize("S", [2, 3, 9, 33, 130])
def test_tensor_core_path_shapes(heads, S):
    """Multi-token bf16 steps with head size 128 run on the tcgen05 kernel for every
    query-head group that tiles a 32-row lane quarter (1, 2, 4, 8, 16, 32); token counts
    leave lane quarters partly filled and cross 128-row query tiles; W=100 puts window
    edges inside key tiles; a ragged batch, one item starting from an empty cache."""
    Nq, Nkv = heads
    if Nq // Nkv >= 16 and S > 33:
        S = 33  # keep the oracle's work bounded
    B, C, W = 2, 110, 100
    sh = wl.Shape("tc", B=B, Nq=Nq, Nkv=Nkv, D=128, W=W, C=C, dtype=wl.BF16)
    pk, pv = wl.cache(sh, 15)
    p = _shape_pair(sh, past_key=pk, past_value=pv)
    T = np.array([0, 77], np.int64)
    for t in range(2):
        q, k, v = wl.step_inputs(sh, S, 1500 + 10 * S + t)
        p.step(q, k, v, T + S - 1)
        T = T + S


@pytest.mark.parametrize("split_keys", [128, 512])
@pytest.mark.parametrize("inplace", [True, False])
def test_tensor_core_path_splits_and_buffers(split_keys, inplace):
    """Forced key splits (merged by the last contributor) and a separate present
    buffer on the tensor-core kernel, with softcap and a bias."""
    sh = wl.Shape("tcs", B=3, Nq=16, Nkv=4, D=128, W=300, C=311, dtype=wl.BF16, softcap=20.0)
    pk, pv = wl.cache(sh, 16)
    p = _shape_pair(sh, past_key=pk, past_value=pv, inplace=inplace, split_keys=split_keys)
    T = np.array([5, 290, 600], np.int64)
    for t, S in enumerate([12, 12, 40]):
        q, k, v = wl.step_inputs(sh, S, 1600 + t)
        total = int(T.max()) + S
        bias = wl.bias(sh.B, sh.Nq, S, total, 1600 + t, std=1.0)
        p.step(q, k, v, T + S - 1, total=total, bias=bias)
        T = T + S


@pytest.mark.parametrize("split_keys", [0, 256])
@pytest.mark.parametrize("inplace", [True, False])
def test_tensor_core_path_more_units_than_sms(split_keys, inplace):
    """The multi-token kernel is persistent (one CTA per SM walking its units): with 4
    items x 8 kv heads x 5 query tiles (S = 130, group 4) there are 160 units -- more with
    key splits -- so CTAs run several units back to back, their key-tile rings and
    barrier phases running on across units.  A ragged batch (one item from an empty
    cache, one crossing a block eviction) and a second step on the advanced cache."""
    sh = wl.Shape("tcu", B=4, Nq=32, Nkv=8, D=128, W=100, C=109, dtype=wl.BF16)
    pk, pv = wl.cache(sh, 17)
    p = _shape_pair(sh, past_key=pk, past_value=pv, inplace=inplace, split_keys=split_keys)
    T = np.array([0, 40, 95, 300], np.int64)
    for t in range(2):
        q, k, v = wl.step_inputs(sh, 130, 1700 + t)
        p.step(q, k, v, T + 130 - 1)
        T = T + 130
