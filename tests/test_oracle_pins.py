"""Pins of the oracle to facts the pages and mathematics fix (no GPU).

Each test names the passage it checks.  The pins are chosen so that a plausible
mistake in the oracle (an off-by-one window, a wrong causal offset, a transposed
head map, a wrong row origin, a bias column taken relative to the cache) fails at
least one of them.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle_driver import OracleCache

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    return np.array(rows)


def _drift_sim(T, C, W):
    """The drifting layout as a mechanism (PR #31142, Key design decisions, "Drifting
    layout"): tokens append at the end; when the buffer is full and one more token
    arrives, a whole block of G = C - W + 1 oldest rows is reclaimed at once."""
    G = C - W + 1
    end = 0
    for _ in range(T):
        if end == C:
            end -= G
        end += 1
    return end


def _rng(seed):
    return np.random.Generator(np.random.Philox(seed))


def _u(rng, shape):
    return rng.uniform(-1.0, 1.0, size=shape).astype(np.float32)


# ---------------------------------------------------------------- L(T) and layout


def test_resident_len_golden_c6_w4():
    """PR #32419, Description: L(T) for C=6, W=4 across eviction boundaries."""
    for T, L in _golden("resident_len_c6_w4.txt"):
        assert oracle.resident_len(int(T), 6, 4) == int(L)


@pytest.mark.parametrize("C,W", [(1, 1), (2, 1), (2, 2), (5, 3), (6, 4), (8, 8), (9, 2), (136, 128)])
def test_resident_len_matches_drifting_mechanism(C, W):
    """PR #31142, "Drifting layout": the closed form equals the block-reclaim mechanism."""
    for T in range(0, 4 * C + 20):
        assert oracle.resident_len(T, C, W) == _drift_sim(T, C, W), (T, C, W)


def test_resident_len_bounds_and_congruence():
    """PR #32419: min(T, W) <= L(T) <= min(T, C).  Beyond C the value lies in [W, C],
    an interval of exactly G integers, and stays congruent to T modulo G (only whole
    G-row blocks are reclaimed), which fixes it uniquely, also near INT32_MAX."""
    for C in range(1, 13):
        for W in range(1, C + 1):
            G = C - W + 1
            for T in list(range(0, 5 * C)) + [2**31 - 1, 2**31, 2**40 + 7]:
                L = oracle.resident_len(T, C, W)
                assert min(T, W) <= L <= min(T, C)
                if T > C:
                    assert (L - T) % G == 0


def test_small_slack_compaction_count():
    """PR #31142, Tests: C = W + 8 with 400 decode steps gives "~44" compaction events
    (here after a 128-token prefill: T = 129 .. 528)."""
    W, C = 128, 136
    events = sum(
        1 for T in range(129, 529) if oracle.resident_len(T, C, W) != oracle.resident_len(T - 1, C, W) + 1
    )
    assert events == 44


def _positions_run(C, W, schedule, D=8):
    """Drive the oracle with keys/values that encode their absolute position and
    return, after each step, (T, present_key rows, present_value rows)."""
    oc = OracleCache(1, 2, 1, D, C, W)
    T = 0
    out = []
    for S in schedule:
        pos = np.arange(T, T + S, dtype=np.float32)
        k = np.repeat(pos[:, None], D, axis=1)[None]  # key of position t: all t
        v = -k - 0.5
        q = np.zeros((1, S, 2 * D), np.float32)
        T += S
        r = oc.step(q, k, v, [T - 1])
        out.append((T, r["present_key"][0, 0, :, 0].copy(), r["present_value"][0, 0, :, 0].copy(),
                    int(r["resident_len"][0])))
    return out


def test_layout_rows_hold_recent_positions():
    """PR #32419, Description: after a step row i holds absolute position T - L + i;
    with C=6, W=4 the run crosses several eviction boundaries, including an 8-token
    prefill (S > C, staged) and a 4-token step.  Keys and values both carry the
    position (the review of that PR asked for present_key to be checked as well)."""
    schedule = [8, 4] + [1] * 12
    seen_not_min = False
    for T, krow, vrow, L in _positions_run(6, 4, schedule):
        assert L == _drift_sim(T, 6, 4)
        if L != min(T, 6):
            seen_not_min = True
        for i in range(L):
            assert krow[i] == T - L + i
            assert vrow[i] == -(T - L + i) - 0.5
    assert seen_not_min  # the test would fail for a cache keeping min(T, C) rows


# ---------------------------------------------------------------- chunk invariance


def test_multi_token_step_equals_single_token_steps():
    """PR #32419, New tests: a 4-token step after an 8-token prefill leaves the same
    present buffers and outputs as four 1-token steps (fp64 oracle: bit-identical)."""
    rng = _rng(1)
    D, Nq, Nkv, C, W = 8, 2, 1, 6, 4
    qp, kp, vp = _u(rng, (1, 8, Nq * D)), _u(rng, (1, 8, Nkv * D)), _u(rng, (1, 8, Nkv * D))
    q4, k4, v4 = _u(rng, (1, 4, Nq * D)), _u(rng, (1, 4, Nkv * D)), _u(rng, (1, 4, Nkv * D))
    a = OracleCache(1, Nq, Nkv, D, C, W)
    b = OracleCache(1, Nq, Nkv, D, C, W)
    a.step(qp, kp, vp, [7])
    b.step(qp, kp, vp, [7])
    ra = a.step(q4, k4, v4, [11])
    for s in range(4):
        rb = b.step(q4[:, s:s + 1], k4[:, s:s + 1], v4[:, s:s + 1], [8 + s])
        assert np.array_equal(ra["output_f64"][:, s], rb["output_f64"][:, 0])
        assert np.array_equal(ra["output"][:, s], rb["output"][:, 0])
    L = int(ra["resident_len"][0])
    assert L == int(rb["resident_len"][0])
    assert np.array_equal(a.pk[:, :, :L], b.pk[:, :, :L])
    assert np.array_equal(a.pv[:, :, :L], b.pv[:, :, :L])


def test_chunk_split_invariance_random_schedules():
    """Same contract, more splits: any split of a token stream into steps gives
    bit-identical outputs and resident rows (layout depends on T only)."""
    rng = _rng(2)
    D, Nq, Nkv = 8, 4, 2
    for C, W in [(6, 4), (5, 5), (9, 3), (12, 4)]:
        total = 40
        q, k, v = _u(rng, (1, total, Nq * D)), _u(rng, (1, total, Nkv * D)), _u(rng, (1, total, Nkv * D))
        outs = []
        for trial in range(3):
            oc = OracleCache(1, Nq, Nkv, D, C, W)
            T, o = 0, []
            while T < total:
                S = int(min(total - T, rng.integers(1, 2 * C + 2)))
                r = oc.step(q[:, T:T + S], k[:, T:T + S], v[:, T:T + S], [T + S - 1])
                o.append(r["output_f64"])
                T += S
            L = int(r["resident_len"][0])
            outs.append((np.concatenate(o, axis=1), oc.pk[:, :, :L].copy(), oc.pv[:, :, :L].copy()))
        for o in outs[1:]:
            assert np.array_equal(o[0], outs[0][0])
            assert np.array_equal(o[1], outs[0][1])
            assert np.array_equal(o[2], outs[0][2])


# ---------------------------------------------------------------- rollback


def test_rollback_exact_iff_formula():
    """PR #32419, Description and New tests: rejecting k of the S tokens of a step
    needs no cache edit and is exact iff L(T - k) == L(T) - k.  Brute force over small
    capacities: the untouched buffer after the S-token step, read as a cache of
    length T - k, equals the buffer built from the accepted tokens only, exactly when
    the formula says so (values encode positions, so equal rows mean equal positions)."""
    cases = exact = 0
    for C in range(1, 8):
        for W in range(1, C + 1):
            for P in range(0, 2 * C + 3):
                for S in range(1, 6):
                    T = P + S
                    for kk in range(0, S + 1):
                        if T - kk < 1:
                            continue
                        full = _positions_run(C, W, ([P] if P else []) + [S])[-1]
                        acc = _positions_run(C, W, ([P] if P else []) + ([S - kk] if S - kk else []))[-1]
                        La = oracle.resident_len(T - kk, C, W)
                        same = bool(np.array_equal(full[1][:La], acc[1][:La]))
                        predicted = oracle.resident_len(T - kk, C, W) == oracle.resident_len(T, C, W) - kk
                        assert same == predicted, (C, W, P, S, kk)
                        cases += 1
                        exact += predicted
    assert cases > 1000 and 0 < exact < cases


def test_rollback_tiny_contract_points():
    """C=6, W=4: the verify step 24 -> 28 accepting 2 (k = 2) is inexact
    (L(26) = 5, L(28) - 2 = 2); 20 -> 24 accepting 2 is exact (L(22) = 4 = 6 - 2)."""
    assert oracle.resident_len(26, 6, 4) != oracle.resident_len(28, 6, 4) - 2
    assert oracle.resident_len(22, 6, 4) == oracle.resident_len(24, 6, 4) - 2


# ---------------------------------------------------------------- masks


def test_causal_worked_example_onehot():
    """PR #34226, Description (repro): Q = K = 0, one-hot values, 2 past keys, 2 new
    keys.  The query at position 2 gives [1/3, 1/3, 1/3, 0]."""
    gold = _golden("causal_onehot_past2.txt")
    D, C, W = 4, 8, 8
    one_hot = np.eye(4, D, dtype=np.float32)
    oc = OracleCache(1, 1, 1, D, C, W)
    oc.pv[0, 0, :2] = one_hot[:2]  # past keys 0, 1 (keys stay zero)
    q = np.zeros((1, 2, D), np.float32)
    k = np.zeros((1, 2, D), np.float32)
    v = one_hot[2:4][None]
    r = oc.step(q, k, v, [3])  # T = 4, S = 2, past P = 2
    for s, row in enumerate(gold):
        assert row[0] == 2 + s
        np.testing.assert_allclose(r["output_f64"][0, s], row[1:], rtol=0, atol=1e-15)
    assert abs(r["output"][0, 0, 3]) == 0.0


@pytest.mark.parametrize("C,W", [(4, 4), (5, 4), (7, 4), (8, 4), (16, 4), (3, 1), (9, 9)])
@pytest.mark.parametrize("S", [1, 3, 5])
def test_window_closed_form_uniform_weights(C, W, S):
    """Local window + causal rule: with Q = 0 every visible key has equal weight, so
    the output is the mean of the visible positions, (max(0, i - W + 1) + i) / 2 when
    the value of position t is t."""
    D = 8
    oc = OracleCache(1, 2, 1, D, C, W)
    T = 0
    for _ in range(6):
        pos = np.arange(T, T + S, dtype=np.float32)
        v = np.repeat(pos[:, None], D, axis=1)[None]
        k = _u(_rng(T), (1, S, D))
        q = np.zeros((1, S, 2 * D), np.float32)
        r = oc.step(q, k, v, [T + S - 1])
        for s in range(S):
            i = T + s
            expect = (max(0, i - W + 1) + i) / 2.0
            np.testing.assert_allclose(r["output_f64"][0, s], expect, rtol=0, atol=1e-12)
        T += S


def _sdpa_reference(q, k, v, Nq, Nkv, D, W, P, scale, bias=None):
    """torch.nn.functional.scaled_dot_product_attention in float64 over the full
    token history (no cache), with the absolute causal + window mask and an additive
    bias; kv heads repeated in contiguous groups."""
    S = q.shape[1]
    T = k.shape[1]
    qt = torch.from_numpy(q.astype(np.float64)).view(1, S, Nq, D).transpose(1, 2)
    kt = torch.from_numpy(k.astype(np.float64)).view(1, T, Nkv, D).transpose(1, 2)
    vt = torch.from_numpy(v.astype(np.float64)).view(1, T, Nkv, D).transpose(1, 2)
    kt = kt.repeat_interleave(Nq // Nkv, dim=1)
    vt = vt.repeat_interleave(Nq // Nkv, dim=1)
    i = torch.arange(S).view(S, 1) + P
    j = torch.arange(T).view(1, T)
    visible = (j <= i) & (j > i - W)
    mask = torch.zeros(S, T, dtype=torch.float64).masked_fill(~visible, float("-inf"))
    mask = mask.view(1, 1, S, T)
    if bias is not None:
        mask = mask + torch.from_numpy(bias.astype(np.float64))
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return out.transpose(1, 2).reshape(1, S, Nq * D).numpy()


@pytest.mark.parametrize("C,W,Nq,Nkv", [(6, 4, 2, 1), (5, 2, 4, 2), (12, 12, 4, 4), (7, 3, 6, 2)])
def test_full_cache_equivalence_and_sdpa(C, W, Nq, Nkv):
    """PR #31142 (results identical to a full-length cache) and the causal rule of
    PR #34226: a windowed cache of capacity C gives bit-identical fp64 outputs to a
    cache that never evicts, and both equal torch's float64 scaled-dot-product
    attention over the full history with the absolute causal + window mask and an
    additive bias (PR #32419: bias columns are absolute key positions)."""
    rng = _rng(10 + C)
    D, total = 8, 30
    q = _u(rng, (1, total, Nq * D))
    k = _u(rng, (1, total, Nkv * D))
    v = _u(rng, (1, total, Nkv * D))
    bias_full = rng.normal(0, 0.5, size=(1, Nq, total, total)).astype(np.float32)
    win = OracleCache(1, Nq, Nkv, D, C, W)
    full = OracleCache(1, Nq, Nkv, D, 64, W)
    T = 0
    for S in [3, 1, 1, 5, 2, 1, 8, 1, 4, 4]:
        bias = np.ascontiguousarray(bias_full[:, :, T:T + S, :T + S])
        rw = win.step(q[:, T:T + S], k[:, T:T + S], v[:, T:T + S], [T + S - 1], bias=bias)
        rf = full.step(q[:, T:T + S], k[:, T:T + S], v[:, T:T + S], [T + S - 1], bias=bias)
        assert np.array_equal(rw["output_f64"], rf["output_f64"])
        ref = _sdpa_reference(q[:, T:T + S], k[:, :T + S], v[:, :T + S], Nq, Nkv, D, W, T,
                              1.0 / math.sqrt(D), bias)
        np.testing.assert_allclose(rw["output_f64"], ref, rtol=0, atol=1e-12)
        T += S


def test_head_grouping_contiguous():
    """Query head h reads kv head h // (Nq / Nkv) (the usual contiguous grouping; the
    pages only say Nq query heads share Nkv kv heads)."""
    D, Nq, Nkv, C, W = 8, 6, 3, 8, 8
    oc = OracleCache(1, Nq, Nkv, D, C, W)
    S = 3
    q = _u(_rng(5), (1, S, Nq * D))
    k = _u(_rng(6), (1, S, Nkv * D))
    v = np.zeros((1, S, Nkv * D), np.float32)
    for kvh in range(Nkv):
        v[:, :, kvh * D:(kvh + 1) * D] = kvh + 1.0
    r = oc.step(q, k, v, [S - 1])
    for h in range(Nq):
        np.testing.assert_allclose(r["output_f64"][0, :, h * D:(h + 1) * D], h // (Nq // Nkv) + 1.0,
                                   rtol=0, atol=1e-14)


def test_bias_absolute_column_ragged_batch():
    """PR #32419, Description: the bias last dimension is total_sequence_length in
    absolute key coordinates.  A +60 bias at absolute column j* makes the output the
    value of position j* (to e^-60); items of a ragged batch each use their own
    absolute column, not one relative to the cache or to the batch maximum."""
    D, C, W = 8, 6, 4
    B = 3
    Ts = [9, 13, 6]  # lengths after the step; total_sequence_length = 13
    total = max(Ts)
    oc = OracleCache(B, 1, 1, D, C, W)
    # Prefill each item to T_b - 1 with position-encoded values, then one decode step.
    for b in range(B):
        one = OracleCache(1, 1, 1, D, C, W)
        P = Ts[b] - 1
        pos = np.arange(P, dtype=np.float32)
        kv = np.repeat(pos[:, None], D, axis=1)[None]
        one.step(np.zeros((1, P, D), np.float32), kv, kv, [P - 1])
        oc.pk[b], oc.pv[b] = one.pk[0], one.pv[0]
    bias = np.zeros((B, 1, 1, total), np.float32)
    targets = [Ts[b] - 3 for b in range(B)]  # visible: within the last W positions
    for b in range(B):
        bias[b, 0, 0, targets[b]] = 60.0
        bias[b, 0, 0, Ts[b]:] = 1e4  # columns beyond T_b are never read
    newpos = np.array([T - 1 for T in Ts], np.float32)
    kv = np.repeat(newpos[:, None], D, axis=1)[:, None, :]
    q = np.zeros((B, 1, D), np.float32)
    r = oc.step(q, kv, kv, [T - 1 for T in Ts], total=total, bias=bias)
    for b in range(B):
        np.testing.assert_allclose(r["output_f64"][b, 0], targets[b], rtol=0, atol=1e-20 + 4 * Ts[b] * math.exp(-60))


def test_softcap_limits():
    """Softcap (mobius issue #111, Part 1.3: "Logit soft-capping (0 = disabled)"):
    a cap of 1e30 is no cap; a cap c bounds every logit to (-c, c), so two visible keys
    never differ in weight by more than e^(2c), however large q.k is."""
    rng = _rng(7)
    D, Nq, Nkv, C, W, S = 8, 2, 1, 8, 8, 8
    q = _u(rng, (1, S, Nq * D)) * 30
    k = _u(rng, (1, S, Nkv * D)) * 30
    v = np.zeros((1, S, Nkv * D), np.float32)
    v[0, :, :] = np.eye(S, D, dtype=np.float32)  # one-hot value: output[d] = weight of key d
    r0 = OracleCache(1, Nq, Nkv, D, C, W, softcap=0.0).step(q, k, v, [S - 1])
    rinf = OracleCache(1, Nq, Nkv, D, C, W, softcap=1e30).step(q, k, v, [S - 1])
    np.testing.assert_allclose(rinf["output_f64"], r0["output_f64"], rtol=0, atol=1e-12)
    c = 0.75
    rc = OracleCache(1, Nq, Nkv, D, C, W, softcap=c).step(q, k, v, [S - 1])
    raw_ratio = 0.0
    for s in range(S):
        for h in range(Nq):
            w = rc["output_f64"][0, s, h * D:h * D + s + 1]
            w0 = r0["output_f64"][0, s, h * D:h * D + s + 1]
            assert w.max() / w.min() <= math.exp(2 * c) * (1 + 1e-12)
            if w0.min() > 0:
                raw_ratio = max(raw_ratio, w0.max() / w0.min())
    assert raw_ratio > math.exp(2 * c) * 10  # the cap did bind


def test_default_scale():
    """The scale attribute defaults to 1/sqrt(head_size) (mobius issue #111, Part 1.3)."""
    rng = _rng(8)
    D, Nq, Nkv, C, W, S = 16, 2, 1, 8, 4, 5
    q, k, v = _u(rng, (1, S, Nq * D)), _u(rng, (1, S, Nkv * D)), _u(rng, (1, S, Nkv * D))
    a = OracleCache(1, Nq, Nkv, D, C, W, scale=0.0).step(q, k, v, [S - 1])
    b = OracleCache(1, Nq, Nkv, D, C, W, scale=0.25).step(q, k, v, [S - 1])
    c = OracleCache(1, Nq, Nkv, D, C, W, scale=0.5).step(q, k, v, [S - 1])
    assert np.array_equal(a["output_f64"], b["output_f64"])
    assert not np.array_equal(a["output_f64"], c["output_f64"])


def test_items_are_independent():
    """Review of PR #32419: T is taken per batch item.  A ragged batch equals its items
    run one by one."""
    rng = _rng(9)
    D, Nq, Nkv, C, W, S, B = 8, 4, 2, 7, 5, 3, 3
    pk, pv = _u(rng, (B, Nkv, C, D)), _u(rng, (B, Nkv, C, D))
    q, k, v = _u(rng, (B, S, Nq * D)), _u(rng, (B, S, Nkv * D)), _u(rng, (B, S, Nkv * D))
    seq = [5, 17, 2]
    rb = OracleCache(B, Nq, Nkv, D, C, W, past_key=pk, past_value=pv).step(q, k, v, seq, total=18)
    for b in range(B):
        r1 = OracleCache(1, Nq, Nkv, D, C, W, past_key=pk[b:b + 1], past_value=pv[b:b + 1]).step(
            q[b:b + 1], k[b:b + 1], v[b:b + 1], seq[b:b + 1], total=18)
        assert np.array_equal(rb["output_f64"][b], r1["output_f64"][0])
        L = int(r1["resident_len"][0])
        assert np.array_equal(rb["present_key"][b, :, :L], r1["present_key"][0, :, :L])


def test_large_positions_int64():
    """PR #31142 review: the planner works in 64-bit; positions near INT32_MAX keep the
    layout (values carry position mod 1024, exact in fp32)."""
    D, C, W = 8, 6, 4
    T = 2**31 - 1
    P = T - 1
    Lp = oracle.resident_len(P, C, W)
    pk = np.zeros((1, 1, C, D), np.float32)
    for r in range(Lp):
        pk[0, 0, r] = (P - Lp + r) % 1024
    oc = OracleCache(1, 1, 1, D, C, W, past_key=pk, past_value=pk)
    newk = np.full((1, 1, D), (T - 1) % 1024, np.float32)
    r = oc.step(np.zeros((1, 1, D), np.float32), newk, newk, [T - 1], total=T)
    L = int(r["resident_len"][0])
    assert L == oracle.resident_len(T, C, W)
    for i in range(L):
        assert r["present_key"][0, 0, i, 0] == (T - L + i) % 1024


def test_errors():
    """A past length below zero ([P2] planner, P = seqlens_k + 1 - S) and T_b above
    total_sequence_length are rejected."""
    z = np.zeros((1, 3, 8), np.float32)
    pk = np.zeros((1, 1, 6, 8), np.float32)
    with pytest.raises(ValueError):
        oracle.step(z, z, z, pk, pk, np.array([1], np.int32), 3, 1, 1, 4)  # T=2 < S=3
    with pytest.raises(ValueError):
        oracle.step(z, z, z, pk, pk, np.array([9], np.int32), 5, 1, 1, 4)  # T=10 > total


def test_round_bf16_matches_torch_on_float_inputs():
    """The oracle's one-step fp64 -> bfloat16 rounding equals torch's float32 ->
    bfloat16 rounding (nearest, ties to even) whenever the input is a float32."""
    rng = _rng(11)
    xs = np.concatenate([
        rng.normal(0, 1, 2000), rng.normal(0, 1e-30, 200), rng.normal(0, 1e30, 200),
        [0.0, -0.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -(1.0 + 2**-8), 3.3895313892515355e38, 3.4e38,
         2**-133, 2**-134, 3 * 2**-135],
    ]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.round_bf16(float(x)) for x in xs], np.uint16)
    assert np.array_equal(got, ref)
    assert oracle.round_bf16(1.0 + 2**-8) == 0x3F80  # tie -> even (1.0)
    assert oracle.round_bf16(1.0 + 2**-8 + 2**-30) == 0x3F81  # above the tie: one fp64 rounding


# ---------------------------------------------------------------- sinks


def test_sink_closed_forms():
    """head_sink / smooth_softmax (mobius issue #111, Part 1.1 input 11 and Part 1.3,
    named only; reading: one more logit per head in the softmax denominator, with no
    value row).  With Q = 0 every visible logit is 0, so each of the n visible keys gets
    weight 1 / (e^sink + n) and the output is the mean of the visible values times
    n / (e^sink + n); smooth_softmax is a sink of 0; a sink of -inf is no sink."""
    D, Nq, Nkv, C, W = 8, 3, 1, 9, 5
    sinks = np.array([0.7, -2.0, 3.0], np.float32)
    for smooth in (False, True):
        oc_ref = OracleCache(1, Nq, Nkv, D, C, W)
        T = 0
        for step, S in enumerate([4, 1, 3, 1]):
            pos = np.arange(T, T + S, dtype=np.float32)
            v = np.repeat(pos[:, None], D, axis=1)[None] + 1.0
            k = _u(_rng(40 + step), (1, S, D))
            q = np.zeros((1, S, Nq * D), np.float32)
            r = oracle.step(q, k, v, oc_ref.pk, oc_ref.pv, np.array([T + S - 1], np.int32), T + S, Nq, Nkv, W,
                            head_sink=None if smooth else sinks, smooth_softmax=smooth)
            oc_ref.step(q, k, v, [T + S - 1])
            for s in range(S):
                i = T + s
                lo = max(0, i - W + 1)
                n = i - lo + 1
                mean = (lo + i) / 2.0 + 1.0
                for h in range(Nq):
                    e_s = 1.0 if smooth else math.exp(float(sinks[h]))
                    np.testing.assert_allclose(r["output_f64"][0, s, h * D:(h + 1) * D], mean * n / (e_s + n),
                                               rtol=1e-13, atol=0)
            T += S
    rng = _rng(41)
    q, k, v = _u(rng, (1, 4, Nq * D)), _u(rng, (1, 4, D)), _u(rng, (1, 4, D))
    pk = np.zeros((1, 1, C, D), np.float32)
    plain = oracle.step(q, k, v, pk, pk, np.array([3], np.int32), 4, Nq, Nkv, W)
    none = oracle.step(q, k, v, pk, pk, np.array([3], np.int32), 4, Nq, Nkv, W,
                       head_sink=np.full(Nq, -np.inf, np.float32))
    zero = oracle.step(q, k, v, pk, pk, np.array([3], np.int32), 4, Nq, Nkv, W, head_sink=np.zeros(Nq, np.float32))
    smooth = oracle.step(q, k, v, pk, pk, np.array([3], np.int32), 4, Nq, Nkv, W, smooth_softmax=True)
    assert np.array_equal(plain["output_f64"], none["output_f64"])
    assert np.array_equal(zero["output_f64"], smooth["output_f64"])
    assert not np.array_equal(plain["output_f64"], smooth["output_f64"])


# ---------------------------------------------------------------- rotary embedding
# mobius issue #111, Part 1.1 (cos_cache, sin_cache, position_ids) and Part 1.3
# (do_rotary, rotary_interleaved) name the fused rotary embedding; the reading is the
# RoFormer rotation of dimension pairs by the angle of the token's position.  The pins
# below use the complex-number form of that rotation (pair (x1, x2) as x1 + i x2,
# multiplied by e^(i theta)), a worked quarter turn, and the relative-position property.


def _rope_tables(npos, half, base=10000.0, dtype=np.float32):
    """cos/sin caches of the usual RoPE angles pos * base^(-i/half)."""
    ang = np.arange(npos)[:, None] * base ** (-np.arange(half)[None, :] / half)
    return np.cos(ang).astype(dtype), np.sin(ang).astype(dtype)


def _pairs(D, rd, interleaved):
    half = rd // 2
    return [(2 * i, 2 * i + 1) if interleaved else (i, i + half) for i in range(half)]


def _turn_complex(x, pos, cos, sin, rd, interleaved):
    """x (D,) turned by the angles of row pos, in complex arithmetic."""
    y = x.astype(np.float64).copy()
    for i, (a, b) in enumerate(_pairs(len(x), rd, interleaved)):
        z = complex(x[a], x[b]) * complex(float(cos[pos, i]), float(sin[pos, i]))
        y[a], y[b] = z.real, z.imag
    return y


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotary_quarter_turn(interleaved):
    """A quarter turn (cos 0, sin 1) of the first pair sends its first unit vector to
    its second and the second to minus the first; other pairs (cos 1, sin 0) stay."""
    D, C, W = 8, 8, 8
    half = D // 2
    cos = np.ones((4, half), np.float32)
    sin = np.zeros((4, half), np.float32)
    cos[2, 0], sin[2, 0] = 0.0, 1.0  # position 2: quarter turn of pair 0
    a, b = _pairs(D, D, interleaved)[0]
    k = np.zeros((1, 3, D), np.float32)
    k[0, 2, a] = 1.0  # token at position 2: unit vector on the pair's first dimension
    k[0, 1, a] = 1.0  # position 1: identity
    r = oracle.step(np.zeros((1, 3, D), np.float32), k, k, np.zeros((1, 1, C, D), np.float32),
                    np.zeros((1, 1, C, D), np.float32), np.array([2], np.int32), 3, 1, 1, W,
                    cos_cache=cos, sin_cache=sin, rotary_interleaved=interleaved)
    pk = r["present_key"][0, 0]
    assert pk[2, b] == 1.0 and pk[2, a] == 0.0 and np.count_nonzero(pk[2]) == 1
    assert pk[1, a] == 1.0 and np.count_nonzero(pk[1]) == 1
    k[0, 2, a], k[0, 2, b] = 0.0, 1.0
    r = oracle.step(np.zeros((1, 3, D), np.float32), k, k, np.zeros((1, 1, C, D), np.float32),
                    np.zeros((1, 1, C, D), np.float32), np.array([2], np.int32), 3, 1, 1, W,
                    cos_cache=cos, sin_cache=sin, rotary_interleaved=interleaved)
    pk = r["present_key"][0, 0]
    assert pk[2, a] == -1.0 and np.count_nonzero(pk[2]) == 1
    # values are not turned
    assert np.array_equal(r["present_value"][0, 0, :3], k[0])


@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("rd", [8, 4])
def test_rotary_cache_rows_are_turned_keys(interleaved, rd):
    """Across compactions and a ragged batch, resident row r holds the key of absolute
    position p = T - L + r turned by the angles of p (complex form); dimensions from
    rd on are the input's bits."""
    D, Nq, Nkv, C, W = 8, 2, 1, 7, 4
    cos, sin = _rope_tables(64, rd // 2)
    rng = _rng(50)
    total = 40
    keys = _u(rng, (2, total, Nkv * D))
    oc = OracleCache(2, Nq, Nkv, D, C, W, cos_cache=cos, sin_cache=sin, rotary_interleaved=interleaved)
    T0 = np.array([0, 5])  # item 1 starts from a zero past of 5 tokens: only rows written here are checked
    T = T0.copy()
    for S in [6, 1, 3, 1, 1, 4, 2]:
        q = _u(rng, (2, S, Nq * D))
        k = np.stack([keys[b, T[b]:T[b] + S] for b in range(2)])
        r = oc.step(q, k, k, T + S - 1)
        T = T + S
        for b in range(2):
            L = int(r["resident_len"][b])
            for row in range(L):
                pos = T[b] - L + row
                if pos < T0[b]:
                    continue
                want = _turn_complex(keys[b, pos], pos, cos, sin, rd, interleaved)
                got = r["present_key"][b, 0, row]
                np.testing.assert_allclose(got[:rd], want[:rd], rtol=0, atol=2e-7)
                assert np.array_equal(got[rd:], keys[b, pos, rd:])


def test_rotary_position_ids_override():
    """position_ids replace the absolute positions: turning by ids equal to P + s gives
    the default's bits, and a shifted id turns the key by the shifted angle."""
    D, C, W = 8, 8, 8
    cos, sin = _rope_tables(32, D // 2)
    rng = _rng(51)
    q, k = _u(rng, (1, 3, D)), _u(rng, (1, 3, D))
    z = np.zeros((1, 1, C, D), np.float32)
    base = oracle.step(q, k, k, z, z, np.array([4], np.int32), 5, 1, 1, W, cos_cache=cos, sin_cache=sin)
    same = oracle.step(q, k, k, z, z, np.array([4], np.int32), 5, 1, 1, W, cos_cache=cos, sin_cache=sin,
                       position_ids=np.array([[2, 3, 4]]))
    assert np.array_equal(base["output_f64"], same["output_f64"])
    assert np.array_equal(base["present_key"], same["present_key"])
    moved = oracle.step(q, k, k, z, z, np.array([4], np.int32), 5, 1, 1, W, cos_cache=cos, sin_cache=sin,
                        position_ids=np.array([[2, 3, 20]]))
    np.testing.assert_allclose(moved["present_key"][0, 0, 4], _turn_complex(k[0, 2], 20, cos, sin, D, False),
                               rtol=0, atol=2e-7)
    with pytest.raises(ValueError):
        oracle.step(q, k, k, z, z, np.array([4], np.int32), 5, 1, 1, W, cos_cache=cos, sin_cache=sin,
                    position_ids=np.array([[2, 3, 32]]))


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotary_relative_position_invariance(interleaved):
    """RoFormer's property: turned q.k depends on the positions' difference only, so
    one prefill step from an empty cache gives the same outputs (to fp64 rounding) at
    positions 0..S-1 and at 1000..1000+S-1.  Fails if the query and keys are turned
    with different positions or conventions."""
    D, Nq, Nkv, S = 16, 4, 2, 9
    cos, sin = _rope_tables(1100, D // 2, dtype=np.float64)
    rng = _rng(52)
    q, k, v = _u(rng, (1, S, Nq * D)), _u(rng, (1, S, Nkv * D)), _u(rng, (1, S, Nkv * D))
    z = np.zeros((1, Nkv, S, D), np.float32)
    outs = []
    for shift in (0, 1000):
        r = oracle.step(q, k, v, z, z, np.array([S - 1], np.int32), S, Nq, Nkv, 6, cos_cache=cos.astype(np.float32),
                        sin_cache=sin.astype(np.float32), position_ids=np.arange(S)[None] + shift,
                        rotary_interleaved=interleaved)
        outs.append(r["output_f64"])
    # the stored keys are rounded to fp32, and the fp32 tables are not exact rotations:
    # agreement to about 1e-6 is all the property promises here
    np.testing.assert_allclose(outs[0], outs[1], rtol=0, atol=5e-6)
    plain = oracle.step(q, k, v, z, z, np.array([S - 1], np.int32), S, Nq, Nkv, 6)["output_f64"]
    assert np.abs(plain - outs[0]).max() > 1e-3  # the rotation does change the outputs


def test_rotary_matches_sdpa_full_history():
    """Multi-step windowed run with rotary embedding == torch float64
    scaled-dot-product attention over the full history of turned queries and keys
    (turned here with torch complex multiplication, non-interleaved pairs)."""
    D, Nq, Nkv, C, W = 8, 4, 2, 7, 5
    cos, sin = _rope_tables(64, D // 2)
    rng = _rng(53)
    total = 30
    q, k, v = _u(rng, (1, total, Nq * D)), _u(rng, (1, total, Nkv * D)), _u(rng, (1, total, Nkv * D))

    def turn(x, heads):
        t = torch.from_numpy(x.astype(np.float64)).view(total, heads, 2, D // 2)
        zc = torch.complex(t[:, :, 0], t[:, :, 1])
        e = torch.complex(torch.from_numpy(cos[:total].astype(np.float64)),
                          torch.from_numpy(sin[:total].astype(np.float64)))[:, None, :]
        y = zc * e
        return torch.stack([y.real, y.imag], dim=2).reshape(1, total, heads * D)

    qt = turn(q[0], Nq).numpy()
    # keys are stored rounded to the cache dtype (fp32) before attention reads them
    kt = turn(k[0], Nkv).numpy().astype(np.float32).astype(np.float64)
    oc = OracleCache(1, Nq, Nkv, D, C, W, cos_cache=cos, sin_cache=sin)
    T = 0
    for S in [3, 1, 4, 1, 6, 1, 2, 5, 1]:
        r = oc.step(q[:, T:T + S], k[:, T:T + S], v[:, T:T + S], [T + S - 1])
        ref = _sdpa_reference(qt[:, T:T + S], kt[:, :T + S], v[:, :T + S], Nq, Nkv, D, W, T, 1.0 / math.sqrt(D),
                              None)
        np.testing.assert_allclose(r["output_f64"], ref, rtol=0, atol=1e-12)
        T += S


def test_rotary_chunk_invariance():
    """With rotary embedding, a 5-token step equals five 1-token steps bit for bit:
    every token is turned by its own absolute position however the stream is split."""
    D, Nq, Nkv, C, W = 8, 2, 1, 6, 4
    cos, sin = _rope_tables(40, D // 2)
    rng = _rng(54)
    qp, kp, vp = _u(rng, (1, 7, Nq * D)), _u(rng, (1, 7, D)), _u(rng, (1, 7, D))
    q5, k5, v5 = _u(rng, (1, 5, Nq * D)), _u(rng, (1, 5, D)), _u(rng, (1, 5, D))
    a = OracleCache(1, Nq, Nkv, D, C, W, cos_cache=cos, sin_cache=sin, rotary_interleaved=True)
    b = OracleCache(1, Nq, Nkv, D, C, W, cos_cache=cos, sin_cache=sin, rotary_interleaved=True)
    a.step(qp, kp, vp, [6])
    b.step(qp, kp, vp, [6])
    ra = a.step(q5, k5, v5, [11])
    for s in range(5):
        rb = b.step(q5[:, s:s + 1], k5[:, s:s + 1], v5[:, s:s + 1], [7 + s])
        assert np.array_equal(ra["output_f64"][:, s], rb["output_f64"][:, 0])
    L = int(ra["resident_len"][0])
    assert np.array_equal(a.pk[:, :, :L], b.pk[:, :, :L])


# ---------------------------------------------------------------- quantized cache
# mobius issue #111, Part 1.1 names k_scale / v_scale ("KV cache quantization scale");
# the reading: int8 or fp8 e4m3 codes, one scale per tensor, code * scale, codes taken
# as x / scale in float rounded to nearest even and saturated.


def test_e4m3_rounding_matches_torch():
    """The oracle's float -> e4m3 rounding equals torch's float8_e4m3fn cast (an
    independent implementation) on random values across the range, ties, subnormals,
    zeros and the largest finite values (torch's cast is not used past 448, where the
    reading saturates)."""
    rng = _rng(60)
    xs = np.concatenate([
        rng.uniform(-448, 448, 4000), rng.normal(0, 1, 4000), rng.normal(0, 0.01, 2000),
        np.ldexp(np.arange(-40, 40, dtype=np.float64) * 0.25 + 0.125, -9),   # ties among subnormals
        np.array([0.0, -0.0, 448.0, -448.0, 1.0625, 1.1875, 240.0, 248.0, 2.0 ** -6, 2.0 ** -9, 2.0 ** -10]),
    ]).astype(np.float32)
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.round_e4m3(float(x)) for x in xs], np.uint8)
    assert np.array_equal(got, want)


def test_e4m3_decode_all_codes():
    """Every e4m3 code decodes to torch's value for it, and every non-NaN code rounds back
    to itself."""
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.decode_e4m3(c)
        if np.isnan(want[c]):
            assert np.isnan(v)
            continue
        assert v == want[c] and math.copysign(1.0, v) == math.copysign(1.0, want[c])
        assert oracle.round_e4m3(v) == c
    assert oracle.round_e4m3(1e6) == 0x7E and oracle.round_e4m3(-1e6) == 0xFE  # saturated
    assert oracle.round_e4m3(float("inf")) == 0x7E


def test_int8_quantizer_rounding_and_saturation():
    """Ties to even, saturation to [-128, 127], the division done in float."""
    q = lambda x, s=1.0: int(np.int8(np.uint8(oracle.quantize(x, s, oracle.I8))))
    assert [q(v) for v in (0.5, 1.5, 2.5, -0.5, -1.5, -2.5)] == [0, 2, 2, 0, -2, -2]
    assert q(126.5) == 126 and q(127.5) == 127 and q(1e9) == 127
    assert q(-127.5) == -128 and q(-128.5) == -128 and q(-1e9) == -128
    assert q(3.0, 2.0) == 2 and q(5.0, 2.0) == 2 and q(7.0, 2.0) == 4  # 1.5, 2.5, 3.5 -> ties to even
    # the quotient is a float: 2.4999998 / 1 stays below the tie, 0.1 / 0.04 = 2.5 in float
    assert q(np.float32(2.4999998)) == 2
    assert q(0.1, 0.04) == int(np.rint(np.float32(0.1) / np.float32(0.04)))


@pytest.mark.parametrize("cache_dtype", [oracle.I8, oracle.E4M3])
def test_quantized_cache_exact_values(cache_dtype):
    """Keys and values that the codes represent exactly (small integers times the scale,
    separate key and value scales): the quantized cache gives fp64-identical outputs to
    the plain fp32 cache across compactions, and its rows hold the codes of the inputs."""
    D, Nq, Nkv, C, W = 8, 4, 2, 7, 5
    ks, vs = 0.25, 0.0625
    rng = _rng(61)
    plain = OracleCache(1, Nq, Nkv, D, C, W)
    quant = OracleCache(1, Nq, Nkv, D, C, W)
    quant.pk = np.zeros((1, Nkv, C, D), np.uint8)
    quant.pv = np.zeros((1, Nkv, C, D), np.uint8)
    T = 0
    for S in [3, 1, 4, 1, 1, 2, 1]:
        q = _u(rng, (1, S, Nq * D))
        k = (rng.integers(-7, 8, size=(1, S, Nkv * D)) * ks).astype(np.float32)
        v = (rng.integers(-7, 8, size=(1, S, Nkv * D)) * vs).astype(np.float32)
        rp = plain.step(q, k, v, [T + S - 1])
        rq = oracle.step(q, k, v, quant.pk, quant.pv, np.array([T + S - 1], np.int32), T + S, Nq, Nkv, W,
                         cache_dtype=cache_dtype, k_scale=ks, v_scale=vs)
        quant.pk, quant.pv = rq["present_key"], rq["present_value"]
        assert np.array_equal(rp["output_f64"], rq["output_f64"])
        T += S
        L = int(rq["resident_len"][0])
        for row in range(L):  # row r holds the codes of the key of position T - L + r
            dec = np.array([(np.int8(np.uint8(c)) if cache_dtype == oracle.I8 else oracle.decode_e4m3(c))
                            for c in quant.pk[0, 0, row]], np.float64) * ks
            assert np.array_equal(dec, plain.pk[0, 0, row].astype(np.float64))


def test_quantized_rounds_and_chunk_invariance():
    """General values: a 4-token step equals four 1-token steps bit for bit (each new row
    is quantized once, and attention reads it as the cache holds it); the outputs differ
    from the unquantized cache only by the quantization (a few percent), and a key scale
    that is doubled halves every key code."""
    D, Nq, Nkv, C, W = 8, 2, 1, 6, 4
    rng = _rng(62)
    qp, kp, vp = _u(rng, (1, 7, Nq * D)), _u(rng, (1, 7, D)), _u(rng, (1, 7, D))
    q4, k4, v4 = _u(rng, (1, 4, Nq * D)), _u(rng, (1, 4, D)), _u(rng, (1, 4, D))
    for ct in (oracle.I8, oracle.E4M3):
        ks, vs = 1.0 / 100, 1.0 / 90

        def run(steps, ks=ks):
            pk = np.zeros((1, 1, C, D), np.uint8)
            pv = np.zeros((1, 1, C, D), np.uint8)
            outs = []
            for (q, k, v, seq) in steps:
                r = oracle.step(q, k, v, pk, pv, np.array([seq], np.int32), seq + 1, Nq, Nkv, W,
                                cache_dtype=ct, k_scale=ks, v_scale=vs)
                pk, pv = r["present_key"], r["present_value"]
                outs.append(r["output_f64"])
            return outs, pk, pv, r

        whole, pk_a, _, ra = run([(qp, kp, vp, 6), (q4, k4, v4, 10)])
        parts, pk_b, _, _ = run([(qp, kp, vp, 6)] + [(q4[:, s:s + 1], k4[:, s:s + 1], v4[:, s:s + 1], 7 + s)
                                                      for s in range(4)])
        for s in range(4):
            assert np.array_equal(whole[1][:, s], parts[1 + s][:, 0])
        L = int(ra["resident_len"][0])
        assert np.array_equal(pk_a[:, :, :L], pk_b[:, :, :L])
        if ct == oracle.I8:
            _, pk_2, _, _ = run([(qp, kp, vp, 6)], ks=2 * ks)
            _, pk_1, _, _ = run([(qp, kp, vp, 6)], ks=ks)
            c1 = pk_1[:, :, :6].view(np.int8).astype(np.int64)
            c2 = pk_2[:, :, :6].view(np.int8).astype(np.int64)
            assert np.all(np.abs(2 * c2 - c1) <= 1)
        ref = OracleCache(1, Nq, Nkv, D, C, W)
        ref.step(qp, kp, vp, [6])
        rr = ref.step(q4, k4, v4, [10])
        err = np.abs(rr["output_f64"] - whole[1]).max() / np.abs(rr["output_f64"]).max()
        assert 0 < err < (0.02 if ct == oracle.I8 else 0.1)
