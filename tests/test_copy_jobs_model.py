"""Model of the cache-update jobs into a separate present buffer (no GPU).

With present a separate buffer, the cache update (PR #31142 "[CPU] Add windowed kv cache
for GQA", Key design decisions, "Drifting layout": present row r <- past row r + seed for
the kept = L(T) - S surviving rows; PR #32419 "Specify GroupQueryAttention windowed KV
cache layout contract", Description: the new rows at [max(kept, 0), L(T))) has no hazard,
and ``finish_copy_kernel`` (csrc/gqaw_finish.cu) cuts it into independent jobs: for each
registered (item, kv head, K or V) slice, segments of R whole rows, numbered
job = slice * segments + segment with segments the most any registered item needs; the
slice's last segment also appends the new rows; an entry flagged "below only" (the
small-step attention kernel wrote the window's rows and the new rows) copies only the
rows below the window, [0, lo_row - seed) with lo_row = L(P) - min(P, W - 1).

This restates that numbering and checks, over random registered sets, that every row the
update must write is written exactly once with the right source and that jobs past an
item's segments do nothing.  L(T) is the library's host function; no oracle.
"""
from __future__ import annotations

import random

from sliding_window_gqa_02_gb300 import gqaw


def item_rows(P, S, C, W, below_only):
    Lp = gqaw.gqaw_resident_len(P, C, W)
    Lt = gqaw.gqaw_resident_len(P + S, C, W)
    kept, seed = Lt - S, Lp + S - Lt
    nwin = min(P, W - 1)
    nrows = Lp - nwin - seed if below_only else kept
    return Lp, Lt, kept, seed, nrows


def run_jobs(items, S, C, W, R, nkv=2):
    """items: list of (P, below_only).  Returns {(item, kvh, tensor, row): source}."""
    plans = [item_rows(P, S, C, W, bo) for P, bo in items]
    nseg = max([(p[4] + R - 1) // R for p in plans if p[4] > 0] or [1])
    nslices = len(items) * nkv * 2
    writes = {}
    for job in range(nslices * nseg):
        slice_, sg = divmod(job, nseg)
        tensor, kvh, ei = slice_ & 1, (slice_ >> 1) % nkv, (slice_ >> 1) // nkv
        Lp, Lt, kept, seed, nrows = plans[ei]
        last = (nrows + R - 1) // R - 1 if nrows > 0 else 0
        if sg > last:
            continue
        if nrows > 0:
            for r in range(sg * R, min(nrows, sg * R + R)):
                key = (ei, kvh, tensor, r)
                assert key not in writes, ("row written twice", key)
                writes[key] = ("past", r + seed)
        if items[ei][1] or sg != last:
            continue
        for r in range(max(kept, 0), Lt):
            key = (ei, kvh, tensor, r)
            assert key not in writes, ("row written twice", key)
            writes[key] = ("new", seed + r - Lp)
    return plans, writes


def check(items, S, C, W, R):
    nkv = 2
    plans, writes = run_jobs(items, S, C, W, R, nkv)
    want = {}
    for ei, ((P, below_only), (Lp, Lt, kept, seed, nrows)) in enumerate(zip(items, plans)):
        for kvh in range(nkv):
            for tensor in range(2):
                for r in range(max(nrows, 0)):
                    want[(ei, kvh, tensor, r)] = ("past", r + seed)
                if not below_only:
                    for r in range(max(kept, 0), Lt):
                        want[(ei, kvh, tensor, r)] = ("new", seed + r - Lp)
    assert writes == want


def test_copy_jobs_random():
    rng = random.Random(11)
    for _ in range(300):
        W = rng.randint(1, 300)
        C = W + rng.randint(0, 120)
        S = rng.randint(1, 40)
        R = rng.choice([1, 3, 16, 64, 128])
        items = [(rng.randint(0, 5 * C), rng.random() < 0.3) for _ in range(rng.randint(1, 6))]
        check(items, S, C, W, R)


def test_copy_jobs_long_context_decode():
    """The Mode A decode shape (C = 5120, W = 4096, S = 1, below-only entries) with the
    kernel's 128-row segments of bf16 rows of head size 128."""
    rng = random.Random(12)
    items = [(rng.randint(4096, 32768), True) for _ in range(8)]
    check(items, 1, 5120, 4096, 128)
