"""Model of the cache update that the small-step kernel does inside the attention pass.

Block compaction (PR #31142 "[CPU] Add windowed kv cache for GQA", Key design decisions,
"Drifting layout": a reclaimed G-row block moves the surviving rows down by seed =
L(P) + S - L(T)) and the append (PR #32419 "Specify GroupQueryAttention windowed KV cache
layout contract", Description: row i holds position T - L + i) are done by the attention
kernel itself for items whose surviving rows all lie in the window it reads: the rows
are written from the key/value tiles already staged in shared memory.

The kernel's CTAs each read a contiguous range of 128-key tiles of an (item, kv head)
slice (stream-K), so a row may be read by one CTA and be the destination of a row read
by another.  The rule the kernel follows, restated here with the same arithmetic:

* a CTA writes a moved row directly when its destination lies in its own range (read by
  itself, earlier) or below the window (read by nobody);
* a destination in an earlier CTA's range (at most seed rows, at the start of a CTA's
  first unit) is written from a stash by the unit's last contributor, once every
  contributor has passed its ticket;
* the CTA that reads the unit's last tile appends the new rows after its tiles; append
  rows in an earlier CTA's range are written by the last contributor.

This test runs that rule over random capacities, windows, step sizes, lengths, tile sizes
and grid splits, and checks that (1) no row is written by one CTA while another CTA
still has to read it, (2) a CTA overwrites its own rows only after reading them, (3)
every row of [0, L(T)) is written exactly once, and (4) the result is the compaction
plus append.  It also checks the host's rule for leaving out the cache-update kernel:
with in-place caches, S <= G, S <= W and G <= the stash rows, every item either
reclaims nothing or is done by the attention kernel.  No GPU; no oracle (L(T) is the
library's host function).
"""
from __future__ import annotations

import random

import pytest

from sliding_window_gqa_02_gb300 import gqaw

STASH_ROWS = 32  # rows a CTA may stash (kMoveStashRows in the kernel)


def L(T, C, W):
    return gqaw.gqaw_resident_len(T, C, W)


def item_plan(P, S, C, W, stash=STASH_ROWS):
    """The kernel's per-item numbers and decision for an in-place cache."""
    Lp, Lt = L(P, C, W), L(P + S, C, W)
    seed, kept = Lp + S - Lt, Lt - S
    nwin = min(P, W - 1)
    lo_row = Lp - nwin
    if seed == 0:
        kind = "append"
    elif 0 <= kept <= nwin and seed <= stash:
        kind = "fused"
    else:
        kind = "finish"
    return dict(Lp=Lp, Lt=Lt, seed=seed, kept=kept, nwin=nwin, lo_row=lo_row, kind=kind)


def owner(x, V, G):
    """The CTA whose stream-K range holds virtual tile x (CTA c: [c*V/G, (c+1)*V/G))."""
    return ((x + 1) * G - 1) // V


def tile_rows(pl, lt, tile):
    """First slice row and valid row count of key tile lt of a unit."""
    return pl["lo_row"] + lt * tile, min(tile, pl["nwin"] - lt * tile)


def stash_rows(pl, lt0, tile):
    """Rows [0, n) of the first tile of a CTA whose range starts at tile lt0 > 0 of a
    fused unit: their destinations lie in the previous CTA's range."""
    if lt0 <= 0:
        return 0
    a, nvalid = tile_rows(pl, lt0, tile)
    return max(0, min(pl["seed"], nvalid))


def run_unit(pl, tiles_of, tile, TPU, u, V, G):
    """Apply the kernel's rule to one fused unit.  tiles_of[c] = (lt0, lt1) of every CTA
    c overlapping the unit.  Returns the list of writes (cta or 'last', step, dst, what)
    and the reads (cta, step, row)."""
    real = (pl["nwin"] + tile - 1) // tile
    seed, kept, Lp, Lt, lo_row = pl["seed"], pl["kept"], pl["Lp"], pl["Lt"], pl["lo_row"]
    reads, writes = [], []
    fx = real - 1 if real > 0 else 0
    cfix = owner(u * TPU + fx, V, G)
    for c, (lt0, lt1) in tiles_of.items():
        nst = stash_rows(pl, lt0, tile)
        for lt in range(lt0, min(lt1, real)):
            r0, nvalid = tile_rows(pl, lt, tile)
            for t in range(nvalid):
                reads.append((c, lt, r0 + t))
            tA = max(0, seed - r0)              # first surviving row of the tile
            first = lt == lt0 and lt0 > 0
            sB = nst if first else 0            # rows [0, sB) went to the stash
            for t in range(max(tA, sB), nvalid):
                writes.append((c, lt, r0 + t - seed, ("past", r0 + t)))
            for t in range(tA, sB):
                writes.append(("last", None, r0 + t - seed, ("past", r0 + t)))
    # appends: the CTA holding the unit's last tile, after its tiles
    lt0f = max(0, tiles_of[cfix][0])
    a_fix = lo_row + tile * lt0f
    for r in range(max(kept, 0), Lt):
        src = ("new", r - kept)
        if r >= a_fix or r < lo_row:
            writes.append((cfix, 10**9, r, src))
        else:
            writes.append(("last", None, r, src))
    return reads, writes


def check_unit(P, S, C, W, tile, TPU, u, V, G):
    pl = item_plan(P, S, C, W)
    if pl["kind"] != "fused":
        return False
    tiles_of = {}
    for x in range(u * TPU, u * TPU + TPU):
        c = owner(x, V, G)
        lt = x - u * TPU
        lo, hi = tiles_of.get(c, (lt, lt + 1))
        tiles_of[c] = (min(lo, lt), max(hi, lt + 1))
    reads, writes = run_unit(pl, tiles_of, tile, TPU, u, V, G)
    readers = {}
    for c, lt, r in reads:
        readers.setdefault(r, []).append((c, lt))
    dsts = {}
    for c, step, dst, src in writes:
        assert dst not in dsts, ("row written twice", dst, P, S, C, W)
        dsts[dst] = src
        if c == "last":
            continue  # after every contributor's ticket: all reads are done
        for rc, rstep in readers.get(dst, []):
            assert rc == c, ("row %d written by CTA %s while CTA %s reads it" % (dst, c, rc), P, S, C, W, tile)
            assert rstep <= step, ("row %d overwritten before its read" % dst, P, S, C, W, tile)
        if src[0] == "past":  # the source was read by the writer itself (in shared memory)
            assert any(rc == c for rc, _ in readers.get(src[1], [])), ("source not staged", src, P, S, C, W)
    # final layout: row i < kept holds past row i + seed, row i >= kept new row i - kept
    for r in range(pl["Lt"]):
        want = ("past", r + pl["seed"]) if r < pl["kept"] else ("new", r - pl["kept"])
        assert dsts.get(r) == want, ("row", r, dsts.get(r), want, P, S, C, W, tile)
    assert set(dsts) == set(range(pl["Lt"])), (P, S, C, W)
    return True


@pytest.mark.parametrize("tile", [32, 64, 128])
def test_fused_rows_random(tile):
    rng = random.Random(1234 + tile)
    fused = 0
    for _ in range(600):
        W = rng.randint(1, 700)
        C = W + rng.randint(0, 80)
        S = rng.randint(1, 32)
        P = rng.randint(S, 6 * C)
        # pre-step length P (seqlens_k + 1 - S); stream-K over several units and CTAs
        TPU = max(1, -(-min(W - 1, P) // tile))
        units = rng.randint(1, 6)
        V = units * TPU
        G = rng.randint(1, min(V, 40))
        for u in range(units):
            fused += check_unit(P, S, C, W, tile, TPU, u, V, G)
    assert fused > 50


def test_fused_rows_workload_shapes():
    """The verify (C = W + S - 1) and small-slack (C = W + 8) shapes with the kernel's
    128-key tiles and grids of up to 152 CTAs."""
    n = 0
    for C, W, S, Ps in [(4103, 4096, 8, range(5990, 6100, 7)), (4099, 4096, 4, range(5990, 6100, 5)),
                        (136, 128, 1, range(128, 600)), (136, 128, 8, range(130, 400, 3))]:
        for P in Ps:
            TPU = max(1, -(-min(W - 1, P) // 128))
            for units, G in [(128, 152), (16, 152), (8, 5), (64, 152)]:
                V = units * TPU
                G = min(G, V)
                for u in (0, units // 2, units - 1):
                    n += check_unit(P, S, C, W, 128, TPU, u, V, G)
    assert n > 100


def test_host_rule_for_skipping_the_cache_update_kernel():
    """In place, S <= G = C - W + 1, S <= W and G <= the stash rows: every item either
    reclaims nothing (append only) or is fused; exhaustive over small shapes."""
    for W in range(1, 40):
        for C in range(W, W + 34):
            G = C - W + 1
            for S in range(1, 33):
                if not (S <= G and S <= W and G <= STASH_ROWS):
                    continue
                for P in range(0, 3 * C + 5):
                    assert item_plan(P, S, C, W)["kind"] in ("append", "fused"), (P, S, C, W)
