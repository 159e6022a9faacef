"""A model of the multi-token tensor-core kernel's barrier protocol (no GPU).

``mma_attend_kernel`` (csrc/gqaw_mma.cu) is persistent: one CTA runs a sequence of units
(a query tile against its key tiles), and its rings and barrier phases run on from one
unit to the next.  Roles, per key tile g numbered across the CTA's units:

  K loader   K(g) into ring stage g % 3 once S(g - 3) is done (k_free); after a unit's
             first K tile, its query tile into the single Q buffer once the previous
             unit's last S product is done (q_free);
  V loader   V(g) into ring stage g % 2 once O += P(g - 2) V(g - 2) is done (pv_done);
  MMA        S(first) of a unit, then per tile S(g + 1) before O += P(g) V(g); S(g) into
             tensor-memory buffer g % 2; O += P V once V(g) and P(g) are ready, and on a
             unit's first tile once the previous unit's O has been read (o_free);
  softmax    reads S(g) (s_full), writes P(g) into buffer g % 2 (p_full); may rescale O
             once O += P(g - 1) V(g - 1) is done; reads O after the unit's last O += P V.

There is no barrier for "the softmax has read S(g - 2)" or "O += P(g - 2) V(g - 2) has
read P buffer g % 2": the MMA thread issues S(g + 1) only after it has seen P(g - 1), and
the commit of S(g) covers the earlier O += P(g - 2) V(g - 2).  The model checks those
hand-overs too.  The roles run as coroutines under a random scheduler; TMA loads and MMAs
complete in any order; a commit arrives once every MMA issued before it has completed
(MMAs into one accumulator run in issue order).  Checked: every parity wait finds its
barrier exactly k or k + 1 phases along, no buffer is rewritten before its last reader
is done, and no deadlock.  Units with no key tile are skipped by every role.
"""
from __future__ import annotations

import random

import pytest


class _Bar:
    def __init__(self):
        self.n = 0  # completed phases (every barrier here has an arrival count of 1)


def _run(units, seed, plant=None, max_steps=400000):
    """Violations of the protocol over units with the given key-tile counts.  ``plant``
    names a deliberate mistake (to show the model catches it)."""
    rnd = random.Random(seed)
    names = [("k_full", i) for i in range(3)] + [("k_free", i) for i in range(3)]
    names += [(n, i) for n in ("v_full", "pv_done", "s_full", "p_full") for i in range(2)]
    names += ["q_full", "q_free", "o_free"]
    bars = {n: _Bar() for n in names}
    errors, mmas, commits, loads = [], [], [], []
    # what each buffer holds: tile numbers (None: nothing yet)
    held = {("K", i): None for i in range(3)}
    held.update({("V", i): None for i in range(2)})
    held.update({("S", i): None for i in range(2)})
    held.update({("P", i): None for i in range(2)})
    held["Q"] = None
    consumed = set()  # (buffer, tile) pairs whose reader is done
    o_state = dict(unit=None, read=True)

    def ready(name, k):
        n = bars[name].n
        if n > k + 1:
            errors.append("wait on %s for phase %d after %d phases (ambiguous)" % (name, k, n))
        if n < k:
            errors.append("wait on %s for phase %d after only %d phases (passes early)" % (name, k, n))
        return n >= k + 1

    def arrive(name):
        bars[name].n += 1

    def in_flight(buf):
        return [m for m in mmas if not m["done"] and (buf in m["reads"] or buf in m["writes"])]

    def overwrite(buf, tile, who):
        """A role or a load replaces the content of buf: its old content must be consumed."""
        old = held[buf]
        if in_flight(buf):
            errors.append("%s overwrites %s while %s uses it" % (who, buf, in_flight(buf)[0]["name"]))
        elif old is not None and (buf, old) not in consumed:
            errors.append("%s overwrites %s holding tile %s before it was consumed" % (who, buf, old))
        held[buf] = tile

    def issue(name, reads, writes, on_done):
        for w in writes:
            if [m for m in in_flight(w) if not (w in m["writes"] and w not in m["reads"])]:
                errors.append("MMA %s writes %s while it is in use" % (name, w))
        mmas.append(dict(name=name, reads=reads, writes=writes, done=False, on_done=on_done))

    def commit(name):
        commits.append((name, [m for m in mmas if not m["done"]]))

    tiles_of = [n for n in units]

    def k_loader():
        g, qi = 0, 0
        for u, nt in enumerate(tiles_of):
            for k in range(nt):
                while g >= 3 and not ready(("k_free", g % 3), g // 3 - 1):
                    yield
                overwrite(("K", g % 3), g, "K load")
                loads.append([("k_full", g % 3), False])
                g += 1
                yield
                if k == 0:
                    while qi > 0 and not ready("q_free", qi - 1):
                        yield
                    overwrite("Q", u, "Q load")
                    loads.append(["q_full", False])
                    qi += 1
                    yield

    def v_loader():
        g = 0
        lag = 3 if plant == "v_reuse_early" else 2
        for nt in tiles_of:
            for _ in range(nt):
                while g >= lag and not ready(("pv_done", (g - lag) % 2), (g - lag) // 2):
                    yield
                overwrite(("V", g % 2), g, "V load")
                loads.append([("v_full", g % 2), False])
                g += 1
                yield

    def mma():
        g, qi = 0, 0

        def s_product(t, u, last):
            kst = t % 3
            if held[("K", kst)] != t or held["Q"] != u:
                errors.append("S(%d) reads K of tile %s, Q of unit %s" % (t, held[("K", kst)], held["Q"]))
            # the buffer's previous S must have been read by the softmax
            overwrite_s = ("S", t & 1)
            old = held[overwrite_s]
            if old is not None and (overwrite_s, old) not in consumed:
                errors.append("S(%d) overwrites S(%d) before the softmax read it" % (t, old))
            held[overwrite_s] = t

            def done(t=t, kst=kst, u=u, last=last):
                consumed.add((("K", kst), t))
                if last:  # the unit's last S product: its query tile is consumed
                    consumed.add(("Q", u))
            issue("S(%d)" % t, [("K", kst), "Q"], [overwrite_s], done)
            commit(("s_full", t & 1))
            commit(("k_free", kst))

        for u, nt in enumerate(tiles_of):
            if nt <= 0:
                continue
            while not ready("q_full", qi):
                yield
            while not ready(("k_full", g % 3), g // 3):
                yield
            s_product(g, u, nt == 1)
            if nt == 1:
                commit("q_free")
            yield
            if nt > 1:
                while not ready(("k_full", (g + 1) % 3), (g + 1) // 3):
                    yield
            for k in range(nt):
                gt = g + k
                if k + 1 < nt:
                    s_product(gt + 1, u, k + 2 == nt)
                    if k + 2 == nt:
                        commit("q_free")
                    yield
                    if k + 2 < nt:
                        while not ready(("k_full", (gt + 2) % 3), (gt + 2) // 3):
                            yield
                while not ready(("v_full", gt & 1), gt >> 1):
                    yield
                while not ready(("p_full", gt & 1), gt >> 1):
                    yield
                while k == 0 and qi > 0 and not ready("o_free", qi - 1):
                    yield
                if held[("V", gt & 1)] != gt or held[("P", gt & 1)] != gt:
                    errors.append("O += P V(%d) reads V of %s, P of %s" % (gt, held[("V", gt & 1)], held[("P", gt & 1)]))
                if k == 0 and not o_state["read"]:
                    errors.append("first O += P V of unit %d overwrites O before it was read" % u)
                if k == 0:
                    o_state.update(unit=u, read=False)

                def done(gt=gt):
                    consumed.add((("V", gt & 1), gt))
                    consumed.add((("P", gt & 1), gt))
                issue("PV(%d)" % gt, [("V", gt & 1), ("P", gt & 1)], ["O"], done)
                commit(("pv_done", gt & 1))
                yield
            g += nt
            qi += 1

    def softmax():
        g = 0
        for u, nt in enumerate(tiles_of):
            if nt <= 0:
                continue
            for k in range(nt):
                gt = g + k
                while not ready(("s_full", gt & 1), gt >> 1):
                    yield
                if in_flight(("S", gt & 1)) or held[("S", gt & 1)] != gt:
                    errors.append("softmax reads S(%d) too early (buffer holds %s)" % (gt, held[("S", gt & 1)]))
                yield
                consumed.add((("S", gt & 1), gt))
                if k > 0 and rnd.random() < 0.3:  # a rescale of O
                    while not ready(("pv_done", (gt - 1) & 1), (gt - 1) >> 1):
                        yield
                    if in_flight("O"):
                        errors.append("rescale at tile %d while O += P V is in flight" % gt)
                overwrite(("P", gt & 1), gt, "softmax P(%d)" % gt)
                arrive(("p_full", gt & 1))
                yield
            last = g + nt - 1
            while not ready(("pv_done", last & 1), last >> 1):
                yield
            if in_flight("O"):
                errors.append("epilogue of unit %d reads O while O += P V is in flight" % u)
            o_state["read"] = True
            arrive("o_free")
            g += nt
            yield

    roles = {"k": k_loader(), "v": v_loader(), "mma": mma(), "softmax": softmax()}
    steps = 0
    while roles and not errors and steps < max_steps:
        steps += 1
        pick = rnd.choice(list(roles) + ["async", "async"])
        if pick == "async":
            pending = [m for m in mmas if not m["done"]] + [x for x in loads if not x[1]]
            if pending:
                x = rnd.choice(pending)
                if isinstance(x, dict):
                    x["done"] = True
                    x["on_done"]()
                else:
                    x[1] = True
                    arrive(x[0])
            for c in list(commits):
                if all(m["done"] for m in c[1]):
                    commits.remove(c)
                    arrive(c[0])
            continue
        try:
            next(roles[pick])
        except StopIteration:
            del roles[pick]
    if not errors and roles:
        errors.append("roles %s never finished (deadlock)" % sorted(roles))
    return errors


def _cases(n, seed):
    rnd = random.Random(seed)
    return [[rnd.randint(0, 5) for _ in range(rnd.randint(1, 6))] for _ in range(n)]


def test_protocol_has_no_hazard_ambiguous_wait_or_deadlock():
    for i, units in enumerate(_cases(600, 3)):
        errors = _run(units, seed=i)
        assert not errors, (units, i, errors[:3])


@pytest.mark.parametrize("units", [[1], [1, 1, 1, 1], [0, 2, 0, 1], [7], [3, 1, 2, 1, 3]])
def test_small_unit_mixes(units):
    for seed in range(200):
        assert not _run(units, seed), (units, seed)


def test_model_catches_early_v_reuse():
    """Loading V(g) once O += P(g - 3) V(g - 3) is done (one tile too early for two ring
    stages) can overwrite a tile still waiting for its O += P V: the model must report it."""
    errors = [e for i, units in enumerate(_cases(200, 4)) for e in _run(units, i, plant="v_reuse_early")]
    assert errors
