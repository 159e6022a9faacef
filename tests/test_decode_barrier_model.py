"""A model of the small-step tensor-core kernel's barrier protocol (no GPU).

``mma_decode_kernel`` (csrc/gqaw_mmad.cuh) runs four roles per CTA that meet only at
mbarriers: the TMA producer, the widening warps, the MMA issuer and the softmax warps.
With a code cache, per key tile k:

  producer   Q of a unit into buffer u & 1 once the unit two back is done with it;
             codes of tile k into stage k % 3 once tile k - 3 is widened;
  widening   K(k) into fp16 K tile k & 1 (tensor memory) once S^T(k - 2) is done;
             V(k) into fp16 V tile k & 1 once P.V(k - 2) is done;
  MMA S      S^T(k) once K(k), Q and S^T buffer k & 1 are ready (its own thread);
  MMA PV     P.V(k) once P(k) and V(k) are ready (and, on a unit's first tile, once the
             previous unit's O has been read), on a second thread;
  softmax    reads S^T(k), frees it; writes P(k) into buffer k & 1 once P.V(k - 2) is
             done; may rescale O once P.V(k - 1) is done; reads O after a unit's last P.V.

With a bf16 cache there are no widening warps: S^T(k) and P.V(k) read the TMA stage of
tile k itself, and the stage is freed by two arrivals: a commit after P.V(k), and the
mover warp once the TMA stores of the rows it moves out of tile k have read the stage
(it waits for tile k's load, issues the stores, waits until they have read shared memory,
then arrives -- on every tile, with or without rows to move).

This model runs the roles as coroutines under a random scheduler, with TMA loads
and MMAs completing in any order and a commit arriving once every MMA its own thread
issued before it has completed (a tcgen05.commit tracks only its thread's MMAs; MMAs
into one accumulator run in issue order).  It checks that every
parity wait finds its barrier exactly k or k + 1 phases along (a parity wait cannot tell
phases two apart), that no buffer is rewritten while an MMA or role still uses it, and
that the roles never deadlock.  A planted early reuse of a V tile, and a mover that
frees a stage before its stores have read it, must be caught, so the model is not
vacuous.
"""
from __future__ import annotations

import random

import pytest


class _Bar:
    def __init__(self, count):
        self.count, self.pending, self.n = count, count, 0

    def arrive(self):
        assert self.pending > 0
        self.pending -= 1
        if self.pending == 0:
            self.n += 1  # one more completed phase
            self.pending = self.count


def _run(units, seed, v_reuse_lag=2, codes=True, max_steps=400000, mover_early=False, empty_by_s=False):
    """Run the protocol over units of the given key-tile counts; returns the violations.
    ``v_reuse_lag``: the widening warps reuse V tile k & 1 once P.V(k - lag) is done (2 is
    the kernel's rule).  ``codes=False``: a bf16 cache, where S^T and P.V read the TMA
    stage itself and a commit after P.V frees it (no widening warps)."""
    rnd = random.Random(seed)
    tiles, kc = [], 0
    for ui, nt in enumerate(units):
        for lt in range(nt):
            tiles.append(dict(kc=kc, ui=ui, first=lt == 0, last=lt == nt - 1))
            kc += 1
    bars = {("full", i): _Bar(1) for i in range(3)}
    bars.update({("empty", i): _Bar(1 if codes else 2) for i in range(3)})
    for i in range(2):
        for name in ("s_full", "s_free", "p_full", "o_done", "q_full", "q_free", "kconv", "vconv"):
            bars[(name, i)] = _Bar(1)
    bars["o_free"] = _Bar(1)
    mmas, commits, loads, errors = [], [], [], []
    held = dict(K16=[None, None], V16=[None, None], P=[None, None], stage=[None, None, None])
    consumed = set()      # ("stage", k): every reader of tile k's stage is done
    stage_reads = {}      # bf16 cache: MMAs done reading tile k's stage (S^T and P.V)

    def ready(name, k):
        n = bars[name].n
        if n > k + 1:
            errors.append("wait on %s for phase %d after %d phases (ambiguous)" % (name, k, n))
        if n < k:
            errors.append("wait on %s for phase %d after only %d phases (passes early)" % (name, k, n))
        return n >= k + 1

    def in_use(buf):
        return [m for m in mmas if not m["done"] and (buf in m["reads"] or buf in m["writes"])]

    def role_writes(buf, who):
        if in_use(buf):
            errors.append("%s rewrites %s while %s uses it" % (who, buf, in_use(buf)[0]["name"]))

    def issue(name, reads, writes, on_done=None, thread=None):
        for w in writes:
            # MMAs into one accumulator run in issue order
            if [m for m in in_use(w) if not (w in m["writes"] and w not in m["reads"])]:
                errors.append("MMA %s writes %s while it is in use" % (name, w))
        mmas.append(dict(name=name, reads=reads, writes=writes, done=False, on_done=on_done, thread=thread))

    def stage_read_done(k):
        stage_reads[k] = stage_reads.get(k, 0) + 1
        if stage_reads[k] == 3:  # S^T, P.V and the mover's stores
            consumed.add(("stage", k))

    def commit(name, thread):
        commits.append((name, [m for m in mmas if not m["done"] and m.get("thread") == thread]))

    def producer():
        for t in tiles:
            k, u = t["kc"], t["ui"]
            if t["first"]:
                while u >= 2 and not ready(("q_free", u & 1), (u - 2) >> 1):
                    yield
                role_writes(("Q", u & 1), "TMA of Q")
                loads.append([("q_full", u & 1), False])
            while k >= 3 and not ready(("empty", k % 3), k // 3 - 1):
                yield
            old = held["stage"][k % 3]
            if old is not None and ("stage", old) not in consumed:
                errors.append("TMA of tile %d overwrites stage %d before tile %d is consumed" % (k, k % 3, old))
            held["stage"][k % 3] = k
            loads.append([("full", k % 3), False])
            yield

    def widening():
        lag = v_reuse_lag
        for t in tiles:
            k = t["kc"]
            while not ready(("full", k % 3), k // 3):
                yield
            while k >= 2 and not ready(("s_full", k & 1), (k - 2) >> 1):
                yield
            role_writes(("K16", k & 1), "widening of K(%d)" % k)
            held["K16"][k & 1] = k
            bars[("kconv", k & 1)].arrive()
            yield
            while k >= lag and not ready(("o_done", (k - lag) & 1), (k - lag) >> 1):
                yield
            role_writes(("V16", k & 1), "widening of V(%d)" % k)
            held["V16"][k & 1] = k
            bars[("vconv", k & 1)].arrive()
            consumed.add(("stage", k))
            bars[("empty", k % 3)].arrive()
            yield

    def mma_s():
        def s_of(t):
            k, u = t["kc"], t["ui"]
            while t["first"] and not ready(("q_full", u & 1), u >> 1):
                yield
            while codes and not ready(("kconv", k & 1), k >> 1):
                yield
            while not codes and not ready(("full", k % 3), k // 3):
                yield
            while k >= 2 and not ready(("s_free", k & 1), (k - 2) >> 1):
                yield
            if codes:
                if held["K16"][k & 1] != k:
                    errors.append("S(%d) reads the K tile of tile %s" % (k, held["K16"][k & 1]))
                issue("S(%d)" % k, [("K16", k & 1), ("Q", u & 1)], [("S", k & 1)], thread="S")
            else:
                if held["stage"][k % 3] != k:
                    errors.append("S(%d) reads stage %d holding tile %s" % (k, k % 3, held["stage"][k % 3]))
                issue("S(%d)" % k, [("stage", k % 3), ("Q", u & 1)], [("S", k & 1)],
                      on_done=lambda k=k: stage_read_done(k), thread="S")
            commit(("s_full", k & 1), "S")
            if empty_by_s and not codes:  # planted: the S^T thread releases the stage
                commit(("empty", k % 3), "S")
            yield

        for t in tiles:
            yield from s_of(t)

    def mma_pv():
        for t in tiles:
            k, u = t["kc"], t["ui"]
            while not ready(("p_full", k & 1), k >> 1):
                yield
            while codes and not ready(("vconv", k & 1), k >> 1):
                yield
            while t["first"] and u >= 1 and not ready("o_free", u - 1):
                yield
            if held["P"][k & 1] != k:
                errors.append("P.V(%d) reads P of tile %s" % (k, held["P"][k & 1]))
            if codes:
                if held["V16"][k & 1] != k:
                    errors.append("P.V(%d) reads V of tile %s" % (k, held["V16"][k & 1]))
                issue("PV(%d)" % k, [("V16", k & 1), ("P", k & 1)], ["O"], thread="PV")
                commit(("o_done", k & 1), "PV")
            else:
                if held["stage"][k % 3] != k:
                    errors.append("P.V(%d) reads stage %d holding tile %s" % (k, k % 3, held["stage"][k % 3]))
                issue("PV(%d)" % k, [("stage", k % 3), ("P", k & 1)], ["O"], on_done=lambda k=k: stage_read_done(k),
                      thread="PV")
                commit(("o_done", k & 1), "PV")
                if not empty_by_s:
                    commit(("empty", k % 3), "PV")
            if t["last"]:
                commit(("q_free", u & 1), "PV")
            yield

    def mover():
        for t in tiles:
            k = t["kc"]
            while not ready(("full", k % 3), k // 3):
                yield
            if held["stage"][k % 3] != k:
                errors.append("mover reads stage %d holding tile %s" % (k % 3, held["stage"][k % 3]))
            store = dict(name="ST(%d)" % k, reads=[("stage", k % 3)], writes=[], done=False,
                         on_done=lambda k=k: stage_read_done(k))
            mmas.append(store)  # an asynchronous reader of the stage, like an MMA
            yield
            while not mover_early and not store["done"]:  # the bulk group has read the stage
                yield
            bars[("empty", k % 3)].arrive()
            yield

    def softmax():
        for t in tiles:
            k, u = t["kc"], t["ui"]
            while not ready(("s_full", k & 1), k >> 1):
                yield
            if in_use(("S", k & 1)):
                errors.append("softmax reads S(%d) before it is complete" % k)
            yield
            bars[("s_free", k & 1)].arrive()
            while k >= 2 and not ready(("o_done", k & 1), (k - 2) >> 1):
                yield
            role_writes(("P", k & 1), "softmax P(%d)" % k)
            held["P"][k & 1] = k
            if not t["first"] and rnd.random() < 0.3:  # a rescale of O
                while not ready(("o_done", (k - 1) & 1), (k - 1) >> 1):
                    yield
                role_writes("O", "rescale at tile %d" % k)
            bars[("p_full", k & 1)].arrive()
            yield
            if t["last"]:
                while not ready(("o_done", k & 1), k >> 1):
                    yield
                role_writes("O", "epilogue of unit %d" % u)
                bars["o_free"].arrive()
                yield

    roles = {"producer": producer(), "mma_s": mma_s(), "mma_pv": mma_pv(), "softmax": softmax()}
    if codes:
        roles["widening"] = widening()
    else:
        roles["mover"] = mover()
    steps = 0
    while roles and not errors and steps < max_steps:
        steps += 1
        pick = rnd.choice(list(roles) + ["async", "async"])
        if pick == "async":  # one TMA load or MMA completes; commits whose MMAs are done arrive
            pending = [m for m in mmas if not m["done"]] + [x for x in loads if not x[1]]
            if pending:
                x = rnd.choice(pending)
                if isinstance(x, dict):
                    x["done"] = True
                    if x["on_done"]:
                        x["on_done"]()
                else:
                    x[1] = True
                    bars[x[0]].arrive()
            for c in list(commits):
                if all(m["done"] for m in c[1]):
                    commits.remove(c)
                    bars[c[0]].arrive()
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
    return [[rnd.randint(1, 6) for _ in range(rnd.randint(1, 6))] for _ in range(n)]


@pytest.mark.parametrize("codes", [True, False])
def test_protocol_has_no_hazard_ambiguous_wait_or_deadlock(codes):
    for i, units in enumerate(_cases(600, 1)):
        errors = _run(units, seed=i, codes=codes)
        assert not errors, (units, i, errors[:3])


@pytest.mark.parametrize("codes", [True, False])
@pytest.mark.parametrize("units", [[1], [1, 1, 1, 1], [7], [2, 1, 3, 1, 2]])
def test_small_unit_mixes(units, codes):
    for seed in range(200):
        assert not _run(units, seed, codes=codes), (units, seed)


def test_model_catches_early_v_reuse():
    """Reusing a V tile once P.V of three tiles back is done (one tile too early for two
    buffers) must be reported; waiting for P.V of the previous tile (one buffer's rule) is
    slower but safe."""
    cases = _cases(200, 2)
    errors = [e for i, units in enumerate(cases) for e in _run(units, i, v_reuse_lag=3)]
    assert any("ambiguous" in e or "rewrites" in e or "reads V" in e for e in errors)
    assert not [e for i, units in enumerate(cases) for e in _run(units, i, v_reuse_lag=1)]


def test_model_catches_mover_freeing_a_stage_early():
    """A mover that frees a stage as soon as it has issued its stores (before they have
    read shared memory) lets the next load overwrite a stage still being read."""
    cases = _cases(300, 3)
    errors = [e for i, units in enumerate(cases) for e in _run(units, i, codes=False, mover_early=True)]
    assert any("before tile" in e or "rewrites" in e for e in errors)


def test_model_catches_stage_released_by_the_wrong_thread():
    """With S^T and P.V on two threads, a commit covers only its own thread's MMAs: the
    S^T thread releasing a stage (its commit does not wait for P.V of the tile) lets the
    next load overwrite a stage that P.V still reads."""
    cases = _cases(300, 4)
    errors = [e for i, units in enumerate(cases) for e in _run(units, i, codes=False, empty_by_s=True)]
    assert any("before tile" in e or "reads stage" in e or "rewrites" in e for e in errors)
