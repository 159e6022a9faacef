"""Steps captured in a CUDA graph (as the benchmark replays them) give the same results
as the same steps launched one by one: both kernels of a step, their programmatic
dependent launch edges and the workspace bookkeeping (item list, tickets) survive
capture and replay."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as wl
from sliding_window_gqa_02_gb300 import gqaw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(sh, S, steps, seed, graph):
    dev = torch.device("cuda:0")
    B = sh.B
    pk, pv = wl.cache(sh, seed)
    ck, cv = pk.to(dev), pv.to(dev)
    T = wl.lengths(B, 120, 600, seed)
    seq = torch.tensor(np.stack([T + t * S + S - 1 for t in range(steps)]).astype(np.int32), device=dev)
    totals = [int(T.max()) + (t + 1) * S for t in range(steps)]
    ins = [tuple(x.to(dev) for x in wl.step_inputs(sh, S, seed * 10 + t)) for t in range(steps)]
    outs = [torch.empty_like(ins[t][0]) for t in range(steps)]
    args = [gqaw.make_args(ins[t][0], ins[t][1], ins[t][2], ck, cv, ck, cv, seq[t], totals[t], sh.Nq, sh.Nkv, sh.W,
                           outs[t]) for t in range(steps)]
    nbytes = max(gqaw.gqaw_workspace_bytes(a) for a in args)
    stream = torch.cuda.Stream()
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    gqaw.check(gqaw.gqaw_workspace_init(int(ws.data_ptr()), nbytes, stream.cuda_stream))
    args = [gqaw.make_args(ins[t][0], ins[t][1], ins[t][2], ck, cv, ck, cv, seq[t], totals[t], sh.Nq, sh.Nkv, sh.W,
                           outs[t], workspace=ws) for t in range(steps)]
    torch.cuda.synchronize()
    if graph:
        # the first call on a device sets function attributes: do it outside capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for a in args:
                gqaw.check(gqaw.gqa_windowed_step(a, stream.cuda_stream))
        g.replay()
    else:
        for a in args:
            gqaw.check(gqaw.gqa_windowed_step(a, stream.cuda_stream))
    torch.cuda.synchronize()
    st, flags = gqaw.gqaw_device_status(int(ws.data_ptr()))
    assert st == 0 and flags == 0
    return [o.cpu() for o in outs], ck.cpu(), cv.cpu()


@pytest.mark.parametrize("name,S", [("slack", 1), ("slack", 6), ("pages", 1)])
def test_graph_replay_equals_eager(name, S):
    sh = wl.SHAPES[name]
    _run(sh, S, 2, 31, graph=False)  # warm: attributes set outside capture
    eager = _run(sh, S, 12, 32, graph=False)
    graph = _run(sh, S, 12, 32, graph=True)
    for a, b in zip(eager[0], graph[0]):
        assert torch.equal(a, b)
    assert torch.equal(eager[1], graph[1]) and torch.equal(eager[2], graph[2])
