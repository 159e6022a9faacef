"""Benchmark of the windowed-GQA step on GB300; prints one JSON line.

Default workload (``longctx-decode``): B=64, 32 query / 8 kv heads, head size 128,
bf16 caches, W=4096, C=5120, per-item contexts ~ U[4096, 32768]; each step is one
decode token for all 64 items through the C ABI.  The K/V window read per step
(about 1.07 GB) is larger than the 129 MB L2, so no flush is needed between steps.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl gqaw|reference]
                    [--workload longctx-decode|longctx-decode-sink|longctx-decode-rope|longctx-decode-i8|
                     longctx-decode-modeA|
                     longctx-decode-e4m3|pages-decode|slack-decode|verify4|verify8|longctx-prefill|
                     longctx-prefill-rope]
                    [--no-extra] [--no-cpu-baseline]

``--impl reference`` times the oracle (the plain fp64 CPU implementation) on this
host's cores on the same workload, each step a bounded sample of items.

Under torchrun (WORLD_SIZE > 1) every rank runs its own independent replica of the
workload (different seeds, no exchange): weak scaling, no collective on the data path.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "windowed-GQA decode tokens/s; KV HBM GB/s as % of GB300 peak"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ workloads


def workload_spec(name):
    import workloads as wl

    if name == "longctx-decode":
        return dict(shape=wl.SHAPES["longctx"], S=1, lo=4096, hi=32768, bias=False, graph=False, accept=False)
    if name == "longctx-decode-sink":  # the same decode with a sink logit per query head
        return dict(shape=wl.SHAPES["longctx"], S=1, lo=4096, hi=32768, bias=False, graph=False, accept=False,
                    sink=True)
    if name in ("longctx-decode-i8", "longctx-decode-e4m3"):  # the same decode on a quantized cache
        return dict(shape=wl.SHAPES["longctx"], S=1, lo=4096, hi=32768, bias=False, graph=False, accept=False,
                    quant=name.rsplit("-", 1)[1])
    if name == "longctx-decode-modeA":  # the same decode into a separate present buffer (ping-pong)
        return dict(shape=wl.SHAPES["longctx"], S=1, lo=4096, hi=32768, bias=False, graph=False, accept=False,
                    separate=True)
    if name == "longctx-decode-rope":  # the same decode with the rotary embedding fused in
        return dict(shape=wl.SHAPES["longctx"], S=1, lo=4096, hi=32768, bias=False, graph=False, accept=False,
                    rope=True)
    if name in ("longctx-prefill", "longctx-prefill-rope"):
        sh = wl.SHAPES["longctx"]
        return dict(shape=sh, S=512, lo=4096, hi=32768, bias=False, graph=False, accept=False, B=8,
                    rope=name.endswith("rope"))
    if name == "pages-decode":
        return dict(shape=wl.SHAPES["pages"], S=1, lo=8192, hi=8192, bias=False, graph=True, accept=False)
    if name == "slack-decode":
        return dict(shape=wl.SHAPES["slack"], S=1, lo=128, hi=160, bias=False, graph=True, accept=False)
    if name in ("verify4", "verify8"):  # speculative verify: C = W + S - 1, softcap, bias, rollbacks
        return dict(shape=wl.SHAPES[name], S=int(name[-1]), lo=6000, hi=6000, bias=True, graph=True, accept=True)
    raise SystemExit("unknown workload " + name)


def workload_config(name, B=None):
    """The `config` object of the JSON line (shared by the GPU and reference arms).
    The step computes in fp32 (accumulation) over caches of `cache_dtype`."""
    spec = workload_spec(name)
    sh = spec["shape"]
    return {"workload": name, "B": B if B else spec.get("B", sh.B), "S": spec["S"], "num_heads": sh.Nq,
            "kv_num_heads": sh.Nkv, "head_size": sh.D, "local_window_size": sh.W, "capacity": sh.C,
            "cache_dtype": sh.dtype, "softcap": sh.softcap, "bias": spec["bias"],
            "head_sink": bool(spec.get("sink", False)), "rotary": bool(spec.get("rope", False)),
            "present": "separate buffer" if spec.get("separate") else "in place",
            "kv_cache": spec.get("quant") or sh.dtype, "contexts": "U[%d,%d]" % (spec["lo"], spec["hi"])}


def resident_len(T, C, W):
    """L(T) through the C ABI (host function of the library)."""
    from sliding_window_gqa_02_gb300 import gqaw

    return gqaw.gqaw_resident_len(int(T), int(C), int(W))


def attention_moves_rows(sh, S, P, separate, quant=None):
    """Does the attention kernel write an item's surviving rows itself (the small-step
    kernel with a bf16 cache: a separate present buffer, or in place with a reclaimed
    block of at most 32 rows whose surviving rows all lie in the window)?  Returns the
    rows it writes that way."""
    if attention_kernel(sh, S, quant) != "mmad" or quant:
        return 0
    Lp, Lt = resident_len(P, sh.C, sh.W), resident_len(P + S, sh.C, sh.W)
    seed, kept, nwin = Lp + S - Lt, Lt - S, min(P, sh.W - 1)
    if separate or (seed > 0 and 0 <= kept <= nwin and seed <= 32):
        return max(0, min(kept, nwin))
    return 0


def algorithmic_bytes(sh, S, T_before, B, cache_bytes=None, separate=False, quant=None):
    """Bytes the step must move, per item from the pre-step lengths: the in-window cache
    rows and the new rows read, the appended rows written, the surviving rows of a
    reclaimed block written at their new place (and read too where they lie below the
    window the attention reads: a surviving row inside the window is read once, for both
    uses), the query read and the output written.  With a ``separate`` present buffer every
    surviving row is written (and read where it lies below the window), reclaimed block
    or not.  Returns (attention kernel bytes, step bytes): the attention kernel's are its
    reads, the query and output, and the rows it writes (appends, and the surviving rows
    it moves from its staged tiles).
    ``cache_bytes``: bytes of a cache element (1 for a quantized cache).  Bias bytes are
    added by the caller."""
    e = 2 if sh.dtype == "bf16" else 4
    row = sh.Nkv * sh.D * (cache_bytes or e) * 2  # K and V of one position, all kv heads
    attn = comp = app = kern_w = 0
    for b in range(B):
        P = int(T_before[b])
        T = P + S
        Lp, Lt = resident_len(P, sh.C, sh.W), resident_len(T, sh.C, sh.W)
        kept = Lt - S
        seed = Lp + S - Lt
        nwin = min(P, sh.W - 1)
        attn += row * (nwin + S)
        app += row * min(S, Lt)
        if (seed > 0 or separate) and kept > 0:
            comp += row * (kept + max(kept - nwin, 0))
        kern_w += row * (min(S, Lt) + attention_moves_rows(sh, S, P, separate, quant))
    qo = B * S * sh.Nq * sh.D * e * 2
    return attn + qo + kern_w, attn + app + comp + qo


def cache_events(sh, S, T_before):
    """Per-step counts of what the cache update does (from the pre-step lengths, through
    the library's L(T)): items that reclaim a block (compaction events, PR #31142 "[CPU]
    Add windowed kv cache for GQA", "Skip compaction on drifting steps"), items whose
    step is hazardous (kept < min(P, W - 1): compaction-first would drop history its own
    first query reads, "Staging for hazardous steps"), and the bytes of rows moved."""
    e = 2 if sh.dtype == "bf16" else 4
    row = sh.Nkv * sh.D * e * 2
    comp = haz = moved = 0
    for P in T_before:
        P = int(P)
        Lp, Lt = resident_len(P, sh.C, sh.W), resident_len(P + S, sh.C, sh.W)
        kept, seed = Lt - S, Lp + S - Lt
        if seed > 0:
            comp += 1
            moved += 2 * row * max(kept, 0)
        haz += int(kept < min(P, sh.W - 1))
    return comp, haz, moved


def events_summary(sh, S, Ts):
    """Mean per step of cache_events over the given pre-step length vectors."""
    c = [cache_events(sh, S, T) for T in Ts]
    n = max(len(c), 1)
    return {"compacting_items_per_step": sum(x[0] for x in c) / n,
            "hazardous_items_per_step": sum(x[1] for x in c) / n,
            "moved_bytes_per_step": sum(x[2] for x in c) / n,
            "steps_with_compaction": sum(1 for x in c if x[0] > 0), "steps": len(c)}


def visible_columns(S, T_before, W):
    n = 0
    for P in T_before:
        for s in range(S):
            n += min(int(P) + s + 1, W)
    return n


def step_flops(sh, S, T_before):
    """Algorithmic FLOPs of one multi-token step: Q.K^T and P.V over the visible keys,
    sum over items and tokens of Nq * 4 * D * min(P + s + 1, W)."""
    return sh.Nq * 4 * sh.D * visible_columns(S, T_before, sh.W)


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms in a background process."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = [r for t, r in self.rows if t0 <= t <= t1]
        window = "timed region"
        if not rows:  # timed region shorter than the sampling period: nearest samples
            rows = [r for t, r in self.rows if t0 - 1.0 <= t <= t1 + 1.0]
            window = "timed region +- 1 s"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if len(r) > 2 and num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if len(r) > 2 and num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, n in enumerate(names):
                if len(r) > 5 + i and r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows), "window": window}


# ------------------------------------------------------------------ profiles (ncu traffic)


# The attention kernel a step runs on (the library's dispatch rule), the short name of
# its profile summaries and the sources that define it.
KERNELS = {
    "mmad": ("mma_decode_kernel (tcgen05)",
             ("gqaw_mmad.cuh", "gqaw_mmad.cu", "gqaw_mmad_q8.cu", "gqaw_tc.cuh", "gqaw_internal.cuh")),
    "mma": ("mma_attend_kernel (tcgen05)", ("gqaw_mma.cu", "gqaw_tc.cuh", "gqaw_internal.cuh")),
    "attend": ("attend_kernel", ("gqaw_attend.cuh", "gqaw_internal.cuh", "gqaw_attend_launch.cuh",
                                 "gqaw_attend_bf16.cu", "gqaw_attend_f32.cu")),
}


def attention_kernel(sh, S, quant=None):
    g = sh.Nq // sh.Nkv
    if sh.dtype == "bf16" and sh.D == 128 and S * g <= 32:
        return "mmad"  # code caches too (widened to fp16 tiles in the kernel)
    if quant:
        return "attend"
    if sh.dtype == "bf16" and sh.D == 128 and S >= 2 and g <= 32 and 32 % g == 0:
        return "mma"
    return "attend"


def kernel_source_hash(kernel="mmad"):
    h = hashlib.sha256()
    for f in KERNELS[kernel][1]:
        with open(os.path.join(ROOT, "sliding_window_gqa_02_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, kernel):
    """DRAM bytes per attention launch from the committed ncu summary of this workload,
    or None if there is none or the kernel's sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (kernel, workload))
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    hm = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    if not m or not hm or hm.group(1) != kernel_source_hash(kernel):
        return None
    return float(m.group(1))


def check_device(h, what):
    """A run whose device status word is non-zero (an expired in-kernel wait, a bad
    seqlens_k) has no valid timing: fail loudly."""
    st, flags = h.gqaw.gqaw_device_status(int(h.ws.data_ptr()), stream=h.stream.cuda_stream)
    if flags:
        raise RuntimeError("%s: device status 0x%x after the timed steps" % (what, flags))


def bf16_peak_tflops():
    """Dense bf16 tensor peak: the burst cuBLAS figure of MEASURED_PEAKS.json, else the
    fallback of 1900 TFLOP/s."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    return 1900.0


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ GPU arm


class Harness:
    """Device buffers and per-step argument structs for one workload replica."""

    def __init__(self, name, steps, warmup, seed, split_keys=0, batch=0):
        import torch

        import workloads as wl
        from sliding_window_gqa_02_gb300 import gqaw

        self.torch, self.wl, self.gqaw = torch, wl, gqaw
        spec = workload_spec(name)
        self.name, self.spec = name, spec
        sh = spec["shape"]
        self.sh = sh
        self.B = batch if batch > 0 else spec.get("B", sh.B)
        self.S = spec["S"]
        self.dev = torch.device("cuda", torch.cuda.current_device())
        self.stream = torch.cuda.Stream()  # every launch and copy of this replica goes here
        n = steps + warmup
        self.n = n
        B, S = self.B, self.S
        self.quant = spec.get("quant")
        pk, pv = wl.code_cache(sh, seed, self.quant, B=self.B) if self.quant else wl.cache(sh, seed, B=self.B)
        self.ks = torch.tensor([0.02 if self.quant == "i8" else 0.01], dtype=torch.float32, device=self.dev)
        self.vs = torch.tensor([0.025 if self.quant == "i8" else 0.005], dtype=torch.float32, device=self.dev)
        self.pk, self.pv = pk.to(self.dev), pv.to(self.dev)
        del pk, pv
        # a separate present buffer: the two caches alternate as past and present
        self.separate = bool(spec.get("separate"))
        self.pk2 = torch.empty_like(self.pk) if self.separate else self.pk
        self.pv2 = torch.empty_like(self.pv) if self.separate else self.pv
        T0 = wl.lengths(B, spec["lo"], spec["hi"], seed)
        # per-step pre-step lengths (decode: +1; verify: + accepted; prefill: +S)
        Ts = [T0.copy()]
        for t in range(n):
            if spec["accept"]:
                Ts.append(Ts[-1] + wl.accepted(B, S, seed * 1000 + t))
            else:
                Ts.append(Ts[-1] + S)
        self.T = np.stack(Ts[:n])  # (n, B) lengths before each step
        seq = (self.T + S - 1).astype(np.int32)
        self.seq_host = torch.from_numpy(seq).pin_memory()
        self.seq = self.seq_host.to(self.dev)
        self.totals = [int(self.T[t].max()) + S for t in range(n)]
        nin = 4
        ins = [wl.step_inputs(sh, S, seed * 100 + i, B=B) for i in range(nin)]
        self.q_host = [x[0].pin_memory() for x in ins]
        self.k_host = [x[1].pin_memory() for x in ins]
        self.v_host = [x[2].pin_memory() for x in ins]
        self.q = [x.to(self.dev) for x in self.q_host]
        self.k = [x.to(self.dev) for x in self.k_host]
        self.v = [x.to(self.dev) for x in self.v_host]
        self.out = torch.empty_like(self.q[0])
        self.out_host = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.bias = None
        self.bias_strides = None
        if spec["bias"]:
            TM = max(self.totals)
            self.bias = wl.bias(B, sh.Nq, S, TM, seed).to(self.dev)
            self.bias_strides = (sh.Nq * S * TM, S * TM, TM)
        self.head_sink = wl.head_sink(sh.Nq, seed).to(self.dev) if spec.get("sink") else None
        self.cos = self.sin = None
        if spec.get("rope"):
            self.cos, self.sin = (x.to(self.dev) for x in wl.rope_tables(int(self.T.max()) + S + 1, sh.D // 2,
                                                                          sh.dtype))
        self.split_keys = split_keys
        self.args = []
        ws_bytes = 0
        for t in range(n):
            a = self._args(t, None)
            ws_bytes = max(ws_bytes, gqaw.gqaw_workspace_bytes(a))
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=self.dev)
        gqaw.check(gqaw.gqaw_workspace_init(int(self.ws.data_ptr()), ws_bytes, self.stream.cuda_stream))
        self.args = [self._args(t, self.ws) for t in range(n)]

    def caches(self, t):
        """(past_key, past_value, present_key, present_value) of step t."""
        if t % 2 == 0:
            return self.pk, self.pv, self.pk2, self.pv2
        return self.pk2, self.pv2, self.pk, self.pv

    def _args(self, t, ws):
        i = t % len(self.q)
        sh = self.sh
        return self.gqaw.make_args(
            self.q[i], self.k[i], self.v[i], *self.caches(t), self.seq[t], self.totals[t],
            sh.Nq, sh.Nkv, sh.W, self.out, workspace=ws, softcap=sh.softcap, attention_bias=self.bias,
            bias_strides=self.bias_strides, split_keys=self.split_keys, head_sink=self.head_sink,
            cos_cache=self.cos, sin_cache=self.sin, k_scale=self.ks, v_scale=self.vs)

    def step(self, t):
        self.gqaw.check(self.gqaw.gqa_windowed_step(self.args[t], self.stream.cuda_stream))

    def step_phases(self, t, ev_mid):
        g = self.gqaw
        g.check(g.gqaw_attend(self.args[t], self.stream.cuda_stream))
        ev_mid.record(self.stream)
        g.check(g.gqaw_update_cache(self.args[t], self.stream.cuda_stream))

    def step_e2e(self, t):
        """One step through the C ABI from pinned host buffers: copy the step's query,
        key, value and seqlens_k in, run the step, copy the output back.  The copies run
        on their own streams (one for input, one for read-back) into one of two device
        slots, so those of step t + 1 overlap the kernels of step t (what a serving loop
        does); events keep each slot's copies, kernels and read-back in order."""
        torch = self.torch
        s, i, cs = t % 2, t % len(self.q), self.cstream
        cs.wait_event(self.ev_done[s])  # step t - 2's kernels have read this slot
        with torch.cuda.stream(cs):
            self.q_e[s].copy_(self.q_host[i], non_blocking=True)
            self.k_e[s].copy_(self.k_host[i], non_blocking=True)
            self.v_e[s].copy_(self.v_host[i], non_blocking=True)
            self.seq[t].copy_(self.seq_host[t], non_blocking=True)
            self.ev_in[s].record(cs)
        self.stream.wait_event(self.ev_in[s])
        self.stream.wait_event(self.ev_out[s])  # step t - 2's output has been read back
        self.gqaw.check(self.gqaw.gqa_windowed_step(self.args_e2e[t], self.stream.cuda_stream))
        self.ev_done[s].record(self.stream)
        ds = self.dstream
        ds.wait_event(self.ev_done[s])
        with torch.cuda.stream(ds):
            self.out_host_e[s].copy_(self.out_e[s], non_blocking=True)
            self.ev_out[s].record(ds)

    def end_e2e(self):
        """The launching stream waits for the last read-backs (end of the timed region)."""
        for s in range(2):
            self.stream.wait_event(self.ev_out[s])

    def prepare_e2e(self):
        torch = self.torch
        sh = self.sh
        self.cstream = torch.cuda.Stream()  # host-to-device copies
        self.dstream = torch.cuda.Stream()  # device-to-host read-back
        self.q_e = [torch.empty_like(self.q[0]) for _ in range(2)]
        self.k_e = [torch.empty_like(self.k[0]) for _ in range(2)]
        self.v_e = [torch.empty_like(self.v[0]) for _ in range(2)]
        self.out_e = [torch.empty_like(self.out) for _ in range(2)]
        self.out_host_e = [torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory() for _ in range(2)]
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_done = [torch.cuda.Event() for _ in range(2)]
        self.ev_out = [torch.cuda.Event() for _ in range(2)]
        for e in self.ev_done + self.ev_out:
            e.record(self.stream)
        self.args_e2e = [self.gqaw.make_args(
            self.q_e[t % 2], self.k_e[t % 2], self.v_e[t % 2], *self.caches(t), self.seq[t],
            self.totals[t], sh.Nq, sh.Nkv, sh.W, self.out_e[t % 2], workspace=self.ws, softcap=sh.softcap,
            attention_bias=self.bias, bias_strides=self.bias_strides, split_keys=self.split_keys,
            head_sink=self.head_sink, cos_cache=self.cos, sin_cache=self.sin, k_scale=self.ks, v_scale=self.vs)
            for t in range(self.n)]
        e = self.q_host[0].element_size()
        self.h2d = (self.q_host[0].numel() + self.k_host[0].numel() + self.v_host[0].numel()) * e + self.B * 4
        self.d2h = self.out.numel() * self.out.element_size()


def run_gpu(args, rank, world):
    import torch

    import workloads as wl  # noqa: F401
    from sliding_window_gqa_02_gb300 import build, gqaw

    build.build()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    name = args.workload
    K, Wm = args.steps, args.warmup
    h = Harness(name, K, Wm, seed=11 + rank, split_keys=args.split_keys, batch=args.batch)
    if args.no_graph:
        h.spec["graph"] = False
    stream = h.stream
    torch.cuda.synchronize()
    torch.cuda.set_stream(stream)

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.5)

    for t in range(Wm):
        h.step(t)
    torch.cuda.synchronize()
    _barrier(world)

    graph = None
    launches0 = gqaw.gqaw_launch_count()
    if h.spec["graph"]:
        # small, launch-bound workloads: the K steps are captured once as a CUDA graph
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for t in range(Wm, Wm + K):
                h.step(t)
        torch.cuda.synchronize()
        launches = gqaw.gqaw_launch_count() - launches0  # the kernels one replay launches
        graph.replay()  # the first replay uploads the graph: untimed
        torch.cuda.synchronize()

    def headline_pass():
        """K whole steps back to back (a graph replay for the launch-bound workloads; else
        stream launches, the kernels of a step overlapping their launch through
        programmatic dependent launch).  Re-running the step indices on the advanced
        cache does the same work per step."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for t in range(Wm, Wm + K):
                h.step(t)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    def phase_pass():
        """The same K steps with an event between the attention and the cache update:
        each attention launch timed alone (no overlap with its neighbours)."""
        ea = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        em = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        for j, t in enumerate(range(Wm, Wm + K)):
            ea[j].record(stream)
            h.step_phases(t, em[j])
        torch.cuda.synchronize()
        return statistics.mean(ea[j].elapsed_time(em[j]) for j in range(K))

    # Repeat the K-step pass until at least half a second has run (every rank runs the
    # same number of passes); the median pass is the reported one.
    t_wall0 = time.time()
    passes = [headline_pass()]
    if graph is None:
        launches = gqaw.gqaw_launch_count() - launches0
    n_pass = int(min(5000, max(5, math.ceil(500.0 / max(passes[0], 1e-3)))))
    n_pass = int(_max_over_ranks(n_pass, world))
    attend_ms = []
    for i in range(1, n_pass):
        passes.append(headline_pass())
        if graph is None and i % 2 == 1:
            attend_ms.append(phase_pass())
    t_wall1 = time.time()
    clocks.stop()
    check_device(h, name)
    med = statistics.median(passes)
    total_ms = _max_over_ranks(med, world)

    sh, B, S = h.sh, h.B, h.S
    tokens = B * S * K * world
    value = tokens / (total_ms / 1e3)
    peak, peak_src = measured_peaks()
    att_bytes = step_bytes = 0.0
    bias_bytes = 0.0
    for t in range(Wm, Wm + K):
        a, s = algorithmic_bytes(sh, S, h.T[t], B, 1 if h.quant else None, h.separate, h.quant)
        att_bytes += a
        step_bytes += s
        if h.bias is not None:
            bias_bytes += 4 * sh.Nq * visible_columns(S, h.T[t], sh.W)
    att_bytes += bias_bytes
    step_bytes += bias_bytes
    qs = sorted(passes)
    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": workload_config(name, B),
        "timing": {
            "passes": n_pass, "reported": "median of %d passes of K=%d steps, max over ranks" % (n_pass, K),
            "pass_ms_median": med, "pass_ms_min": qs[0], "pass_ms_max": qs[-1],
            "pass_ms_p10": qs[len(qs) // 10], "pass_ms_p90": qs[(9 * len(qs)) // 10],
            "window_s": t_wall1 - t_wall0,
            "l2": "no flush: K/V window per step %.0f MB > 129 MB L2" % (step_bytes / K / 1e6)
            if step_bytes / K > 129e6 else "CUDA-graph replay, working set L2-resident",
            "launch": "CUDA graph of K steps" if graph is not None else "stream launches",
            "parallelism": "replicas x%d" % world},
        "gpu_launches": launches,
        "clocks": clocks.summary(t_wall0, t_wall1),
        "cache_events": events_summary(sh, S, [h.T[t] for t in range(Wm, Wm + K)]),
    }
    step_gbs = step_bytes / (total_ms / 1e3) / 1e9
    result["step_hbm"] = {"achieved_gbs": step_gbs, "frac_of_peak": step_gbs / peak, "peak_gbs": peak,
                          "peak_source": peak_src, "bytes_per_step": step_bytes / K}
    if attend_ms:
        am = statistics.median(attend_ms)
        kern = attention_kernel(sh, S, h.quant)
        # a committed figure is for the workload's own batch; another batch has none
        traffic = profiled_traffic(name, kern) if not args.batch else None
        timing_note = ("median over %d passes of the mean CUDA-event time of the attention launch, each launch "
                       "timed alone (an event on each side: no overlap with the neighbouring kernels); "
                       "avg_step_ms is the headline's whole step" % len(attend_ms))
        if kern == "mma":  # multi-token steps on the tensor-core kernel: tensor bound
            flops = sum(step_flops(sh, S, h.T[t]) for t in range(Wm, Wm + K)) / K
            ach = flops / (am / 1e3) / 1e12
            tpk = bf16_peak_tflops()
            result["roofline"] = {"kernel": KERNELS[kern][0], "bound": "tensor", "achieved": ach, "peak": tpk,
                                  "unit": "TFLOP/s", "frac": ach / tpk, "traffic": traffic,
                                  "algorithmic_flops_per_launch": flops, "avg_launch_ms": am,
                                  "avg_step_ms": total_ms / K, "timing": timing_note,
                                  "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)"}
        else:
            ach = att_bytes / K / (am / 1e3) / 1e9
            result["roofline"] = {"kernel": KERNELS[kern][0], "bound": "hbm", "achieved": ach, "peak": peak,
                                  "unit": "GB/s", "frac": ach / peak, "traffic": traffic,
                                  "algorithmic_bytes_per_launch": att_bytes / K, "avg_launch_ms": am,
                                  "avg_step_ms": total_ms / K, "timing": timing_note,
                                  "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs, burst copy)"}
    # end-to-end through the C ABI with host buffers (the e2e passes re-run the same
    # step indices on the advanced cache: the step function is defined for any buffer)
    h.prepare_e2e()
    for t in range(min(Wm, 3)):
        h.step_e2e(t)
    torch.cuda.synchronize()

    def e2e_pass():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        h.cstream.wait_event(e0)  # no copy of the timed steps starts before the timed region
        for t in range(Wm, Wm + K):
            h.step_e2e(t)
        h.end_e2e()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    e2e_passes = [e2e_pass()]
    n_e2e = int(_max_over_ranks(int(min(2000, max(3, math.ceil(250.0 / max(e2e_passes[0], 1e-3))))), world))
    for _ in range(1, n_e2e):
        e2e_passes.append(e2e_pass())
    e2e_ms = _max_over_ranks(statistics.median(e2e_passes), world)
    check_device(h, name + " (e2e)")
    result["e2e"] = {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h.h2d,
                     "d2h_bytes_per_step": h.d2h, "ms_per_step": e2e_ms / K, "passes": n_e2e}
    torch.cuda.set_stream(torch.cuda.default_stream())
    del h
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        result["cpu_baseline"] = cpu_baseline(name, budget_s=args.cpu_seconds)
    if rank == 0 and not args.no_extra:
        result["workloads"] = extra_workloads(name, args)
    return result


def extra_workloads(main, args):
    """Short measurements of the other workloads (context; not the headline)."""
    import torch

    out = {}
    for name in ("pages-decode", "slack-decode", "verify4", "verify8", "longctx-prefill", "longctx-decode-modeA",
                 "longctx-decode-sink",
                 "longctx-decode-rope", "longctx-prefill-rope", "longctx-decode-i8", "longctx-decode-e4m3"):
        if name == main:
            continue
        K = 8 if name.startswith("longctx-prefill") else 64
        Wm = 3
        h = Harness(name, K, Wm, seed=5)
        torch.cuda.synchronize()
        torch.cuda.set_stream(h.stream)
        for t in range(Wm):
            h.step(t)
        torch.cuda.synchronize()
        if h.spec["graph"]:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=h.stream):
                for t in range(Wm, Wm + K):
                    h.step(t)
            torch.cuda.synchronize()
            g.replay()  # the first replay uploads the graph: untimed
            torch.cuda.synchronize()
        passes = []
        for _ in range(5):  # the median of five passes of K steps
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(h.stream)
            if h.spec["graph"]:
                g.replay()
            else:
                for t in range(Wm, Wm + K):
                    h.step(t)
            e1.record(h.stream)
            torch.cuda.synchronize()
            passes.append(e0.elapsed_time(e1) / K)
        check_device(h, name)
        ms = statistics.median(passes)
        _, sb = algorithmic_bytes(h.sh, h.S, h.T[Wm], h.B, 1 if h.quant else None, h.separate, h.quant)
        if h.bias is not None:
            sb += 4 * h.sh.Nq * visible_columns(h.S, h.T[Wm], h.sh.W)
        hbm, _ = measured_peaks()
        entry = {"ms_per_step": ms, "tokens_per_s": h.B * h.S / (ms / 1e3),
                 "step_gbs": sb / (ms / 1e3) / 1e9, "hbm_frac": sb / (ms / 1e3) / 1e9 / hbm,
                 "B": h.B, "S": h.S, "cache_dtype": h.sh.dtype,
                 "launch": "CUDA graph" if h.spec["graph"] else "stream",
                 "cache_events": events_summary(h.sh, h.S, [h.T[t] for t in range(Wm, Wm + K)])}
        if h.S > 1:
            flops = step_flops(h.sh, h.S, h.T[Wm])
            entry["tflops"] = flops / (ms / 1e3) / 1e12
            entry["tensor_frac"] = entry["tflops"] / bf16_peak_tflops()
        entry["kernel"] = KERNELS[attention_kernel(h.sh, h.S, h.quant)][0]
        out[name] = entry
        torch.cuda.synchronize()
        torch.cuda.set_stream(torch.cuda.default_stream())
        del h
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ CPU oracle (baseline / reference arm)


_ORACLE_INPUTS = {}


def oracle_item_step(name, seed, b_items, t_index=0):
    """Run the oracle on items ``b_items`` of one step of ``name``; returns seconds."""
    import oracle
    import workloads as wl

    spec = workload_spec(name)
    sh = spec["shape"]
    B = spec.get("B", sh.B)
    S = spec["S"]
    T0 = wl.lengths(B, spec["lo"], spec["hi"], seed) + t_index * S
    key = ("inputs", name, seed, t_index % 4)
    if key not in _ORACLE_INPUTS:
        q, k, v = wl.step_inputs(sh, S, seed * 100 + (t_index % 4), B=B)
        _ORACLE_INPUTS[key] = (wl.to_numpy(q), wl.to_numpy(k), wl.to_numpy(v))
    nq, nk, nv = _ORACLE_INPUTS[key]
    odt = oracle.F32 if sh.dtype == wl.F32 else oracle.BF16
    el = 0.0
    for b in b_items:
        ckey = ("cache", name, seed, b % 8)  # eight distinct caches serve every item: timing only
        if ckey not in _ORACLE_INPUTS:
            pk, pv = (wl.code_cache(sh, seed * 7919 + b % 8, spec["quant"], B=1) if spec.get("quant")
                      else wl.cache(sh, seed * 7919 + b % 8, B=1))
            _ORACLE_INPUTS[ckey] = (wl.to_numpy(pk), wl.to_numpy(pv))
        npk, npv = _ORACLE_INPUTS[ckey]
        seq = (T0[b:b + 1] + S - 1).astype(np.int32)
        total = int(seq.max()) + 1
        bias = None
        if spec["bias"]:
            bias = wl.to_numpy(wl.bias(1, sh.Nq, S, total, seed + b))
        sink = wl.to_numpy(wl.head_sink(sh.Nq, seed)) if spec.get("sink") else None
        rope = {}
        if spec.get("rope"):
            cos, sin = wl.rope_tables(int(seq.max()) + 1, sh.D // 2, sh.dtype)
            rope = dict(cos_cache=wl.to_numpy(cos), sin_cache=wl.to_numpy(sin))
        t0 = time.perf_counter()
        quant = {}
        if spec.get("quant"):
            quant = dict(cache_dtype=oracle.I8 if spec["quant"] == "i8" else oracle.E4M3,
                         k_scale=0.02 if spec["quant"] == "i8" else 0.01,
                         v_scale=0.025 if spec["quant"] == "i8" else 0.005)
        oracle.step(nq[b:b + 1], nk[b:b + 1], nv[b:b + 1], npk, npv, seq, total, sh.Nq, sh.Nkv, sh.W,
                    softcap=sh.softcap, attention_bias=bias, dtype=odt, head_sink=sink, **rope, **quant)
        el += time.perf_counter() - t0
    return el


def _oracle_worker(task):
    """One process of the parallel CPU baseline: item-steps of the oracle, timed."""
    name, seed, items = task
    el = 0.0
    for b, t in items:
        el += oracle_item_step(name, seed, [b], t)
    return el, len(items)


def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def oracle_parallel(name, item_steps, cores, seed=11):
    """The oracle as it stands on ``cores`` host cores: ``item_steps`` ((item, step)
    pairs, independent) dealt out to that many spawned processes (spawn: the parent
    holds a CUDA context); returns (oracle seconds of the slowest process, item-steps)."""
    import multiprocessing as mp

    chunks = [item_steps[c::cores] for c in range(cores)]
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_oracle_worker, [(name, seed, ch) for ch in chunks if ch], chunksize=1)
    return max(r[0] for r in res), sum(r[1] for r in res)


def cpu_baseline(name, budget_s=15.0):
    """The oracle as it stands on items of the same workload: on every host core (item-steps
    dealt out to spawned processes, about ``budget_s`` seconds each; tokens/s = tokens
    computed / the slowest process's oracle time) and, beside it, on one thread."""
    spec = workload_spec(name)
    B = spec.get("B", spec["shape"].B)
    S = spec["S"]
    done, el = 0, 0.0
    while el < budget_s / 3 and done < 64 * B:  # single thread: item after item, step after step
        el += oracle_item_step(name, 11, [done % B], done // B)
        done += 1
    single = done * S / el
    cores = host_cores()
    per = max(1, int(budget_s / max(el / done, 1e-6)))
    pairs = [(i % B, i // B) for i in range(cores * per)]
    pel, n = oracle_parallel(name, pairs, cores)
    return {"value": n * S / pel, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "%d item-steps of %s (%d items per step, %d token(s) each), fp64 C oracle, %d processes "
                      "x ~%.1f s" % (n, name, B, S, cores, pel),
            "single_thread": {"value": single, "cores": 1,
                              "sample": "%d item-steps, 1 thread, %.1f s" % (done, el)}}


def run_reference(args):
    """The reference arm: the oracle on every host core, each step a bounded sample of its
    items dealt out to spawned processes (step time = the slowest process's oracle time)."""
    spec = workload_spec(args.workload)
    B = spec.get("B", spec["shape"].B)
    S = spec["S"]
    K, Wm = args.steps, args.warmup
    cores = host_cores()
    t_item = oracle_item_step(args.workload, 11, [0])
    per_step = max(1, min(B, int(120.0 * cores / max(K + Wm, 1) / max(t_item, 1e-6))))
    for t in range(Wm):
        oracle_item_step(args.workload, 11, [(t * per_step) % B], t)
    pairs = [(((Wm + t) * per_step + j) % B, Wm + t) for t in range(K) for j in range(per_step)]
    el, n = oracle_parallel(args.workload, pairs, cores)
    tokens = n * S
    value = tokens / el
    sample = "%d of %d items per step, %d steps, fp64 C oracle, %d processes" % (per_step, B, K, cores)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": K,
            "warmup": Wm, "ms_per_step": el / K * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, B),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ distributed helpers


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if not dist.is_initialized():
            backend = os.environ.get("GQAW_DIST_BACKEND", "nccl")
            if backend == "nccl":
                import torch

                torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
            dist.init_process_group(backend)
    return rank, world


def _barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def _max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gqaw", choices=["gqaw", "reference"])
    ap.add_argument("--workload", default="longctx-decode")
    ap.add_argument("--split-keys", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch size (profiling)")
    ap.add_argument("--no-graph", action="store_true", help="launch every step from the host (no CUDA graph)")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    rank, world = _dist()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    res = run_gpu(args, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
