"""Test helper: drive the CUDA library across steps, and compare with the oracle.

The CUDA side is called only through the C ABI (``sliding_window_gqa_02_gb300.gqaw``);
torch supplies device memory and the stream.  Nothing here computes any part of the
step.
"""
from __future__ import annotations

import numpy as np
import torch

import workloads as wl
from sliding_window_gqa_02_gb300 import gqaw

TOL = {wl.F32: 1e-5, wl.BF16: 2e-2}


class GpuCache:
    def __init__(self, B, Nq, Nkv, D, C, W, dtype, scale=0.0, softcap=0.0, past_key=None, past_value=None,
                 inplace=True, split_keys=0, head_sink=None, smooth_softmax=False, cos_cache=None, sin_cache=None,
                 rotary_interleaved=False, cache_dtype=None, k_scale=1.0, v_scale=1.0):
        self.dev = torch.device("cuda:0")
        self.cache_dtype = cache_dtype
        self.ks = torch.tensor([k_scale], dtype=torch.float32, device=self.dev)
        self.vs = torch.tensor([v_scale], dtype=torch.float32, device=self.dev)
        self.cos = None if cos_cache is None else cos_cache.to(self.dev).contiguous()
        self.sin = None if sin_cache is None else sin_cache.to(self.dev).contiguous()
        self.rotary_interleaved = rotary_interleaved
        self.head_sink = None if head_sink is None else head_sink.to(self.dev).contiguous()
        self.smooth_softmax = smooth_softmax
        self.B, self.Nq, self.Nkv, self.D, self.C, self.W = B, Nq, Nkv, D, C, W
        self.dtype, self.scale, self.softcap = dtype, scale, softcap
        self.inplace, self.split_keys = inplace, split_keys
        td = wl.TORCH_DTYPE[dtype]
        if cache_dtype == "i8":
            td = torch.int8
        elif cache_dtype == "e4m3":
            td = torch.float8_e4m3fn
        z = torch.zeros((B, Nkv, C, D), dtype=torch.uint8).view(td) if cache_dtype else torch.zeros((B, Nkv, C, D), dtype=td)
        self.pk = (z if past_key is None else past_key).to(self.dev).contiguous()
        self.pv = (z if past_value is None else past_value).to(self.dev).contiguous()
        if not inplace:
            # stale rows (bytes 7 throughout): must never be read
            nbytes = self.pk.element_size()
            shape = (*self.pk.shape[:-1], self.pk.shape[-1] * nbytes)
            self.rk = torch.full(shape, 7, dtype=torch.uint8, device=self.dev).view(self.pk.dtype)
            self.rv = torch.full(shape, 7, dtype=torch.uint8, device=self.dev).view(self.pv.dtype)

    def step(self, q, k, v, seqlens, total=None, bias=None, bias_strides=None, phases=False, position_ids=None):
        seqlens = np.asarray(seqlens, np.int64)
        if total is None:
            total = int(seqlens.max()) + 1
        dq, dk, dv = (t.to(self.dev).contiguous() for t in (q, k, v))
        seq = torch.tensor(seqlens.astype(np.int32), device=self.dev)
        out = torch.full_like(dq, float("nan"))
        res = torch.full((self.B,), -1, dtype=torch.int32, device=self.dev)
        dbias = None if bias is None else bias.to(self.dev)
        rk, rv = (self.pk, self.pv) if self.inplace else (self.rk, self.rv)
        kw = dict(scale=self.scale, softcap=self.softcap, attention_bias=dbias, bias_strides=bias_strides,
                  resident_len_out=res, split_keys=self.split_keys, head_sink=self.head_sink,
                  smooth_softmax=self.smooth_softmax, cos_cache=self.cos, sin_cache=self.sin,
                  rotary_interleaved=self.rotary_interleaved, k_scale=self.ks, v_scale=self.vs,
                  position_ids=None if position_ids is None else
                  torch.as_tensor(np.asarray(position_ids, np.int64)).to(self.dev).contiguous())
        args = gqaw.make_args(dq, dk, dv, self.pk, self.pv, rk, rv, seq, total, self.Nq, self.Nkv, self.W,
                              out, **kw)
        stream = torch.cuda.current_stream().cuda_stream
        ws = gqaw.new_workspace(args, self.dev, stream)
        args = gqaw.make_args(dq, dk, dv, self.pk, self.pv, rk, rv, seq, total, self.Nq, self.Nkv, self.W,
                              out, workspace=ws, **kw)
        if phases:
            gqaw.check(gqaw.gqaw_attend(args, stream))
            gqaw.check(gqaw.gqaw_update_cache(args, stream))
        else:
            gqaw.check(gqaw.gqa_windowed_step(args, stream))
        torch.cuda.synchronize()
        st, flags = gqaw.gqaw_device_status(int(ws.data_ptr()), stream=stream)
        if not self.inplace:
            self.pk, self.rk = self.rk, self.pk
            self.pv, self.rv = self.rv, self.pv
        return {
            "output": out.cpu(),
            "resident_len": res.cpu().numpy(),
            "present_key": wl.to_numpy(self.pk.cpu()),
            "present_value": wl.to_numpy(self.pv.cpu()),
            "device_flags": flags,
        }


def oracle_dtype(dtype):
    import oracle

    return oracle.F32 if dtype == wl.F32 else oracle.BF16


def _values(a, dtype):
    """Host cache array (float32, or bfloat16 bit patterns) as float64 values."""
    if dtype == wl.F32:
        return np.asarray(a, np.float32).astype(np.float64)
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _spacing(x, dtype):
    """The spacing of the cache dtype's numbers at |x| (normal range)."""
    s = np.spacing(np.abs(x).astype(np.float32)).astype(np.float64)
    return s if dtype == wl.F32 else s * 65536.0  # bfloat16 keeps 16 fewer significand bits


def codes_close(got, want, cache_dtype):
    """Key codes of a quantized cache whose keys were turned (rotary): the turn is fp32 on
    the device and fp64 in the oracle, so a code may differ by one step (adjacent codes
    of the same sign for e4m3)."""
    g, w = np.asarray(got, np.uint8), np.asarray(want, np.uint8)
    if cache_dtype == "i8":
        return bool(np.all(np.abs(g.view(np.int8).astype(np.int32) - w.view(np.int8).astype(np.int32)) <= 1))
    same_sign = (g & 0x80) == (w & 0x80)
    near = np.abs((g & 0x7F).astype(np.int32) - (w & 0x7F).astype(np.int32)) <= 1
    zero = ((g & 0x7F) == 0) & ((w & 0x7F) <= 1) | ((w & 0x7F) == 0) & ((g & 0x7F) <= 1)
    return bool(np.all((same_sign & near) | zero))


def keys_close(got, want, dtype):
    """Turned key rows (rotary embedding): the kernel turns in fp32, the oracle in fp64,
    each rounds once to the cache dtype.  Allowed: one spacing of the dtype at the
    oracle's value plus 2^-21 of the row scale (the fp32 error of x1 c - x2 s)."""
    gw, ww = _values(got, dtype), _values(want, dtype)
    if gw.size == 0:
        return True
    scale = float(np.abs(ww).max())
    return bool(np.all(np.abs(gw - ww) <= _spacing(ww, dtype) + scale * 2.0 ** -21))


def compare(gpu, ref, dtype, items=None, rows=None, check_layout=True, turned_keys=False, cache_dtype=None):
    """Assert parity: resident lengths equal, present rows [0, L_b) bit-exact for the
    given items (all by default), output within TOL relative to the output's scale
    (max |oracle|) over the given items and token rows.  Returns the output error.
    With ``turned_keys`` (rotary embedding) the present key rows are floating-point
    results and are held to ``keys_close`` instead of bit equality."""
    B = len(ref["resident_len"])
    items = list(range(B)) if items is None else list(items)
    assert gpu["device_flags"] == 0, "device status 0x%x" % gpu["device_flags"]
    for b in items:
        assert gpu["resident_len"][b] == ref["resident_len"][b], (b, gpu["resident_len"][b], ref["resident_len"][b])
        if check_layout:
            n = int(ref["resident_len"][b])
            if turned_keys and cache_dtype:
                assert codes_close(gpu["present_key"][b, :, :n], ref["present_key"][b, :, :n], cache_dtype), \
                    "present_key item %d" % b
            elif turned_keys:
                assert keys_close(gpu["present_key"][b, :, :n], ref["present_key"][b, :, :n], dtype), \
                    "present_key item %d" % b
            else:
                assert np.array_equal(gpu["present_key"][b, :, :n], ref["present_key"][b, :, :n]), \
                    "present_key item %d" % b
            assert np.array_equal(gpu["present_value"][b, :, :n], ref["present_value"][b, :, :n]), "present_value item %d" % b
    got = gpu["output"].float().numpy()[items]
    exp = ref["output_f64"][items]
    if rows is not None:
        got, exp = got[:, rows[0]:rows[1]], exp[:, rows[0]:rows[1]]
    assert np.all(np.isfinite(got)), "non-finite output"
    scale = float(np.abs(exp).max())
    err = float(np.abs(got - exp).max()) / (scale if scale > 0 else 1.0)
    assert err <= TOL[dtype], "output error %.3g > %.3g" % (err, TOL[dtype])
    return err
