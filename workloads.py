"""Seeded synthetic inputs shaped like the workloads of the windowed-GQA pages.

This module only draws random numbers and describes shapes.  It holds none of the
step's arithmetic (no resident-length formula, no attention), so both the oracle
side and the CUDA side of a test can take their inputs from here.

Every draw comes from a CPU ``torch.Generator`` seeded explicitly, so a test and the
benchmark see the same bits on every machine.  bfloat16 tensors are drawn in
float32 and rounded once by torch (round to nearest even).

Workloads (PR #31142 "[CPU] Add windowed kv cache for GQA", Performance Results and
Tests; PR #32419 "Specify GroupQueryAttention windowed KV cache layout contract",
New tests):

``tiny``      B=1, Nq=2, Nkv=1, D=8, fp32, C=6, W=4; U[-1,1] values
``pages``     B=1, Nq=64, Nkv=8, D=64, fp32, W=128, C=384; N(0,1) values
``slack``     B=8, Nq=32, Nkv=8, D=128, bf16, W=128, C=136; N(0,1) values
``verify``    B=16, Nq=32, Nkv=8, D=128, bf16, W=4096, C=W+S-1, S in {4, 8};
              softcap 30, fp32 attention_bias ~ N(0, 0.5)
``longctx``   B=64, Nq=32, Nkv=8, D=128, bf16, W=4096, C=5120; contexts U[4096, 32768]
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

F32 = "f32"
BF16 = "bf16"

TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}


@dataclass(frozen=True)
class Shape:
    """Static sizes of one windowed GQA layer."""

    name: str
    B: int
    Nq: int
    Nkv: int
    D: int
    W: int
    C: int
    dtype: str
    softcap: float = 0.0
    dist: str = "normal"  # "normal" N(0,1) or "uniform" U[-1,1]
    extra: dict = field(default_factory=dict)


SHAPES = {
    "tiny": Shape("tiny", B=1, Nq=2, Nkv=1, D=8, W=4, C=6, dtype=F32, dist="uniform"),
    "pages": Shape("pages", B=1, Nq=64, Nkv=8, D=64, W=128, C=384, dtype=F32),
    "slack": Shape("slack", B=8, Nq=32, Nkv=8, D=128, W=128, C=136, dtype=BF16),
    "verify4": Shape("verify4", B=16, Nq=32, Nkv=8, D=128, W=4096, C=4096 + 4 - 1, dtype=BF16,
                     softcap=30.0, extra={"S": 4, "T0": 6000}),
    "verify8": Shape("verify8", B=16, Nq=32, Nkv=8, D=128, W=4096, C=4096 + 8 - 1, dtype=BF16,
                     softcap=30.0, extra={"S": 8, "T0": 6000}),
    "longctx": Shape("longctx", B=64, Nq=32, Nkv=8, D=128, W=4096, C=5120, dtype=BF16,
                     extra={"T_lo": 4096, "T_hi": 32768, "prefill_items": 8, "prefill_S": 512}),
}


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def draw(shape, dtype: str, seed: int, dist: str = "normal", std: float = 1.0) -> torch.Tensor:
    """A CPU tensor of ``shape`` with N(0, std^2) or U[-1, 1] entries, in ``dtype``."""
    g = generator(seed)
    if dist == "normal":
        t = torch.randn(tuple(shape), generator=g, dtype=torch.float32) * std
    elif dist == "uniform":
        t = torch.rand(tuple(shape), generator=g, dtype=torch.float32) * 2.0 - 1.0
    else:
        raise ValueError(dist)
    return t.to(TORCH_DTYPE[dtype])


def step_inputs(sh: Shape, S: int, seed: int, B: int | None = None):
    """Query/key/value of one step: (B,S,Nq*D), (B,S,Nkv*D), (B,S,Nkv*D)."""
    B = sh.B if B is None else B
    q = draw((B, S, sh.Nq * sh.D), sh.dtype, seed * 3 + 0, sh.dist)
    k = draw((B, S, sh.Nkv * sh.D), sh.dtype, seed * 3 + 1, sh.dist)
    v = draw((B, S, sh.Nkv * sh.D), sh.dtype, seed * 3 + 2, sh.dist)
    return q, k, v


def cache(sh: Shape, seed: int, B: int | None = None, capacity: int | None = None):
    """A (B, Nkv, C, D) key cache and value cache with every row drawn at random.

    A cache "seeded at length T" needs nothing more: the layout contract fixes only
    rows [0, L(T)), and any content is a valid past for the step function."""
    B = sh.B if B is None else B
    C = sh.C if capacity is None else capacity
    k = draw((B, sh.Nkv, C, sh.D), sh.dtype, seed * 2 + 100001, sh.dist)
    v = draw((B, sh.Nkv, C, sh.D), sh.dtype, seed * 2 + 100002, sh.dist)
    return k, v


def bias(B: int, Nq: int, S: int, total: int, seed: int, std: float = 0.5) -> torch.Tensor:
    """fp32 attention_bias (B, Nq, S, total) ~ N(0, std^2)."""
    return draw((B, Nq, S, total), F32, seed + 200003, "normal", std)


def head_sink(Nq: int, seed: int, mean: float = 0.0, std: float = 2.0) -> torch.Tensor:
    """fp32 sink logits (Nq,) ~ N(mean, std^2), one per query head."""
    return draw((Nq,), F32, seed + 400009, "normal", std) + mean


def rope_tables(max_pos: int, half: int, dtype: str, base: float = 10000.0):
    """cos/sin caches (max_pos, half) of the usual rotary angles pos * base^(-i/half),
    computed in float64 and rounded once to ``dtype``: inputs of the step, as a model
    would supply them."""
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * base ** (
        -torch.arange(half, dtype=torch.float64)[None, :] / half)
    td = TORCH_DTYPE[dtype]
    return torch.cos(ang).to(td).contiguous(), torch.sin(ang).to(td).contiguous()


def code_cache(sh: Shape, seed: int, cache_dtype: str, B: int | None = None):
    """Random quantized-cache contents (B, Nkv, C, D): int8 codes ~ U{-100..100}, or fp8
    e4m3 codes drawn as bytes with the two NaN codes replaced by zero."""
    B = sh.B if B is None else B
    g = generator(seed + 500009)
    shape = (B, sh.Nkv, sh.C, sh.D)
    out = []
    for _ in range(2):
        if cache_dtype == "i8":
            out.append(torch.randint(-100, 101, shape, generator=g, dtype=torch.int8))
        else:
            c = torch.randint(0, 256, shape, generator=g, dtype=torch.int16).to(torch.uint8)
            c[(c == 0x7F) | (c == 0xFF)] = 0
            out.append(c.view(torch.float8_e4m3fn))
    return out[0], out[1]


def lengths(B: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Per-item token counts T_b ~ U{lo..hi} (inclusive), int64."""
    rng = np.random.Generator(np.random.Philox(seed + 300007))
    return rng.integers(lo, hi + 1, size=B, dtype=np.int64)


def accepted(B: int, S: int, seed: int) -> np.ndarray:
    """Accepted draft counts k_b ~ U{0..S} for a speculative verify step."""
    rng = np.random.Generator(np.random.Philox(seed + 400009))
    return rng.integers(0, S + 1, size=B, dtype=np.int64)


def to_numpy(t: torch.Tensor) -> np.ndarray:
    """Host array for the oracle: float32 as is, bfloat16 as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype == torch.int32:
        return t.numpy()
    if t.dtype == torch.int8 or str(t.dtype) == "torch.float8_e4m3fn":  # quantized-cache codes
        return t.view(torch.uint8).numpy()
    raise TypeError(t.dtype)


def from_numpy(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Inverse of :func:`to_numpy`."""
    if dtype == BF16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))
