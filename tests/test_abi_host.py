"""The C-ABI library without a GPU: it builds, loads, exports every declared symbol,
its pure host functions agree with the oracle, and malformed arguments are rejected
on the host before anything is enqueued."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sliding_window_gqa_02_gb300 import build, gqaw

    build.build()
    return gqaw


def _declared():
    src = open(os.path.join(ROOT, "include", "gqaw.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(gqaw?_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "gqa_windowed_step" in names and len(names) >= 10
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(so, n), n
    assert sorted(lib.EXPORTED) == names


def test_struct_layout_matches(lib):
    lib.load()  # raises on a size mismatch
    assert lib.load().gqaw_step_args_size() == ctypes.sizeof(lib.gqaw_step_args)


def test_resident_len_and_rollback_agree_with_oracle(lib):
    for C in range(1, 14):
        for W in range(1, C + 1):
            for T in list(range(0, 4 * C)) + [2**31 - 1, 2**35 + 3]:
                assert lib.gqaw_resident_len(T, C, W) == oracle.resident_len(T, C, W)
                for k in range(0, min(T, 6) + 1):
                    exact = oracle.resident_len(T - k, C, W) == oracle.resident_len(T, C, W) - k
                    assert lib.gqaw_rollback_exact(T, k, C, W) == int(exact)
    assert lib.gqaw_resident_len(-1, 4, 2) == -1
    assert lib.gqaw_resident_len(3, 4, 5) == -1
    assert lib.gqaw_rollback_exact(3, 4, 8, 4) == -1


FAKE = 1 << 20  # a 16-byte-aligned non-null address: these tests never reach the device


def _args(lib, **over):
    a = lib.gqaw_step_args()
    base = dict(batch_size=2, sequence_length=1, num_heads=8, kv_num_heads=2, head_size=64, capacity=40,
                local_window_size=32, dtype=lib.GQAW_BF16, total_sequence_length=50)
    base.update({k: v for k, v in over.items() if not k.startswith("p_")})
    for k, v in base.items():
        setattr(a, k, v)
    # disjoint fake device buffers, 1 MiB apart
    ptrs = ["query", "key", "value", "past_key", "past_value", "present_key", "present_value", "seqlens_k",
            "output", "workspace"]
    for i, n in enumerate(ptrs):
        setattr(a, n, FAKE * (i + 1) * 16)
    a.workspace_bytes = 1 << 20
    for k, v in over.items():
        if k.startswith("p_"):
            setattr(a, k[2:], v)
    return a


def test_workspace_bytes(lib):
    a = _args(lib)
    n = lib.gqaw_workspace_bytes(a)
    assert n >= 256 and n % 256 == 0
    assert lib.gqaw_workspace_bytes(_args(lib, head_size=96)) == 0
    assert "head_size 96" in lib.gqaw_last_error()
    # fewer, longer attention ranges need fewer partial-result slots
    big = _args(lib, batch_size=64, local_window_size=40, total_sequence_length=5000)
    assert lib.gqaw_workspace_bytes(_args(lib, batch_size=64, local_window_size=40, total_sequence_length=5000,
                                          split_keys=100000)) < lib.gqaw_workspace_bytes(big)


@pytest.mark.parametrize("over,status,msg", [
    (dict(sequence_length=0), 1, "sequence_length"),
    (dict(batch_size=-1), 1, "batch_size"),
    (dict(num_heads=6, kv_num_heads=4), 1, "multiple"),
    (dict(head_size=96), 2, "head_size"),
    (dict(local_window_size=41), 1, "local_window_size"),
    (dict(local_window_size=0), 1, "local_window_size"),
    (dict(capacity=0, local_window_size=0), 1, "capacity"),
    (dict(dtype=7), 1, "dtype"),
    (dict(total_sequence_length=0), 1, "total_sequence_length"),
    (dict(scale=-1.0), 1, "scale"),
    (dict(softcap=float("inf")), 1, "softcap"),
    (dict(split_keys=-3), 1, "split_keys"),
    (dict(p_query=0), 1, "query is NULL"),
    (dict(p_seqlens_k=0), 1, "seqlens_k is NULL"),
    (dict(p_key=FAKE * 16 * 2 + 8), 1, "key is not 16-byte aligned"),
    (dict(p_workspace=0), 4, "workspace is NULL"),
    (dict(p_workspace=FAKE * 160 + 64), 4, "256-byte"),
    (dict(p_workspace_bytes=16), 4, "workspace_bytes"),
    (dict(p_present_key=FAKE * 16 * 4 + 4096), 1, "overlaps"),
    (dict(p_output=FAKE * 16 * 1), 1, "overlaps"),
    (dict(p_attention_bias=FAKE * 300 + 2), 1, "attention_bias"),
    (dict(p_attention_bias=FAKE * 300, p_bias_stride_h=-1), 1, "strides"),
    (dict(p_head_sink=FAKE * 300 + 2), 1, "head_sink"),
    (dict(p_cache_dtype=5), 1, "cache_dtype"),
    (dict(p_cache_dtype=2, dtype=0), 2, "GQAW_BF16"),
    (dict(p_cache_dtype=3, head_size=32), 2, "head_size 64, 128 or 256"),
    (dict(p_cache_dtype=2), 1, "k_scale and v_scale"),
    (dict(p_cache_dtype=2, p_k_scale=FAKE * 300 + 2, p_v_scale=FAKE * 301), 1, "4-byte aligned"),
    (dict(p_do_rotary=1, p_rotary_dim=5, p_rotary_cache_len=8), 1, "rotary_dim"),
    (dict(p_do_rotary=1, p_rotary_dim=66, p_rotary_cache_len=8), 1, "rotary_dim"),
    (dict(p_do_rotary=1, p_rotary_cache_len=0), 1, "rotary_cache_len"),
    (dict(p_do_rotary=1, p_rotary_cache_len=8), 1, "cos_cache and sin_cache"),
    (dict(p_do_rotary=1, p_rotary_cache_len=8, p_cos_cache=FAKE * 300 + 1, p_sin_cache=FAKE * 301), 1,
     "2-byte aligned"),
    (dict(p_do_rotary=1, p_rotary_cache_len=8, p_cos_cache=FAKE * 300, p_sin_cache=FAKE * 301,
          p_position_ids=FAKE * 302 + 4), 1, "position_ids"),
])
def test_rejected_on_host(lib, over, status, msg):
    a = _args(lib, **over)
    for fn in (lib.gqa_windowed_step, lib.gqaw_attend, lib.gqaw_update_cache):
        assert fn(a, 0) == status
        assert msg in lib.gqaw_last_error(), lib.gqaw_last_error()


def test_rotary_workspace(lib):
    """The turned query and key rows (B*S*(Nq+Nkv)*D elements) live in the workspace."""
    plain = lib.gqaw_workspace_bytes(_args(lib, sequence_length=4))
    rot = lib.gqaw_workspace_bytes(_args(lib, sequence_length=4, p_do_rotary=1, p_rotary_cache_len=64))
    assert rot - plain >= 2 * 4 * (8 + 2) * 64 * 2


def test_empty_batch_returns_ok_without_pointers(lib):
    a = lib.gqaw_step_args()
    a.batch_size, a.sequence_length, a.num_heads, a.kv_num_heads = 0, 1, 1, 1
    a.head_size, a.capacity, a.local_window_size, a.total_sequence_length = 8, 6, 4, 1
    before = lib.gqaw_launch_count()
    assert lib.gqa_windowed_step(a, 0) == lib.GQAW_OK
    assert lib.gqaw_launch_count() == before


def test_product_path_has_no_oracle_or_fallback():
    """The package never imports the oracle, and loads only libgqaw.so."""
    pkg = os.path.join(ROOT, "sliding_window_gqa_02_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "oracle_" not in text, f
