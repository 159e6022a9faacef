"""The oracle's pins catch plausible mistakes (no GPU).

Each mutant below plants one mistake in a temporary copy of the oracle (its C source
or its Python marshalling) and runs ``tests/test_oracle_pins.py`` against that copy,
which must then fail.  The unmodified copy must pass, so a broken harness cannot
pass for a caught mutant.  Every mutant stays within the buffers the oracle is given
(no mistake here reads or writes out of bounds), and all of them run on the CPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
C_SRC = "oracle/gqaw_oracle.c"
PY_SRC = "oracle/__init__.py"

# name -> (file, [(old, new, occurrences of old)]); each `old` must occur exactly that
# many times, so a change of the oracle's text shows up here as a failure, not as a
# silently unapplied mutant.
MUTANTS = {
    # L(T), the drifting-layout resident count (PR #32419 Description, the formula)
    "resident_len_floor_plus_one": (C_SRC, [("blocks = (T - C + G - 1) / G;", "blocks = (T - C) / G + 1;", 1)]),
    "resident_len_block_off_by_one": (C_SRC, [("G = C - W + 1;\n  blocks", "G = C - W + 2;\n  blocks", 1)]),
    # the local window and the causal rule (PR #34226 Description; PR #32419 Description)
    "window_one_key_narrower": (C_SRC, [("int64_t jlo = i - W + 1;", "int64_t jlo = i - W + 2;", 1)]),
    "causal_excludes_own_key": (C_SRC, [("for (j = jlo; j <= i; ++j) {", "for (j = jlo; j < i; ++j) {", 2)]),
    # grouped heads: query head h reads kv head h / (Nq / Nkv)
    "head_map_modulo": (C_SRC, [("kvh = h / group;", "kvh = h % Nkv;", 1)]),
    # attention_bias in absolute key columns (PR #32419 Description)
    "bias_column_relative_to_cache": (C_SRC, [("s * a->bias_stride_s + j];", "s * a->bias_stride_s + (j - first_pos)];", 1)]),
    # softcap (mobius issue #111, Part 1.3)
    "softcap_ignored": (C_SRC, [("zj = a->softcap * tanh(zj / a->softcap);", "zj = zj;", 1)]),
    # default scale 1/sqrt(head_size) (mobius issue #111, Part 1.3)
    "default_scale_over_d": (PY_SRC, [("1.0 / math.sqrt(D)", "1.0 / D", 1)]),
    # present rows: row r holds position T - L + r (PR #32419 Description, row layout)
    "present_rows_shifted_by_one": (C_SRC, [("const int64_t xr = Lp + S - Lt + r;",
                                             "const int64_t xr = (Lp + S - Lt + r + 1) % (Lp + S);", 1)]),
    # the output's single rounding to bf16, ties to even
    "bf16_ties_away_from_zero": (C_SRC, [("r = nearbyint(ldexp(a, -q));", "r = floor(ldexp(a, -q) + 0.5);", 1)]),
    # sinks (mobius issue #111, Part 1.1 input head_sink, Part 1.3 smooth_softmax)
    "sink_one_head_for_all": (C_SRC, [("a->head_sink[h]", "a->head_sink[0]", 1)]),
    "sink_left_out_of_denominator": (C_SRC, [("denom += exp(sink - zmax);", "(void)denom;", 1)]),
    "sink_scaled_like_a_logit": (C_SRC, [("a->head_sink ? (double)a->head_sink[h] : 0.0;",
                                          "a->head_sink ? a->scale * (double)a->head_sink[h] : 0.0;", 1)]),
    # rotary embedding (mobius issue #111, Part 1.1 cos_cache / sin_cache / position_ids,
    # Part 1.3 do_rotary / rotary_interleaved)
    "rotary_turns_backwards": (C_SRC, [("y[i1] = x1 * c - x2 * sn;", "y[i1] = x1 * c + x2 * sn;", 1),
                                       ("y[i2] = x2 * c + x1 * sn;", "y[i2] = x2 * c - x1 * sn;", 1)]),
    "rotary_pairings_swapped": (C_SRC, [("a->rotary_interleaved ? 2 * i : i;", "a->rotary_interleaved ? i : 2 * i;", 1),
                                        ("a->rotary_interleaved ? 2 * i + 1 : i + half;",
                                         "a->rotary_interleaved ? i + half : 2 * i + 1;", 1)]),
    "rotary_query_one_position_late": (C_SRC, [("rotate_row(a, a->query, off, pos, qrot + off);",
                                                "rotate_row(a, a->query, off, pos + 1 < a->rotary_cache_len ? pos + 1 : pos, "
                                                "qrot + off);", 1)]),
    "rotary_positions_relative_to_step": (C_SRC, [("a->position_ids[b * S + s] : P + s;",
                                                   "a->position_ids[b * S + s] : s;", 1)]),
    "rotary_keys_stored_unturned": (C_SRC, [("ksrc = krot;", "ksrc = a->key;", 1)]),
    "rotary_cos_column_reversed": (C_SRC, [("load_elem(a->cos_cache, pos * half + i, a->dtype);",
                                            "load_elem(a->cos_cache, pos * half + (half - 1 - i), a->dtype);", 1)]),
    # quantized cache (mobius issue #111, Part 1.1 k_scale / v_scale)
    "int8_ties_half_up": (C_SRC, [("return (uint8_t)(int8_t)(int)nearbyintf(q);",
                                   "return (uint8_t)(int8_t)(int)floorf(q + 0.5f);", 1)]),
    "e4m3_subnormal_ties_half_up": (C_SRC, [("r = (int)nearbyint(ldexp(a, 9));", "r = (int)floor(ldexp(a, 9) + 0.5);", 1)]),
    "e4m3_exponent_bias_8": (C_SRC, [("return sign * ldexp(1.0 + m / 8.0, e - 7);",
                                      "return sign * ldexp(1.0 + m / 8.0, e - 8);", 1)]),
    "keys_read_with_value_scale": (C_SRC, [("load_kv(a, kb, koff + d, a->k_scale);", "load_kv(a, kb, koff + d, a->v_scale);", 1)]),
    "attention_reads_unquantized_new_keys": (C_SRC, [("qrot, quant ? (const void *)knew : ksrc,", "qrot, ksrc,", 1)]),
}

# what the pins need besides the oracle itself
_COPY = ["oracle/gqaw_oracle.c", "oracle/__init__.py", "tests/conftest.py", "tests/test_oracle_pins.py",
         "tests/oracle_driver.py", "workloads.py"]


def _run(name):
    """Copy, mutate (unless `name` is None) and run the pins; returns (returncode, tail)."""
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        for rel in _COPY:
            os.makedirs(os.path.dirname(os.path.join(tmp, rel)) or tmp, exist_ok=True)
            shutil.copy(os.path.join(ROOT, rel), os.path.join(tmp, rel))
        shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(tmp, "tests", "golden"))
        if name is not None:
            path, edits = MUTANTS[name]
            text = open(os.path.join(tmp, path)).read()
            for old, new, count in edits:
                if text.count(old) != count:
                    return -1, "mutant text not found %d times: %r" % (count, old)
                text = text.replace(old, new)
            open(os.path.join(tmp, path), "w").write(text)
        env = dict(os.environ)
        env.pop("PYTHONPATH", None)
        r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q",
                            "-p", "no:cacheprovider", "-m", "not gpu"],
                           cwd=tmp, env=env, capture_output=True, text=True, timeout=600)
        return r.returncode, (r.stdout + r.stderr)[-1500:]
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


@pytest.fixture(scope="module")
def results():
    names = [None] + sorted(MUTANTS)
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        return dict(zip(names, ex.map(_run, names)))


def test_unmodified_copy_passes(results):
    rc, tail = results[None]
    assert rc == 0, tail


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(results, name):
    rc, tail = results[name]
    assert rc != -1, tail  # the mutant applied
    assert rc != 0, "the pins pass with the mistake '%s' planted" % name
    assert " failed" in tail, tail  # a pin failed (a crash of the copy would not count)
