"""The oracle's pins catch plausible mistakes in the oracle.

Each case below plants one mistake in a copy of ``oracle/quat_oracle.c``: a
flipped sign, a dropped term, a transposed operand, a wrong index or a missing
conjugate.  It compiles the copy with gcc into a temporary library, points the
oracle's ctypes binding at it, and runs every pin in ``test_oracle_pins.py``.
At least one pin must fail, and among the failures must be the pin named as
the one that guards that part of the method.  The mistakes follow burn-mamba
``mamba3/quat_scan/backward.rs``, module documentation, "Gradient math":
Hamilton's product, the left-multiplied scan ``cum[t] = q_t (x) cum[t-1]``, the
VJP rules ``grad_a = g (x) conj(b)``, ``grad_b = conj(a) (x) g``, the reverse
recurrence, and the unit-quaternion closed form.

The unmodified source, built the same way, must pass every pin: that is the
control that the harness itself is sound.  Every planted mistake keeps every
memory access inside its buffer (the index mistakes only move reads and writes
within the same array), so a mutant cannot crash the test process.

Everything here runs on the CPU; nothing touches the CUDA library.
"""
from __future__ import annotations

import ctypes
import inspect
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "quat_oracle.c")
GCC = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-pthread",
       "-ffp-contract=off", "-fno-fast-math"]

# (name, text in the oracle's source, replacement, the pin that must catch it)
MUTANTS = [
    # Hamilton's product and the conjugate
    ("product_cross_sign",
     "out[1] = aw * bx + ax * bw + ay * bz - az * by;",
     "out[1] = aw * bx + ax * bw - ay * bz + az * by;",
     "test_hamilton_basis_table"),
    ("product_drops_a_term",
     "out[0] = aw * bw - ax * bx - ay * by - az * bz;",
     "out[0] = aw * bw - ax * bx - ay * by;",
     "test_hamilton_basis_table"),
    ("product_operands_transposed",
     "static void hamilton(const double *a, const double *b, double *out)",
     "static void hamilton(const double *b, const double *a, double *out)",
     "test_hamilton_basis_table"),
    ("conj_keeps_z",
     "out[3] = -a[3];",
     "out[3] = a[3];",
     "test_conjugate_norm_identities"),
    # forward scan
    ("fwd_multiplies_on_the_right",
     "hamilton(qt, c, next);",
     "hamilton(c, qt, next);",
     "test_fwd_left_multiplication_matches_rotation_chain"),
    ("fwd_ignores_init",
     "memcpy(c, init, sizeof c);\n    for (int64_t t = 0; t < S; ++t) {\n        const double *qt",
     "c[0] = 1.0; c[1] = c[2] = c[3] = 0.0;\n    for (int64_t t = 0; t < S; ++t) {\n"
     "        const double *qt",
     "test_fwd_identity_q_keeps_init"),
    ("fwd_stores_the_previous_carry",
     "memcpy(c, next, sizeof c);\n        memcpy(cum + 4 * t * stride, c, sizeof c);",
     "memcpy(cum + 4 * t * stride, c, sizeof c);\n        memcpy(c, next, sizeof c);",
     "test_fwd_single_step_is_one_product"),
    ("fwd_step_stride_of_one",
     "const double *qt = q + 4 * t * stride;",
     "const double *qt = q + 4 * t;",
     "test_fwd_layout_lanes_independent"),
    ("lane_base_drops_the_batch",
     "const int64_t base = (b * S * HJ + hj) * 4;",
     "const int64_t base = hj * 4; (void)b;",
     "test_fwd_layout_lanes_independent"),
    # backward by the reverse recurrence
    ("bwd_recompute_multiplies_on_the_right",
     "hamilton(q + 4 * t * stride, c, tmp);",
     "hamilton(c, q + 4 * t * stride, tmp);",
     "test_bwd_central_finite_differences"),
    ("bwd_seed_dropped",
     "memcpy(G, d_cum + 4 * (S - 1) * stride, sizeof G);",
     "memset(G, 0, sizeof G);",
     "test_bwd_central_finite_differences"),
    ("bwd_d_q_uses_cum_t",
     "const double *prev = (t == 0) ? init : cumbuf + 4 * (t - 1);",
     "const double *prev = cumbuf + 4 * t;",
     "test_bwd_central_finite_differences"),
    ("bwd_d_q_without_conj",
     "hamilton(G, cprev, d_q + 4 * t * stride);\n        /* Cotangent",
     "hamilton(G, prev, d_q + 4 * t * stride);\n        /* Cotangent",
     "test_bwd_central_finite_differences"),
    ("bwd_d_q_operands_transposed",
     "hamilton(G, cprev, d_q + 4 * t * stride);\n        /* Cotangent",
     "hamilton(cprev, G, d_q + 4 * t * stride);\n        /* Cotangent",
     "test_bwd_central_finite_differences"),
    ("bwd_cotangent_without_conj",
     "hamilton(cq, G, back);",
     "hamilton(q + 4 * t * stride, G, back);",
     "test_bwd_central_finite_differences"),
    ("bwd_cotangent_operands_transposed",
     "hamilton(cq, G, back);",
     "hamilton(G, cq, back);",
     "test_bwd_central_finite_differences"),
    ("bwd_drops_d_cum",
     "G[k] = d[k] + back[k];",
     "G[k] = back[k];",
     "test_bwd_central_finite_differences"),
    ("bwd_d_cum_index_off_by_one",
     "const double *d = d_cum + 4 * (t - 1) * stride;",
     "const double *d = d_cum + 4 * t * stride;",
     "test_bwd_central_finite_differences"),
    ("bwd_d_init_skips_the_last_factor",
     "memcpy(d_init, back, sizeof back);",
     "memcpy(d_init, G, sizeof G);",
     "test_bwd_central_finite_differences"),
    ("bwd_empty_sequence_leaves_d_init_unset",
     "    if (S == 0) {\n        memset(d_init, 0, 4 * sizeof(double));\n        return;\n    }\n"
     "    /* Recompute",
     "    if (S == 0) {\n        d_init[0] = 1.0; d_init[1] = d_init[2] = d_init[3] = 0.0;\n"
     "        return;\n    }\n    /* Recompute",
     "test_bwd_empty_and_degenerate_shapes"),
    # the page's closed form, which the recurrence is pinned against
    ("closed_form_prefix_not_conjugated",
     "conjugate(pbuf + 4 * t, cp);",
     "memcpy(cp, pbuf + 4 * t, sizeof cp);",
     "test_bwd_recurrence_equals_closed_form_for_unit_q"),
    ("closed_form_d_init_from_the_wrong_end",
     "memcpy(d_init, sbuf, 4 * sizeof(double));",
     "memcpy(d_init, sbuf + 4 * (S - 1), 4 * sizeof(double));",
     "test_bwd_recurrence_equals_closed_form_for_unit_q"),
]


def _pin_calls():
    """Every pin of ``test_oracle_pins`` as (id, zero-argument call)."""
    calls = []
    for name, fn in sorted(vars(pins).items()):
        if not (name.startswith("test_") and inspect.isfunction(fn)):
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            assert not inspect.signature(fn).parameters, name
            calls.append((name, fn))
            continue
        assert len(marks) == 1, name
        argnames, argvalues = marks[0].args[:2]
        argnames = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
        for vals in argvalues:
            vals = vals if len(argnames) > 1 else (vals,)
            kw = dict(zip(argnames, vals))
            calls.append((f"{name}{list(vals)}", lambda fn=fn, kw=kw: fn(**kw)))
    return calls


PIN_CALLS = _pin_calls()


def _failing_pins(lib_path, monkeypatch):
    """Run every pin against the oracle built at ``lib_path``; return the failing pins' names."""
    monkeypatch.setattr(oracle, "_LIB_PATH", lib_path)
    monkeypatch.setattr(oracle, "build", lambda force=False: lib_path)
    monkeypatch.setattr(oracle, "_lib", None)
    failed = set()
    for pid, call in PIN_CALLS:
        try:
            call()
        except AssertionError:
            failed.add(pid.split("[")[0])
        except pytest.skip.Exception:
            pass
    return failed


def _build(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(GCC + [str(src), "-o", str(lib)], check=True)
    # a fresh file name per build, so dlopen never hands back an earlier library
    assert ctypes.CDLL(str(lib)) is not None
    return str(lib)


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def test_pins_cover_every_part_named_by_a_mutant():
    names = {pid.split("[")[0] for pid, _ in PIN_CALLS}
    assert {m[3] for m in MUTANTS} <= names


def test_unmodified_source_passes_every_pin(source, tmp_path, monkeypatch):
    assert _failing_pins(_build(tmp_path, "control", source), monkeypatch) == set()


@pytest.mark.parametrize("name,old,new,guard", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(source, tmp_path, monkeypatch, name, old, new, guard):
    assert source.count(old) == 1, f"{name}: the text to mutate is not unique in the oracle"
    failed = _failing_pins(_build(tmp_path, name, source.replace(old, new)), monkeypatch)
    assert guard in failed, f"{name}: caught by {sorted(failed)}, not by {guard}"
