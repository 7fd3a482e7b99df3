"""Pins of the fp64 oracle against what the page and the mathematics fix.

The oracle (``oracle/``) follows burn-mamba ``mamba3/quat_scan/backward.rs``,
module documentation, "Gradient math".  None of these tests re-types the
oracle's formulas: the quaternion product used here is built from Hamilton's
multiplication table and bilinearity (a different formulation from the
oracle's component formulas), and the other references are library routines
(scipy rotation composition, numpy complex ``cumprod`` / ``cumsum``), closed
forms, exact rational arithmetic, hand-derived fixtures, finite differences and
an exact forward-mode JVP.
"""
from __future__ import annotations

import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_derived_scans.txt")

# --------------------------------------------------------------------------
# Test-side quaternion product from the multiplication table of 1, i, j, k.
# e_a (x) e_b = sign * e_index  (Hamilton: i^2 = j^2 = k^2 = ijk = -1).
# --------------------------------------------------------------------------
_NAMES = "1ijk"
_TABLE = {
    ("1", "1"): (1, "1"), ("1", "i"): (1, "i"), ("1", "j"): (1, "j"), ("1", "k"): (1, "k"),
    ("i", "1"): (1, "i"), ("i", "i"): (-1, "1"), ("i", "j"): (1, "k"), ("i", "k"): (-1, "j"),
    ("j", "1"): (1, "j"), ("j", "i"): (-1, "k"), ("j", "j"): (-1, "1"), ("j", "k"): (1, "i"),
    ("k", "1"): (1, "k"), ("k", "i"): (1, "j"), ("k", "j"): (-1, "i"), ("k", "k"): (-1, "1"),
}
_STRUCT = np.zeros((4, 4, 4))
for (a, b), (s, c) in _TABLE.items():
    _STRUCT[_NAMES.index(a), _NAMES.index(b), _NAMES.index(c)] = s


def tmul(x, y):
    """Bilinear extension of the table; works on [...,4] arrays (broadcasting)."""
    return np.einsum("...a,...b,abc->...c", np.asarray(x, np.float64),
                     np.asarray(y, np.float64), _STRUCT)


def tmul_exact(x, y):
    out = [Fraction(0)] * 4
    for a, b in itertools.product(range(4), range(4)):
        s, c = _TABLE[(_NAMES[a], _NAMES[b])]
        out[_NAMES.index(c)] += s * Fraction(x[a]) * Fraction(y[b])
    return out


def tconj(x):
    x = np.array(x, np.float64, copy=True)
    x[..., 1:] *= -1
    return x


def basis(name):
    v = np.zeros(4)
    v[_NAMES.index(name)] = 1.0
    return v


def rand_quat(rng, *shape, unit=False):
    v = rng.standard_normal(shape + (4,))
    if unit:
        v /= np.linalg.norm(v, axis=-1, keepdims=True)
    return v


# --------------------------------------------------------------------------
# Hamilton product and conjugate.
# --------------------------------------------------------------------------
def test_hamilton_basis_table():
    for (a, b), (s, c) in _TABLE.items():
        got = oracle.hamilton(basis(a), basis(b))
        np.testing.assert_array_equal(got, s * basis(c), err_msg=f"{a}*{b}")
    # ijk = -1 (Hamilton's defining relation)
    ijk = oracle.hamilton(oracle.hamilton(basis("i"), basis("j")), basis("k"))
    np.testing.assert_array_equal(ijk, -basis("1"))


def test_hamilton_bilinear_exact_integers():
    rng = np.random.default_rng(11)
    for _ in range(200):
        a = rng.integers(-50, 51, 4)
        b = rng.integers(-50, 51, 4)
        want = np.array([float(v) for v in tmul_exact(a, b)])
        np.testing.assert_array_equal(oracle.hamilton(a, b), want)


def test_hamilton_matches_rotation_composition():
    Rotation = pytest.importorskip("scipy.spatial.transform").Rotation
    rng = np.random.default_rng(12)
    for _ in range(50):
        a, b = rand_quat(rng, unit=True), rand_quat(rng, unit=True)
        ab = oracle.hamilton(a, b)
        ra = Rotation.from_quat(np.roll(a, -1))      # scipy is scalar-last
        rb = Rotation.from_quat(np.roll(b, -1))
        rab = Rotation.from_quat(np.roll(ab, -1))
        np.testing.assert_allclose(rab.as_matrix(), (ra * rb).as_matrix(), atol=1e-12)


def test_conjugate_norm_identities():
    rng = np.random.default_rng(13)
    for _ in range(100):
        a, b = rand_quat(rng), rand_quat(rng)
        n2 = float(a @ a)
        np.testing.assert_allclose(oracle.hamilton(oracle.conj(a), a), [n2, 0, 0, 0], atol=1e-12)
        np.testing.assert_allclose(oracle.hamilton(a, oracle.conj(a)), [n2, 0, 0, 0], atol=1e-12)
        ab = oracle.hamilton(a, b)
        assert abs(np.linalg.norm(ab) - np.linalg.norm(a) * np.linalg.norm(b)) < 1e-12
        # conj is an anti-automorphism: conj(a b) = conj(b) conj(a)
        np.testing.assert_allclose(oracle.conj(ab), oracle.hamilton(oracle.conj(b), oracle.conj(a)),
                                   atol=1e-12)
        # unit q: conj(q) (x) q = 1
        u = a / np.linalg.norm(a)
        np.testing.assert_allclose(oracle.hamilton(oracle.conj(u), u), [1, 0, 0, 0], atol=1e-15)


# --------------------------------------------------------------------------
# Golden, hand-derived worked examples.
# --------------------------------------------------------------------------
def _read_golden():
    cases, cur, name = {}, None, None
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("case "):
                name, cur = line.split()[1], {}
            elif line == "end":
                cases[name] = cur
            else:
                key, *vals = line.split()
                arr, idx = key.rstrip("]").split("[")
                cur.setdefault(arr, {})[int(idx)] = [float(v) for v in vals]
    out = {}
    for name, c in cases.items():
        S = len(c["q"])
        q = np.array([c["q"][t] for t in range(S)]).reshape(1, S, 1, 1, 4)
        d_cum = np.array([c["d_cum"][t] for t in range(S)]).reshape(1, S, 1, 1, 4)
        cum = np.array([c["cum"][t] for t in range(S)]).reshape(1, S, 1, 1, 4)
        d_q = np.array([c["d_q"][t] for t in range(S)]).reshape(1, S, 1, 1, 4)
        init = np.array(c["init"][0]).reshape(1, 1, 1, 4)
        d_init = np.array(c["d_init"][0]).reshape(1, 1, 1, 4)
        out[name] = (q, init, d_cum, cum, d_q, d_init)
    return out


@pytest.mark.parametrize("name", ["basis", "nonunit"])
def test_golden_hand_derived(name):
    q, init, d_cum, cum, d_q, d_init = _read_golden()[name]
    np.testing.assert_array_equal(oracle.fwd(q, init), cum)
    gq, gi = oracle.bwd(q, init, d_cum)
    np.testing.assert_array_equal(gq, d_q)
    np.testing.assert_array_equal(gi, d_init)


# --------------------------------------------------------------------------
# Forward scan pins.
# --------------------------------------------------------------------------
def test_fwd_identity_q_keeps_init():
    rng = np.random.default_rng(21)
    q = np.zeros((2, 7, 2, 3, 4))
    q[..., 0] = 1
    init = rand_quat(rng, 2, 2, 3)
    cum = oracle.fwd(q, init)
    np.testing.assert_array_equal(cum, np.broadcast_to(init[:, None], cum.shape))


def test_fwd_single_step_is_one_product():
    rng = np.random.default_rng(22)
    q = rand_quat(rng, 3, 1, 2, 2)
    init = rand_quat(rng, 3, 2, 2)
    np.testing.assert_allclose(oracle.fwd(q, init)[:, 0], tmul(q[:, 0], init), atol=1e-14)


def test_fwd_exact_rational_bruteforce():
    """S <= 3 integer quaternions: nested products in exact arithmetic."""
    rng = np.random.default_rng(23)
    for S in (1, 2, 3):
        q = rng.integers(-9, 10, (1, S, 1, 2, 4))
        init = rng.integers(-9, 10, (1, 1, 2, 4))
        got = oracle.fwd(q, init)
        for j in range(2):
            c = list(init[0, 0, j])
            for t in range(S):
                c = tmul_exact(q[0, t, 0, j], c)
                np.testing.assert_array_equal(got[0, t, 0, j], [float(v) for v in c])


def test_fwd_single_axis_closed_form_and_complex_cumprod():
    """Commuting rotations about one axis: P_t = (cos T_t/2, sin T_t/2 u), T = cumsum(theta)."""
    rng = np.random.default_rng(24)
    S = 500
    theta = rng.uniform(0, 0.3, S)
    u = rng.standard_normal(3)
    u /= np.linalg.norm(u)
    q = np.zeros((1, S, 1, 1, 4))
    q[0, :, 0, 0, 0] = np.cos(theta / 2)
    q[0, :, 0, 0, 1:] = np.sin(theta / 2)[:, None] * u
    init = np.array([1.0, 0, 0, 0]).reshape(1, 1, 1, 4)
    cum = oracle.fwd(q, init)[0, :, 0, 0]
    T = np.cumsum(theta)
    np.testing.assert_allclose(cum[:, 0], np.cos(T / 2), atol=1e-12)
    np.testing.assert_allclose(cum[:, 1:], np.sin(T / 2)[:, None] * u, atol=1e-12)
    # Axis i with an init in span{1, i}: the scan is numpy's complex cumprod.
    zq = np.exp(0.5j * theta) * rng.uniform(0.9, 1.1, S)     # not unit on purpose
    z0 = complex(*rng.standard_normal(2))
    q2 = np.zeros((1, S, 1, 1, 4))
    q2[0, :, 0, 0, 0], q2[0, :, 0, 0, 1] = zq.real, zq.imag
    init2 = np.array([z0.real, z0.imag, 0, 0]).reshape(1, 1, 1, 4)
    want = z0 * np.cumprod(zq)
    got = oracle.fwd(q2, init2)[0, :, 0, 0]
    np.testing.assert_allclose(got[:, 0] + 1j * got[:, 1], want, rtol=1e-12)
    np.testing.assert_array_equal(got[:, 2:], 0)


def test_fwd_left_multiplication_matches_rotation_chain():
    """cum[t] = q_t (x) ... (x) q_0 (x) init  <=>  R(cum[t]) = R(q_t) ... R(q_0) R(init)."""
    Rotation = pytest.importorskip("scipy.spatial.transform").Rotation
    rng = np.random.default_rng(25)
    S = 12
    q = rand_quat(rng, 1, S, 1, 1, unit=True)
    init = rand_quat(rng, 1, 1, 1, unit=True)
    cum = oracle.fwd(q, init)[0, :, 0, 0]
    r = Rotation.from_quat(np.roll(init[0, 0, 0], -1))
    for t in range(S):
        r = Rotation.from_quat(np.roll(q[0, t, 0, 0], -1)) * r
        np.testing.assert_allclose(Rotation.from_quat(np.roll(cum[t], -1)).as_matrix(),
                                   r.as_matrix(), atol=1e-12)


def test_fwd_norm_preservation_unit_q():
    rng = np.random.default_rng(26)
    q = rand_quat(rng, 2, 3000, 2, 2, unit=True)
    init = rand_quat(rng, 2, 2, 2) * 3.0
    cum = oracle.fwd(q, init)
    np.testing.assert_allclose(np.linalg.norm(cum, axis=-1),
                               np.broadcast_to(np.linalg.norm(init, axis=-1)[:, None], cum.shape[:-1]),
                               rtol=1e-12)


def test_fwd_linear_in_init():
    rng = np.random.default_rng(27)
    q = rand_quat(rng, 2, 40, 1, 3)
    i1, i2 = rand_quat(rng, 2, 1, 3), rand_quat(rng, 2, 1, 3)
    a, b = 0.7, -1.3
    lhs = oracle.fwd(q, a * i1 + b * i2)
    rhs = a * oracle.fwd(q, i1) + b * oracle.fwd(q, i2)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-10, atol=1e-10)


def test_fwd_layout_lanes_independent():
    """A [B,S,H,J] call equals per-lane calls (catches stride / index mistakes)."""
    rng = np.random.default_rng(28)
    B, S, H, J = 2, 9, 2, 3
    q = rand_quat(rng, B, S, H, J)
    init = rand_quat(rng, B, H, J)
    d_cum = rand_quat(rng, B, S, H, J)
    cum = oracle.fwd(q, init)
    d_q, d_init = oracle.bwd(q, init, d_cum)
    for b, h, j in itertools.product(range(B), range(H), range(J)):
        ql = q[b:b + 1, :, h:h + 1, j:j + 1]
        il = init[b:b + 1, h:h + 1, j:j + 1]
        dl = d_cum[b:b + 1, :, h:h + 1, j:j + 1]
        np.testing.assert_array_equal(cum[b, :, h, j], oracle.fwd(ql, il)[0, :, 0, 0])
        gq, gi = oracle.bwd(ql, il, dl)
        np.testing.assert_array_equal(d_q[b, :, h, j], gq[0, :, 0, 0])
        np.testing.assert_array_equal(d_init[b, h, j], gi[0, 0, 0])


def test_fwd_threads_do_not_change_result():
    rng = np.random.default_rng(29)
    q = rand_quat(rng, 3, 50, 2, 5)
    init = rand_quat(rng, 3, 2, 5)
    np.testing.assert_array_equal(oracle.fwd(q, init, nthreads=1), oracle.fwd(q, init, nthreads=7))


# --------------------------------------------------------------------------
# Backward pins.
# --------------------------------------------------------------------------
def _loss(q, init, d_cum):
    return float(np.sum(oracle.fwd(q, init) * d_cum))


@pytest.mark.parametrize("S,J", [(1, 1), (3, 2), (6, 2)])
def test_bwd_central_finite_differences(S, J):
    """Every component of q and init, L = <cum, d_cum>, non-unit q (all quaternions)."""
    rng = np.random.default_rng(31 + S)
    q = rand_quat(rng, 1, S, 1, J) * 1.2
    init = rand_quat(rng, 1, 1, J)
    d_cum = rand_quat(rng, 1, S, 1, J)
    d_q, d_init = oracle.bwd(q, init, d_cum)
    h = 1e-6
    for idx in np.ndindex(q.shape):
        qp, qm = q.copy(), q.copy()
        qp[idx] += h
        qm[idx] -= h
        fd = (_loss(qp, init, d_cum) - _loss(qm, init, d_cum)) / (2 * h)
        assert abs(fd - d_q[idx]) < 1e-7 * max(1.0, abs(fd)), idx
    for idx in np.ndindex(init.shape):
        ip, im = init.copy(), init.copy()
        ip[idx] += h
        im[idx] -= h
        fd = (_loss(q, ip, d_cum) - _loss(q, im, d_cum)) / (2 * h)
        assert abs(fd - d_init[idx]) < 1e-7 * max(1.0, abs(fd)), idx


def test_bwd_adjoint_dot_test_exact_jvp():
    """<d_q, dq> + <d_init, dinit> = <d_cum, dcum> with dcum from forward-mode JVP.

    dcum[t] = dq_t (x) cum[t-1] + q_t (x) dcum[t-1], dcum[-1] = dinit (product rule).
    """
    rng = np.random.default_rng(41)
    B, S, H, J = 2, 300, 1, 3
    q = rand_quat(rng, B, S, H, J) * 1.05
    init = rand_quat(rng, B, H, J)
    d_cum = rand_quat(rng, B, S, H, J)
    dq = rand_quat(rng, B, S, H, J)
    dinit = rand_quat(rng, B, H, J)
    cum = oracle.fwd(q, init)
    dcum = np.empty_like(cum)
    prev, dprev = init, dinit
    for t in range(S):
        dprev = tmul(dq[:, t], prev) + tmul(q[:, t], dprev)
        prev = cum[:, t]
        dcum[:, t] = dprev
    d_q, d_init = oracle.bwd(q, init, d_cum)
    lhs = np.sum(d_q * dq) + np.sum(d_init * dinit)
    rhs = np.sum(d_cum * dcum)
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs))


def test_bwd_recurrence_equals_closed_form_for_unit_q():
    rng = np.random.default_rng(42)
    q = rand_quat(rng, 2, 2000, 2, 2, unit=True)
    init = rand_quat(rng, 2, 2, 2, unit=True)
    d_cum = rand_quat(rng, 2, 2000, 2, 2)
    a_q, a_i = oracle.bwd(q, init, d_cum)
    b_q, b_i = oracle.bwd_closed_form(q, init, d_cum)
    scale = np.abs(a_q).max()
    assert np.abs(a_q - b_q).max() <= 1e-11 * scale
    assert np.abs(a_i - b_i).max() <= 1e-11 * np.abs(a_i).max()
    # and the closed form is NOT exact once |q| != 1 (the test is sensitive)
    c_q, _ = oracle.bwd_closed_form(q * 1.001, init, d_cum)
    d_q2, _ = oracle.bwd(q * 1.001, init, d_cum)
    assert np.abs(c_q - d_q2).max() > 1e-3 * np.abs(d_q2).max()


def test_bwd_generalised_closed_form_for_any_quaternions():
    """The page's closed form, extended to non-unit q, against the literal recurrence.

    With M = q_s (x) ... (x) q_{t+1} = P_s (x) P_t^-1 and P^-1 = conj(P) / |P|^2,
    the cotangent of cum[t] is G[t] = sum_{s>=t} conj(M) (x) d_cum[s]
    = P_t (x) S[t] / |P_t|^2, S[t] = sum_{s>=t} conj(P_s) (x) d_cum[s], and the
    cotangent of init is S[0] exactly (cum[s] = P_s (x) init).  So the page's
    d_init = S[0] holds for every non-zero q, and its G = P (x) S only for unit P.
    Everything here is computed with the test-side table product.
    """
    rng = np.random.default_rng(46)
    B, S, H, J = 2, 200, 1, 3
    q = rand_quat(rng, B, S, H, J)
    q *= (rng.uniform(0.8, 1.25, (B, S, H, J, 1)) / np.linalg.norm(q, axis=-1, keepdims=True))
    init = rand_quat(rng, B, H, J)
    d_cum = rand_quat(rng, B, S, H, J)
    P = np.empty_like(q)
    acc = np.broadcast_to(np.array([1.0, 0, 0, 0]), (B, H, J, 4))
    for t in range(S):
        acc = tmul(q[:, t], acc)
        P[:, t] = acc
    terms = tmul(tconj(P), d_cum)
    Ssuf = np.flip(np.cumsum(np.flip(terms, axis=1), axis=1), axis=1)
    G = tmul(P, Ssuf) / np.sum(P * P, axis=-1, keepdims=True)
    cum_prev = np.concatenate([init[:, None], tmul(P[:, :-1], init[:, None])], axis=1)
    want_q = tmul(G, tconj(cum_prev))
    d_q, d_init = oracle.bwd(q, init, d_cum)
    assert np.abs(d_q - want_q).max() <= 1e-10 * np.abs(want_q).max()
    assert np.abs(d_init - Ssuf[:, 0]).max() <= 1e-10 * np.abs(Ssuf[:, 0]).max()
    # the norms really vary: the unnormalised G = P (x) S would be far off
    assert np.ptp(np.sum(P * P, axis=-1)) > 1.0


def test_bwd_identity_q_is_reverse_cumsum():
    rng = np.random.default_rng(43)
    B, S, H, J = 2, 64, 2, 2
    q = np.zeros((B, S, H, J, 4))
    q[..., 0] = 1
    init = rand_quat(rng, B, H, J)
    d_cum = rand_quat(rng, B, S, H, J)
    G = np.flip(np.cumsum(np.flip(d_cum, axis=1), axis=1), axis=1)
    d_q, d_init = oracle.bwd(q, init, d_cum)
    np.testing.assert_allclose(d_q, tmul(G, tconj(init)[:, None]), atol=1e-12)
    np.testing.assert_allclose(d_init, G[:, 0], atol=1e-12)


def test_bwd_complex_case_by_division_formula():
    """q, init, d_cum in span{1, i}: grad_k = sum_{t>=k} d_t conj(cum_t / q_k)."""
    rng = np.random.default_rng(44)
    S = 200
    zq = np.exp(1j * rng.uniform(0, 0.5, S)) * rng.uniform(0.95, 1.05, S)
    z0 = complex(*rng.standard_normal(2))
    zd = rng.standard_normal(S) + 1j * rng.standard_normal(S)
    cumz = z0 * np.cumprod(zq)
    rev = np.flip(np.cumsum(np.flip(zd * np.conj(cumz))))
    want_q = rev / np.conj(zq)
    want_init = rev[0] / np.conj(z0)

    def emb(z, shape):
        a = np.zeros(shape + (4,))
        a[..., 0], a[..., 1] = z.real, z.imag
        return a

    q = emb(zq, (S,)).reshape(1, S, 1, 1, 4)
    init = emb(np.array(z0), ()).reshape(1, 1, 1, 4)
    d_cum = emb(zd, (S,)).reshape(1, S, 1, 1, 4)
    d_q, d_init = oracle.bwd(q, init, d_cum)
    got_q = d_q[0, :, 0, 0, 0] + 1j * d_q[0, :, 0, 0, 1]
    np.testing.assert_allclose(got_q, want_q, rtol=1e-10)
    np.testing.assert_allclose(d_init[0, 0, 0, 0] + 1j * d_init[0, 0, 0, 1], want_init, rtol=1e-10)
    np.testing.assert_array_equal(d_q[..., 2:], 0)


def test_bwd_empty_and_degenerate_shapes():
    for shape in [(0, 5, 1, 1), (1, 0, 2, 2), (2, 3, 0, 4)]:
        B, S, H, J = shape
        q = np.zeros((B, S, H, J, 4))
        init = np.ones((B, H, J, 4))
        assert oracle.fwd(q, init).shape == q.shape
        d_q, d_init = oracle.bwd(q, init, q)
        assert d_q.shape == q.shape and d_init.shape == init.shape
        if S == 0 and d_init.size:
            np.testing.assert_array_equal(d_init, 0)


def test_bwd_zero_cotangent_gives_zero():
    rng = np.random.default_rng(45)
    q = rand_quat(rng, 1, 30, 2, 2)
    init = rand_quat(rng, 1, 2, 2)
    d_q, d_init = oracle.bwd(q, init, np.zeros_like(q))
    assert not d_q.any() and not d_init.any()
    assert math.isfinite(float(np.abs(d_q).sum()))
