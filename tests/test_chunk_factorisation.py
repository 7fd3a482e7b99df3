"""The chunk factorisation the GPU design rests on, pinned in fp64 against the oracle.

burn-mamba ``mamba3/quat_scan/backward.rs``, module documentation, "Gradient
math": the forward is the left-multiplied prefix product
cum[t] = q_t (x) cum[t-1], and the backward the reverse recurrence
G[t] = d_cum[t] + conj(q_{t+1}) (x) G[t+1], d_q[t] = G[t] (x) conj(cum[t-1]);
for unit quaternions the page also gives the closed form through the prefix
product P and the suffix sum S[t] = sum_{s>=t} conj(P_s) (x) d_cum[s].

The CUDA kernels never run those loops over a whole lane.  They cut the
sequence into chunks, reduce every chunk on its own, chain the chunk results,
and finish each chunk from its carry.  This file writes that chunked algorithm
out step by step in fp64 numpy, with the test-side quaternion product built
from Hamilton's table, and checks it against the oracle's sequential loops for
any chunk length (1, ragged, whole sequence, longer than the sequence):

* forward: chunk products L_c and local prefixes; carries
  carry_{c+1} = L_c (x) carry_c from init; cum[t] = local_t (x) carry_c;
* backward, any non-zero q (the kernels' form): each chunk alone gives the
  affine map h_{c-1} = W_c + conj(L_c) (x) h_c of the cotangent h_c entering
  it from the right, and G[t] = A_t + B_t (x) h_c inside it; the maps are
  chained from h_last = 0, and d_init = h_{-1};
* backward, unit q (the page's form): W_c = sum conj(local_s) (x) d_cum[s],
  R_c = conj(L_c) (x) (W_{c+1} + R_{c+1}), G[t] = local_t (x) (W_c^{>=t} + R_c),
  d_init = W_0 + R_0.  This rests on conj(P_s) = conj(P_{c-1}) (x) conj(local_s).

Nothing here comes from the CUDA sources.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from test_oracle_pins import rand_quat, tconj, tmul

ONE = np.array([1.0, 0.0, 0.0, 0.0])


def chunks(S, T):
    return [(t0, min(t0 + T, S)) for t0 in range(0, S, T)]


def lanes(x):
    """[B,S,H,J,4] -> [S, lanes, 4] (lane = (b,h,j))."""
    B, S, H, J, _ = x.shape
    return x.transpose(1, 0, 2, 3, 4).reshape(S, B * H * J, 4)


def unlanes(x, B, H, J):
    S = x.shape[0]
    return x.reshape(S, B, H, J, 4).transpose(1, 0, 2, 3, 4)


def chunked_fwd(q, init, T):
    """q [S,n,4], init [n,4] -> (cum [S,n,4], local prefixes per chunk, carries)."""
    S, n, _ = q.shape
    bounds = chunks(S, T)
    local, L = [], []
    for t0, t1 in bounds:              # every chunk on its own
        loc = np.empty((t1 - t0, n, 4))
        acc = np.broadcast_to(ONE, (n, 4))
        for t in range(t0, t1):
            acc = tmul(q[t], acc)
            loc[t - t0] = acc
        local.append(loc)
        L.append(acc)
    carry = [np.asarray(init, np.float64)]
    for c in range(len(bounds) - 1):   # the chain across chunks
        carry.append(tmul(L[c], carry[c]))
    cum = np.empty((S, n, 4))
    for c, (t0, t1) in enumerate(bounds):
        cum[t0:t1] = tmul(local[c], carry[c][None])
    return cum, local, carry, L


def cum_prev(local, carry, c, k):
    """cum[t-1] for step k of chunk c: local_{t-1} (x) carry_c, local_{t0-1} = 1."""
    return carry[c] if k == 0 else tmul(local[c][k - 1], carry[c])


def chunked_bwd_affine(q, init, d_cum, T, swap_chain=False):
    """(d_q, d_init) through the affine chunk maps; exact for any non-zero q.

    ``swap_chain`` multiplies h_c by conj(L_c) on the wrong side (a planted
    mistake for the sensitivity check)."""
    S, n, _ = q.shape
    bounds = chunks(S, T)
    _, local, carry, L = chunked_fwd(q, init, T)
    A_all, B_all, W = [], [], []
    for t0, t1 in bounds:              # every chunk on its own: G[t] = A_t + B_t (x) h
        A = np.empty((t1 - t0, n, 4))
        Bm = np.empty((t1 - t0, n, 4))
        A[-1] = d_cum[t1 - 1]
        Bm[-1] = ONE
        for t in range(t1 - 2, t0 - 1, -1):
            cq = tconj(q[t + 1])
            A[t - t0] = d_cum[t] + tmul(cq, A[t - t0 + 1])
            Bm[t - t0] = tmul(cq, Bm[t - t0 + 1])
        A_all.append(A)
        B_all.append(Bm)
        W.append(tmul(tconj(q[t0]), A[0]))   # h_{c-1} = conj(q_t0) (x) G[t0]
    # chain from the right: h_last = 0, h_{c-1} = W_c + conj(L_c) (x) h_c
    h = [None] * len(bounds)
    hc = np.zeros((n, 4))
    for c in range(len(bounds) - 1, -1, -1):
        h[c] = hc
        hc = W[c] + (tmul(hc, tconj(L[c])) if swap_chain else tmul(tconj(L[c]), hc))
    d_init = hc
    d_q = np.empty((S, n, 4))
    for c, (t0, t1) in enumerate(bounds):
        for k in range(t1 - t0):
            G = A_all[c][k] + tmul(B_all[c][k], h[c])
            d_q[t0 + k] = tmul(G, tconj(cum_prev(local, carry, c, k)))
    return d_q, d_init


def chunked_bwd_page(q, init, d_cum, T):
    """(d_q, d_init) by the page's closed form, chunked; exact for unit q only."""
    S, n, _ = q.shape
    bounds = chunks(S, T)
    _, local, carry, L = chunked_fwd(q, init, T)
    Wsuf = []                            # W_c^{>=t} for every t of chunk c, on its own
    for c, (t0, t1) in enumerate(bounds):
        terms = tmul(tconj(local[c]), d_cum[t0:t1])
        Wsuf.append(np.flip(np.cumsum(np.flip(terms, 0), 0), 0))
    R = [None] * len(bounds)
    R[-1] = np.zeros((n, 4))
    for c in range(len(bounds) - 2, -1, -1):
        R[c] = tmul(tconj(L[c]), Wsuf[c + 1][0] + R[c + 1])
    d_init = Wsuf[0][0] + R[0]
    d_q = np.empty((S, n, 4))
    for c, (t0, t1) in enumerate(bounds):
        for k in range(t1 - t0):
            G = tmul(local[c][k], Wsuf[c][k] + R[c])
            d_q[t0 + k] = tmul(G, tconj(cum_prev(local, carry, c, k)))
    return d_q, d_init


def rel(a, b):
    return float(np.abs(a - b).max() / np.abs(b).max())


B, S, H, J = 2, 203, 1, 3
CHUNKS = [1, 7, 64, S, S + 50]


@pytest.fixture(scope="module")
def data():
    rng = np.random.default_rng(2024)
    q = rand_quat(rng, B, S, H, J) * rng.uniform(0.8, 1.25, (B, S, H, J, 1))   # not unit
    qu = rand_quat(rng, B, S, H, J, unit=True)
    init = rand_quat(rng, B, H, J)
    d_cum = rand_quat(rng, B, S, H, J)
    return q, qu, init, d_cum


@pytest.mark.parametrize("T", CHUNKS)
def test_chunked_forward_matches_sequential(data, T):
    q, _, init, _ = data
    cum, *_ = chunked_fwd(lanes(q), init.reshape(-1, 4), T)
    want = oracle.fwd(q, init)
    assert rel(unlanes(cum, B, H, J), want) <= 1e-12


@pytest.mark.parametrize("T", CHUNKS)
def test_affine_chunk_maps_match_literal_recurrence(data, T):
    q, _, init, d_cum = data
    d_q, d_init = chunked_bwd_affine(lanes(q), init.reshape(-1, 4), lanes(d_cum), T)
    want_q, want_i = oracle.bwd(q, init, d_cum)
    assert rel(unlanes(d_q, B, H, J), want_q) <= 1e-11
    assert rel(d_init.reshape(want_i.shape), want_i) <= 1e-11


@pytest.mark.parametrize("T", CHUNKS)
def test_page_chunked_closed_form_for_unit_q(data, T):
    _, qu, init, d_cum = data
    d_q, d_init = chunked_bwd_page(lanes(qu), init.reshape(-1, 4), lanes(d_cum), T)
    want_q, want_i = oracle.bwd(qu, init, d_cum)
    assert rel(unlanes(d_q, B, H, J), want_q) <= 1e-11
    assert rel(d_init.reshape(want_i.shape), want_i) <= 1e-11


def test_page_chunked_closed_form_needs_unit_q(data):
    """The same chunked closed form on non-unit q is far off: the pin is sensitive."""
    q, _, init, d_cum = data
    d_q, _ = chunked_bwd_page(lanes(q), init.reshape(-1, 4), lanes(d_cum), 7)
    want_q, _ = oracle.bwd(q, init, d_cum)
    assert rel(unlanes(d_q, B, H, J), want_q) > 1e-3


def test_forward_carry_on_the_wrong_side_is_caught(data):
    """Chaining the chunk products with the operands swapped changes the result."""
    q, _, init, d_cum = data
    ql, il, dl = lanes(q), init.reshape(-1, 4), lanes(d_cum)
    S_, n, _ = ql.shape
    # forward carries multiplied on the wrong side: carry_c (x) L_c
    bounds = chunks(S_, 7)
    _, local, carry, L = chunked_fwd(ql, il, 7)
    wrong = [il]
    for c in range(len(bounds) - 1):
        wrong.append(tmul(wrong[c], L[c]))
    cum_wrong = np.concatenate([tmul(local[c], wrong[c][None]) for c in range(len(bounds))])
    assert rel(unlanes(cum_wrong, B, H, J), oracle.fwd(q, init)) > 1e-3


def test_backward_chain_on_the_wrong_side_is_caught(data):
    q, _, init, d_cum = data
    d_q, _ = chunked_bwd_affine(lanes(q), init.reshape(-1, 4), lanes(d_cum), 7, swap_chain=True)
    want_q, _ = oracle.bwd(q, init, d_cum)
    assert rel(unlanes(d_q, B, H, J), want_q) > 1e-3


def test_chunked_algorithm_on_random_shapes():
    """Random (B, S, H, J), chunk length and quaternion scale: the chunked forward
    and the affine-map backward equal the oracle's sequential loops."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    @hyp.settings(max_examples=60, deadline=None, derandomize=True)
    @hyp.given(B=st.integers(1, 3), S=st.integers(1, 90), H=st.integers(1, 2), J=st.integers(1, 3),
               T=st.integers(1, 100), scale=st.floats(0.5, 1.5), seed=st.integers(0, 2**31 - 1))
    def check(B, S, H, J, T, scale, seed):
        rng = np.random.default_rng(seed)
        q = rand_quat(rng, B, S, H, J)
        q *= scale / np.linalg.norm(q, axis=-1, keepdims=True)
        init = rand_quat(rng, B, H, J)
        d_cum = rand_quat(rng, B, S, H, J)
        cum, *_ = chunked_fwd(lanes(q), init.reshape(-1, 4), T)
        want = oracle.fwd(q, init)
        assert rel(unlanes(cum, B, H, J), want) <= 1e-11
        d_q, d_init = chunked_bwd_affine(lanes(q), init.reshape(-1, 4), lanes(d_cum), T)
        want_q, want_i = oracle.bwd(q, init, d_cum)
        assert rel(unlanes(d_q, B, H, J), want_q) <= 1e-10
        assert rel(d_init.reshape(want_i.shape), want_i) <= 1e-10

    check()
