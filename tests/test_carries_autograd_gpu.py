"""GPU: forward with saved chunk carries, backward from them, and the autograd wrapper.

Everything is compared with the fp64 oracle at the parity tolerance (normwise
relative error <= 1e-4 per output tensor).  The carries are checked against
the oracle's own ``cum`` rows: ``carries[:, c] = cum[:, 64c - 1]`` and
``init`` for ``c = 0``.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import quaternion_cumulative_product_gb300 as qs
from quaternion_cumulative_product_gb300 import workloads

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TOL = 1e-4
STEPS = qs.QS_CARRY_STEPS


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    qs.load_library()
    return torch.device("cuda", 0)


@pytest.fixture(autouse=True)
def reset_hooks():
    lib = qs.load_library()
    yield
    lib.quat_cumprod_debug_set_variant(-1, -1)


def normwise(got, ref):
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    scale = float(np.abs(ref).max())
    return float(np.abs(np.asarray(got, np.float64) - ref).max()) / (scale if scale > 0 else 1.0)


def expected_carries(cum, init):
    B, S, H, J, _ = cum.shape
    C = (S + STEPS - 1) // STEPS
    out = np.empty((B, C, H, J, 4))
    out[:, 0] = init
    for c in range(1, C):
        out[:, c] = cum[:, c * STEPS - 1]
    return out


def to_dev(dev, *arrays):
    return [torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in arrays]


# Both designs on each shape: the walk (variant 4) and aggregate / carry /
# apply (variant 0); configurations with another chunk length fall back to
# their design's default, which is also exercised here (variants 1 and 6).
SHAPES = [(2, 333, 3, 16), (1, 64, 2, 4), (1, 63, 1, 1), (3, 1100, 1, 40), (2, 4096, 2, 32)]


@pytest.mark.parametrize("variant", [0, 4, 1, 6])
@pytest.mark.parametrize("dims", SHAPES)
def test_forward_writes_carries_and_backward_uses_them(dev, variant, dims):
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(variant, variant) == qs.QS_OK
    w = workloads.custom("carries", *dims, q_kind="rotation", theta_max=0.7, seed=variant + 3)
    q, init, d_cum = workloads.make_inputs(w)
    tq, ti, td = to_dev(dev, q, init, d_cum)
    cum, carries = qs.quat_cumprod_fwd_carries(tq, ti)
    d_q, d_init = qs.quat_cumprod_bwd_carries(tq, carries, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    ref_cum = oracle.fwd(q, init)
    ref_dq, ref_di = oracle.bwd(q, init, d_cum)
    assert normwise(cum.cpu().numpy(), ref_cum) <= TOL
    assert normwise(carries.cpu().numpy(), expected_carries(ref_cum, init)) <= TOL
    assert normwise(d_q.cpu().numpy(), ref_dq) <= TOL
    assert normwise(d_init.cpu().numpy(), ref_di) <= TOL


def test_carry_calls_at_full_size_match_the_plain_calls(dev):
    """mamba3 at full size, in the configuration the library picks (walk)."""
    w = workloads.WORKLOADS["mamba3"]
    assert qs.quat_cumprod_plan("bwd_carries", w.B, w.S, w.H, w.J, device=dev)[1] == 1
    q, init, d_cum = workloads.make_inputs(w)
    tq, ti, td = to_dev(dev, q, init, d_cum)
    cum_a = qs.quat_cumprod_fwd(tq, ti)
    cum_b, carries = qs.quat_cumprod_fwd_carries(tq, ti)
    dq_a, di_a = qs.quat_cumprod_bwd(tq, ti, td)
    dq_b, di_b = qs.quat_cumprod_bwd_carries(tq, carries, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    assert torch.equal(cum_a, cum_b)   # the same kernel, writing the carries on the side
    for a, b in ((dq_a, dq_b), (di_a, di_b)):
        assert normwise(b.cpu().numpy(), a.cpu().numpy().astype(np.float64)) <= TOL
    # and sampled whole lanes against the oracle
    lanes = np.random.default_rng(7).choice(w.lanes, 24, replace=False)
    sq, si, sd = workloads.sample_lanes((q, init, d_cum), lanes, w.H, w.J)
    rq, ri = oracle.bwd(sq, si, sd)
    gq, gi = workloads.sample_lanes((dq_b.cpu().numpy(), di_b.cpu().numpy()), lanes, w.H, w.J)
    assert normwise(gq, rq) <= TOL and normwise(gi, ri) <= TOL


def test_plan_counts_the_kernels_of_the_carry_calls(dev):
    # few lanes: the segmented walks, which write and read the carries themselves
    assert qs.quat_cumprod_plan("fwd_carries", 1, 4096, 1, 4, device=dev)[1] == 1
    assert qs.quat_cumprod_plan("bwd_carries", 1, 4096, 1, 4, device=dev)[1] == 1
    assert qs.quat_cumprod_plan("bwd", 1, 4096, 1, 4, device=dev)[1] == 3   # recompute: aggregate / carry / apply
    assert qs.quat_cumprod_plan("bwd", 1, 4096, 32, 32, device=dev)[1] == 2  # 64 groups: + the carries-only pass
    assert qs.quat_cumprod_plan("fwd_carries", 8, 4096, 16, 32, device=dev)[1] == 1
    # forced aggregate / carry / apply: plus the carry export for the forward
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(0, 0) == qs.QS_OK
    assert qs.quat_cumprod_plan("fwd_carries", 1, 4096, 1, 4, device=dev)[1] == 4
    assert qs.quat_cumprod_plan("bwd_carries", 1, 4096, 1, 4, device=dev)[1] == 3


# The segmented walks of both directions (forward 12: one role, 14:
# warp-specialised; backward 11-14) write and read the carries themselves.
@pytest.mark.parametrize("fv,bv", [(12, 11), (14, 11), (12, 12), (14, 13), (14, 14), (9, 11)])
@pytest.mark.parametrize("dims", [(2, 333, 3, 16), (1, 63, 1, 1), (1, 20000, 1, 3), (2, 17000, 2, 5)])
def test_segmented_walks_write_and_read_carries(dev, fv, bv, dims):
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(fv, bv) == qs.QS_OK
    assert qs.quat_cumprod_plan("bwd_carries", *dims, device=dev) == (bv, 1)
    w = workloads.custom("segcarries", *dims, q_kind="rotation", theta_max=0.5, seed=fv * 16 + bv)
    q, init, d_cum = workloads.make_inputs(w)
    tq, ti, td = to_dev(dev, q, init, d_cum)
    cum, carries = qs.quat_cumprod_fwd_carries(tq, ti)
    d_q, d_init = qs.quat_cumprod_bwd_carries(tq, carries, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    ref_cum = oracle.fwd(q, init)
    ref_dq, ref_di = oracle.bwd(q, init, d_cum)
    assert normwise(cum.cpu().numpy(), ref_cum) <= TOL
    assert normwise(carries.cpu().numpy(), expected_carries(ref_cum, init)) <= TOL
    assert normwise(d_q.cpu().numpy(), ref_dq) <= TOL
    assert normwise(d_init.cpu().numpy(), ref_di) <= TOL


# The short-sequence kernels write the carries (forward) and start from
# carries[:, 0] (backward, which recomputes the rest).
@pytest.mark.parametrize("fv,bv", [(25, 25), (26, 26), (27, 27), (28, 28), (26, 25)])
@pytest.mark.parametrize("dims", [(2, 333, 3, 16), (1, 63, 1, 1), (3, 64, 1, 5), (1, 500, 2, 3)])
def test_short_sequences_write_and_read_carries(dev, fv, bv, dims):
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(fv, bv) == qs.QS_OK
    assert qs.quat_cumprod_plan("fwd_carries", *dims, device=dev) == (fv, 1)
    assert qs.quat_cumprod_plan("bwd_carries", *dims, device=dev) == (bv, 1)
    w = workloads.custom("shortcarries", *dims, q_kind="rotation", theta_max=0.5, seed=fv * 16 + bv)
    q, init, d_cum = workloads.make_inputs(w)
    tq, ti, td = to_dev(dev, q, init, d_cum)
    cum, carries = qs.quat_cumprod_fwd_carries(tq, ti)
    d_q, d_init = qs.quat_cumprod_bwd_carries(tq, carries, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    ref_cum = oracle.fwd(q, init)
    ref_dq, ref_di = oracle.bwd(q, init, d_cum)
    assert normwise(cum.cpu().numpy(), ref_cum) <= TOL
    assert normwise(carries.cpu().numpy(), expected_carries(ref_cum, init)) <= TOL
    assert normwise(d_q.cpu().numpy(), ref_dq) <= TOL
    assert normwise(d_init.cpu().numpy(), ref_di) <= TOL


def test_long_from_saved_carries_full_size_sampled_lanes(dev):
    """The long workload (1 x 131072 x 16 x 16) at full size through the
    segmented walks of both directions, compared on sampled whole lanes."""
    w = workloads.WORKLOADS["long"]
    assert qs.quat_cumprod_plan("bwd_carries", w.B, w.S, w.H, w.J, device=dev) == (31, 1)
    q, init, d_cum = workloads.make_inputs(w)
    tq, ti, td = to_dev(dev, q, init, d_cum)
    _, carries = qs.quat_cumprod_fwd_carries(tq, ti)
    d_q, d_init = qs.quat_cumprod_bwd_carries(tq, carries, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    lanes = np.unique(np.concatenate([[0, 15, 16, w.lanes - 1],
                                      np.random.default_rng(8).choice(w.lanes, 24, replace=False)]))
    sq, si, sd = workloads.sample_lanes((q, init, d_cum), lanes, w.H, w.J)
    rq, ri = oracle.bwd(sq, si, sd)
    gq, gi = workloads.sample_lanes((d_q.cpu().numpy(), d_init.cpu().numpy()), lanes, w.H, w.J)
    assert normwise(gq, rq) <= TOL and normwise(gi, ri) <= TOL


# ---------------------------------------------------------------------------
# autograd wrapper
# ---------------------------------------------------------------------------
from quaternion_cumulative_product_gb300 import autograd as qa  # noqa: E402


@pytest.mark.parametrize("save_carries", [False, True])
@pytest.mark.parametrize("dims", [(2, 300, 3, 5), (4, 1024, 8, 16)])
def test_autograd_matches_oracle(dev, save_carries, dims):
    w = workloads.custom("ag", *dims, q_kind="gauss4", seed=31)
    q, init, W = workloads.make_inputs(w)
    tq, ti, tW = to_dev(dev, q, init, W)
    tq.requires_grad_(True)
    ti.requires_grad_(True)
    cum = qa.quat_cumprod(tq, ti, save_carries=save_carries)
    (cum * tW).sum().backward()     # L = <cum, W>: the cotangent of cum is W
    ref_cum = oracle.fwd(q, init)
    ref_dq, ref_di = oracle.bwd(q, init, W)
    assert normwise(cum.detach().cpu().numpy(), ref_cum) <= TOL
    assert normwise(tq.grad.cpu().numpy(), ref_dq) <= TOL
    assert normwise(ti.grad.cpu().numpy(), ref_di) <= TOL


@pytest.mark.parametrize("save_carries", [False, True])
def test_final_carry_cotangent_folds_into_the_last_step(dev, save_carries):
    """The page's final carry is a slice of cum: its cotangent adds into d_cum[:, S-1]."""
    w = workloads.custom("final", 2, 200, 2, 3, q_kind="rotation", theta_max=0.9, seed=41)
    q, init, W = workloads.make_inputs(w)
    V = np.random.default_rng(5).standard_normal(init.shape).astype(np.float32)
    tq, ti, tW, tV = to_dev(dev, q, init, W, V)
    tq.requires_grad_(True)
    ti.requires_grad_(True)
    cum, final = qa.quat_cumprod_recalculated(tq, ti, save_carries=save_carries)
    ((cum * tW).sum() + (final * tV).sum()).backward()
    folded = W.astype(np.float64).copy()
    folded[:, -1] += V
    ref_dq, ref_di = oracle.bwd(q, init, folded)
    assert normwise(final.detach().cpu().numpy(), oracle.fwd(q, init)[:, -1]) <= TOL
    assert normwise(tq.grad.cpu().numpy(), ref_dq) <= TOL
    assert normwise(ti.grad.cpu().numpy(), ref_di) <= TOL


def test_autograd_partial_requirements_and_no_grad(dev):
    w = workloads.custom("partial", 1, 130, 2, 2, seed=51)
    q, init, W = workloads.make_inputs(w)
    tq, ti, tW = to_dev(dev, q, init, W)
    ti.requires_grad_(True)                       # only init
    (qa.quat_cumprod(tq, ti) * tW).sum().backward()
    assert tq.grad is None
    assert normwise(ti.grad.cpu().numpy(), oracle.bwd(q, init, W)[1]) <= TOL
    with torch.no_grad():                         # untracked: nothing kept
        cum = qa.quat_cumprod(tq.requires_grad_(True), ti, save_carries=True)
    assert cum.grad_fn is None
    assert normwise(cum.cpu().numpy(), oracle.fwd(q, init)) <= TOL
