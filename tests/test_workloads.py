"""The seeded input generator follows the workload table (CPU only).

The table is restated here, independently of ``workloads.py``: shapes, seeds,
the kind of ``q`` (normalized Gaussian quaternions, or rotations by an angle
drawn uniformly below a bound about a uniformly drawn axis), the kind of
``init`` and the spread of ``d_cum``.  The distribution checks run on a
shortened copy of each workload (same recipe, fewer steps).
"""
from __future__ import annotations

import math

import numpy as np
import pytest

from quaternion_cumulative_product_gb300 import workloads

# name: (B, S, H, J), q kind, theta_max, init kind, d_cum sigma, seed
TABLE = {
    "tiny": ((1, 64, 2, 4), "gauss4", None, "gauss4", 1.0, 0),
    "small": ((4, 1024, 8, 16), "rotation", 0.1, "gauss4", 1.0, 1),
    "mamba3": ((8, 4096, 16, 32), "rotation", math.pi / 8, "identity", 0.02, 2),
    "large": ((16, 8192, 32, 32), "gauss4", None, "gauss4", 1.0, 3),
    "long": ((1, 131072, 16, 16), "rotation", 0.05, "gauss4", 1.0, 4),
}


def test_table_matches():
    assert set(workloads.WORKLOADS) == set(TABLE)
    for name, (dims, qk, th, ik, sigma, seed) in TABLE.items():
        w = workloads.WORKLOADS[name]
        assert (w.B, w.S, w.H, w.J) == dims
        assert (w.q_kind, w.init_kind, w.seed) == (qk, ik, seed)
        assert w.dcum_sigma == sigma
        if th is not None:
            assert w.theta_max == pytest.approx(th)


@pytest.mark.parametrize("name", sorted(TABLE))
def test_distributions(name):
    dims, qk, th, ik, sigma, seed = TABLE[name]
    B, S, H, J = dims
    S_short = max(1, min(S, (1 << 16) // (B * H * J)))
    w = workloads.custom(name, B, S_short, H, J, q_kind=qk, theta_max=th or 0.0, init_kind=ik,
                         dcum_sigma=sigma, seed=seed)
    q, init, d_cum = workloads.make_inputs(w)
    assert q.dtype == init.dtype == d_cum.dtype == np.float32
    assert q.shape == (B, S_short, H, J, 4) and init.shape == (B, H, J, 4) and d_cum.shape == q.shape
    qq = q.reshape(-1, 4).astype(np.float64)
    np.testing.assert_allclose(np.linalg.norm(qq, axis=1), 1.0, atol=2e-6)
    if qk == "rotation":
        theta = 2 * np.arccos(np.clip(qq[:, 0], -1, 1))
        assert theta.min() >= -1e-6 and theta.max() <= th + 1e-3
        assert abs(theta.mean() - th / 2) < 0.05 * th          # uniform on [0, th]
        axis = qq[:, 1:] / np.linalg.norm(qq[:, 1:], axis=1, keepdims=True)
        assert np.abs(axis.mean(axis=0)).max() < 0.05          # uniform on the sphere
    else:
        assert np.abs(qq.mean(axis=0)).max() < 0.05            # uniform on the 3-sphere
        assert (qq[:, 0] < 0).any()
    ii = init.reshape(-1, 4)
    if ik == "identity":
        assert (ii == np.array([1, 0, 0, 0], np.float32)).all()
    else:
        np.testing.assert_allclose(np.linalg.norm(ii.astype(np.float64), axis=1), 1.0, atol=2e-6)
    assert abs(d_cum.std() / sigma - 1) < 0.02 and abs(d_cum.mean()) < 0.02 * sigma


def test_seeds_give_distinct_streams():
    a = workloads.make_inputs(workloads.custom("a", 1, 8, 1, 2, seed=0))
    b = workloads.make_inputs(workloads.custom("b", 1, 8, 1, 2, seed=1))
    assert not np.array_equal(a[0], b[0])


@pytest.mark.parametrize("name", ["tiny", "small", "identity-init"])
def test_device_draws_follow_the_same_recipe(name):
    """make_inputs_device (the bench's draws for the other workloads) on the CPU:
    shapes, unit q and init (or identity init), rotation angles within their
    bound, d_cum's spread."""
    torch = pytest.importorskip("torch")
    w = (workloads.WORKLOADS[name] if name in workloads.WORKLOADS else
         workloads.custom(name, 2, 4096, 4, 8, q_kind="rotation", theta_max=math.pi / 8,
                          init_kind="identity", dcum_sigma=0.02, seed=2))
    q, init, d_cum = workloads.make_inputs_device(w, torch.device("cpu"))
    assert q.shape == (w.B, w.S, w.H, w.J, 4) and d_cum.shape == q.shape and init.shape == (w.B, w.H, w.J, 4)
    assert q.dtype == init.dtype == d_cum.dtype == torch.float32
    assert torch.allclose(q.double().norm(dim=-1), torch.ones(()).double(), atol=1e-6)
    if w.init_kind == "identity":
        assert torch.equal(init, torch.tensor([1.0, 0, 0, 0]).expand_as(init))
    else:
        assert torch.allclose(init.double().norm(dim=-1), torch.ones(()).double(), atol=1e-6)
    if w.q_kind == "rotation":
        theta = 2 * torch.acos(q[..., 0].double().clamp(-1, 1))
        assert float(theta.max()) <= w.theta_max + 1e-5
    sd = float(d_cum.double().std())
    assert abs(sd - w.dcum_sigma) < 0.05 * w.dcum_sigma
    again = workloads.make_inputs_device(w, torch.device("cpu"))
    assert all(torch.equal(a, b) for a, b in zip((q, init, d_cum), again))   # seeded
