"""GPU: one forward + backward step on host buffers (quat_cumprod_fwd_bwd_host).

The step is cut into slices of whole batch entries whose copies overlap the
kernels; it must compute exactly the forward and the backward, so every output
is compared with the fp64 oracle at the parity tolerance (normwise relative
error <= 1e-4 per output tensor).
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


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    qs.load_library()
    return torch.device("cuda", 0)


def normwise(got, ref):
    ref = np.asarray(ref, np.float64)
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    return float(np.abs(np.asarray(got, np.float64) - ref).max()) / (scale if scale > 0 else 1.0) if ref.size else 0.0


def host(a, pinned):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory() if pinned else t


# Slices hold about 32 MB of one tensor.  (6, 8192, 4, 32): 16.8 MB per batch
# entry, two entries per slice (3 slices); (7, 6000, 4, 32): two entries per
# slice and a ragged last one (4 slices, a staging slot reused); (1, 2048, 8,
# 100): 8 lane ranges of 112 lanes and a ragged last range of 16 (pitched
# copies); (3, 5000, 2, 32): two ranges of 32 lanes per entry (6 slices);
# (2, 333, 3, 16): one slice; (1, 64, 2, 4): one entry.
@pytest.mark.parametrize("dims", [(6, 8192, 4, 32), (1, 2048, 8, 100), (7, 6000, 4, 32), (3, 5000, 2, 32),
                                  (2, 333, 3, 16), (1, 64, 2, 4)])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_step_matches_oracle(dev, dims, pinned):
    w = workloads.custom("host", *dims, q_kind="rotation", theta_max=0.4, seed=101)
    q, init, d_cum = workloads.make_inputs(w)
    cum, d_q, d_init = qs.quat_cumprod_fwd_bwd_host(host(q, pinned), host(init, pinned), host(d_cum, pinned),
                                                    device=dev)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    rq, ri = oracle.bwd(q, init, d_cum)
    assert normwise(cum.numpy(), oracle.fwd(q, init)) <= TOL
    assert normwise(d_q.numpy(), rq) <= TOL
    assert normwise(d_init.numpy(), ri) <= TOL


def test_host_step_repeated_and_async(dev):
    """Back-to-back calls without synchronizing in between reuse the staging safely."""
    w1 = workloads.custom("h1", 6, 8192, 4, 32, q_kind="gauss4", seed=5)
    w2 = workloads.custom("h2", 6, 8192, 4, 32, q_kind="rotation", theta_max=0.9, seed=6)
    ins1 = [host(a, True) for a in workloads.make_inputs(w1)]
    ins2 = [host(a, True) for a in workloads.make_inputs(w2)]
    out1 = qs.quat_cumprod_fwd_bwd_host(*ins1, device=dev, synchronize=False)
    out2 = qs.quat_cumprod_fwd_bwd_host(*ins2, device=dev, synchronize=False)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK   # synchronizes the stream
    for ins, out in ((ins1, out1), (ins2, out2)):
        q, init, d_cum = (t.numpy() for t in ins)
        rq, ri = oracle.bwd(q, init, d_cum)
        assert normwise(out[0].numpy(), oracle.fwd(q, init)) <= TOL
        assert normwise(out[1].numpy(), rq) <= TOL
        assert normwise(out[2].numpy(), ri) <= TOL


def test_host_step_matches_device_calls_at_full_size(dev):
    """mamba3 at full size through host buffers, against the device calls (sampled lanes vs the oracle)."""
    w = workloads.WORKLOADS["mamba3"]
    q, init, d_cum = workloads.make_inputs(w)
    cum, d_q, d_init = qs.quat_cumprod_fwd_bwd_host(host(q, True), host(init, True), host(d_cum, True), device=dev)
    lanes = np.random.default_rng(11).choice(w.lanes, 24, replace=False)
    sq, si, sd = workloads.sample_lanes((q, init, d_cum), lanes, w.H, w.J)
    gc, gq, gi = workloads.sample_lanes((cum.numpy(), d_q.numpy(), d_init.numpy()), lanes, w.H, w.J)
    rq, ri = oracle.bwd(sq, si, sd)
    assert normwise(gc, oracle.fwd(sq, si)) <= TOL
    assert normwise(gq, rq) <= TOL and normwise(gi, ri) <= TOL


def test_host_step_empty_sequence_and_bad_tensors(dev):
    q0 = torch.zeros(2, 0, 2, 1, 4)
    i0 = torch.ones(2, 2, 1, 4)
    _, _, di = qs.quat_cumprod_fwd_bwd_host(q0, i0, q0.clone(), device=dev)
    assert float(di.abs().max()) == 0.0
    with pytest.raises(ValueError):
        qs.quat_cumprod_fwd_bwd_host(torch.zeros(1, 4, 1, 1, 4, device=dev), torch.zeros(1, 1, 1, 4),
                                     torch.zeros(1, 4, 1, 1, 4), device=dev)
    with pytest.raises(TypeError):
        qs.quat_cumprod_fwd_bwd_host(torch.zeros(1, 4, 1, 1, 4, dtype=torch.float64), torch.zeros(1, 1, 1, 4),
                                     torch.zeros(1, 4, 1, 1, 4), device=dev)
