"""GPU: the bfloat16-I/O calls against the fp64 oracle.

The inputs are bfloat16, and the oracle runs on exactly those values
(widened to fp64).  The kernels compute in fp32 and round each output once to
the nearest bfloat16.

Tolerance, normwise per output tensor:

- bfloat16 has 8 significant bits, so rounding to nearest moves a value by at
  most half an ulp, 2^-8 of its magnitude, hence at most 2^-8 of max|ref|.
- The fp32 arithmetic before the rounding is within the fp32 calls'
  tolerance of 1e-4.
- So |out - ref| <= 2^-8 (1 + 1e-4) max|ref| + 1e-4 max|ref|, which gives
  TOL_BF16 = 2^-8 + 1.1e-4 (about 4.0e-3).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import parity_log
import quaternion_cumulative_product_gb300 as qs
from quaternion_cumulative_product_gb300 import workloads

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TOL_BF16 = 2.0 ** -8 + 1.1e-4


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    qs.load_library()
    return torch.device("cuda", 0)


def normwise(got, ref, what="", tol=None):
    """Normwise error; with QS_PARITY_LOG set, both measures are logged."""
    err = parity_log.normwise(got, ref)
    parity_log.record(what, "bf16", got, ref, TOL_BF16 if tol is None else tol, err)
    return err


def bf16_inputs(dev, w):
    """The workload's inputs rounded to bfloat16, on the device, and the same values as fp64."""
    arrays = workloads.make_inputs(w)
    tb = [torch.from_numpy(a).to(dev).to(torch.bfloat16) for a in arrays]
    exact = [t.float().cpu().numpy().astype(np.float64) for t in tb]
    return tb, exact


# Compiled configurations: forward 0-3 walks, 4 three kernels, 5 segmented
# chained walk, 6 the same with self-describing look-back values, 7 its
# warp-specialised form; backward 0-3 walks, 4 three kernels, 5 walk with
# registers capped for three CTAs per SM, 6 and 7 the segmented walk after its
# carries pass (segments of 4 and 2 chunks); forward 8, 9 and backward 8-10
# short sequences (the whole sequence of a few lanes in one CTA, up to 1024,
# 2048 / 1024, 512, 2048 steps); forward 10 the segmented walk with per-unit
# tables (32 lanes).
N_BF16_FWD, N_BF16_BWD = 11, 11


@pytest.fixture(autouse=True)
def reset_bf16_variant():
    yield
    qs.load_library().quat_cumprod_debug_set_variant_bf16(-1, -1)


@pytest.mark.parametrize("variant", range(max(N_BF16_FWD, N_BF16_BWD)))
@pytest.mark.parametrize("dims", [(1, 64, 2, 4), (2, 333, 3, 16), (3, 1100, 1, 40), (1, 70, 5, 2),
                                  (2, 1, 1, 2), (1, 5000, 2, 32), (1, 512, 1, 6), (1, 1024, 3, 2),
                                  (1, 2048, 1, 2)])
def test_bf16_matches_oracle(dev, dims, variant):
    fv = variant if variant < N_BF16_FWD else -1
    bv = variant if variant < N_BF16_BWD else -1
    assert qs.load_library().quat_cumprod_debug_set_variant_bf16(fv, bv) == qs.QS_OK
    w = workloads.custom("bf16", *dims, q_kind="rotation", theta_max=0.6, seed=61)
    (tq, ti, td), (q, init, d_cum) = bf16_inputs(dev, w)
    cum = qs.quat_cumprod_fwd_bf16(tq, ti)
    d_q, d_init = qs.quat_cumprod_bwd_bf16(tq, ti, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    assert cum.dtype == d_q.dtype == d_init.dtype == torch.bfloat16
    ref_cum = oracle.fwd(q, init)
    ref_dq, ref_di = oracle.bwd(q, init, d_cum)
    for got, ref, name in ((cum, ref_cum, "cum"), (d_q, ref_dq, "d_q"), (d_init, ref_di, "d_init")):
        err = normwise(got.float().cpu().numpy(), ref, name)
        assert err <= TOL_BF16, f"{name}: {err:.3e} > {TOL_BF16:.3e}"


def test_bf16_full_size_sampled_lanes(dev):
    """mamba3 at full size (bench launch configuration) on sampled whole lanes."""
    w = workloads.WORKLOADS["mamba3"]
    (tq, ti, td), _ = bf16_inputs(dev, w)
    cum = qs.quat_cumprod_fwd_bf16(tq, ti)
    d_q, d_init = qs.quat_cumprod_bwd_bf16(tq, ti, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    lanes = np.random.default_rng(3).choice(w.lanes, 24, replace=False)
    host = [t.float().cpu().numpy() for t in (tq, ti, td, cum, d_q, d_init)]
    sq, si, sd = (a.astype(np.float64) for a in workloads.sample_lanes(host[:3], lanes, w.H, w.J))
    gc, gq, gi = workloads.sample_lanes(host[3:], lanes, w.H, w.J)
    ref_dq, ref_di = oracle.bwd(sq, si, sd)
    assert normwise(gc, oracle.fwd(sq, si)) <= TOL_BF16
    assert normwise(gq, ref_dq) <= TOL_BF16
    assert normwise(gi, ref_di) <= TOL_BF16


def test_bf16_rounding_is_the_only_difference_from_fp32(dev):
    """On bfloat16-representable inputs the bf16 call is the fp32 call rounded."""
    w = workloads.custom("bf16fp32", 2, 500, 4, 4, q_kind="gauss4", seed=62)
    (tq, ti, td), _ = bf16_inputs(dev, w)
    c16 = qs.quat_cumprod_fwd_bf16(tq, ti).float()
    c32 = qs.quat_cumprod_fwd(tq.float(), ti.float())
    g16, i16 = qs.quat_cumprod_bwd_bf16(tq, ti, td)
    g32, i32 = qs.quat_cumprod_bwd(tq.float(), ti.float(), td.float())
    for a, b in ((c16, c32), (g16.float(), g32), (i16.float(), i32)):
        assert normwise(a.cpu().numpy(), b.cpu().numpy().astype(np.float64), "vs fp32", 2.0 ** -8 + 1e-5) \
            <= 2.0 ** -8 + 1e-5


@pytest.mark.parametrize("name,walk", [("mamba3", True), ("large", True), ("long", False), ("small", False)])
def test_bf16_plan_picks_the_design_by_lane_groups(dev, name, walk):
    """Walks for many lane groups (the forward only from three 16-lane groups per
    SM: large, not mamba3); else, for short sequences, the whole sequence of a
    few lanes in one CTA; else the segmented walk with per-unit tables forward
    (10), three kernels backward."""
    w = workloads.WORKLOADS[name]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fvariant, fkernels = qs.quat_cumprod_plan("fwd_bf16", w.B, w.S, w.H, w.J, device=dev)
    assert fkernels == 1
    fwalk = w.B * ((w.H * w.J + 15) // 16) >= 3 * sms
    assert fvariant == (1 if fwalk else 8 if w.S <= 1024 else 9 if w.S <= 2048 else 10), (name, fvariant)
    variant, kernels = qs.quat_cumprod_plan("bwd_bf16", w.B, w.S, w.H, w.J, device=dev)
    assert kernels == (1 if walk or w.S <= 2048 else 3)
    if not walk and w.S <= 2048:
        assert variant == (9 if w.S <= 512 else 8 if w.S <= 1024 else 10), (name, variant)
    if walk:   # more lane groups than two CTAs per SM hold: the register-capped walk (5)
        groups = w.B * ((w.H * w.J + 15) // 16)
        assert variant == (5 if groups > 2 * sms else 0), (name, variant, groups)


def test_bf16_long_sequence_sampled_lanes(dev):
    """The long workload (few lanes: aggregate / carry / apply) at full size, sampled lanes."""
    w = workloads.WORKLOADS["long"]
    (tq, ti, td), _ = bf16_inputs(dev, w)
    cum = qs.quat_cumprod_fwd_bf16(tq, ti)
    d_q, d_init = qs.quat_cumprod_bwd_bf16(tq, ti, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    lanes = np.random.default_rng(4).choice(w.lanes, 6, replace=False)
    host = [t.float().cpu().numpy() for t in (tq, ti, td, cum, d_q, d_init)]
    sq, si, sd = (a.astype(np.float64) for a in workloads.sample_lanes(host[:3], lanes, w.H, w.J))
    gc, gq, gi = workloads.sample_lanes(host[3:], lanes, w.H, w.J)
    ref_dq, ref_di = oracle.bwd(sq, si, sd)
    assert normwise(gc, oracle.fwd(sq, si)) <= TOL_BF16
    assert normwise(gq, ref_dq) <= TOL_BF16
    assert normwise(gi, ref_di) <= TOL_BF16


@pytest.mark.parametrize("name", ["tiny", "small", "mamba3", "large", "long"])
def test_bf16_named_workloads(dev, name):
    """Every workload in bfloat16, in the configuration the library picks: the
    two smallest compared in full, the others (at full size) on sampled whole
    lanes."""
    w = workloads.WORKLOADS[name]
    (tq, ti, td), exact = bf16_inputs(dev, w)
    cum = qs.quat_cumprod_fwd_bf16(tq, ti)
    d_q, d_init = qs.quat_cumprod_bwd_bf16(tq, ti, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    got = [t.float().cpu().numpy() for t in (cum, d_q, d_init)]
    if w.elements <= 1 << 20:
        q, init, d_cum = exact
        ref = [oracle.fwd(q, init), *oracle.bwd(q, init, d_cum)]
    else:
        lanes = np.unique(np.concatenate([[0, w.lanes - 1],
                                          np.random.default_rng(5).choice(w.lanes, 12, replace=False)]))
        sq, si, sd = workloads.sample_lanes(exact, lanes, w.H, w.J)
        ref = [oracle.fwd(sq, si), *oracle.bwd(sq, si, sd)]
        got = list(workloads.sample_lanes(got, lanes, w.H, w.J))
    for g, r, t in zip(got, ref, ("cum", "d_q", "d_init")):
        err = normwise(g, r, t)
        assert err <= TOL_BF16, f"{name} {t}: {err:.3e} > {TOL_BF16:.3e}"


def test_bf16_unknown_variant_is_rejected(dev):
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant_bf16(N_BF16_FWD, 0) == qs.QS_ERR_DIMS
    assert lib.quat_cumprod_debug_set_variant_bf16(0, N_BF16_BWD) == qs.QS_ERR_DIMS


def test_bf16_rejects_odd_lane_count_and_wrong_dtype(dev):
    q = torch.zeros(1, 8, 3, 1, 4, device=dev, dtype=torch.bfloat16)
    init = torch.zeros(1, 3, 1, 4, device=dev, dtype=torch.bfloat16)
    with pytest.raises(qs.QuatScanError) as ei:
        qs.quat_cumprod_fwd_bf16(q, init)
    assert ei.value.status == qs.QS_ERR_DIMS
    with pytest.raises(TypeError):
        qs.quat_cumprod_fwd_bf16(q.float(), init.float())
    # S == 0: d_init is zero
    q0 = torch.zeros(2, 0, 2, 1, 4, device=dev, dtype=torch.bfloat16)
    i0 = torch.ones(2, 2, 1, 4, device=dev, dtype=torch.bfloat16)
    _, di = qs.quat_cumprod_bwd_bf16(q0, i0, q0.clone())
    torch.cuda.synchronize(dev)
    assert float(di.float().abs().max()) == 0.0


def test_bf16_graph_capture_replays_match_the_oracle(dev):
    """A bf16 forward and backward captured into a CUDA graph, replayed on new inputs.

    Eagerly the forward for few lane groups is the segmented walk, whose status
    words are tied to one launch; under capture it is the three-kernel forward."""
    dims = (1, 20000, 2, 16)

    def inputs(seed):
        return bf16_inputs(dev, workloads.custom("graph16", *dims, q_kind="rotation", theta_max=0.3, seed=seed))

    (tq, ti, td), _ = inputs(140)
    cum, dq, di = torch.empty_like(tq), torch.empty_like(tq), torch.empty_like(ti)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):   # sizes the capture stream's scratch
        qs.quat_cumprod_fwd_bf16(tq, ti, cum)
        qs.quat_cumprod_bwd_bf16(tq, ti, td, dq, di)
    assert qs.quat_cumprod_status(stream=s, device=dev) == qs.QS_OK
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        qs.quat_cumprod_fwd_bf16(tq, ti, cum)
        qs.quat_cumprod_bwd_bf16(tq, ti, td, dq, di)
    for seed in (141, 142):
        (nq, ni, nd), (eq, ei, ed) = inputs(seed)
        tq.copy_(nq)
        ti.copy_(ni)
        td.copy_(nd)
        g.replay()
        torch.cuda.synchronize(dev)
        assert qs.quat_cumprod_status(stream=s, device=dev) == qs.QS_OK
        assert normwise(cum.float().cpu().numpy(), oracle.fwd(eq, ei)) <= TOL_BF16
        rq, ri = oracle.bwd(eq, ei, ed)
        assert normwise(dq.float().cpu().numpy(), rq) <= TOL_BF16
        assert normwise(di.float().cpu().numpy(), ri) <= TOL_BF16
