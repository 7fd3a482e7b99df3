"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerance: for every output tensor, the normwise relative error
``max_i |gpu_i - ref_i| / max_i |ref_i|`` must be <= 1e-4 (fp32 I/O and fp32
arithmetic against the exact-input fp64 oracle).  Workloads are the seeded
synthetic ones of ``workloads.py``; the two largest are run at full size in the
benchmark's launch configuration and compared on whole sampled lanes (lanes
are independent, so the oracle on a lane subset is exact).
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
import parity_log
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


@pytest.fixture(autouse=True)
def reset_hooks():
    lib = qs.load_library()
    yield
    lib.quat_cumprod_debug_set_timeout_ns(0)
    lib.quat_cumprod_debug_stall_tile(-1)
    lib.quat_cumprod_debug_set_variant(-1, -1)
    lib.quat_cumprod_debug_set_walk_cap(-1)


normwise = parity_log.normwise


def run_gpu(dev, q, init, d_cum, stream=None):
    tq, ti, td = (torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in (q, init, d_cum))
    cum = qs.quat_cumprod_fwd(tq, ti, stream=stream)
    d_q, d_init = qs.quat_cumprod_bwd(tq, ti, td, stream=stream)
    st = qs.quat_cumprod_status(stream=stream, device=dev)
    assert st == qs.QS_OK, qs.quat_cumprod_strerror(st)
    return cum.cpu().numpy(), d_q.cpu().numpy(), d_init.cpu().numpy()


def assert_parity(got, ref, what):
    """The pass criterion (normwise); with QS_PARITY_LOG set, both measures are logged."""
    err = normwise(got, ref)
    parity_log.record(what, "fp32", got, ref, TOL, err)
    assert err <= TOL, f"{what}: normwise relative error {err:.3e} > {TOL}"
    return err


def check_against_oracle(dev, q, init, d_cum, stream=None):
    cum, d_q, d_init = run_gpu(dev, q, init, d_cum, stream)
    ref_cum = oracle.fwd(q, init)
    ref_dq, ref_di = oracle.bwd(q, init, d_cum)
    return (assert_parity(cum, ref_cum, "cum"), assert_parity(d_q, ref_dq, "d_q"),
            assert_parity(d_init, ref_di, "d_init"))


# ---------------------------------------------------------------------------
# Named workloads.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["tiny", "small", "mamba3"])
def test_named_workload_full_parity(dev, name):
    w = workloads.WORKLOADS[name]
    check_against_oracle(dev, *workloads.make_inputs(w))


def _sampled_lane_parity(dev, w, nlanes, seed):
    q, init, d_cum = workloads.make_inputs(w)
    tq, ti, td = (torch.from_numpy(a).to(dev) for a in (q, init, d_cum))
    cum = qs.quat_cumprod_fwd(tq, ti)
    d_q, d_init = qs.quat_cumprod_bwd(tq, ti, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    rng = np.random.default_rng(seed)
    HJ = w.H * w.J
    lanes = np.unique(np.concatenate([[0, 31, 32, HJ - 1, w.lanes - 1],
                                      rng.choice(w.lanes, nlanes, replace=False)]))
    b = torch.from_numpy(lanes // HJ).to(dev)
    hj = torch.from_numpy(lanes % HJ).to(dev)
    g_cum = cum.view(w.B, w.S, HJ, 4)[b, :, hj].cpu().numpy()        # [n, S, 4]
    g_dq = d_q.view(w.B, w.S, HJ, 4)[b, :, hj].cpu().numpy()
    g_di = d_init.view(w.B, HJ, 4)[b, hj].cpu().numpy()
    del cum, d_q, d_init, tq, td
    sq, si, sd = workloads.sample_lanes((q, init, d_cum), lanes, w.H, w.J)
    ref_cum = oracle.fwd(sq, si)[0, :, :, 0].transpose(1, 0, 2)
    ref_dq, ref_di = oracle.bwd(sq, si, sd)
    assert_parity(g_cum, ref_cum, "cum (sampled lanes)")
    assert_parity(g_dq, ref_dq[0, :, :, 0].transpose(1, 0, 2), "d_q (sampled lanes)")
    assert_parity(g_di, ref_di[0, :, 0], "d_init (sampled lanes)")


def test_large_full_size_sampled_lanes(dev):
    _sampled_lane_parity(dev, workloads.WORKLOADS["large"], 48, 5)


def test_long_sequence_full_size(dev):
    w = workloads.WORKLOADS["long"]
    _sampled_lane_parity(dev, w, 60, 6)


def test_mamba3_full_size_sampled_lanes(dev):
    _sampled_lane_parity(dev, workloads.WORKLOADS["mamba3"], 64, 7)


# ---------------------------------------------------------------------------
# Edge shapes: ragged sequence tails, lane counts that are not multiples of
# 32 (partial lane groups, groups of several batch entries), S < tile, S = 1.
# ---------------------------------------------------------------------------
EDGE = [(1, 1, 1, 1), (1, 2, 1, 1), (2, 33, 1, 1), (1, 100, 2, 3), (3, 257, 5, 8),
        (2, 31, 40, 1), (1, 64, 4, 8), (2, 500, 1, 32), (1, 1000, 3, 17), (4, 65, 2, 16),
        (1, 4099, 1, 33), (2, 129, 8, 8)]


@pytest.mark.parametrize("dims", EDGE)
def test_edge_shapes(dev, dims):
    B, S, H, J = dims
    w = workloads.custom("edge", B, S, H, J, seed=sum(dims))
    check_against_oracle(dev, *workloads.make_inputs(w))


def test_non_unit_quaternions(dev):
    """The backward is exact for all quaternions (no unit assumption)."""
    rng = np.random.default_rng(3)
    B, S, H, J = 2, 700, 2, 20
    q = rng.standard_normal((B, S, H, J, 4))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    q *= rng.uniform(0.995, 1.005, (B, S, H, J, 1))
    init = (rng.standard_normal((B, H, J, 4)) * 2).astype(np.float32)
    d_cum = rng.standard_normal((B, S, H, J, 4)).astype(np.float32)
    check_against_oracle(dev, q.astype(np.float32), init, d_cum)
    # strongly non-unit on a short sequence
    q2 = (rng.standard_normal((1, 24, 3, 7, 4)) * 1.5).astype(np.float32)
    init2 = rng.standard_normal((1, 3, 7, 4)).astype(np.float32)
    check_against_oracle(dev, q2, init2, rng.standard_normal(q2.shape).astype(np.float32))


def test_identity_q_is_reverse_cumsum(dev):
    rng = np.random.default_rng(4)
    B, S, H, J = 2, 300, 1, 40
    q = np.zeros((B, S, H, J, 4), np.float32)
    q[..., 0] = 1
    init = rng.standard_normal((B, H, J, 4)).astype(np.float32)
    d_cum = rng.standard_normal((B, S, H, J, 4)).astype(np.float32)
    cum, d_q, d_init = run_gpu(dev, q, init, d_cum)
    np.testing.assert_array_equal(cum, np.broadcast_to(init[:, None], cum.shape))
    G = np.flip(np.cumsum(np.flip(d_cum.astype(np.float64), 1), 1), 1)
    assert_parity(d_init, G[:, 0], "d_init")


def test_empty_sizes(dev):
    z = torch.zeros(0, device=dev)
    for B, S, H, J in [(0, 5, 2, 2), (2, 5, 0, 2), (2, 5, 2, 0)]:
        q = torch.zeros(B, S, H, J, 4, device=dev)
        init = torch.zeros(B, H, J, 4, device=dev)
        assert qs.quat_cumprod_fwd(q, init).shape == q.shape
        gq, gi = qs.quat_cumprod_bwd(q, init, q)
        assert gq.shape == q.shape and gi.shape == init.shape
    q = torch.zeros(3, 0, 2, 2, 4, device=dev)
    init = torch.randn(3, 2, 2, 4, device=dev)
    gi = torch.full_like(init, 7.0)
    qs.quat_cumprod_bwd(q, init, q, d_init=gi)
    torch.cuda.synchronize()
    assert torch.count_nonzero(gi).item() == 0
    del z


# Variants 0-3: aggregate / carry / apply kernels; the rest: walk kernels
# (forward 8: chained scan; 9: segmented chained walk; 10, 11: the same,
# warp-specialised; 12: as 9, look-back values that carry their own state, read
# in one round trip; 13, 14: as 10, 11 with those values; backward 10: at most
# two CTAs per SM, more lane groups in waves; backward 11-14: the segmented
# walk of the backward, after its carries-only forward pass; forward and
# backward 25-29: short sequences, a lane group's whole sequence in one CTA;
# backward 30-33: the segmented walk of the backward with walk 2 two or three
# units behind).
N_FWD_VARIANTS, N_BWD_VARIANTS = 30, 34
SEGWALK_FWD = [9, 10, 11, 12, 13, 14, 15, 16, 17, 18, 19, 20, 21, 22, 23, 24]
SEGWALK_BWD = [11, 12, 13, 14, 15, 16, 17, 18, 19, 20, 21, 22, 23, 24, 30, 31, 32, 33]


@pytest.mark.parametrize("variant", range(max(N_FWD_VARIANTS, N_BWD_VARIANTS)))
@pytest.mark.parametrize("dims", [(2, 333, 3, 16), (1, 70, 5, 9), (3, 1100, 1, 40), (1, 5000, 2, 32)])
def test_every_compiled_variant(dev, variant, dims):
    """Each compiled configuration (lane-group width, steps per thread, cluster size, stages).

    The sizes give chunk counts below, at and above the cluster sizes, ragged
    lane groups and ragged last chunks.
    """
    lib = qs.load_library()
    fv = variant if variant < N_FWD_VARIANTS else -1
    bv = variant if variant < N_BWD_VARIANTS else -1
    assert lib.quat_cumprod_debug_set_variant(fv, bv) == qs.QS_OK
    B, S, H, J = dims
    w = workloads.custom("variant", B, S, H, J, q_kind="rotation", theta_max=0.5, seed=variant)
    check_against_oracle(dev, *workloads.make_inputs(w))


@pytest.mark.parametrize("variant", [0, 1])   # 64- and 32-step chunks
@pytest.mark.parametrize("dims", [(1, 20000, 1, 3), (2, 17000, 2, 5)])
def test_many_chunks_per_lane_carry_scan(dev, variant, dims):
    """More than 256 chunks per lane: the carry step scans 256 chunk ranges per lane."""
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(variant, variant) == qs.QS_OK
    w = workloads.custom("chunks", *dims, q_kind="rotation", theta_max=0.3, seed=71 + variant)
    check_against_oracle(dev, *workloads.make_inputs(w))


@pytest.mark.parametrize("cap", [1, 2, 3, 5])
@pytest.mark.parametrize("variant", [4, 8, 10])   # fold by segments 0 and 1, every thread folds, capped
def test_backward_walk_in_waves(dev, variant, cap):
    """A CTA walks several lane groups one after another (grid capped below the group count).

    3 x 48 lanes: 9 groups of 16 lanes; caps 1, 2, 3, 5 give one CTA
    walking every group, and waves whose last one is ragged.  The backward from
    saved carries (the reverse walk alone) runs under the same cap.
    """
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(-1, variant) == qs.QS_OK
    assert lib.quat_cumprod_debug_set_walk_cap(cap) == qs.QS_OK
    w = workloads.custom("waves", 3, 333, 2, 24, q_kind="rotation", theta_max=0.6, seed=80 + cap)
    q, init, d_cum = workloads.make_inputs(w)
    check_against_oracle(dev, q, init, d_cum)
    tq, ti, td = (torch.from_numpy(a).to(dev) for a in (q, init, d_cum))
    _, carries = qs.quat_cumprod_fwd_carries(tq, ti)
    d_q, d_init = qs.quat_cumprod_bwd_carries(tq, carries, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    rq, ri = oracle.bwd(q, init, d_cum)
    assert_parity(d_q.cpu().numpy(), rq, "d_q (from carries)")
    assert_parity(d_init.cpu().numpy(), ri, "d_init (from carries)")


def test_stall_in_a_later_wave_reports_timeout_then_recovers(dev):
    """2 x 32 lanes = 4 groups of 16, cap 3: two CTAs walk two groups each.

    The stalled tile is chunk 0 of group 2, the second group of CTA 0.
    """
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(-1, 4) == qs.QS_OK
    assert lib.quat_cumprod_debug_set_walk_cap(3) == qs.QS_OK
    w = workloads.custom("stall_wave", 2, 600, 2, 16, seed=22)
    q, init, d_cum = workloads.make_inputs(w)
    tq, ti, td = (torch.from_numpy(a).to(dev) for a in (q, init, d_cum))
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    lib.quat_cumprod_debug_set_timeout_ns(50_000_000)    # 50 ms
    lib.quat_cumprod_debug_stall_tile(2)                 # item c * NG + g = 0 * 4 + 2
    qs.quat_cumprod_bwd(tq, ti, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_ERR_TIMEOUT
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    lib.quat_cumprod_debug_stall_tile(-1)
    lib.quat_cumprod_debug_set_timeout_ns(0)
    check_against_oracle(dev, q, init, d_cum)


@pytest.mark.parametrize("variant", SEGWALK_FWD)
@pytest.mark.parametrize("dims", [(1, 20000, 1, 3), (2, 17000, 2, 5), (1, 131072 // 8, 2, 16)])
def test_segmented_walk_long_sequences(dev, variant, dims):
    """Many segments per lane (up to 40): the look-back chains over segments."""
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(variant, -1) == qs.QS_OK
    w = workloads.custom("segwalk", *dims, q_kind="rotation", theta_max=0.3, seed=90 + variant)
    q, init, d_cum = workloads.make_inputs(w)
    tq, ti = (torch.from_numpy(a).to(dev) for a in (q, init))
    for _ in range(2):   # a second launch reuses the status words and the ticket counter
        cum = qs.quat_cumprod_fwd(tq, ti)
        assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
        assert_parity(cum.cpu().numpy(), oracle.fwd(q, init), "cum")


def test_segmented_walk_alternating_layouts(dev):
    """Configuration 12 keeps its look-back values between launches on a stream
    (two buffers, each launch resetting the one the next reads): shapes that
    alternate change the layout, repeats reuse it, and every result must match."""
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(12, -1) == qs.QS_OK
    cases = []
    for i, dims in enumerate([(1, 20000, 1, 3), (2, 17000, 2, 5), (1, 9000, 2, 16)]):
        w = workloads.custom("seg_alt", *dims, q_kind="rotation", theta_max=0.3, seed=110 + i)
        q, init, _ = workloads.make_inputs(w)
        cases.append((q, init, oracle.fwd(q, init)))
    for k in [0, 0, 1, 0, 2, 2, 2, 1, 1, 0]:
        q, init, ref = cases[k]
        cum = qs.quat_cumprod_fwd(*(torch.from_numpy(a).to(dev) for a in (q, init)))
        assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
        assert_parity(cum.cpu().numpy(), ref, f"cum (case {k})")


@pytest.mark.parametrize("variant", [9, 10, 12, 13, 19, 20, 22, 24])   # one CTA role, warp-specialised, each with self-describing values; per-unit tables
def test_segmented_walk_stall_reports_timeout_then_recovers(dev, variant):
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(variant, -1) == qs.QS_OK
    w = workloads.custom("segstall", 2, 3000, 2, 16, seed=23)
    q, init, d_cum = workloads.make_inputs(w)
    tq, ti = (torch.from_numpy(a).to(dev) for a in (q, init))
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    lib.quat_cumprod_debug_set_timeout_ns(50_000_000)    # 50 ms
    lib.quat_cumprod_debug_stall_tile(1)                 # chunk 0 of lane group 1
    qs.quat_cumprod_fwd(tq, ti)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_ERR_TIMEOUT
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    lib.quat_cumprod_debug_stall_tile(-1)
    lib.quat_cumprod_debug_set_timeout_ns(0)
    cum = qs.quat_cumprod_fwd(tq, ti)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    assert_parity(cum.cpu().numpy(), oracle.fwd(q, init), "cum")


def test_segmented_walk_from_concurrent_threads(dev):
    """Host threads enqueue the segmented-walk forward (few lane groups) on
    streams of their own at the same time: each stream keeps its own look-back
    buffers and workspace, and every result must match the oracle."""
    import threading
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(-1, -1) == qs.QS_OK
    cases = []
    for i, dims in enumerate([(1, 20000, 2, 16), (2, 9000, 1, 32), (1, 30000, 1, 16)]):
        w = workloads.custom("seg_threads", *dims, q_kind="rotation", theta_max=0.3, seed=150 + i)
        q, init, _ = workloads.make_inputs(w)
        cases.append((torch.from_numpy(q).to(dev), torch.from_numpy(init).to(dev), oracle.fwd(q, init)))
    torch.cuda.synchronize(dev)
    errors = []

    def worker(k):
        try:
            torch.cuda.set_device(dev)
            s = torch.cuda.Stream(device=dev)
            tq, ti, ref = cases[k]
            with torch.cuda.stream(s):
                for _ in range(4):
                    cum = qs.quat_cumprod_fwd(tq, ti)
                    assert qs.quat_cumprod_status(stream=s, device=dev) == qs.QS_OK
                    errors.append((k, normwise(cum.cpu().numpy(), ref)))
        except Exception as e:   # reported below
            errors.append((k, repr(e)))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert len(errors) == 4 * len(cases), errors
    for k, e in errors:
        assert isinstance(e, float) and e <= 1e-4, (k, e)


@pytest.mark.parametrize("dims", [(1, 20000, 2, 16), (2, 1000, 3, 8)])
def test_graph_capture_replays_match_the_oracle(dev, dims):
    """A forward and a backward captured into a CUDA graph, replayed on new inputs.

    Both shapes have few lane groups.  On the long one an eager forward is the
    segmented walk, whose look-back values are tied to the launch that reads
    them; under capture the library takes the aggregate / carry / apply
    forward instead.  The short one runs the short-sequence kernels, which keep
    no state and are captured as they are.  Every replay must match the
    oracle."""
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(-1, -1) == qs.QS_OK

    def inputs(seed):
        return workloads.make_inputs(workloads.custom("graph", *dims, q_kind="rotation", theta_max=0.3, seed=seed))

    q, init, d_cum = inputs(130)
    tq, ti, td = (torch.from_numpy(a).to(dev) for a in (q, init, d_cum))
    cum, dq, di = torch.empty_like(tq), torch.empty_like(tq), torch.empty_like(ti)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):   # sizes the capture stream's scratch
        qs.quat_cumprod_fwd(tq, ti, cum)
        qs.quat_cumprod_bwd(tq, ti, td, dq, di)
    assert qs.quat_cumprod_status(stream=s, device=dev) == qs.QS_OK
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        qs.quat_cumprod_fwd(tq, ti, cum)
        qs.quat_cumprod_bwd(tq, ti, td, dq, di)
    for seed in (131, 132, 133):
        q, init, d_cum = inputs(seed)
        tq.copy_(torch.from_numpy(q))
        ti.copy_(torch.from_numpy(init))
        td.copy_(torch.from_numpy(d_cum))
        g.replay()
        torch.cuda.synchronize(dev)
        assert qs.quat_cumprod_status(stream=s, device=dev) == qs.QS_OK
        assert_parity(cum.cpu().numpy(), oracle.fwd(q, init), "cum (replay)")
        rq, ri = oracle.bwd(q, init, d_cum)
        assert_parity(dq.cpu().numpy(), rq, "d_q (replay)")
        assert_parity(di.cpu().numpy(), ri, "d_init (replay)")


def test_unknown_variant_is_rejected(dev):
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(N_FWD_VARIANTS, 0) == qs.QS_ERR_DIMS
    assert lib.quat_cumprod_debug_set_variant(0, N_BWD_VARIANTS) == qs.QS_ERR_DIMS


def test_repeated_calls_and_side_stream(dev):
    w = workloads.WORKLOADS["small"]
    q, init, d_cum = workloads.make_inputs(w)
    s = torch.cuda.Stream(device=dev)
    for _ in range(3):
        check_against_oracle(dev, q, init, d_cum)
    with torch.cuda.stream(s):
        check_against_oracle(dev, q, init, d_cum, stream=s)


def test_unaligned_base_views(dev):
    """Tensors that start 16 bytes into an allocation (TMA base alignment is 16 B)."""
    w = workloads.custom("view", 2, 77, 3, 5, seed=12)
    q, init, d_cum = workloads.make_inputs(w)
    n = q.size
    big = torch.zeros(n + 4, device=dev)
    big[4:] = torch.from_numpy(q.ravel()).to(dev)
    tq = big[4:].view(q.shape)
    ti = torch.from_numpy(init).to(dev)
    bigd = torch.zeros(n + 8, device=dev)
    bigd[8:] = torch.from_numpy(d_cum.ravel()).to(dev)
    td = bigd[8:].view(q.shape)
    cum = qs.quat_cumprod_fwd(tq, ti)
    d_q, d_init = qs.quat_cumprod_bwd(tq, ti, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    assert_parity(cum.cpu().numpy(), oracle.fwd(q, init), "cum")
    rq, ri = oracle.bwd(q, init, d_cum)
    assert_parity(d_q.cpu().numpy(), rq, "d_q")
    assert_parity(d_init.cpu().numpy(), ri, "d_init")


def test_binding_rejects_bad_tensors(dev):
    q = torch.zeros(1, 4, 1, 1, 4, device=dev)
    init = torch.zeros(1, 1, 1, 4, device=dev)
    with pytest.raises(TypeError):
        qs.quat_cumprod_fwd(q.double(), init)
    with pytest.raises(ValueError):
        qs.quat_cumprod_fwd(q.cpu(), init)
    with pytest.raises(ValueError):
        qs.quat_cumprod_fwd(q, init[:, :, :, :3])
    with pytest.raises(ValueError):
        qs.quat_cumprod_fwd(torch.zeros(1, 4, 1, 2, 4, device=dev)[:, :, :, :1], init)
    with pytest.raises(qs.QuatScanError) as ei:
        qs.quat_cumprod_fwd(q, init, cum=q)
    assert ei.value.status == qs.QS_ERR_ALIAS


# Short-sequence configurations: variant -> longest sequence.
SHORT_FWD = {25: 1024, 26: 1024, 27: 1024, 28: 2048, 29: 256}
SHORT_BWD = {25: 1024, 26: 1024, 27: 512, 28: 2048, 29: 256}
SHORT_PAIRS = [(25, 25), (26, 26), (27, 27), (28, 28), (29, 29), (26, 25)]


@pytest.mark.parametrize("fv,bv", SHORT_PAIRS)
@pytest.mark.parametrize("at", ["one", "chunk-1", "chunk", "chunk+1", "max-1", "max"])
def test_short_sequences(dev, fv, bv, at):
    """A lane group's whole sequence in one CTA: lengths from one step to the
    configuration's longest (one chunk of the carries and one step either side),
    lane groups ragged on both sides (H*J = 3 x 7 is no multiple of the lanes)."""
    lib = qs.load_library()
    smax = min(SHORT_FWD[fv], SHORT_BWD[bv])
    S = {"one": 1, "chunk-1": 63, "chunk": 64, "chunk+1": 65, "max-1": smax - 1, "max": smax}[at]
    assert lib.quat_cumprod_debug_set_variant(fv, bv) == qs.QS_OK
    assert qs.quat_cumprod_plan("fwd", 2, S, 3, 7, device=dev) == (fv, 1)
    assert qs.quat_cumprod_plan("bwd", 2, S, 3, 7, device=dev) == (bv, 1)
    w = workloads.custom("short", 2, S, 3, 7, q_kind="gauss4", seed=fv * 8 + len(at))
    check_against_oracle(dev, *workloads.make_inputs(w))


@pytest.mark.parametrize("fv,bv", SHORT_PAIRS)
def test_short_sequences_non_unit_quaternions(dev, fv, bv):
    """The scans compose segment products and affine cotangent maps exactly for
    every quaternion: norms drifting along the configuration's longest sequence,
    a large init, and ragged lane groups."""
    lib = qs.load_library()
    S = min(SHORT_FWD[fv], SHORT_BWD[bv])
    rng = np.random.default_rng(fv * 31 + bv)
    q = rng.standard_normal((2, S, 3, 5, 4))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    q *= rng.uniform(0.999, 1.001, (2, S, 3, 5, 1))
    init = (rng.standard_normal((2, 3, 5, 4)) * 3).astype(np.float32)
    d_cum = rng.standard_normal(q.shape).astype(np.float32)
    assert lib.quat_cumprod_debug_set_variant(fv, bv) == qs.QS_OK
    assert qs.quat_cumprod_plan("fwd", 2, S, 3, 5, device=dev) == (fv, 1)
    assert qs.quat_cumprod_plan("bwd", 2, S, 3, 5, device=dev) == (bv, 1)
    check_against_oracle(dev, q.astype(np.float32), init, d_cum)


@pytest.mark.parametrize("fv,bv", [(25, 25), (28, 28)])
def test_short_sequences_past_their_length_take_another_design(dev, fv, bv):
    """A short-sequence configuration asked for a longer sequence is not used."""
    lib = qs.load_library()
    fmax, bmax = SHORT_FWD[fv], SHORT_BWD[bv]
    assert lib.quat_cumprod_debug_set_variant(fv, bv) == qs.QS_OK
    assert qs.quat_cumprod_plan("fwd", 1, fmax + 1, 2, 4, device=dev)[0] != fv
    assert qs.quat_cumprod_plan("bwd", 1, bmax + 1, 2, 4, device=dev)[0] != bv
    w = workloads.custom("short-past", 1, bmax + 1, 2, 4, q_kind="rotation", theta_max=0.5, seed=fv)
    check_against_oracle(dev, *workloads.make_inputs(w))


@pytest.mark.parametrize("variant", SEGWALK_BWD)
@pytest.mark.parametrize("dims", [(1, 20000, 1, 3), (2, 17000, 2, 5), (1, 131072 // 8, 2, 16), (3, 64 * 9 + 1, 1, 33)])
def test_segmented_backward_long_sequences(dev, variant, dims):
    """Many segments per lane (up to 79): the backward's look-back chains the
    segments' affine maps from the right end; ragged last chunk and lane group.
    Two launches in a row read the two sets of look-back buffers in turn."""
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(-1, variant) == qs.QS_OK
    w = workloads.custom("segbwd", *dims, q_kind="rotation", theta_max=0.3, seed=170 + variant)
    q, init, d_cum = workloads.make_inputs(w)
    tq, ti, td = (torch.from_numpy(a).to(dev) for a in (q, init, d_cum))
    rq, ri = oracle.bwd(q, init, d_cum)
    for _ in range(2):
        d_q, d_init = qs.quat_cumprod_bwd(tq, ti, td)
        assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
        assert_parity(d_q.cpu().numpy(), rq, "d_q")
        assert_parity(d_init.cpu().numpy(), ri, "d_init")
    _, carries = qs.quat_cumprod_fwd_carries(tq, ti)   # and from saved carries
    d_q, d_init = qs.quat_cumprod_bwd_carries(tq, carries, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    assert_parity(d_q.cpu().numpy(), rq, "d_q (from carries)")
    assert_parity(d_init.cpu().numpy(), ri, "d_init (from carries)")


@pytest.mark.parametrize("cap", [1, 2, 5])
@pytest.mark.parametrize("variant", [22, 24, 31])
def test_segmented_backward_few_ctas(dev, variant, cap):
    """The persistent grid capped below the units in flight (one CTA takes every
    unit in ticket order): a unit waits only on units taken before it, also with
    walk 2 two units behind walk 1; recomputing and from saved carries."""
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(-1, variant) == qs.QS_OK
    assert lib.quat_cumprod_debug_set_walk_cap(cap) == qs.QS_OK
    w = workloads.custom("segbwd_cap", 2, 3000, 2, 16, q_kind="rotation", theta_max=0.4, seed=90 + cap)
    q, init, d_cum = workloads.make_inputs(w)
    check_against_oracle(dev, q, init, d_cum)
    tq, ti, td = (torch.from_numpy(a).to(dev) for a in (q, init, d_cum))
    _, carries = qs.quat_cumprod_fwd_carries(tq, ti)
    d_q, d_init = qs.quat_cumprod_bwd_carries(tq, carries, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    rq, ri = oracle.bwd(q, init, d_cum)
    assert_parity(d_q.cpu().numpy(), rq, "d_q (from carries)")
    assert_parity(d_init.cpu().numpy(), ri, "d_init (from carries)")


@pytest.mark.parametrize("fv,bv", [(-1, 11), (24, 31), (22, 24)])
def test_segmented_backward_non_unit_quaternions(dev, fv, bv):
    """The affine segment maps are exact for every quaternion: strongly non-unit
    q over many segments (norms drift far from one along the sequence); the
    table forward and the backward with walk 2 two units behind as well."""
    rng = np.random.default_rng(9)
    B, S, H, J = 1, 5000, 2, 8
    q = rng.standard_normal((B, S, H, J, 4))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    q *= rng.uniform(0.999, 1.0012, (B, S, H, J, 1))
    q = q.astype(np.float32)
    init = (rng.standard_normal((B, H, J, 4)) * 3).astype(np.float32)
    d_cum = rng.standard_normal(q.shape).astype(np.float32)
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(fv, bv) == qs.QS_OK
    check_against_oracle(dev, q, init, d_cum)


def test_segmented_backward_alternating_layouts(dev):
    """Forward, backward and the backward's carries pass each keep their own
    look-back buffers between launches on a stream: shapes that alternate
    change the layouts, repeats reuse them, and every result must match."""
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(-1, 11) == qs.QS_OK
    cases = []
    for i, dims in enumerate([(1, 20000, 1, 3), (2, 17000, 2, 5), (1, 9000, 2, 16)]):
        w = workloads.custom("segbwd_alt", *dims, q_kind="rotation", theta_max=0.3, seed=180 + i)
        q, init, d_cum = workloads.make_inputs(w)
        cases.append((q, init, d_cum, oracle.fwd(q, init), *oracle.bwd(q, init, d_cum)))
    for k in [0, 0, 1, 0, 2, 2, 2, 1, 1, 0]:
        q, init, d_cum, rc, rq, ri = cases[k]
        tq, ti, td = (torch.from_numpy(a).to(dev) for a in (q, init, d_cum))
        cum = qs.quat_cumprod_fwd(tq, ti)
        d_q, d_init = qs.quat_cumprod_bwd(tq, ti, td)
        assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
        assert_parity(cum.cpu().numpy(), rc, f"cum (case {k})")
        assert_parity(d_q.cpu().numpy(), rq, f"d_q (case {k})")
        assert_parity(d_init.cpu().numpy(), ri, f"d_init (case {k})")


@pytest.mark.parametrize("variant", [11, 22, 31])   # one look-back warp, two; walk 2 two units behind
@pytest.mark.parametrize("saved", [False, True])
def test_segmented_backward_stall_reports_timeout_then_recovers(dev, saved, variant):
    """The stall hook holds the first kernel of the call: the carries-only pass
    of the recompute backward, or the segmented backward itself when it starts
    from saved carries.  Either way the call reports QS_ERR_TIMEOUT, and the
    next calls (which read the other set of look-back buffers) are clean."""
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(-1, variant) == qs.QS_OK
    w = workloads.custom("segbwd_stall", 2, 3000, 2, 16, seed=24)
    q, init, d_cum = workloads.make_inputs(w)
    tq, ti, td = (torch.from_numpy(a).to(dev) for a in (q, init, d_cum))
    assert qs.quat_cumprod_plan(True, 2, 3000, 2, 16, device=dev) == (variant, 2)
    _, carries = qs.quat_cumprod_fwd_carries(tq, ti)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    lib.quat_cumprod_debug_set_timeout_ns(50_000_000)    # 50 ms
    lib.quat_cumprod_debug_stall_tile(1)                 # chunk 0 of lane group 1
    if saved:
        qs.quat_cumprod_bwd_carries(tq, carries, td)
    else:
        qs.quat_cumprod_bwd(tq, ti, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_ERR_TIMEOUT
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    lib.quat_cumprod_debug_stall_tile(-1)
    lib.quat_cumprod_debug_set_timeout_ns(0)
    rq, ri = oracle.bwd(q, init, d_cum)
    for _ in range(2):
        d_q, d_init = (qs.quat_cumprod_bwd_carries(tq, carries, td) if saved else qs.quat_cumprod_bwd(tq, ti, td))
        assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
        assert_parity(d_q.cpu().numpy(), rq, "d_q")
        assert_parity(d_init.cpu().numpy(), ri, "d_init")


def test_segmented_backward_from_concurrent_threads(dev):
    """Host threads enqueue the segmented backward on streams of their own at
    the same time: each stream keeps its own look-back buffers and workspace."""
    import threading
    lib = qs.load_library()
    assert lib.quat_cumprod_debug_set_variant(-1, 11) == qs.QS_OK
    cases = []
    for i, dims in enumerate([(1, 20000, 2, 16), (2, 9000, 1, 32), (1, 30000, 1, 16)]):
        w = workloads.custom("segbwd_threads", *dims, q_kind="rotation", theta_max=0.3, seed=190 + i)
        q, init, d_cum = workloads.make_inputs(w)
        cases.append((*(torch.from_numpy(a).to(dev) for a in (q, init, d_cum)), oracle.bwd(q, init, d_cum)[0]))
    torch.cuda.synchronize(dev)
    errors = []

    def worker(k):
        try:
            torch.cuda.set_device(dev)
            s = torch.cuda.Stream(device=dev)
            tq, ti, td, ref = cases[k]
            with torch.cuda.stream(s):
                for _ in range(4):
                    d_q, _ = qs.quat_cumprod_bwd(tq, ti, td)
                    assert qs.quat_cumprod_status(stream=s, device=dev) == qs.QS_OK
                    errors.append((k, normwise(d_q.cpu().numpy(), ref)))
        except Exception as e:   # reported below
            errors.append((k, repr(e)))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert len(errors) == 4 * len(cases), errors
    for k, e in errors:
        assert isinstance(e, float) and e <= 1e-4, (k, e)


# ---------------------------------------------------------------------------
# Failure detection: a tile whose wait is made to expect bytes that never come
# runs out its bounded wait; the call reports QS_ERR_TIMEOUT (no hang) and the
# next call is clean.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("variant", [0, 4, 8])   # aggregate / carry / apply, walk, chained scan (fwd)
@pytest.mark.parametrize("which", ["fwd", "bwd"])
def test_stalled_tile_reports_timeout_then_recovers(dev, which, variant):
    lib = qs.load_library()
    if which == "bwd" and variant == 8:
        variant = 4   # the chained scan is a forward design
    assert lib.quat_cumprod_debug_set_variant(variant, variant) == qs.QS_OK
    w = workloads.custom("stall", 2, 600, 2, 16, seed=21)
    q, init, d_cum = workloads.make_inputs(w)
    tq, ti, td = (torch.from_numpy(a).to(dev) for a in (q, init, d_cum))
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    lib.quat_cumprod_debug_set_timeout_ns(50_000_000)    # 50 ms
    lib.quat_cumprod_debug_stall_tile(0)
    if which == "fwd":
        qs.quat_cumprod_fwd(tq, ti)
    else:
        qs.quat_cumprod_bwd(tq, ti, td)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_ERR_TIMEOUT
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK   # cleared
    lib.quat_cumprod_debug_stall_tile(-1)
    lib.quat_cumprod_debug_set_timeout_ns(0)
    check_against_oracle(dev, q, init, d_cum)


# ---------------------------------------------------------------------------
# Automatic choice of design: walk kernels when the lane groups fill the GPU,
# the three-kernel path otherwise.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name,walk", [("mamba3", True), ("large", True), ("long", False),
                                       ("small", False), ("tiny", False)])
def test_plan_picks_the_design_by_lane_groups(dev, name, walk):
    w = workloads.WORKLOADS[name]
    for bwd in (False, True):
        variant, kernels = qs.quat_cumprod_plan(bwd, w.B, w.S, w.H, w.J, device=dev)
        if not walk and w.S <= 2048:
            # short sequences: the whole sequence of a few lanes in one CTA,
            # the configuration that fits S (backward: 8 lanes up to 512 steps)
            assert kernels == 1, (name, bwd, variant, kernels)
            assert variant == ((27 if w.S <= 512 else 25) if bwd else 26), (name, bwd, variant)
            continue
        # few lane groups: the segmented chained walk forward (one kernel); the
        # backward: on long sequences (at least 4 units of 4 chunks per SM) the
        # carries pass and the segmented walk with walk 2 two units behind (31)
        units4 = w.B * ((w.H * w.J + 15) // 16) * ((w.S + 255) // 256)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        seg = bwd and not walk and units4 >= 4 * sms
        assert kernels == (1 if walk or not bwd else 2 if seg else 3), (name, bwd, variant, kernels)
        if not walk and not bwd:
            # the segmented walk with per-unit tables, segments of 2 chunks:
            # 32-lane groups (24) when there are at most 32 of them, else 16 (22)
            groups32 = w.B * ((w.H * w.J + 31) // 32)
            assert variant == (24 if groups32 <= 32 else 22), (name, variant)
        if not walk and bwd:
            assert variant == (31 if seg else 0), (name, variant)
    assert qs.quat_cumprod_plan(True, 2, 0, 3, 4, device=dev) == (-1, 0)


def test_plan_picks_the_segmented_backward_for_many_groups(dev):
    """64 or more 16-lane groups, too few for a walk: the recompute backward is
    the carries pass and the segmented walk (segments of 2 chunks)."""
    assert qs.quat_cumprod_plan(True, 1, 4096, 32, 32, device=dev) == (24, 2)   # 64 groups
    assert qs.quat_cumprod_plan(True, 1, 4096, 31, 32, device=dev) == (31, 2)   # 62 groups, 992 units
    assert qs.quat_cumprod_plan(True, 1, 4096, 16, 16, device=dev) == (0, 3)    # 16 groups, 256 units
    # from saved carries: the segmented walk whatever the group count
    assert qs.quat_cumprod_plan("bwd_carries", 1, 131072, 16, 16, device=dev) == (31, 1)
    assert qs.quat_cumprod_plan("bwd_carries", 4, 4096, 8, 16, device=dev) == (24, 1)   # few units
    assert qs.quat_cumprod_plan("bwd_carries", 4, 1024, 8, 16, device=dev) == (25, 1)   # short sequences
    w = workloads.custom("manygroups", 1, 2100, 32, 33, q_kind="rotation", theta_max=0.4, seed=200)
    assert qs.quat_cumprod_plan(True, w.B, w.S, w.H, w.J, device=dev) == (24, 2)
    check_against_oracle(dev, *workloads.make_inputs(w))
