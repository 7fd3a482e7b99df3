"""quat_cumprod_bwd_noalloc: the backward with a fixed scratch array, no allocation.

The GPU tests compare it, through the C ABI, with quat_cumprod_bwd on the same
inputs (normwise relative error <= 1e-4, the tolerance of the parity tests) on
two calls in a row that share the one scratch array.  The file is named to be
collected last, and its tests pass alone in a fresh process as well.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import quaternion_cumulative_product_gb300 as qs
from quaternion_cumulative_product_gb300 import build as qbuild
from quaternion_cumulative_product_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TOL = 1e-4


def normwise(got, ref):
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    scale = float(np.abs(ref).max())
    return float(np.abs(np.asarray(got, np.float64) - ref).max()) / (scale if scale > 0 else 1.0)


def _p(addr):
    return ctypes.c_void_p(addr)


# ---------------------------------------------------------------------------
# Host-side checks (no GPU): every case below returns before any CUDA call.
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def host_lib():
    qbuild.build()
    return qs.load_library()


def test_header_states_the_limit():
    text = open(os.path.join(ROOT, "include", "quat_cumprod.h")).read()
    m = re.search(r"#define\s+QS_NOALLOC_MAX_TILES\s+(\d+)", text)
    assert m and int(m.group(1)) == qs.QS_NOALLOC_MAX_TILES == 8192
    assert re.search(r"QS_ERR_SCRATCH\s*=\s*-9", text)


def test_noalloc_rejects_sizes_beyond_the_scratch(host_lib):
    f = host_lib.quat_cumprod_bwd_noalloc
    # buffers 2^40 bytes apart: no two overlap for any of these sizes
    q, d, gq, i, gi = (k << 40 for k in (1, 2, 3, 4, 5))
    # B * ceil(H*J/32) * ceil(S/64): 8193 tiles (one step past 8192 chunks)
    assert f(_p(q), _p(i), _p(d), _p(gq), _p(gi), 1, 64 * 8192 + 1, 1, 32, None) == qs.QS_ERR_SCRATCH
    # 33 lanes are two lane groups: 2 * 4097 tiles
    assert f(_p(q), _p(i), _p(d), _p(gq), _p(gi), 1, 64 * 4097, 1, 33, None) == qs.QS_ERR_SCRATCH
    # twice the 8 x 4096 x 16 x 32 problem that fills the scratch exactly
    assert f(_p(q), _p(i), _p(d), _p(gq), _p(gi), 16, 4096, 16, 32, None) == qs.QS_ERR_SCRATCH
    # the largest sizes the other limits allow (about 2^49 tiles); the
    # [B,S,1,1,4] tensors span < 2^59 bytes, placed so that none overlap
    B, S = (1 << 31) - 1, 1 << 24
    assert f(_p(1 << 59), _p(1 << 62), _p(1 << 60), _p(1 << 61), _p((1 << 62) + (1 << 40)),
             B, S, 1, 1, None) == qs.QS_ERR_SCRATCH
    msg = qs.quat_cumprod_strerror(qs.QS_ERR_SCRATCH)
    assert "8192" in msg and "noalloc" in msg


def test_noalloc_argument_checks_match_bwd(host_lib):
    f = host_lib.quat_cumprod_bwd_noalloc
    q, i, d, gq, gi = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000
    assert f(_p(q), _p(i), _p(d), _p(gq), _p(gi), 1, -1, 1, 1, None) == qs.QS_ERR_DIMS
    assert f(None, None, None, None, None, 0, 5, 2, 2, None) == qs.QS_OK
    assert f(None, None, None, None, None, 2, 0, 2, 2, None) == qs.QS_ERR_NULL
    assert f(None, None, None, None, _p(gi + 4), 2, 0, 2, 2, None) == qs.QS_ERR_MISALIGNED
    for k in range(5):
        ptrs = [_p(q), _p(i), _p(d), _p(gq), _p(gi)]
        ptrs[k] = None
        assert f(*ptrs, 1, 4, 1, 1, None) == qs.QS_ERR_NULL
        ptrs = [_p(q), _p(i), _p(d), _p(gq), _p(gi)]
        ptrs[k] = _p([q, i, d, gq, gi][k] + 4)
        assert f(*ptrs, 1, 4, 1, 1, None) == qs.QS_ERR_MISALIGNED
    assert f(_p(q), _p(i), _p(d), _p(q + 16), _p(gi), 1, 4, 1, 1, None) == qs.QS_ERR_ALIAS
    assert f(_p(q), _p(i), _p(d), _p(gq), _p(i), 1, 4, 1, 1, None) == qs.QS_ERR_ALIAS


# ---------------------------------------------------------------------------
# GPU: the no-alloc entry point against the allocating one.
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    lib = qs.load_library()
    lib.quat_cumprod_debug_set_variant(-1, -1)
    lib.quat_cumprod_debug_stall_tile(-1)
    lib.quat_cumprod_debug_set_timeout_ns(0)
    return torch.device("cuda", 0)


def _to_dev(dev, arrays):
    import torch
    return [torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in arrays]


def _noalloc(q, init, d_cum, d_q, d_init, stream):
    """Calls the C ABI directly (no binding-side allocation, no checks)."""
    B, S, H, J, _ = q.shape
    return qs.load_library().quat_cumprod_bwd_noalloc(
        _p(q.data_ptr()), _p(init.data_ptr()), _p(d_cum.data_ptr()), _p(d_q.data_ptr()),
        _p(d_init.data_ptr()), B, S, H, J, _p(stream.cuda_stream))


# Two problems of different shapes: one that fills the scratch exactly
# (8 * 512/32 * 4096/64 = 8192 tiles) and a ragged one.
FULL = workloads.WORKLOADS["mamba3"]
RAGGED = workloads.custom("ragged", 3, 1000, 3, 7, seed=11)


@pytest.mark.gpu
def test_noalloc_matches_bwd_on_two_calls_in_a_row(dev):
    import torch
    stream = torch.cuda.current_stream(dev)
    cases = []
    for w in (FULL, RAGGED):
        q, init, d_cum = _to_dev(dev, workloads.make_inputs(w))
        ref_dq, ref_di = qs.quat_cumprod_bwd(q, init, d_cum)          # the allocating entry point
        assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
        d_q = torch.full_like(q, float("nan"))
        d_init = torch.full_like(init, float("nan"))
        cases.append((w, q, init, d_cum, d_q, d_init, ref_dq, ref_di))
    torch.cuda.synchronize(dev)
    # Two calls in a row on one stream, no synchronization between them.
    for w, q, init, d_cum, d_q, d_init, _, _ in cases:
        rc = _noalloc(q, init, d_cum, d_q, d_init, stream)
        assert rc == qs.QS_OK, qs.quat_cumprod_strerror(rc)
    torch.cuda.synchronize(dev)
    for w, q, init, d_cum, d_q, d_init, ref_dq, ref_di in cases:
        e_q = normwise(d_q.cpu().numpy(), ref_dq.cpu().numpy())
        e_i = normwise(d_init.cpu().numpy(), ref_di.cpu().numpy())
        assert e_q <= TOL and e_i <= TOL, f"{w.name}: d_q {e_q:.3e}, d_init {e_i:.3e}"


@pytest.mark.gpu
def test_noalloc_repeated_call_and_oracle(dev):
    import torch
    stream = torch.cuda.current_stream(dev)
    arrays = workloads.make_inputs(RAGGED)
    q, init, d_cum = _to_dev(dev, arrays)
    outs = []
    for _ in range(2):   # the same problem twice in a row; each call reuses the scratch
        d_q, d_init = torch.empty_like(q), torch.empty_like(init)
        rc = _noalloc(q, init, d_cum, d_q, d_init, stream)
        assert rc == qs.QS_OK, qs.quat_cumprod_strerror(rc)
        outs.append((d_q, d_init))
    torch.cuda.synchronize(dev)
    ref_dq, ref_di = qs.quat_cumprod_bwd(q, init, d_cum)
    ora_dq, ora_di = oracle.bwd(*arrays)
    for d_q, d_init in outs:
        assert normwise(d_q.cpu().numpy(), ref_dq.cpu().numpy()) <= TOL
        assert normwise(d_init.cpu().numpy(), ref_di.cpu().numpy()) <= TOL
        assert normwise(d_q.cpu().numpy(), ora_dq) <= TOL
        assert normwise(d_init.cpu().numpy(), ora_di) <= TOL


@pytest.mark.gpu
def test_noalloc_binding_and_empty_sequence(dev):
    import torch
    q, init, d_cum = _to_dev(dev, workloads.make_inputs(workloads.WORKLOADS["tiny"]))
    d_q, d_init = torch.empty_like(q), torch.empty_like(init)
    qs.quat_cumprod_bwd_noalloc(q, init, d_cum, d_q, d_init)
    ref_dq, ref_di = qs.quat_cumprod_bwd(q, init, d_cum)
    assert normwise(d_q.cpu().numpy(), ref_dq.cpu().numpy()) <= TOL
    assert normwise(d_init.cpu().numpy(), ref_di.cpu().numpy()) <= TOL
    # S == 0: d_init is written as zero
    q0 = torch.empty((2, 0, 3, 5, 4), device=dev)
    i0 = torch.ones((2, 3, 5, 4), device=dev)
    g0 = torch.full_like(i0, 7.0)
    qs.quat_cumprod_bwd_noalloc(q0, i0, torch.empty_like(q0), torch.empty_like(q0), g0)
    torch.cuda.synchronize(dev)
    assert float(g0.abs().max()) == 0.0
    # beyond the scratch: a clear error, nothing enqueued
    w = workloads.custom("over", 1, 64 * 8192 + 64, 1, 32)
    qb = torch.zeros((w.B, w.S, w.H, w.J, 4), device=dev)
    ib = torch.zeros((w.B, w.H, w.J, 4), device=dev)
    with pytest.raises(qs.QuatScanError) as ei:
        qs.quat_cumprod_bwd_noalloc(qb, ib, qb.clone(), torch.empty_like(qb), torch.empty_like(ib))
    assert ei.value.status == qs.QS_ERR_SCRATCH


@pytest.mark.gpu
@pytest.mark.parametrize("dims", [(1, 40000, 1, 32), (1, 20000, 1, 33)])
def test_noalloc_many_chunks_per_lane(dev, dims):
    """More than 256 chunks per lane (625 and 313 chunks, the second with a
    ragged lane group) but within the 8192 tiles: the carry step is the scan
    over chunk ranges, as in quat_cumprod_bwd."""
    import torch
    w = workloads.custom("noalloc_long", *dims, q_kind="rotation", theta_max=0.3, seed=sum(dims))
    arrays = workloads.make_inputs(w)
    q, init, d_cum = _to_dev(dev, arrays)
    d_q, d_init = torch.empty_like(q), torch.empty_like(init)
    stream = torch.cuda.current_stream(dev)
    rc = _noalloc(q, init, d_cum, d_q, d_init, stream)
    assert rc == qs.QS_OK, qs.quat_cumprod_strerror(rc)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    ref_dq, ref_di = qs.quat_cumprod_bwd(q, init, d_cum)
    ora_dq, ora_di = oracle.bwd(*arrays)
    assert normwise(d_q.cpu().numpy(), ref_dq.cpu().numpy()) <= TOL
    assert normwise(d_init.cpu().numpy(), ref_di.cpu().numpy()) <= TOL
    assert normwise(d_q.cpu().numpy(), ora_dq) <= TOL
    assert normwise(d_init.cpu().numpy(), ora_di) <= TOL


@pytest.mark.gpu
def test_noalloc_timeout_is_reported_then_clears(dev):
    """A tile whose copy never completes (the stall hook) makes the wait run
    out; quat_cumprod_status reports it once, and the next call is clean."""
    import torch
    lib = qs.load_library()
    stream = torch.cuda.current_stream(dev)
    arrays = workloads.make_inputs(RAGGED)
    q, init, d_cum = _to_dev(dev, arrays)
    d_q, d_init = torch.empty_like(q), torch.empty_like(init)
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    try:
        lib.quat_cumprod_debug_set_timeout_ns(50_000_000)   # 50 ms
        lib.quat_cumprod_debug_stall_tile(0)
        assert _noalloc(q, init, d_cum, d_q, d_init, stream) == qs.QS_OK
        assert qs.quat_cumprod_status(device=dev) == qs.QS_ERR_TIMEOUT
        assert qs.quat_cumprod_status(device=dev) == qs.QS_OK   # read once, then cleared
    finally:
        lib.quat_cumprod_debug_stall_tile(-1)
        lib.quat_cumprod_debug_set_timeout_ns(0)
    assert _noalloc(q, init, d_cum, d_q, d_init, stream) == qs.QS_OK
    assert qs.quat_cumprod_status(device=dev) == qs.QS_OK
    ora_dq, ora_di = oracle.bwd(*arrays)
    assert normwise(d_q.cpu().numpy(), ora_dq) <= TOL
    assert normwise(d_init.cpu().numpy(), ora_di) <= TOL


_CAPTURE_FIRST = r"""
import ctypes, sys, torch
sys.path.insert(0, {root!r})
import quaternion_cumulative_product_gb300 as qs
lib = qs.load_library()
dev = torch.device("cuda", 0)
q = torch.zeros(1, 64, 1, 4, 4, device=dev); q[..., 0] = 1
init = torch.zeros(1, 1, 4, 4, device=dev); init[..., 0] = 1
d_cum, d_q, d_init = torch.ones_like(q), torch.empty_like(q), torch.empty_like(init)
s = torch.cuda.Stream(device=dev)
g = torch.cuda.CUDAGraph()
p = lambda t: ctypes.c_void_p(t.data_ptr())
with torch.cuda.graph(g, stream=s):
    rc = lib.quat_cumprod_bwd_noalloc(p(q), p(init), p(d_cum), p(d_q), p(d_init), 1, 64, 1, 4,
                                      ctypes.c_void_p(s.cuda_stream))
print("first", rc)
rc2 = lib.quat_cumprod_bwd_noalloc(p(q), p(init), p(d_cum), p(d_q), p(d_init), 1, 64, 1, 4,
                                   ctypes.c_void_p(s.cuda_stream))
print("second", rc2, lib.quat_cumprod_status(ctypes.c_void_p(s.cuda_stream)))
"""


@pytest.mark.gpu
def test_noalloc_first_call_during_capture_is_refused(dev):
    """In a fresh process, a first call made while its stream is being captured
    returns QS_ERR_NOMEM (its set-up is not done under a capture) and enqueues
    nothing; the same call outside the capture then works."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "-c", _CAPTURE_FIRST.format(root=ROOT)], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert f"first {qs.QS_ERR_NOMEM}" in r.stdout, r.stdout
    assert f"second {qs.QS_OK} {qs.QS_OK}" in r.stdout, r.stdout
