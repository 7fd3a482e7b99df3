"""Host-side tests of the C ABI (no GPU needed).

The library must load and export every function ``include/*.h`` declares; the
argument checks that run before any CUDA call must return the documented
status codes.
"""
from __future__ import annotations

import ctypes
import glob
import os
import re
import subprocess

import numpy as np
import pytest

import quaternion_cumulative_product_gb300 as qs
from quaternion_cumulative_product_gb300 import build as qbuild
from quaternion_cumulative_product_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qs.load_library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?\w+\s*\*?\s*(quat_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("quat_cumprod_fwd", "quat_cumprod_bwd", "quat_cumprod_status",
                     "quat_cumprod_strerror"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", qs.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = _declared_functions() - exported
    assert not missing, f"declared but not exported: {sorted(missing)}"
    for name in _declared_functions():
        assert hasattr(lib, name)


def test_strerror_covers_all_codes(lib):
    seen = set()
    for code in (qs.QS_OK, qs.QS_ERR_NULL, qs.QS_ERR_DIMS, qs.QS_ERR_MISALIGNED, qs.QS_ERR_ALIAS,
                 qs.QS_ERR_CUDA, qs.QS_ERR_TIMEOUT, qs.QS_ERR_NOMEM, qs.QS_ERR_DEVICE):
        msg = qs.quat_cumprod_strerror(code)
        assert msg and msg != "unknown status"
        seen.add(msg)
    assert len(seen) == 9
    assert qs.quat_cumprod_strerror(12345) == "unknown status"


def _p(addr):
    return ctypes.c_void_p(addr)


def test_fwd_argument_checks_before_any_cuda_call(lib):
    A, Bp, Cp = 0x10000, 0x20000000, 0x40000000
    # negative sizes
    assert lib.quat_cumprod_fwd(_p(A), _p(Bp), _p(Cp), -1, 4, 1, 1, None) == qs.QS_ERR_DIMS
    assert lib.quat_cumprod_fwd(_p(A), _p(Bp), _p(Cp), 1, -4, 1, 1, None) == qs.QS_ERR_DIMS
    # sizes beyond the limits
    assert lib.quat_cumprod_fwd(_p(A), _p(Bp), _p(Cp), 1, 1 << 32, 1, 1, None) == qs.QS_ERR_DIMS
    assert lib.quat_cumprod_fwd(_p(A), _p(Bp), _p(Cp), 1, 1 << 20, 1 << 12, 1 << 10, None) == qs.QS_ERR_DIMS
    # empty problems are no-ops (NULL pointers allowed)
    for dims in [(0, 4, 1, 1), (1, 0, 1, 1), (1, 4, 0, 1), (1, 4, 1, 0)]:
        assert lib.quat_cumprod_fwd(None, None, None, *dims, None) == qs.QS_OK
    # NULL pointers
    assert lib.quat_cumprod_fwd(None, _p(Bp), _p(Cp), 1, 4, 1, 1, None) == qs.QS_ERR_NULL
    assert lib.quat_cumprod_fwd(_p(A), None, _p(Cp), 1, 4, 1, 1, None) == qs.QS_ERR_NULL
    assert lib.quat_cumprod_fwd(_p(A), _p(Bp), None, 1, 4, 1, 1, None) == qs.QS_ERR_NULL
    # 16-byte alignment
    assert lib.quat_cumprod_fwd(_p(A + 4), _p(Bp), _p(Cp), 1, 4, 1, 1, None) == qs.QS_ERR_MISALIGNED
    assert lib.quat_cumprod_fwd(_p(A), _p(Bp + 8), _p(Cp), 1, 4, 1, 1, None) == qs.QS_ERR_MISALIGNED
    assert lib.quat_cumprod_fwd(_p(A), _p(Bp), _p(Cp + 12), 1, 4, 1, 1, None) == qs.QS_ERR_MISALIGNED
    # outputs overlapping inputs (q is 1*4*1*1*16 = 64 bytes)
    assert lib.quat_cumprod_fwd(_p(A), _p(Bp), _p(A + 48), 1, 4, 1, 1, None) == qs.QS_ERR_ALIAS
    assert lib.quat_cumprod_fwd(_p(A), _p(Bp), _p(Bp - 48), 1, 4, 1, 1, None) == qs.QS_ERR_ALIAS
    # adjacent but not overlapping is not aliasing: the call then goes on to
    # the device (not exercised here)


def test_bwd_argument_checks_before_any_cuda_call(lib):
    q, i, d, gq, gi = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000
    f = lib.quat_cumprod_bwd
    assert f(_p(q), _p(i), _p(d), _p(gq), _p(gi), 1, -1, 1, 1, None) == qs.QS_ERR_DIMS
    assert f(None, None, None, None, None, 0, 5, 2, 2, None) == qs.QS_OK
    assert f(None, None, None, None, None, 2, 5, 0, 2, None) == qs.QS_OK
    # S == 0 with lanes: d_init must be written -> needs a valid pointer
    assert f(None, None, None, None, None, 2, 0, 2, 2, None) == qs.QS_ERR_NULL
    assert f(None, None, None, None, _p(gi + 4), 2, 0, 2, 2, None) == qs.QS_ERR_MISALIGNED
    for k in range(5):
        ptrs = [_p(q), _p(i), _p(d), _p(gq), _p(gi)]
        ptrs[k] = None
        assert f(*ptrs, 1, 4, 1, 1, None) == qs.QS_ERR_NULL
        ptrs = [_p(q), _p(i), _p(d), _p(gq), _p(gi)]
        ptrs[k] = _p([q, i, d, gq, gi][k] + 4)
        assert f(*ptrs, 1, 4, 1, 1, None) == qs.QS_ERR_MISALIGNED
    # q/d_cum/d_q are 64 bytes, init/d_init 16 bytes
    assert f(_p(q), _p(i), _p(d), _p(q + 16), _p(gi), 1, 4, 1, 1, None) == qs.QS_ERR_ALIAS
    assert f(_p(q), _p(i), _p(d), _p(d), _p(gi), 1, 4, 1, 1, None) == qs.QS_ERR_ALIAS
    assert f(_p(q), _p(i), _p(d), _p(gq), _p(i), 1, 4, 1, 1, None) == qs.QS_ERR_ALIAS
    assert f(_p(q), _p(i), _p(d), _p(gq), _p(gq + 32), 1, 4, 1, 1, None) == qs.QS_ERR_ALIAS


def test_debug_hooks_return_ok(lib):
    assert lib.quat_cumprod_debug_set_timeout_ns(1000) == qs.QS_OK
    assert lib.quat_cumprod_debug_set_timeout_ns(0) == qs.QS_OK
    assert lib.quat_cumprod_debug_stall_tile(3) == qs.QS_OK
    assert lib.quat_cumprod_debug_stall_tile(-1) == qs.QS_OK
    assert lib.quat_cumprod_debug_set_variant(1, 2) == qs.QS_OK
    assert lib.quat_cumprod_debug_set_variant(-1, -1) == qs.QS_OK
    assert lib.quat_cumprod_debug_set_variant(99, 0) == qs.QS_ERR_DIMS
    assert lib.quat_cumprod_debug_set_walk_cap(100) == qs.QS_OK
    assert lib.quat_cumprod_debug_set_walk_cap(-1) == qs.QS_OK


def test_workload_generator_is_seeded_and_shaped():
    w = workloads.WORKLOADS["tiny"]
    a = workloads.make_inputs(w)
    b = workloads.make_inputs(w)
    for x, y in zip(a, b):
        assert x.dtype.name == "float32" and (x == y).all()
    q, init, d_cum = a
    assert q.shape == (1, 64, 2, 4, 4) and init.shape == (1, 2, 4, 4) and d_cum.shape == q.shape
    import numpy as np
    assert np.allclose(np.linalg.norm(q, axis=-1), 1, atol=1e-6)
    w3 = workloads.custom("c", 2, 10, 1, 3, q_kind="rotation", theta_max=0.1, init_kind="identity")
    q3, i3, _ = workloads.make_inputs(w3)
    assert np.all(q3[..., 0] >= np.cos(0.05) - 1e-6) and np.all(i3[..., 0] == 1)
    lanes = [0, 4, 5]
    sq, si, sd = workloads.sample_lanes(a, lanes, 2, 4)
    assert sq.shape == (1, 64, 3, 1, 4) and si.shape == (1, 3, 1, 4)
    assert (sq[0, :, 1, 0] == q[0, :, 1, 0]).all() and (si[0, 2, 0] == init[0, 1, 1]).all()


def test_plan_query_argument_checks(lib):
    v, k = ctypes.c_int(7), ctypes.c_int(7)
    assert lib.quat_cumprod_plan(0, 1, 4, 1, 1, None, ctypes.byref(k)) == qs.QS_ERR_NULL
    assert lib.quat_cumprod_plan(1, 1, 4, 1, 1, ctypes.byref(v), None) == qs.QS_ERR_NULL
    assert lib.quat_cumprod_plan(0, 1, -4, 1, 1, ctypes.byref(v), ctypes.byref(k)) == qs.QS_ERR_DIMS
    assert lib.quat_cumprod_plan(1, 0, 4, 1, 1, ctypes.byref(v), ctypes.byref(k)) == qs.QS_OK
    assert (v.value, k.value) == (-1, 0)


def test_carry_calls_argument_checks_before_any_cuda_call(lib):
    # [1, 100, 1, 1, 4]: q / cum / d_cum are 1600 bytes, carries 2 chunks = 32 bytes
    q, i, c, car, d, gq, gi = (k << 20 for k in range(1, 8))
    f = lib.quat_cumprod_fwd_carries
    assert f(_p(q), _p(i), _p(c), _p(car), 1, -1, 1, 1, None) == qs.QS_ERR_DIMS
    assert f(None, None, None, None, 0, 100, 1, 1, None) == qs.QS_OK
    for k in range(4):
        ptrs = [_p(q), _p(i), _p(c), _p(car)]
        ptrs[k] = None
        assert f(*ptrs, 1, 100, 1, 1, None) == qs.QS_ERR_NULL
        ptrs = [_p(q), _p(i), _p(c), _p(car)]
        ptrs[k] = _p([q, i, c, car][k] + 8)
        assert f(*ptrs, 1, 100, 1, 1, None) == qs.QS_ERR_MISALIGNED
    assert f(_p(q), _p(i), _p(c), _p(c + 16), 1, 100, 1, 1, None) == qs.QS_ERR_ALIAS     # carries in cum
    assert f(_p(q), _p(i), _p(c), _p(q + 1584), 1, 100, 1, 1, None) == qs.QS_ERR_ALIAS   # carries in q
    assert f(_p(q), _p(i), _p(c), _p(i - 16), 1, 100, 1, 1, None) == qs.QS_ERR_ALIAS     # overlaps init
    g = lib.quat_cumprod_bwd_carries
    assert g(_p(q), _p(car), _p(d), _p(gq), _p(gi), 1, -1, 1, 1, None) == qs.QS_ERR_DIMS
    assert g(None, None, None, None, None, 2, 0, 2, 2, None) == qs.QS_ERR_NULL   # S == 0 writes d_init
    for k in range(5):
        ptrs = [_p(q), _p(car), _p(d), _p(gq), _p(gi)]
        ptrs[k] = None
        assert g(*ptrs, 1, 100, 1, 1, None) == qs.QS_ERR_NULL
        ptrs = [_p(q), _p(car), _p(d), _p(gq), _p(gi)]
        ptrs[k] = _p([q, car, d, gq, gi][k] + 4)
        assert g(*ptrs, 1, 100, 1, 1, None) == qs.QS_ERR_MISALIGNED
    assert g(_p(q), _p(car), _p(d), _p(car - 1584), _p(gi), 1, 100, 1, 1, None) == qs.QS_ERR_ALIAS
    assert g(_p(q), _p(car), _p(d), _p(gq), _p(car + 16), 1, 100, 1, 1, None) == qs.QS_ERR_ALIAS


def test_plan_rejects_unknown_call(lib):
    v, k = ctypes.c_int(0), ctypes.c_int(0)
    assert lib.quat_cumprod_plan(4, 1, 4, 1, 1, ctypes.byref(v), ctypes.byref(k)) == qs.QS_ERR_DIMS
    assert lib.quat_cumprod_plan(-1, 1, 4, 1, 1, ctypes.byref(v), ctypes.byref(k)) == qs.QS_ERR_DIMS
    assert lib.quat_cumprod_plan(3, 0, 4, 1, 1, ctypes.byref(v), ctypes.byref(k)) == qs.QS_OK


def test_bf16_calls_argument_checks_before_any_cuda_call(lib):
    q, i, c, d, gq, gi = (k << 20 for k in range(1, 7))
    f, g = lib.quat_cumprod_fwd_bf16, lib.quat_cumprod_bwd_bf16
    assert f(_p(q), _p(i), _p(c), 1, 16, 3, 5, None) == qs.QS_ERR_DIMS        # H*J odd
    assert g(_p(q), _p(i), _p(d), _p(gq), _p(gi), 1, 16, 1, 1, None) == qs.QS_ERR_DIMS
    assert f(None, None, None, 0, 16, 2, 2, None) == qs.QS_OK
    assert f(None, _p(i), _p(c), 1, 16, 2, 2, None) == qs.QS_ERR_NULL
    assert f(_p(q + 8), _p(i), _p(c), 1, 16, 2, 2, None) == qs.QS_ERR_MISALIGNED
    assert f(_p(q), _p(i), _p(q + 64), 1, 16, 2, 2, None) == qs.QS_ERR_ALIAS    # 1*16*4 quats * 8 B
    assert g(None, None, None, None, None, 2, 0, 2, 2, None) == qs.QS_ERR_NULL
    assert g(_p(q), _p(i), _p(d), _p(d + 256), _p(gi), 1, 16, 2, 2, None) == qs.QS_ERR_ALIAS


def test_host_step_argument_checks(lib):
    """quat_cumprod_fwd_bwd_host rejects bad arguments before any CUDA call (host buffers)."""
    f = lib.quat_cumprod_fwd_bwd_host
    big = np.zeros((1, 4, 1, 1, 4), np.float32)
    small = np.zeros((1, 1, 1, 4), np.float32)
    bufs = [big, small, big.copy(), big.copy(), big.copy(), small.copy()]
    ptrs = [b.ctypes.data for b in bufs]
    assert f(*ptrs, 1, -1, 1, 1, None) == qs.QS_ERR_DIMS
    for k in range(6):
        p = list(ptrs)
        p[k] = None
        assert f(*p, 1, 4, 1, 1, None) == qs.QS_ERR_NULL
    p = list(ptrs)
    p[3] = ptrs[0]              # cum over q
    assert f(*p, 1, 4, 1, 1, None) == qs.QS_ERR_ALIAS
    p = list(ptrs)
    p[4] = ptrs[3]              # d_q over cum
    assert f(*p, 1, 4, 1, 1, None) == qs.QS_ERR_ALIAS
    p = list(ptrs)
    p[5] = ptrs[1]              # d_init over init
    assert f(*p, 1, 4, 1, 1, None) == qs.QS_ERR_ALIAS
    assert f(*ptrs, 0, 4, 1, 1, None) == qs.QS_OK   # no lanes: nothing to do


def test_size_limits_at_their_boundaries(lib):
    """Just past each documented limit the size check rejects the call; at the
    limit it passes, and with no device here the call then stops at its first
    CUDA query.  Fake device pointers are far apart so that no range overlaps."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("the accepted calls would reach a GPU with fake device pointers")
    q, i, c = _p(1 << 44), _p(1 << 46), _p(1 << 45)
    f = lib.quat_cumprod_fwd

    def accepted(*dims):
        rc = f(q, i, c, *dims, None)
        assert rc not in (qs.QS_ERR_DIMS, qs.QS_OK), dims
        assert rc in (qs.QS_ERR_CUDA, qs.QS_ERR_DEVICE), (dims, rc)

    # S*H*J*16 < 2^40 bytes per batch entry
    accepted(1, (1 << 26) - 1, 32, 32)
    assert f(q, i, c, 1, 1 << 26, 32, 32, None) == qs.QS_ERR_DIMS
    # H*J*4 < 2^32
    accepted(1, 1, 1 << 15, (1 << 15) - 1)
    assert f(q, i, c, 1, 1, 1 << 15, 1 << 15, None) == qs.QS_ERR_DIMS
    # every size below 2^31
    accepted((1 << 31) - 1, 1, 1, 1)
    assert f(q, i, c, 1 << 31, 1, 1, 1, None) == qs.QS_ERR_DIMS
    assert f(q, i, c, 1, 1, 1, 1 << 31, None) == qs.QS_ERR_DIMS
