"""Seeded synthetic workloads for the quaternion cumulative-product scan.

This module only draws random inputs; it holds none of the scan's arithmetic
and imports neither the CUDA binding nor the oracle, so that both sides can
use the same inputs.

Shapes follow burn-mamba ``mamba3/quat_scan/backward.rs`` (``q`` is
``[b,s,h,j,4]``, ``init`` is ``[b,h,j,4]``, ``d_cum`` has the shape of ``q``).
The page prints no workload, so five synthetic ones are defined here:

======  ==================  ==========================================================
name    (B, S, H, J)        q / init / d_cum
======  ==================  ==========================================================
tiny    (1, 64, 2, 4)       q = normalize(N(0,1)^4); init = normalize(N(0,1)^4); d_cum ~ N(0,1)
small   (4, 1024, 8, 16)    q = (cos th/2, sin th/2 u), th ~ U(0, 0.1); init unit; d_cum ~ N(0,1)
mamba3  (8, 4096, 16, 32)   th ~ U(0, pi/8); init = (1,0,0,0); d_cum ~ N(0, 0.02^2)
large   (16, 8192, 32, 32)  q = normalize(N(0,1)^4); init unit; d_cum ~ N(0,1)
long    (1, 131072, 16, 16) th ~ U(0, 0.05); init unit; d_cum ~ N(0,1)
======  ==================  ==========================================================

``u`` is ``normalize(N(0,1)^3)`` (uniform on the sphere), "init unit" is
``normalize(N(0,1)^4)``.  Seeds are 0..4 in the order above.

Draw recipe (numpy ``default_rng(seed)``, PCG64, fp64 draws cast to fp32):
the quaternions of ``q`` are drawn in blocks of ``BLOCK`` quaternions along
the flattened ``[B,S,H,J]`` order; a normalized-Gaussian block draws ``4n``
normals (row-major ``[n,4]``); a rotation block draws ``n`` uniforms for the
angles, then ``3n`` normals for the axes.  ``init`` is drawn next (one block),
then ``d_cum`` block by block (``4n`` normals each).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BLOCK = 1 << 22  # quaternions per generation block


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    H: int
    J: int
    q_kind: str          # "gauss4" (normalized N(0,1)^4) or "rotation"
    theta_max: float     # rotation angle upper bound (q_kind == "rotation")
    init_kind: str       # "gauss4" or "identity"
    dcum_sigma: float
    seed: int

    @property
    def elements(self) -> int:
        return self.B * self.S * self.H * self.J

    @property
    def lanes(self) -> int:
        return self.B * self.H * self.J

    def describe(self) -> str:
        return f"{self.name}: B={self.B},S={self.S},H={self.H},J={self.J}"


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny", 1, 64, 2, 4, "gauss4", 0.0, "gauss4", 1.0, 0),
        Workload("small", 4, 1024, 8, 16, "rotation", 0.1, "gauss4", 1.0, 1),
        Workload("mamba3", 8, 4096, 16, 32, "rotation", math.pi / 8, "identity", 0.02, 2),
        Workload("large", 16, 8192, 32, 32, "gauss4", 0.0, "gauss4", 1.0, 3),
        Workload("long", 1, 131072, 16, 16, "rotation", 0.05, "gauss4", 1.0, 4),
    )
}


def custom(name: str, B: int, S: int, H: int, J: int, *, q_kind="gauss4",
           theta_max=0.0, init_kind="gauss4", dcum_sigma=1.0, seed=0) -> Workload:
    """A workload with arbitrary sizes (edge cases in tests)."""
    return Workload(name, B, S, H, J, q_kind, theta_max, init_kind, dcum_sigma, seed)


def _gauss4(rng: np.random.Generator, n: int) -> np.ndarray:
    v = rng.standard_normal((n, 4))
    v /= np.linalg.norm(v, axis=1, keepdims=True)
    return v


def _rotation(rng: np.random.Generator, n: int, theta_max: float) -> np.ndarray:
    theta = rng.uniform(0.0, theta_max, n)
    u = rng.standard_normal((n, 3))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    out = np.empty((n, 4))
    out[:, 0] = np.cos(theta / 2)
    out[:, 1:] = np.sin(theta / 2)[:, None] * u
    return out


def _fill_blocks(out: np.ndarray, draw) -> None:
    flat = out.reshape(-1, 4)
    n = flat.shape[0]
    for start in range(0, n, BLOCK):
        stop = min(n, start + BLOCK)
        flat[start:stop] = draw(stop - start)


def make_inputs(w: Workload):
    """(q, init, d_cum) as contiguous float32 numpy arrays."""
    rng = np.random.default_rng(w.seed)
    q = np.empty((w.B, w.S, w.H, w.J, 4), np.float32)
    if w.q_kind == "gauss4":
        _fill_blocks(q, lambda n: _gauss4(rng, n))
    elif w.q_kind == "rotation":
        _fill_blocks(q, lambda n: _rotation(rng, n, w.theta_max))
    else:
        raise ValueError(w.q_kind)
    init = np.empty((w.B, w.H, w.J, 4), np.float32)
    if w.init_kind == "gauss4":
        init.reshape(-1, 4)[:] = _gauss4(rng, w.lanes)
    elif w.init_kind == "identity":
        init[...] = 0.0
        init[..., 0] = 1.0
    else:
        raise ValueError(w.init_kind)
    d_cum = np.empty_like(q)
    _fill_blocks(d_cum, lambda n: w.dcum_sigma * rng.standard_normal((n, 4)))
    return q, init, d_cum


def make_inputs_device(w: Workload, device):
    """(q, init, d_cum) as float32 torch tensors drawn on ``device``.

    The same distributions as ``make_inputs`` (and the same draw order: q,
    init, d_cum) from torch's generator on the device seeded with ``w.seed``,
    so the values differ from ``make_inputs``'s.  For timing only: the kernels
    do the same work whatever the values, and drawing the largest workloads on
    the host would take longer than timing them.
    """
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    n = w.elements

    def gauss4(m):
        v = torch.randn((m, 4), generator=g, device=device, dtype=torch.float64)
        return v / v.norm(dim=1, keepdim=True)

    if w.q_kind == "gauss4":
        q = gauss4(n)
    elif w.q_kind == "rotation":
        theta = torch.rand(n, generator=g, device=device, dtype=torch.float64) * w.theta_max
        u = torch.randn((n, 3), generator=g, device=device, dtype=torch.float64)
        u /= u.norm(dim=1, keepdim=True)
        q = torch.cat([torch.cos(theta / 2)[:, None], torch.sin(theta / 2)[:, None] * u], dim=1)
        del theta, u
    else:
        raise ValueError(w.q_kind)
    q = q.float().reshape(w.B, w.S, w.H, w.J, 4)
    if w.init_kind == "gauss4":
        init = gauss4(w.lanes).float()
    elif w.init_kind == "identity":
        init = torch.zeros((w.lanes, 4), device=device)
        init[:, 0] = 1.0
    else:
        raise ValueError(w.init_kind)
    init = init.reshape(w.B, w.H, w.J, 4)
    d_cum = (torch.randn((w.B, w.S, w.H, w.J, 4), generator=g, device=device) * w.dcum_sigma)
    return q.contiguous(), init.contiguous(), d_cum.contiguous()


def sample_lanes(arrays, lanes, H: int, J: int):
    """Gather whole lanes (b,h,j) of [B,S,H,J,4] / [B,H,J,4] arrays.

    ``lanes`` are flat lane ids ``(b*H + h)*J + j``.  Returns the same arrays
    reshaped to one batch of ``len(lanes)`` lanes: ``[1,S,len,1,4]`` and
    ``[1,len,1,4]``.  Lanes are independent in the scan, so any subset is a
    valid smaller problem.
    """
    lanes = np.asarray(lanes, dtype=np.int64)
    b = lanes // (H * J)
    hj = lanes % (H * J)
    out = []
    for a in arrays:
        if a.ndim == 5:
            B, S = a.shape[:2]
            v = a.reshape(B, S, H * J, 4)[b, :, hj, :]      # [n, S, 4]
            out.append(np.ascontiguousarray(np.transpose(v, (1, 0, 2)))[None, :, :, None, :])
        else:
            B = a.shape[0]
            v = a.reshape(B, H * J, 4)[b, hj, :]
            out.append(np.ascontiguousarray(v)[None, :, None, :])
    return out
