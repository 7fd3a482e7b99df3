"""Error measures of the GPU parity tests against the oracle, and their opt-in log.

Two measures per output tensor (quaternions along the last axis of size 4):

* normwise: ``max_i |got_i - ref_i| / max_i |ref_i|`` over all components;
  the pass criterion (tolerance 1e-4 for fp32, ``2**-8 + 1.1e-4`` for bf16);
* per quaternion: ``max_q ||got_q - ref_q|| / max(||ref_q||, 1e-6 * max_q ||ref_q||)``
  (2-norms of whole quaternions), which shows the local precision that the
  tensor-wide normwise figure can hide: a small quaternion next to large ones
  is held to its own size, down to a floor of 1e-6 of the largest.

With ``QS_PARITY_LOG`` set to a file name, every comparison appends one JSON
object per line (test, tensor, dtype, elements, both measures, tolerance).
``python tests/parity_log.py LOG`` prints the margins of such a log as a
Markdown table, one row per (workload, dtype, tensor), keeping the worst case.
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

PARITY_LOG = os.environ.get("QS_PARITY_LOG")
QUAT_FLOOR = 1e-6


def normwise(got, ref) -> float:
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    scale = float(np.abs(ref).max())
    return float(np.abs(np.asarray(got, np.float64) - ref).max()) / (scale if scale > 0 else 1.0)


def per_quaternion(got, ref, floor: float = QUAT_FLOOR) -> float:
    ref = np.asarray(ref, np.float64).reshape(-1, 4)
    if ref.size == 0:
        return 0.0
    diff = np.asarray(got, np.float64).reshape(-1, 4) - ref
    rn = np.linalg.norm(ref, axis=1)
    top = float(rn.max())
    den = np.maximum(rn, floor * top) if top > 0 else np.ones_like(rn)
    return float((np.linalg.norm(diff, axis=1) / den).max())


def record(tensor: str, dtype: str, got, ref, tol: float, err: float) -> None:
    """Appends one comparison to the log (nothing unless QS_PARITY_LOG is set)."""
    if not PARITY_LOG:
        return
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    ref = np.asarray(ref)
    line = {"test": test, "tensor": tensor, "dtype": dtype, "elements": int(ref.size // 4),
            "normwise": err, "per_quaternion": per_quaternion(got, ref), "tol": tol}
    with open(PARITY_LOG, "a") as f:
        f.write(json.dumps(line) + "\n")


WORKLOAD_OF_TEST = [
    # (substring of the test id, workload row)
    ("test_named_workload_full_parity[tiny]", "tiny (1x64x2x4), full"),
    ("test_named_workload_full_parity[small]", "small (4x1024x8x16), full"),
    ("test_named_workload_full_parity[mamba3]", "mamba3 (8x4096x16x32), full"),
    ("test_mamba3_full_size_sampled_lanes", "mamba3, sampled lanes"),
    ("test_large_full_size_sampled_lanes", "large (16x8192x32x32), sampled lanes"),
    ("test_long_sequence_full_size", "long (1x131072x16x16), sampled lanes"),
    ("test_bf16_named_workloads[tiny]", "tiny (1x64x2x4), full"),
    ("test_bf16_named_workloads[small]", "small (4x1024x8x16), full"),
    ("test_bf16_named_workloads[mamba3]", "mamba3, sampled lanes"),
    ("test_bf16_named_workloads[large]", "large (16x8192x32x32), sampled lanes"),
    ("test_bf16_named_workloads[long]", "long (1x131072x16x16), sampled lanes"),
]


def margin_table(path: str) -> str:
    rows = {}
    every = {"fp32": [0.0, 0.0, 0], "bf16": [0.0, 0.0, 0]}
    with open(path) as f:
        for ln in f:
            d = json.loads(ln)
            dt = d.get("dtype", "fp32")
            every.setdefault(dt, [0.0, 0.0, 0])
            every[dt][0] = max(every[dt][0], d["normwise"] / d["tol"])
            every[dt][1] = max(every[dt][1], d["per_quaternion"])
            every[dt][2] += 1
            for key, wl in WORKLOAD_OF_TEST:
                if key in d["test"]:
                    k = (wl, dt, d["tensor"].split(" ")[0])
                    r = rows.setdefault(k, [0.0, 0.0, d["tol"], 0])
                    r[0] = max(r[0], d["normwise"])
                    r[1] = max(r[1], d["per_quaternion"])
                    r[3] = max(r[3], d["elements"])
    out = ["| workload | dtype | tensor | quaternions compared | normwise error | tolerance | "
           "normwise / tolerance | per-quaternion error (max) |",
           "|---|---|---|---:|---:|---:|---:|---:|"]
    order = {wl: i for i, (_, wl) in enumerate(WORKLOAD_OF_TEST)}
    for (wl, dt, t), (nw, pq, tol, n) in sorted(rows.items(), key=lambda kv: (kv[0][1], order[kv[0][0]], kv[0][2])):
        out.append(f"| {wl} | {dt} | {t} | {n} | {nw:.2e} | {tol:.2e} | {nw / tol:.3f} | {pq:.2e} |")
    out.append("")
    out.append("| every comparison logged | count | worst normwise / tolerance | worst per-quaternion error |")
    out.append("|---|---:|---:|---:|")
    for dt, (ratio, pq, cnt) in every.items():
        if cnt:
            out.append(f"| {dt} | {cnt} | {ratio:.3f} | {pq:.2e} |")
    return "\n".join(out)


if __name__ == "__main__":
    print(margin_table(sys.argv[1]))
