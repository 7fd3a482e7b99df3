"""Host logic of bench.py's multi-rank path, run as world-size-2 gloo ranks on CPU.

On N GPUs every rank scans its own batch (independent lanes: no data
exchange); the only collectives are the barrier around the timed region and
the max of the per-rank step times.  These tests run that logic without a
GPU.
"""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest

import bench
from quaternion_cumulative_product_gb300 import workloads

torch = pytest.importorskip("torch")
dist = pytest.importorskip("torch.distributed")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        bench.barrier()
        # rank r "measured" 1 + r ms: every rank must see the slowest one
        slowest = bench.reduce_max(1.0 + rank)
        # each rank draws its own batch
        w = workloads.WORKLOADS["tiny"]
        wr = workloads.custom(w.name, w.B, w.S, w.H, w.J, seed=bench.rank_seed(w.seed, rank))
        q, _, _ = workloads.make_inputs(wr)
        digest = float(np.abs(q).sum())
        gathered = [None] * world
        dist.all_gather_object(gathered, digest)
        bench.barrier()
        results[rank] = (slowest, gathered)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_max_time_and_draw_different_batches():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    world, port = 2, _free_port()
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        for p in procs:
            if p.is_alive():
                p.kill()
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(results)
    assert sorted(res) == [0, 1]
    for rank in range(world):
        slowest, gathered = res[rank]
        assert slowest == 2.0                        # the max over ranks
        assert gathered[0] != gathered[1]            # independent batches
    assert res[0][1] == res[1][1]


def test_single_process_helpers_need_no_process_group():
    assert bench.reduce_max(3.5) == 3.5
    bench.barrier()   # no-op without a process group
    assert bench.rank_seed(2, 0) == 2 and bench.rank_seed(2, 1) != bench.rank_seed(2, 0)


def test_weak_scaling_value_counts_every_rank():
    E = 8 * 4096 * 16 * 32
    assert bench.weak_scaling_value(1, E, 0.5) == pytest.approx(E / 0.5e-3)
    assert bench.weak_scaling_value(4, E, 0.5) == pytest.approx(4 * E / 0.5e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_warmup_below_three_is_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_source_hash_ignores_comments_and_blank_lines():
    import bench
    assert bench._code_only("a = 1; // note\n\n/* block\n comment */ b = 2;\n") == "a = 1;\n b = 2;"
    assert bench._code_only("x\n// only a comment\ny") == "x\ny"


def test_design_names_follow_the_plan():
    """The forward for few lane groups is one segmented-walk kernel."""
    assert bench.design_name("quat_cumprod_fwd", 1, 12) == "quat_cumprod_fwd (segmented chained walk kernel)"
    assert bench.design_name("quat_cumprod_fwd", 1, 9) == "quat_cumprod_fwd (segmented chained walk kernel)"
    assert bench.design_name("quat_cumprod_bwd", 3, 0) == "quat_cumprod_bwd (aggregate + carry + apply kernels)"
    assert bench.design_name("quat_cumprod_fwd", 1, 4) == "quat_cumprod_fwd (walk kernel)"


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    """Rank 0 times the fp64 oracle on a lane sample and prints one JSON line with
    the base contract's keys, its own cpu_baseline and an e2e without copies."""
    import json
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3",
                       "--cpu-lanes", "8"]) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == 2 and d["warmup"] == 3 and d["ms_per_step"] > 0
    assert d["config"]["workload"].startswith("tiny") and d["config"]["elements"] == 1 * 64 * 2 * 4
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_every_timed_loop_is_bracketed_and_starts_on_a_busy_stream():
    """Each device-timed loop over ``range(args.steps)`` in the bench has a
    synchronize and a barrier before and after it, and the lead spin right before it (the first
    step's events then exclude the host's enqueue of its first call)."""
    import ast

    def call_name(stmt):
        if isinstance(stmt, ast.Expr) and isinstance(stmt.value, ast.Call):
            return ast.unparse(stmt.value.func)
        if isinstance(stmt, ast.Assign) and isinstance(stmt.value, ast.Call):
            return ast.unparse(stmt.value.func)
        return None

    tree = ast.parse(open(bench.__file__).read())
    loops = 0
    for node in ast.walk(tree):
        for field in ("body", "orelse"):
            stmts = getattr(node, field, None)
            if not isinstance(stmts, list):
                continue
            for k, st in enumerate(stmts):
                if not (isinstance(st, ast.For) and ast.unparse(st.iter) == "range(args.steps)"
                        and ".record(stream)" in ast.unparse(st)):
                    continue   # only the device-timed loops (the oracle arm times on the host)
                loops += 1
                before = [call_name(s) for s in stmts[max(0, k - 6):k]]
                after = [call_name(s) for s in stmts[k + 1:k + 4]]
                assert before[-1] == "lead_spin", ast.unparse(st)[:60]
                assert "torch.cuda.synchronize" in before and "barrier" in before
                assert after[0] == "torch.cuda.synchronize" and "barrier" in after
    assert loops == 3   # the step, the saved-carries step, the bf16 step
