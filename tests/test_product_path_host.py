"""The product path has no CPU fallback and no route through the oracle (CPU checks).

* The package (binding, build script, workload generator, CUDA sources) never
  imports or includes the oracle, and the oracle never imports the package:
  they meet only in the seeded input generator, which holds none of the scan's
  arithmetic.
* ``bench.py`` imports the oracle only inside ``time_oracle``, the CPU-baseline
  and reference-arm leg.
* Every public call of the binding refuses CPU tensors before anything runs,
  and a missing CUDA library makes the first call raise instead of computing
  anything elsewhere.
"""
from __future__ import annotations

import ast
import glob
import os
import re

import pytest

import quaternion_cumulative_product_gb300 as qs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "quaternion_cumulative_product_gb300")


def _imported_modules(tree):
    """(top-level module name, enclosing function name or None) for every import in ``tree``."""
    out = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            name = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else fn
            if isinstance(child, ast.Import):
                out.extend((a.name.split(".")[0], fn) for a in child.names)
            elif isinstance(child, ast.ImportFrom) and child.module and child.level == 0:
                out.append((child.module.split(".")[0], fn))
            visit(child, name)

    visit(tree, None)
    return out


def _parse(path):
    with open(path) as f:
        return ast.parse(f.read(), path)


def test_package_never_imports_the_oracle():
    files = glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True)
    assert files
    for path in files:
        mods = {m for m, _ in _imported_modules(_parse(path))}
        assert "oracle" not in mods, path
    for path in glob.glob(os.path.join(PKG, "csrc", "*")):
        with open(path) as f:
            includes = re.findall(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', f.read(), flags=re.M)
        assert not any("oracle" in inc for inc in includes), path


def test_oracle_never_imports_the_package():
    mods = {m for m, _ in _imported_modules(_parse(os.path.join(ROOT, "oracle", "__init__.py")))}
    assert not mods & {"quaternion_cumulative_product_gb300", "torch", "bench"}
    with open(os.path.join(ROOT, "oracle", "quat_oracle.c")) as f:
        includes = re.findall(r'^\s*#\s*include\s*([<"][^>"]+[>"])', f.read(), flags=re.M)
    assert includes and all(inc.startswith("<") for inc in includes), includes


def test_bench_imports_the_oracle_only_in_its_cpu_leg():
    uses = [fn for m, fn in _imported_modules(_parse(os.path.join(ROOT, "bench.py"))) if m == "oracle"]
    assert uses and set(uses) == {"time_oracle"}


def test_public_calls_refuse_cpu_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 4, 1, 2, 4)
    init = torch.zeros(1, 1, 2, 4)
    carries = torch.zeros(1, 1, 1, 2, 4)
    with pytest.raises(ValueError, match="no CPU path"):
        qs.quat_cumprod_fwd(q, init)
    with pytest.raises(ValueError, match="no CPU path"):
        qs.quat_cumprod_bwd(q, init, q)
    with pytest.raises(ValueError, match="no CPU path"):
        qs.quat_cumprod_fwd_carries(q, init)
    with pytest.raises(ValueError, match="no CPU path"):
        qs.quat_cumprod_bwd_carries(q, carries, q)
    with pytest.raises(ValueError, match="no CPU path"):
        qs.quat_cumprod_bwd_noalloc(q, init, q, torch.zeros_like(q), torch.zeros_like(init))
    qb, ib = q.to(torch.bfloat16), init.to(torch.bfloat16)
    with pytest.raises(ValueError, match="no CPU path"):
        qs.quat_cumprod_fwd_bf16(qb, ib)
    with pytest.raises(ValueError, match="no CPU path"):
        qs.quat_cumprod_bwd_bf16(qb, ib, qb)


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(qs, "_lib", None)
    monkeypatch.setattr(qs, "library_path", lambda: str(tmp_path / "libquatscan.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        qs.load_library()
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        qs.quat_cumprod_strerror(0)
