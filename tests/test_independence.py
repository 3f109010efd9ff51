"""Static checks that the CUDA path and the CPU oracle stay apart.

The product path (the CUDA library and its Python binding) never imports,
includes or calls the oracle; the oracle uses nothing but the standard library
and NumPy; in ``bench.py`` the oracle is reached only by the CPU-baseline and
reference legs; and the binding refuses to run without its compiled library
instead of falling back to anything on the CPU.
"""
import ast
import glob
import os
import re

import pytest

from newton_schulz_bucket_gb300 import _capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "newton_schulz_bucket_gb300")


def _product_sources():
    out = []
    for pat in ("*.py", "csrc/*.cu", "csrc/*.cuh", "csrc/*.cpp", "csrc/*.h"):
        out += glob.glob(os.path.join(PKG, pat))
    out += glob.glob(os.path.join(ROOT, "include", "*.h"))
    return sorted(out)


def test_product_path_never_reaches_the_oracle():
    files = _product_sources()
    assert any(f.endswith(".cu") for f in files) and any(f.endswith("_capi.py") for f in files)
    imp = re.compile(r"^\s*(from\s+oracle\b|import\s+oracle\b|#\s*include\s*[<\"].*oracle)", re.M)
    for f in files:
        src = open(f, encoding="utf-8").read()
        assert not imp.search(src), f
        if f.endswith(".py"):
            for node in ast.walk(ast.parse(src)):
                if isinstance(node, ast.Call) and isinstance(node.func, ast.Name):
                    assert node.func.id not in ("__import__",), f
                if isinstance(node, ast.Constant) and isinstance(node.value, str):
                    assert not re.fullmatch(r"oracle(\.\w+)*", node.value), (f, node.value)


def test_oracle_uses_only_numpy_and_the_standard_library():
    allowed = {"__future__", "math", "typing", "numpy"}
    for f in sorted(glob.glob(os.path.join(ROOT, "oracle", "*.py"))):
        tree = ast.parse(open(f, encoding="utf-8").read())
        for node in ast.walk(tree):
            if isinstance(node, ast.Import):
                names = [a.name.split(".")[0] for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                if node.level:  # within the oracle package itself
                    continue
                names = [node.module.split(".")[0]]
            else:
                continue
            for n in names:
                assert n in allowed, (f, n)


def _parents(tree):
    par = {}
    for node in ast.walk(tree):
        for ch in ast.iter_child_nodes(node):
            par[ch] = node
    return par


def _enclosing(node, par, kind):
    while node in par:
        node = par[node]
        if isinstance(node, kind):
            return node
    return None


def test_bench_reaches_the_oracle_only_from_its_cpu_legs():
    """bench.py imports the oracle inside `time_members` only; that function
    is called from the oracle estimate and the reference arm, and the estimate
    from the reference arm and from main's CPU-baseline block (which the flag
    turns off)."""
    tree = ast.parse(open(os.path.join(ROOT, "bench.py"), encoding="utf-8").read())
    par = _parents(tree)
    importers = set()
    calls = {"time_members": [], "oracle_estimate": []}
    for node in ast.walk(tree):
        mod = None
        if isinstance(node, ast.ImportFrom):
            mod = node.module or ""
        elif isinstance(node, ast.Import):
            mod = ",".join(a.name for a in node.names)
        if mod is not None and re.search(r"\boracle\b", mod):
            fn = _enclosing(node, par, ast.FunctionDef)
            assert fn is not None, "bench.py imports the oracle at module level"
            importers.add(fn.name)
        if isinstance(node, ast.Call) and isinstance(node.func, ast.Name) and node.func.id in calls:
            calls[node.func.id].append(node)
    assert importers == {"time_members"}
    callers = {k: {_enclosing(c, par, ast.FunctionDef).name for c in v} for k, v in calls.items()}
    assert callers["time_members"] == {"oracle_estimate", "run_reference"}
    assert callers["oracle_estimate"] == {"run_reference", "main"}
    for call in calls["oracle_estimate"]:
        if _enclosing(call, par, ast.FunctionDef).name == "main":
            guard = _enclosing(call, par, ast.If)
            assert guard is not None and "no_cpu_baseline" in ast.unparse(guard.test)


def test_binding_raises_without_its_library(monkeypatch):
    monkeypatch.setattr(_capi, "_lib", None)
    monkeypatch.setattr(_capi, "lib_path", lambda: os.path.join(ROOT, "no-such-dir", "libmuon.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _capi.load()
