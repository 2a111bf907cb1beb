"""The oracle stays test infrastructure and shares nothing with the CUDA path.

Static checks over the source tree: outside tests/ the oracle is imported only
by the entry points allowed to run it (the build step that compiles it, the
smoke check, and the benchmark's CPU-baseline and reference legs); the product
package never names it; the oracle's C source includes only system headers and
the CUDA sources include nothing of the oracle's.
"""
from __future__ import annotations

import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "w8a8_quantized_decode_gb300")

# file -> functions that may import the oracle
ALLOWED = {
    "__graft_entry__.py": {"build", "smoke"},
    "bench.py": {"time_oracle_steps", "run_reference", "cpu_baseline"},
}
# functions that run the oracle, and the only functions that may call them
ORACLE_RUNNERS = {"bench.py": ({"time_oracle_steps"}, {"run_reference", "cpu_baseline"})}


def _py_files():
    """Python files of the repository outside tests/ and oracle/: the files
    git tracks, or, in a copy without git metadata, the top-level scripts and
    the product packages."""
    import subprocess
    skip = ("tests", "oracle", "baseline")
    try:
        out = subprocess.run(["git", "ls-files", "*.py"], cwd=ROOT, capture_output=True,
                             text=True, check=True).stdout.split()
    except (OSError, subprocess.CalledProcessError):
        out = []
    if not out:
        out = [f for f in os.listdir(ROOT) if f.endswith(".py")]
        for pkg in ("w8a8_quantized_decode_gb300", "synth"):
            out += [os.path.relpath(p, ROOT)
                    for p in glob.glob(os.path.join(ROOT, pkg, "**", "*.py"), recursive=True)]
    for rel in out:
        if rel.split("/")[0] not in skip:
            yield os.path.join(ROOT, rel)


def _imports_oracle(node) -> bool:
    if isinstance(node, ast.Import):
        return any(a.name == "oracle" or a.name.startswith("oracle.") for a in node.names)
    if isinstance(node, ast.ImportFrom):
        return (node.module or "").split(".")[0] == "oracle" and node.level == 0
    return False


def _function_scopes(tree):
    """(function name, node) for every node, the innermost enclosing def."""
    out = []

    def walk(node, fn):
        for child in ast.iter_child_nodes(node):
            name = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else fn
            out.append((name, child))
            walk(child, name)
    walk(tree, None)
    return out


def test_oracle_imported_only_where_allowed():
    seen = {}
    for path in _py_files():
        rel = os.path.relpath(path, ROOT)
        tree = ast.parse(open(path).read(), rel)
        for fn, node in _function_scopes(tree):
            if _imports_oracle(node):
                assert fn in ALLOWED.get(rel, set()), f"{rel}: oracle imported in {fn!r}"
                seen.setdefault(rel, set()).add(fn)
    assert seen.get("bench.py") and seen.get("__graft_entry__.py")


def test_oracle_runners_called_only_from_the_baseline_legs():
    for rel, (runners, callers) in ORACLE_RUNNERS.items():
        tree = ast.parse(open(os.path.join(ROOT, rel)).read(), rel)
        for fn, node in _function_scopes(tree):
            if isinstance(node, ast.Call) and getattr(node.func, "id", None) in runners:
                assert fn in callers, f"{rel}: {node.func.id} called from {fn!r}"


def test_product_package_never_names_the_oracle():
    for path in glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True):
        tree = ast.parse(open(path).read(), path)
        for node in ast.walk(tree):
            assert not _imports_oracle(node), path
            if isinstance(node, ast.Name):
                assert node.id != "oracle", path
    for path in glob.glob(os.path.join(PKG, "csrc", "*")):
        src = open(path).read()
        for inc in re.findall(r'#include\s+[<"]([^>"]+)[>"]', src):
            assert "oracle" not in inc, (path, inc)
        assert "a8w8_oracle" not in src and "or_" + "decode" not in src, path


def test_oracle_c_source_includes_only_system_headers():
    src = open(os.path.join(ROOT, "oracle", "a8w8_oracle.c")).read()
    incs = re.findall(r"#include\s+([<\"][^>\"]+[>\"])", src)
    assert incs and all(i.startswith("<") for i in incs), incs
    assert "a8w8.h" not in src and "kernels.cuh" not in src
