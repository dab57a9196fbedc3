"""The oracle and the CUDA path share nothing, and only the allowed places run
the oracle: checked on the sources, without a GPU.

- The package (Python binding, build, input generators, kernels, C ABI) never
  imports, includes or names the oracle.
- The oracle never imports the package, includes its headers or loads its
  library.
- The benchmark imports the oracle only inside its CPU-baseline leg and its
  reference arm; ``__graft_entry__`` only inside ``smoke()``.
"""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "tensor_gemm_reduction_gb300")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "_lib" in d or "__pycache__" in d or "_build" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def test_package_never_touches_the_oracle():
    for path in list(_files(PKG, (".py", ".cu", ".cuh", ".h"))) + [os.path.join(ROOT, "include", "gsr.h")]:
        text = open(path).read()
        assert not re.search(r"\boracle\b", text, re.I), path


def test_oracle_never_touches_the_package():
    for path in _files(os.path.join(ROOT, "oracle"), (".py", ".c", ".h")):
        text = open(path).read()
        assert "tensor_gemm_reduction_gb300" not in text, path
        assert "libgsr.so" not in text, path
        assert not re.search(r'#include\s+"gsr(_params|_device)?\.(h|cuh)"', text), path
        if path.endswith(".py"):
            for node in ast.walk(ast.parse(text)):
                if isinstance(node, (ast.Import, ast.ImportFrom)):
                    mods = [a.name for a in node.names] if isinstance(node, ast.Import) else [node.module or ""]
                    assert not any(m.startswith(("tensor_gemm_reduction_gb300", "bench")) for m in mods), path


def _oracle_import_sites(path):
    tree = ast.parse(open(path).read())
    sites = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            name = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else fn
            if isinstance(child, ast.Import) and any(a.name.split(".")[0] == "oracle" for a in child.names):
                sites.append(fn)
            if isinstance(child, ast.ImportFrom) and (child.module or "").split(".")[0] == "oracle":
                sites.append(fn)
            visit(child, name)

    visit(tree, None)
    return sites


def test_bench_runs_the_oracle_only_in_its_baseline_legs():
    sites = _oracle_import_sites(os.path.join(ROOT, "bench.py"))
    assert sites and set(sites) <= {"cpu_oracle_rate", "run_reference"}, sites


def test_graft_entry_runs_the_oracle_only_in_smoke_and_build():
    sites = _oracle_import_sites(os.path.join(ROOT, "__graft_entry__.py"))
    # build() compiles the oracle (building the checker is not using it).
    assert sites and set(sites) <= {"smoke", "build"}, sites
