"""CPU checks that the oracle and the product stay apart: the library and its
Python package never import, include or load anything under oracle/, the
oracle never imports the product, and the benchmark touches the oracle only in
its CPU-baseline and reference legs."""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "rank_adapter_apply_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _sources(top, exts):
    for d, dirs, files in os.walk(top):
        dirs[:] = [x for x in dirs if not x.startswith(("_build", "__pycache__"))]
        for f in files:
            if f.endswith(exts):
                yield os.path.join(d, f)


def _imported_modules(path):
    tree = ast.parse(open(path).read(), path)
    for n in ast.walk(tree):
        if isinstance(n, ast.Import):
            for a in n.names:
                yield a.name.split(".")[0], n
        elif isinstance(n, ast.ImportFrom) and n.module and n.level == 0:
            yield n.module.split(".")[0], n


def test_product_never_imports_the_oracle():
    for path in _sources(PKG, (".py",)):
        mods = {m for m, _ in _imported_modules(path)}
        assert "oracle" not in mods and "tests" not in mods, path


def test_native_sources_never_include_the_oracle():
    inc = re.compile(r'#\s*include\s*[<"]([^>"]+)[>"]')
    for path in _sources(PKG, (".cu", ".cuh", ".cpp", ".h")):
        for name in inc.findall(open(path).read()):
            assert "oracle" not in name, (path, name)
        assert "lora_oracle" not in open(path).read(), path


def test_oracle_never_imports_the_product():
    for path in _sources(ORACLE, (".py",)):
        mods = {m for m, _ in _imported_modules(path)}
        assert not mods & {"rank_adapter_apply_gb300", "bench", "tests", "torch"}, path
    inc = re.compile(r'#\s*include\s*[<"]([^>"]+)[>"]')
    for path in _sources(ORACLE, (".c", ".h")):
        for name in inc.findall(open(path).read()):
            assert "/" not in name and "rank_adapter" not in name and "cuda" not in name, (path, name)


def test_bench_uses_the_oracle_only_for_cpu_timing():
    """bench.py imports the oracle inside the two functions that time it on the
    host (the cpu_baseline leg and the reference arm) and nowhere else."""
    path = os.path.join(ROOT, "bench.py")
    tree = ast.parse(open(path).read(), path)
    allowed = {"oracle_tokens_per_s", "run_reference"}
    owners = set()
    for f in ast.walk(tree):
        if isinstance(f, ast.FunctionDef):
            for n in ast.walk(f):
                if isinstance(n, (ast.Import, ast.ImportFrom)):
                    names = [a.name for a in n.names] if isinstance(n, ast.Import) else [n.module]
                    if any(x and x.split(".")[0] == "oracle" for x in names):
                        owners.add(f.name)
    top = {m for m, n in _imported_modules(path) if n.col_offset == 0}
    assert "oracle" not in top
    assert owners and owners <= allowed, owners
