"""Separation of the product path, the oracle and the input generators, checked on the source (no GPU).

* The oracle imports nothing but numpy, the standard library and its own modules: it shares no code with
  the CUDA path or the input generators.
* Nothing in the product package (the binding, the build script, the CUDA sources and the header) names
  the oracle, and the input generators do not import it either.
* `bench.py` imports the oracle in one function only, reached from the reference arm alone (the GPU
  run's CPU baseline runs that arm as a child process).
* A missing library makes the binding raise: there is no fallback to run instead.
"""
import ast
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "w4afp8_mixture_experts_gb300")


def _py_files(d):
    for base, _, files in os.walk(d):
        if "_lib" in base or "__pycache__" in base:
            continue
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(base, f)


def _imports(path):
    """(top-level module name or '.' for relative, enclosing function name or None) of every import."""
    tree = ast.parse(open(path).read(), path)
    out = []

    def visit(node, func):
        for ch in ast.iter_child_nodes(node):
            f = ch.name if isinstance(ch, (ast.FunctionDef, ast.AsyncFunctionDef)) else func
            if isinstance(ch, ast.Import):
                out.extend((a.name.split(".")[0], func) for a in ch.names)
            elif isinstance(ch, ast.ImportFrom):
                out.append(("." if ch.level else ch.module.split(".")[0], func))
            visit(ch, f)

    visit(tree, None)
    return out


def test_oracle_imports_only_numpy_the_standard_library_and_itself():
    allowed = {"numpy", "."} | set(sys.stdlib_module_names)
    found = {m for p in _py_files(os.path.join(ROOT, "oracle")) for m, _ in _imports(p)}
    assert "numpy" in found
    assert found <= allowed, found - allowed


def test_product_package_and_input_generators_never_name_the_oracle():
    for p in _py_files(PKG):
        assert "oracle" not in {m for m, _ in _imports(p)}, p
    for p in _py_files(os.path.join(ROOT, "inputs")):
        assert "oracle" not in {m for m, _ in _imports(p)}, p
    native = [os.path.join(PKG, "csrc", f) for f in os.listdir(os.path.join(PKG, "csrc"))]
    native += [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    for p in native:
        assert "oracle" not in open(p).read().lower(), p


def test_bench_imports_the_oracle_only_in_its_cpu_timing_leg():
    users = {func for m, func in _imports(os.path.join(ROOT, "bench.py")) if m == "oracle"}
    assert users == {"oracle_sample"}
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    callers = {}
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for n in ast.walk(fn):
                if isinstance(n, ast.Name) and n.id in ("oracle_sample", "_oracle_worker", "oracle_on_host_cores"):
                    callers.setdefault(n.id, set()).add(fn.name)
    assert callers["oracle_sample"] == {"_oracle_worker"}
    assert callers["_oracle_worker"] == {"oracle_on_host_cores"}
    assert callers["oracle_on_host_cores"] == {"run_reference"}
    # the GPU run's cpu_baseline is that reference arm, run as a child process of its own
    src = ast.get_source_segment(open(os.path.join(ROOT, "bench.py")).read(),
                                 next(f for f in ast.walk(tree) if isinstance(f, ast.FunctionDef)
                                      and f.name == "cpu_baseline"))
    assert '"--impl", "reference"' in src


def test_missing_library_raises(monkeypatch, tmp_path):
    import w4afp8_mixture_experts_gb300._binding as b
    monkeypatch.setattr(b, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        b.load(str(tmp_path / "libw4a8moe.so"))
