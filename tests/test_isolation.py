"""Static checks that the product path and the oracle stay apart.

The package (kivi_bit_kv_gb300/, its Python and its CUDA sources) never
imports, includes or loads anything under oracle/, and the oracle never
imports the package.  In bench.py only the CPU-baseline leg and the reference
arm may reach the oracle.  The only module both sides share is the seeded
input generator, kivi_bit_kv_gb300/workloads.py, which holds no quantization
arithmetic: it must not call the library either.
"""
import ast
import glob
import os
import re

from conftest import ROOT

PKG = os.path.join(ROOT, "kivi_bit_kv_gb300")


def _imports(path):
    """(module, enclosing function or None) for every import in a file."""
    tree = ast.parse(open(path).read(), filename=path)
    found = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)):
                visit(child, child.name)
                continue
            if isinstance(child, ast.Import):
                found.extend((a.name, fn) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                found.append((child.module or "", fn))
            visit(child, fn)

    visit(tree, None)
    return found


def test_package_python_never_imports_the_oracle():
    for path in glob.glob(os.path.join(PKG, "*.py")):
        for mod, _ in _imports(path):
            assert not mod.startswith("oracle"), (path, mod)
        src = open(path).read()
        assert "libkivi_ref" not in src and "kivi_ref" not in src, path


def test_cuda_sources_never_include_the_oracle():
    for path in glob.glob(os.path.join(PKG, "csrc", "*")):
        src = open(path).read()
        for inc in re.findall(r'#include\s*[<"]([^>"]+)[>"]', src):
            assert "kivi_ref" not in inc and "oracle" not in inc, (path, inc)


def test_oracle_never_imports_the_package():
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        for mod, _ in _imports(path):
            assert not mod.startswith("kivi_bit_kv_gb300"), (path, mod)
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.[ch]")):
        src = open(path).read()
        for inc in re.findall(r'#include\s*[<"]([^>"]+)[>"]', src):
            assert inc.startswith(("kivi_ref", "std", "math", "string")), (path, inc)


def test_bench_reaches_the_oracle_only_from_the_cpu_legs():
    for mod, fn in _imports(os.path.join(ROOT, "bench.py")):
        if mod.startswith("oracle"):
            assert fn in ("cpu_baseline", "run_reference"), fn


def test_input_generator_holds_no_library_call():
    for mod, _ in _imports(os.path.join(PKG, "workloads.py")):
        assert not mod.startswith(("oracle", "kivi_bit_kv_gb300", ".")), mod
        assert mod.split(".")[0] not in ("ctypes",), mod
