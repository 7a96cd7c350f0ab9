"""The oracle and the CUDA path share no code: neither imports, loads or
includes the other, and the product package carries no CPU fallback into the
oracle.  Only the seeded input recipes (workloads.py, random numbers only) serve
both sides, and they hold none of the method's arithmetic.  This scans the
sources as text, on the CPU."""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "test_neural_memory_titans_b300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(top, exts):
    for dirpath, dirnames, filenames in os.walk(top):
        dirnames[:] = [d for d in dirnames if not d.startswith((".", "_")) and d != "__pycache__"]
        for f in filenames:
            if f.endswith(exts):
                yield os.path.join(dirpath, f)


def _imports(path):
    tree = ast.parse(open(path).read(), path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom):
            yield ("." * node.level) + (node.module or "")


def test_product_package_never_reaches_the_oracle():
    for path in _files(PKG, (".py",)):
        for name in _imports(path):
            assert not name.split(".")[0] == "oracle", (path, name)
        src = open(path).read()
        assert "liboracle" not in src and "nm_oracle" not in src, path
    for path in _files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".h", ".cpp", ".c")):
        src = open(path).read()
        assert not re.search(r'#\s*include\s*[<"][^>"]*oracle', src), path
        assert "liboracle" not in src and "oracle_" not in src, path


def test_oracle_never_reaches_the_product():
    for path in _files(ORACLE, (".py",)):
        for name in _imports(path):
            assert name.split(".")[0] != "test_neural_memory_titans_b300", (path, name)
        assert "libnm" not in open(path).read(), path
    for path in _files(ORACLE, (".c", ".h", ".cpp")):
        src = open(path).read()
        for inc in re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', src):
            assert not inc.startswith(("nm", "tc_")) and "csrc" not in inc, (path, inc)


def test_shared_input_recipes_hold_no_arithmetic_of_the_method():
    """workloads.py imports only the standard library and torch, and calls none
    of the method's steps (no gradient, momentum, forgetting or retrieval)."""
    path = os.path.join(PKG, "workloads.py")
    for name in _imports(path):
        assert name.split(".")[0] in ("__future__", "dataclasses", "typing", "torch"), name
    src = open(path).read()
    for word in ("silu", "sigmoid", "autograd", "backward(", "libnm", "oracle."):
        assert word not in src, word


def test_product_path_fails_loudly_without_its_library():
    """The binding raises when libnm.so is missing instead of falling back."""
    src = open(os.path.join(PKG, "__init__.py")).read()
    assert "raise ImportError" in src
    assert not re.search(r"\bexcept\s+(ImportError|OSError)\b[^\n]*:\s*\n\s*(pass|return None)", src)
