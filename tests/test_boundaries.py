"""The oracle and the CUDA path stay apart (CPU only, static checks).

The library (package, CUDA sources, headers) never imports, links or reads the
oracle; the oracle imports nothing from the library.  Only the seeded input
generators (workloads.py) serve both sides, and they hold none of the
method's arithmetic.
"""

import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "speculative_drafting_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "__pycache__" in d or "_build" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def _imports(path):
    tree = ast.parse(open(path).read())
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            yield from (a.name for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            yield ("." * node.level) + (node.module or "")


def test_library_never_imports_the_oracle():
    for f in _files(PKG, (".py",)):
        for mod in _imports(f):
            assert not mod.split(".")[0] == "oracle", f"{f} imports {mod}"


def test_cuda_sources_and_headers_never_name_the_oracle():
    tops = [os.path.join(PKG, "csrc"), os.path.join(ROOT, "include")]
    for top in tops:
        for f in _files(top, (".cu", ".cuh", ".h", ".cc", ".cpp")):
            text = open(f).read()
            assert not re.search(r"\boracle\b|pe_oracle|pe_cod\.py", text), f


def test_oracle_imports_nothing_from_the_library():
    allowed = {"numpy", "scipy", "math", "__future__", "dataclasses", "functools", "itertools",
               "collections", "typing", "os", "concurrent"}
    for f in _files(ORACLE, (".py",)):
        for mod in _imports(f):
            top = mod.lstrip(".").split(".")[0]
            assert top in allowed or mod.startswith("."), f"{f} imports {mod}"


def test_input_generators_hold_no_method_arithmetic():
    # workloads.py draws and lays out numbers; it names none of the step's ops
    text = open(os.path.join(PKG, "workloads.py")).read()
    for word in ("rmsnorm", "softmax", "argmax", "rope", "silu", "swiglu", "einsum", "matmul"):
        assert not re.search(rf"\b{word}\s*\(", text, re.I), word
