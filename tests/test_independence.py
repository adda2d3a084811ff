"""The oracle and the CUDA path share no code (CPU only): no module of the
product package imports the oracle, no oracle module imports the product
package or the tests, the native sources include nothing from the oracle, and
the seeded input generators that serve both sides import neither."""

import ast
import glob
import os
import re

from tests.conftest import ROOT

PKG = "pagedattention_decode_attention_gb300"


def imported_modules(path):
    """Top-level names of every module a Python file imports (at any depth:
    imports inside functions count too).  Relative imports are reported as
    ``.`` so they stay inside their own package."""
    tree = ast.parse(open(path).read(), filename=path)
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom):
            names.add("." if node.level else node.module.split(".")[0])
    return names


def py_files(folder):
    return sorted(glob.glob(os.path.join(ROOT, folder, "**", "*.py"), recursive=True))


def test_product_package_never_imports_the_oracle():
    files = py_files(PKG)
    assert files
    offenders = [f for f in files if {"oracle", "tests"} & imported_modules(f)]
    assert not offenders, offenders


def test_oracle_never_imports_the_product_or_the_tests():
    files = py_files("oracle")
    assert files
    offenders = [f for f in files if {PKG, "tests", "bench", "__graft_entry__"} & imported_modules(f)]
    assert not offenders, offenders


def test_native_sources_include_nothing_from_the_oracle():
    sources = []
    for ext in ("cu", "cuh", "cpp", "h"):
        sources += glob.glob(os.path.join(ROOT, PKG, "csrc", f"*.{ext}"))
    sources += glob.glob(os.path.join(ROOT, "include", "*.h"))
    assert sources
    include = re.compile(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', re.M)
    for path in sources:
        for target in include.findall(open(path).read()):
            assert "oracle" not in target, (path, target)


def test_input_generators_import_neither_side():
    """The seeded generators feed both sides, so they hold none of the
    method's arithmetic: they import neither the oracle nor the library's
    binding, kernels or pool."""
    mods = imported_modules(os.path.join(ROOT, PKG, "workloads.py"))
    assert "oracle" not in mods and "." not in mods and PKG not in mods, mods
