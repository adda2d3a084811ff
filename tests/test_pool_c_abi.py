"""The host pool driven from plain C through the public header and the built
library (CPU): tests/pool_abi_check.c compiled with the system C compiler."""

import os
import shutil
import subprocess

import pytest

from tests.conftest import ROOT


def test_pool_from_c(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from pagedattention_decode_attention_gb300 import build, capi
    if not os.path.exists(capi.LIB_PATH):
        build.build()
    libdir = os.path.dirname(capi.LIB_PATH)
    exe = tmp_path / "pool_abi_check"
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "pool_abi_check.c"), "-o", str(exe),
                    "-L", libdir, "-lpagedattn", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "all checks passed" in out.stdout
