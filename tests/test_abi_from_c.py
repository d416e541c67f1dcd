"""The C ABI used from plain C: tests/c/abi_from_c.c includes include/dion3.h as C11 (so the
header carries no C++), links libdion3.so and calls its host-side paths (sizes, validation)."""

import os
import shutil
import subprocess

import pytest

from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_header_compiles_as_c11_and_library_links(tmp_path):
    lib = _build.build()
    libdir = os.path.dirname(lib)
    exe = tmp_path / "abi_from_c"
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_from_c.c"), "-o", str(exe), "-L", libdir, "-ldion3",
           f"-Wl,-rpath,{libdir}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip() == "ok"
