"""The C ABI from plain C: include/rpa.h compiles as pedantic C99, and a C
program linked against librpa.so gets the documented codes on the host-only
paths (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_gets_the_documented_codes(tmp_path):
    from ragged_paged_attention_kv_gb300 import _lib, build
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    libdir = os.path.dirname(_lib.LIB_PATH)
    exe = str(tmp_path / "abi_from_c")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "abi_from_c.c"),
           "-o", exe, os.path.join(libdir, "librpa.so"), f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
