"""The C ABI from C: `tests/c_client/kda_c_client.c` is compiled as strict
C99 against include/kda.h, linked against the built libkda.so, and run (it
needs no GPU: it checks the version and status strings, the dispatch policy
queries and the host-side contract checks)."""

import os
import shutil
import subprocess

import pytest

from linear_attention_decode_02_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib_dir():
    build.build()
    return os.path.join(ROOT, "linear_attention_decode_02_gb300")


def test_c_client_compiles_links_and_runs(lib_dir, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "kda_c_client"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_client", "kda_c_client.c"),
                    "-L", lib_dir, "-lkda", "-Wl,-rpath," + lib_dir, "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "all checks passed" in r.stdout
