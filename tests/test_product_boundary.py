"""The product path stands alone (CPU only): it has no fallback when the
CUDA library is missing, and nothing in the package reaches the oracle."""

import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "linear_attention_decode_02_gb300")


def test_missing_library_fails_loudly():
    code = ("from linear_attention_decode_02_gb300 import binding\n"
            "binding.library('/nonexistent/dir/libkda.so')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0
    assert "libkda.so is not built" in r.stderr


def test_package_never_imports_the_oracle():
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if not f.endswith((".py", ".cu", ".cuh", ".h")):
                continue
            with open(os.path.join(dirpath, f)) as fh:
                text = fh.read()
            assert not re.search(r"^\s*(from|import)\s+oracle\b", text, re.M), f
            assert "kda_oracle" not in text, f


def test_oracle_imports_nothing_from_the_package():
    with open(os.path.join(ROOT, "oracle", "kda_oracle.py")) as fh:
        text = fh.read()
    assert "linear_attention_decode_02_gb300" not in text
    assert not re.search(r"^\s*import\s+torch|^\s*from\s+torch", text, re.M)
