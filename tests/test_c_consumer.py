"""The boundary as a C library: a plain C program built against the public
header and the shared library runs its host-side checks (no GPU needed)."""

import os
import shutil
import subprocess

import pytest

import deepseek_sparse_attention_ragged_gb300 as ds

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_links_and_calls_the_library(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = ds.build()
    exe = tmp_path / "abi_consumer"
    src = os.path.join(ROOT, "tests", "c", "abi_consumer.c")
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src, "-o", str(exe),
                    "-L", os.path.dirname(lib), "-ldsrows", "-Wl,-rpath," + os.path.dirname(lib)],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "all checks passed" in r.stdout
