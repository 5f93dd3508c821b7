"""include/pa.h from plain C (CPU only): the header compiles as C11 with warnings as
errors, a C program links libpa.so, and its GPU-free calls answer as the Python
binding's do."""
import os
import shutil
import subprocess

import pytest

import paged_kv_attention_pa_gb300 as pa
from paged_kv_attention_pa_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "abi_check.c")


def test_c_consumer():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = pa_build.build()
    os.makedirs(pa_build.BUILD_DIR, exist_ok=True)
    exe = os.path.join(pa_build.BUILD_DIR, "abi_check")  # the in-tree build folder
    libdir = os.path.dirname(lib)
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I" + os.path.join(ROOT, "include"), SRC, "-o", exe,
                    "-L" + libdir, "-l:" + os.path.basename(lib), "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {line.split()[0]: line.split()[1:] for line in out if line.strip()}
    assert got["version"] == [pa.version()]
    assert got["status"][0] == str(pa.PA_ERR_WORKSPACE)
    assert " ".join(got["status"][1:]) == pa.status_string(pa.PA_ERR_WORKSPACE)
    S, P = pa.plan(1, 24, 4, 256, 784, 32768, sm_count=152)
    assert got["plan"] == [str(pa.PA_OK), str(S), str(P)]
    assert got["invalid"] == [str(pa.PA_ERR_INVALID_ARG)]
    assert got["deterministic_plan"] == [str(pa.PA_OK)]
    assert got["header_bytes"] == [str(pa.PA_WORKSPACE_HEADER_BYTES)]
