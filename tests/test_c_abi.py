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


@pytest.mark.gpu
def test_c_program_decodes_on_the_gpu():
    # abi_decode.c allocates device memory with the CUDA runtime, runs pa_decode and
    # writes its host-generated inputs and the output; the float64 oracle checks the
    # output here
    import numpy as np
    from harness import assert_parity
    from oracle import decode_ref

    cc = shutil.which("gcc") or shutil.which("cc")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if cc is None or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime_api.h")):
        pytest.skip("no C compiler or CUDA runtime headers")
    lib = pa_build.build()
    os.makedirs(pa_build.BUILD_DIR, exist_ok=True)
    exe = os.path.join(pa_build.BUILD_DIR, "abi_decode")
    libdir = os.path.dirname(lib)
    cudalib = next(d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                   if os.path.isdir(d))
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror",
                    "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(cuda, "include"),
                    os.path.join(ROOT, "tests", "c_abi", "abi_decode.c"), "-o", exe,
                    "-L" + libdir, "-l:" + os.path.basename(lib), "-L" + cudalib, "-lcudart",
                    "-Wl,-rpath," + libdir + ":" + cudalib],
                   check=True, capture_output=True, text=True)
    dump = os.path.join(pa_build.BUILD_DIR, "abi_decode.bin")
    r = subprocess.run([exe, dump], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stderr)
    B, HQ, HKV, D = 2, 8, 2, 128
    raw = open(dump, "rb").read()

    def take(n, dt):
        nonlocal raw
        a = np.frombuffer(raw[:n * np.dtype(dt).itemsize], dtype=dt)
        raw = raw[n * np.dtype(dt).itemsize:]
        return a

    def bf16(bits):  # bf16 bits -> float64
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    lens = [1000, 37]
    q = bf16(take(B * HQ * D, np.uint16)).reshape(B, HQ, D)
    kc = bf16(take(sum(lens) * HKV * D, np.uint16)).reshape(sum(lens), HKV, D)
    vc = bf16(take(sum(lens) * HKV * D, np.uint16)).reshape(sum(lens), HKV, D)
    sl = take(B, np.int32)
    out = bf16(take(B * HQ * D, np.uint16)).reshape(B, HQ, D)
    assert not raw and list(sl) == lens
    # each sequence's K and V in token order, as the program generated them
    K = [kc[:lens[0]], kc[lens[0]:]]
    V = [vc[:lens[0]], vc[lens[0]:]]
    ref = decode_ref(q, K, V, float(np.float32(0.08838834764831845)))
    assert_parity(out, ref, what="C program")
