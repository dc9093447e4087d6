"""The C ABI from a C99 program (tests/c_abi_client.c), with no Python or C++ in between.

On the CPU: the header compiles as C99 with every warning an error, a C program links
against libfgemm.so, and the library's host-only queries and argument checks answer
as the header says.  On a GPU: the same program copies a seeded problem to the
device, calls fgemm_sgemm_bias_relu on a stream of its own and writes C back; the
result must equal the FP64 oracle's bit for bit (small-integer data).
"""

import glob
import os
import struct
import subprocess

import numpy as np
import pytest

import oracle
from dense_fp32_gemm_sm_gb300 import _build, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_client.c")


def _cuda_lib_dir(cuda):
    for d in [os.path.join(cuda, "lib64")] + sorted(glob.glob(os.path.join(cuda, "targets", "*", "lib"))):
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    pytest.skip("no shared CUDA runtime library found")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    lib = _build.build()
    cuda = os.path.dirname(os.path.dirname(_build.nvcc()))
    libdir, cudalib = os.path.dirname(lib), _cuda_lib_dir(cuda)
    exe = str(tmp_path_factory.mktemp("c_abi") / "c_abi_client")
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror",
           "-isystem", os.path.join(cuda, "include"), "-I", os.path.join(ROOT, "include"),
           SRC, "-o", exe, "-L", libdir, "-lfgemm", "-Wl,-rpath," + libdir,
           "-L", cudalib, "-lcudart", "-Wl,-rpath," + cudalib]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_header_compiles_as_c_and_host_calls_answer(client):
    r = subprocess.run([client, "host"], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok host", r.stdout + r.stderr


CASES = [  # ta, tb, M, N, K, alpha, beta, bias, relu, seed
    (0, 0, 150, 131, 77, 1.5, 0.5, True, True, 40),
    (1, 0, 300, 260, 333, -1.0, 0.0, False, False, 41),
    (0, 1, 129, 257, 64, 2.0, -0.25, True, False, 42),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES)
def test_c_program_gemm_matches_the_oracle(client, tmp_path, case):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    ta, tb, M, N, K, alpha, beta, bias, relu, seed = case
    g = workloads.generator(seed)
    A = workloads.small_ints(g, (K, M) if ta else (M, K)).numpy()
    B = workloads.small_ints(g, (N, K) if tb else (K, N)).numpy()
    C0 = workloads.small_ints(g, (M, N)).numpy()
    b = workloads.small_ints(g, (N,)).numpy() if bias else None
    src, dst = tmp_path / "problem.bin", tmp_path / "c.bin"
    with open(src, "wb") as f:
        f.write(struct.pack("<7i2f", ta, tb, M, N, K, int(bias), int(relu), alpha, beta))
        for x in (A, B, C0) + ((b,) if bias else ()):
            f.write(np.ascontiguousarray(x, dtype="<f4").tobytes())
    r = subprocess.run([client, "run", str(src), str(dst)], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok run", r.stdout + r.stderr
    got = np.fromfile(dst, dtype="<f4").reshape(M, N).astype(np.float64)
    want, _ = oracle.gemm(ta, tb, M, N, K, alpha, A.reshape(-1), M if ta else K, B.reshape(-1),
                          K if tb else N, beta=beta, C0=C0.reshape(-1), ldc=N, bias=b, relu=relu,
                          want_mag=False)
    assert np.array_equal(got, want)
