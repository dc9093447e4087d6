"""Calls from several host threads at once, each thread on its own stream.

The header promises that calls from several host threads are safe (except the no-alloc
split-K entry, whose calls share one scratch array, and the tensor-core test hook).  The
test runs in a fresh Python process, so every first-use setup of the library -- kernel
attributes, the SM count, the tensor-map encoder, the device error word -- happens while
the threads race: eight threads wait at a barrier, then each makes a different mix of
calls on its own stream and data, three times over: plain calls in every transpose
layout (single and strided-batch, whole tiles and the last-wave splits), the staged call
with its own workspace, split-K with its own workspace, the row-bias entry and both
tensor-core modes.  Every result is compared with the FP64 oracle element by element;
the data are small integers, so each must match bit for bit.
"""

import os
import subprocess
import sys
import threading

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
THREADS = 8
REPEATS = 3

# (entry, ta, tb, M, N, K, batch, alpha, beta, bias, relu, extra)
TEMPLATES = [
    ("plain", 0, 0, 300, 260, 333, 1, 1.5, 0.5, True, True, None),
    ("plain", 0, 1, 200, 172, 96, 3, 1.0, 0.0, False, False, None),
    ("plain", 1, 0, 2000, 1900, 256, 1, 1.0, -1.0, False, False, None),  # whole tiles + last wave
    ("plain", 1, 1, 129, 257, 77, 1, -0.5, 0.0, True, False, None),
    ("staged", 0, 1, 520, 600, 300, 2, 1.0, 0.0, False, False, -1),
    ("staged", 0, 0, 700, 300, 200, 1, 2.0, 0.0, True, True, 3),
    ("splitk", 0, 0, 256, 256, 1024, 1, 1.0, 0.5, True, True, 4),
    ("row_bias", 1, 0, 333, 222, 111, 1, 1.0, 0.25, False, True, None),
    ("tf32", 0, 0, 384, 256, 128, 1, 1.0, 0.0, True, False, None),
    ("3xtf32", 0, 1, 256, 384, 160, 2, -1.0, 0.5, False, False, None),
]


def _child():
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch

    import dense_fp32_gemm_sm_gb300 as fg
    import oracle
    from dense_fp32_gemm_sm_gb300 import workloads

    torch.cuda.init()
    fg.library()  # load the shared object; no CUDA call of the library has run yet

    def make(t, i):
        entry, ta, tb, M, N, K, batch, alpha, beta, bias, relu, extra = TEMPLATES[i]
        g = workloads.generator(1000 * t + i)
        a_shape = (K, M) if ta else (M, K)
        b_shape = (N, K) if tb else (K, N)
        c = dict(entry=entry, ta=ta, tb=tb, M=M, N=N, K=K, batch=batch, alpha=alpha, beta=beta,
                 relu=relu, extra=extra)
        c["A"] = workloads.small_ints(g, (batch,) + a_shape)
        c["B"] = workloads.small_ints(g, (batch,) + b_shape)
        c["C0"] = workloads.small_ints(g, (batch, M, N))
        c["bias"] = workloads.small_ints(g, (M if entry == "row_bias" else N,)) if (
            bias or entry == "row_bias") else None
        c["lda"], c["ldb"] = a_shape[1], b_shape[1]
        return c

    def to_device(c):
        d = {k: (v.cuda() if hasattr(v, "cuda") else v) for k, v in c.items()}
        d["C"] = d["C0"].clone()
        if d["entry"] == "staged":
            need = fg.staged_workspace_size(c["ta"], c["tb"], c["M"], c["N"], c["K"], c["batch"])
            d["ws"], d["need"] = torch.empty((need + 3) // 4, device="cuda"), need
        if d["entry"] == "splitk":
            need = fg.splitk_workspace_size(c["M"], c["N"], c["K"], c["extra"])
            d["ws"], d["need"] = torch.empty((need + 3) // 4, device="cuda"), need
        return d

    def call(d, s):
        ta, tb, M, N, K, b = d["ta"], d["tb"], d["M"], d["N"], d["K"], d["batch"]
        A, B, C, lda, ldb = d["A"], d["B"], d["C"], d["lda"], d["ldb"]
        sA, sB, sC = A[0].numel(), B[0].numel(), M * N
        al, be, bias, relu = d["alpha"], d["beta"], d["bias"], d["relu"]
        C.copy_(d["C0"])  # on stream s: every repeat starts from the same C
        e = d["entry"]
        if e == "plain":
            fg.gemm_explicit(-1, ta, tb, M, N, K, al, A, lda, sA, B, ldb, sB, be, C, N, sC, b,
                             bias=bias, apply_relu=relu, stream=s)
        elif e == "staged":
            fg.sgemm_staged(ta, tb, M, N, K, al, A, lda, sA, B, ldb, sB, be, C, N, sC, b, bias,
                            relu, d["extra"], d["ws"], d["need"], stream=s)
        elif e == "splitk":
            fg.sgemm_splitk(ta, tb, M, N, K, al, A, lda, B, ldb, be, C, N, bias, relu, d["extra"],
                            d["ws"], d["need"], stream=s)
        elif e == "row_bias":
            fg.sgemm_row_bias_relu(ta, tb, M, N, K, al, A, lda, B, ldb, be, C, N, bias, relu,
                                   stream=s)
        else:
            math = fg.MATH_TF32 if e == "tf32" else fg.MATH_3XTF32
            assert fg.math_supported(math, ta, tb, M, N, K, al, A, lda, sA, B, ldb, sB, b) == 1
            fg.gemm_math(math, ta, tb, M, N, K, al, A, lda, sA, B, ldb, sB, be, C, N, sC, b,
                         bias=bias, apply_relu=relu, stream=s)

    host = [[make(t, (t + j) % len(TEMPLATES)) for j in range(len(TEMPLATES))]
            for t in range(THREADS)]
    dev = [[to_device(c) for c in row] for row in host]
    torch.cuda.synchronize()

    barrier = threading.Barrier(THREADS)
    errors = []

    def work(t):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                barrier.wait()
                for _ in range(REPEATS):
                    for d in dev[t]:
                        call(d, s)
            s.synchronize()
        except Exception as exc:  # reported by the parent through the exit status
            errors.append("thread %d: %r" % (t, exc))
            barrier.abort()

    threads = [threading.Thread(target=work, args=(t,)) for t in range(THREADS)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    if errors:
        print("\n".join(errors))
        sys.exit(1)
    assert fg.device_status() == fg.OK

    checked = 0
    for t in range(THREADS):
        for c, d in zip(host[t], dev[t]):
            M, N, K, b = c["M"], c["N"], c["K"], c["batch"]
            got = d["C"].cpu().numpy().astype(np.float64)
            for p in range(b):
                want, _ = oracle.gemm(c["ta"], c["tb"], M, N, K, c["alpha"],
                                      c["A"][p].numpy().reshape(-1), c["lda"],
                                      c["B"][p].numpy().reshape(-1), c["ldb"], beta=c["beta"],
                                      C0=c["C0"][p].numpy().reshape(-1), ldc=N,
                                      bias=None if c["entry"] == "row_bias" else c["bias"],
                                      row_bias=c["bias"] if c["entry"] == "row_bias" else None,
                                      relu=c["relu"], want_mag=False)
                if not np.array_equal(got[p], want):
                    bad = np.argwhere(got[p] != want)[0]
                    print("thread %d, %s %s: element %s is %r, the oracle says %r" % (
                        t, c["entry"], (c["ta"], c["tb"], M, N, K, b), tuple(bad),
                        got[p][tuple(bad)], want[tuple(bad)]))
                    sys.exit(1)
                checked += 1
    print("ok: %d threads x %d repeats, %d problems checked" % (THREADS, REPEATS, checked))


@pytest.mark.gpu
def test_calls_from_many_host_threads():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    r = subprocess.run([sys.executable, os.path.abspath(__file__)], cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok:"), r.stdout


if __name__ == "__main__":
    _child()
