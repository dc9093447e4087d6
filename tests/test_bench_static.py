"""Static check of bench.py: every name it reads is bound somewhere in the file, imported,
or a builtin.  The GPU arm of the benchmark cannot run without a GPU, so this catches a
stale variable name there before a GPU run does."""

import ast
import builtins
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_reads_only_bound_names():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py"), encoding="utf-8").read())
    bound = set(dir(builtins)) | {"__file__", "__name__"}
    for n in ast.walk(tree):
        if isinstance(n, ast.Name) and isinstance(n.ctx, (ast.Store, ast.Del)):
            bound.add(n.id)
        elif isinstance(n, (ast.FunctionDef, ast.AsyncFunctionDef, ast.ClassDef)):
            bound.add(n.name)
        elif isinstance(n, (ast.Import, ast.ImportFrom)):
            bound |= {a.asname or a.name.split(".")[0] for a in n.names}
        elif isinstance(n, ast.arg):
            bound.add(n.arg)
        elif isinstance(n, ast.ExceptHandler) and n.name:
            bound.add(n.name)
    loads = {n.id for n in ast.walk(tree) if isinstance(n, ast.Name) and isinstance(n.ctx, ast.Load)}
    assert not sorted(loads - bound)


def test_launch_count():
    # the library's own count of the kernel launches of one call (bench.py reports it)
    import sys
    sys.path.insert(0, ROOT)
    import dense_fp32_gemm_sm_gb300 as fg
    cfg = {fg.config_name(i): i for i in range(fg.num_configs())}
    lc = fg.launch_count
    assert lc(cfg["simt_128x128_t8x8"], 0, 0, 4096, 4096, 4096, 1, True, 152) == 1
    assert lc(cfg["simt_128x128_t8x8_split"], 0, 0, 4096, 4096, 4096, 1, True, 152) == 2
    assert lc(cfg["simt_128x128_t8x8_ksplit"], 0, 0, 4096, 4864, 4096, 1, True, 152) == 1
    assert lc(cfg["simt_128x128_t8x8_ksplit"], 0, 0, 1024, 1024, 1024, 1, True, 152) == 1
    assert lc(cfg["simt_128x128_t8x8_ksplit"], 0, 0, 2048, 128, 2048, 128, True, 152) == 2
    # the k-chain: whole tiles, then one launch per k-slice of the last wave: four for
    # the 112 tiles of 4096^3, three for 44 tiles at K = 1024, five for 120 at 3072, seven
    # for 16 at 4096; two for the 136 tiles 148 SMs leave at 4096^3
    assert lc(cfg["simt_128x128_t8x8_kchain"], 0, 0, 4096, 4096, 4096, 1, True, 152) == 1 + 4
    assert lc(cfg["simt_128x128_t8x8_kchain"], 0, 0, 1792, 1792, 1024, 1, True, 152) == 1 + 3
    assert lc(cfg["simt_128x128_t8x8_kchain"], 0, 0, 3072, 3072, 3072, 1, True, 152) == 1 + 5
    assert lc(cfg["simt_128x128_t8x8_kchain"], 0, 0, 4096, 3648, 4096, 1, True, 152) == 1 + 7
    assert lc(cfg["simt_128x128_t8x8_kchain"], 0, 0, 4096, 4096, 4096, 1, True, 148) == 1 + 2
    assert lc(cfg["simt_128x128_t8x8_kchain"], 0, 0, 4096, 4864, 4096, 1, True, 152) == 1
    # the per-problem grid splits a batch into chunks of 65535 problems
    assert lc(cfg["simt_32x32x16_t4x4_s4"], 0, 0, 64, 64, 64, 65535, True, 152) == 1
    assert lc(cfg["simt_32x32x16_t4x4_s4"], 0, 0, 64, 64, 64, 65536, True, 152) == 2
    assert lc(cfg["simt_128x128_t8x8"], 0, 0, 64, 64, 64, 65536, True, 152) == 2
    # TT whole tiles: linear-order launches of up to 2^31 - 1 CTAs
    assert lc(cfg["simt_128x128_t8x8"], 1, 1, 64, 64, 64, 65536, True, 152) == 1
    assert lc(cfg["simt_128x128_t8x8"], 1, 1, 256, 256, 64, 2**29, True, 152) == 2  # 4 tiles a problem
    # selection, empty problems and bad arguments
    assert lc(-1, 0, 0, 4096, 4096, 4096, 1, True, 152) == 5
    assert lc(-1, 0, 0, 0, 4096, 4096, 1, True, 152) == 0
    assert lc(-1, 0, 0, -1, 4096, 4096, 1, True, 152) == -1
    assert lc(fg.num_configs(), 0, 0, 8, 8, 8, 1, True, 152) == -1
