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


def test_call_launches():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    # whole tiles only, two launches, or only the split tiles
    assert bench.call_launches("simt_128x128_t8x8", 4096, 4096, 1, 152) == 1
    assert bench.call_launches("simt_128x128_t8x8_split", 4096, 4096, 1, 152) == 2  # 912 + 112
    assert bench.call_launches("simt_128x128_t8x8_ksplit", 4096, 4864, 1, 152) == 1  # 8 x 152
    assert bench.call_launches("simt_128x128_t8x8_ksplit", 1024, 1024, 1, 152) == 1  # 64 < 152
    assert bench.call_launches("simt_128x128_t8x8_ksplit", 2048, 128, 128, 152) == 2
    # the k-chain: whole tiles, then one launch per k-slice of the last wave
    assert bench.call_launches("simt_128x128_t8x8_kchain", 4096, 4096, 1, 152) == 1 + 4
    assert bench.call_launches("simt_128x128_t8x8_kchain", 4096, 4864, 1, 152) == 1
    assert bench.call_launches("simt_128x128_t8x8_kchain", 1024, 1024, 1, 152) == 4
    # the per-problem grid splits a batch into chunks of 65535 problems
    assert bench.call_launches("simt_32x32x16_t4x4_s4", 64, 64, 65535, 152) == 1
    assert bench.call_launches("simt_32x32x16_t4x4_s4", 64, 64, 65536, 152) == 2
