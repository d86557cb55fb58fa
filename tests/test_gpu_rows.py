"""Parity of the short-row direct path (one block per row, the row in
registers: n <= 32768, k <= 1024) with the CPU oracle, bit-exact.

Covers the candidate path (the k-th largest per-thread maximum bounds the
candidates), the many-ties path (every element at one value: the exact k-th
value and position-ordered ties), ragged and tiny rows, both dtypes and both
directions.
"""
import zlib

import pytest

from oracle import plain
from top_selection_prof_gb300 import workloads

from .gpu_util import assert_same, to_device

pytestmark = pytest.mark.gpu

# (kind, rows, n, k)
ROWS = [
    ("normal", 300, 32768, 64),          # the many-rows benchmark shape, fewer rows
    ("normal", 200, 32768, 1024),        # largest k of the path
    ("normal", 200, 32768, 1),
    ("uniform", 170, 30001, 333),        # ragged rows: scalar loads
    ("ties1000", 160, 32768, 700),       # many equal values
    ("constant", 160, 32768, 100),       # all equal: the many-ties path
    ("constant", 3, 5000, 1024),
    ("specials", 160, 4099, 50),         # NaN, infinities, signed zeros
    ("normal", 160, 100, 64),            # fewer threads hold elements than k
    ("normal", 160, 500, 500),           # k = n
    ("int20", 155, 65536 // 2, 10),
    ("relu_normal_bf16", 160, 32768, 256),
    ("relu_normal_bf16", 160, 20000, 999),
]


@pytest.mark.parametrize("kind,rows,n,k", ROWS)
@pytest.mark.parametrize("largest", [True, False])
def test_rows_parity(kind, rows, n, k, largest):
    import top_selection_prof_gb300 as tk
    x = workloads.make(kind, rows, n, seed=zlib.crc32(("rows/%s/%d/%d/%d" % (kind, rows, n, k)).encode()) % 1000)
    v, i, st = tk.select_ex(to_device(x), k, largest=largest)
    assert st["path_name"] == "direct", st
    ov, oi = plain.topk(x, k, largest=largest)
    assert_same(v, i, ov, oi, "%s rows=%d n=%d k=%d largest=%s" % (kind, rows, n, k, largest))
