"""topk_select_noalloc against the pooled entry points and the oracle (collected last on purpose).

topk_select_noalloc serves callers that cannot allocate device memory while
they run (their memory belongs to another allocator, or cudaMalloc's implicit
synchronisation is not allowed in their loop).  It takes all scratch from a
static 8 MiB device array inside the library and runs the pooled entry
points' pipeline on it.  These tests call it through the C ABI and require
its results to equal those of topk_select / topk_select_global and of the CPU
oracle bit for bit (the tolerance every selection test uses, 0), on two calls
in a row, so stale contents of the shared array would show.
"""
import ctypes

import numpy as np
import pytest

from oracle import plain
from top_selection_prof_gb300 import workloads

from .gpu_util import bits, oracle_bits, to_device

pytestmark = pytest.mark.gpu

NOALLOC_BYTES = 8 << 20


def _lib():
    from top_selection_prof_gb300 import _lib as L
    lib = L.get()
    f = lib.topk_select_noalloc
    vp = ctypes.c_void_p
    f.argtypes = [vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_double, vp, vp, ctypes.c_int, vp]
    f.restype = ctypes.c_int
    return lib, L


def _run(fn_name, x, k, eps, global_, largest, lib, L):
    import torch
    rows, n = x.shape
    shape = (k,) if global_ else (rows, k)
    vals = torch.empty(shape, dtype=x.dtype, device=x.device)
    idx = torch.empty(shape, dtype=torch.int64, device=x.device)
    code = L.TOPK_BF16 if x.dtype == torch.bfloat16 else L.TOPK_F32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if fn_name == "noalloc":
        rc = lib.topk_select_noalloc(x.data_ptr(), code, rows, n, k, int(largest), eps, vals.data_ptr(),
                                     idx.data_ptr(), int(global_), stream)
    else:
        fn = lib.topk_select_global if global_ else lib.topk_select
        rc = fn(x.data_ptr(), code, rows, n, k, int(largest), eps, vals.data_ptr(), idx.data_ptr(), stream)
    torch.cuda.synchronize()
    assert rc == 0, (fn_name, rc)
    assert lib.topk_last_status(stream) == 0, fn_name
    return bits(vals), idx.cpu().numpy()


CASES = [
    ("pareto15", 1, 1 << 22, 1024, 1e-6, False),          # Prof-K, f32 single row
    ("relu_normal_bf16", 256, 65536, 8192, 1e-3, True),   # Prof-K, bf16 batch-global, grid refinement
    ("normal", 1, 1 << 22, 65536, 1e-3, False),           # f32 single row, large k: grid refinement + bin sort
    ("normal", 64, 32768, 64, 1e-3, False),               # direct per-row path
    ("ties1000", 1, 1 << 23, 5000, 0.0, False),           # grid-wide exact path (eps = 0)
]


@pytest.mark.parametrize("largest", [True, False])
@pytest.mark.parametrize("kind,rows,n,k,eps,global_", CASES)
def test_noalloc_matches_the_pooled_entry_point_and_the_oracle_twice(kind, rows, n, k, eps, global_, largest):
    lib, L = _lib()
    for call, seed in enumerate((11, 12)):      # two calls in a row, different inputs
        xh = workloads.make(kind, rows, n, seed)
        x = to_device(xh)
        v_ref, i_ref = _run("pooled", x, k, eps, global_, largest, lib, L)
        v_na, i_na = _run("noalloc", x, k, eps, global_, largest, lib, L)
        assert np.array_equal(i_na, i_ref), "call %d: indices differ from topk_select" % call
        assert np.array_equal(v_na, v_ref), "call %d: values differ from topk_select" % call
        ov, oi = plain.topk(xh, k, largest=largest, global_=global_)
        assert np.array_equal(i_na, oi), "call %d: indices differ from the oracle" % call
        assert np.array_equal(v_na, oracle_bits(ov)), "call %d: values differ from the oracle" % call


@pytest.mark.slow
@pytest.mark.parametrize("largest", [True, False])
def test_noalloc_batchtopk_full_size(largest):
    """The 4096 x 65536 bf16 BatchTopK selection (K = 131072) fits the array."""
    lib, L = _lib()
    xh = workloads.make("relu_normal_bf16", 4096, 65536, 5)
    x = to_device(xh)
    for _ in range(2):
        v_na, i_na = _run("noalloc", x, 131072, 1e-3, True, largest, lib, L)
    del x
    ov, oi = plain.topk(xh, 131072, largest=largest, global_=True)
    assert np.array_equal(i_na, oi)
    assert np.array_equal(v_na, oracle_bits(ov))


def test_noalloc_rejects_requests_beyond_its_scratch():
    import torch
    from oracle import params
    lib, L = _lib()
    rows, n, k, eps = 32, 1 << 20, 2000, 1e-3
    s, t, m = params.exact(n, k, eps)
    assert rows * (s + m) * 8 > NOALLOC_BYTES            # per-row samples + buffers alone exceed it
    x = torch.zeros((rows, n), dtype=torch.float32, device="cuda")
    vals = torch.empty((rows, k), dtype=torch.float32, device="cuda")
    idx = torch.empty((rows, k), dtype=torch.int64, device="cuda")
    rc = lib.topk_select_noalloc(x.data_ptr(), L.TOPK_F32, rows, n, k, 1, eps, vals.data_ptr(), idx.data_ptr(),
                                 0, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == L.TOPK_EUNSUPPORTED
