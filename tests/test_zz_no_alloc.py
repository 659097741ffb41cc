"""The allocation-free scheduling entry point gives the same admission as the
workspace one.

dspark_schedule_noalloc serves callers that cannot hand the library device
scratch memory -- a serving loop that must never block on a cudaMalloc, or a
host whose device memory is wholly reserved by another allocator.  Its scratch
is one fixed array inside the library (the status header) that every call
reuses, so this test calls it twice in a row on different pools (the second
call finds the first call's status header and must clear it) and checks each
result against dspark_schedule with a workspace of its own, bit for bit, as the
other scheduling tests do.  It also checks that a pool beyond the entry point's
limit is refused before any launch.
"""
import ctypes

import numpy as np
import pytest

from workloads import sps_table

pytestmark = pytest.mark.gpu


def _pool(B, N, seed):
    rng = np.random.default_rng(seed)
    c = rng.beta(rng.uniform(1, 9), rng.uniform(0.5, 3), size=(B, N)).astype(np.float32)
    c[rng.random((B, N)) < 0.1] = 1.0                      # ties in survival
    return c


def _noalloc(ds, c, sps, K_in):
    import torch
    B, N = c.shape
    dc = torch.from_numpy(c).cuda()
    dsps = torch.from_numpy(sps).cuda() if sps is not None else None
    surv = torch.full((B, N), -1.0, device="cuda")
    K = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    lens = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    sel = torch.full((B * N,), -7, dtype=torch.int32, device="cuda")
    L = ds.lib()
    L.dspark_schedule_noalloc.restype = ctypes.c_int
    L.dspark_schedule_noalloc.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 5
    ptr = lambda t: ctypes.c_void_p(t.data_ptr() if t is not None else 0)
    st = L.dspark_schedule_noalloc(ptr(dc), ptr(dsps), 0 if sps is None else len(sps), B, N, K_in,
                                   ptr(surv), ptr(K), ptr(lens), ptr(sel),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, L.dspark_last_error()
    torch.cuda.synchronize()
    return surv.cpu().numpy(), int(K.item()), lens.cpu().numpy(), sel.cpu().numpy()


def _with_workspace(ds, c, sps, K_in):
    import torch
    surv, K, lens, sel = ds.dspark_schedule(torch.from_numpy(c).cuda(),
                                            torch.from_numpy(sps).cuda() if sps is not None else None,
                                            K_in)
    return surv.cpu().numpy(), int(K.item()), lens.cpu().numpy(), sel.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_twice_in_a_row(cuda_lib):
    ds = cuda_lib
    cases = [(_pool(1024, 16, 1), sps_table(16384), -1),      # the full-size admission pool
             (_pool(37, 5, 2), None, 60)]                      # then a small, fixed-capacity pool
    for c, sps, K_in in cases:
        a = _noalloc(ds, c, sps, K_in)
        b = _with_workspace(ds, c, sps, K_in)
        np.testing.assert_array_equal(a[0], b[0])
        assert a[1] == b[1]
        np.testing.assert_array_equal(a[2], b[2])
        np.testing.assert_array_equal(a[3], b[3])


def test_noalloc_refuses_pools_beyond_its_scratch(cuda_lib):
    import torch
    L = cuda_lib.lib()
    L.dspark_schedule_noalloc.restype = ctypes.c_int
    L.dspark_schedule_noalloc.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 5
    x = torch.zeros(16, device="cuda")
    p = ctypes.c_void_p(x.data_ptr())
    st = L.dspark_schedule_noalloc(p, p, 1, 16385, 1, 5, p, p, p, p, None)
    assert st == 1 and b"16384" in L.dspark_last_error()
