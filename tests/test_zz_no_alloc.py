"""The allocation-free RMSNorm entry point, called through the C ABI.

fuse_rmsnorm_unfused_static() is for callers that cannot allocate device memory where they call
(their memory budget is owned by someone else, or cudaMalloc is not allowed on their path): it
keeps its row statistics in one fixed array owned by the library instead of a caller workspace.
Its output must match the regular entry point, fuse_rmsnorm(..., FUSE_UNFUSED, workspace), within
the RMSNorm tolerance of the other tests (1e-5 relative per element), on two calls in a row with
different shapes, so that nothing left in the shared array by the first call leaks into the
second.  The output is also compared with the CPU oracle directly.  This file is collected
last on purpose.
"""
import ctypes

import numpy as np
import pytest

import epilogue_chains_gb300 as fc
import oracle
from epilogue_chains_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _close(a, b, rtol=1e-5):
    a = a.astype(np.float64)
    b = b.astype(np.float64)
    assert np.all(np.abs(a - b) <= rtol * np.abs(b) + 1e-30)


def _regular(lib, x, w, eps, stream):
    import torch
    rows, hidden = x.shape
    y = torch.empty_like(x)
    nbytes = lib.fuse_rmsnorm_workspace_bytes(rows, hidden, fc.FUSE_UNFUSED)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    rc = lib.fuse_rmsnorm(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, hidden, eps,
                          fc.FUSE_UNFUSED, ws.data_ptr(), nbytes, stream)
    assert rc == fc.FUSE_OK
    return y


def test_static_scratch_matches_workspace_entry_point_twice(cuda_device):
    import torch
    lib = fc._load()
    stream = torch.cuda.current_stream().cuda_stream
    shapes = [(wl.RMS_ROWS, wl.RMS_HIDDEN, 1), (1000, 1536, 2)]   # second call: fewer, narrower rows
    for rows, hidden, salt in shapes:
        xh, wh = wl.rmsnorm_input(rows, hidden, salt=salt)
        x = torch.from_numpy(xh).cuda()
        w = torch.from_numpy(wh).cuda()
        y = torch.full_like(x, float("nan"))
        rc = lib.fuse_rmsnorm_unfused_static(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows,
                                             hidden, ctypes.c_float(wl.RMS_EPS), stream)
        assert rc == fc.FUSE_OK, fc.fuse_strerror(rc)
        ref = _regular(lib, x, w, wl.RMS_EPS, stream)
        torch.cuda.synchronize()
        assert lib.fuse_check(stream) == fc.FUSE_OK
        got = y.cpu().numpy()
        _close(got, ref.cpu().numpy())
        _close(got, oracle.rmsnorm(xh, wh, wl.RMS_EPS))


def test_static_scratch_rejects_rows_beyond_its_size(cuda_device):
    # Every buffer is valid for the full over-limit shape, so a call that got past the size check
    # would return a status or a result, never touch memory outside its buffers.
    import torch
    lib = fc._load()
    rows, hidden = fc.FUSE_RMSNORM_STATIC_MAX_ROWS + 1, 8
    x = torch.ones(rows, hidden, device="cuda")
    w = torch.ones(hidden, device="cuda")
    y = torch.full_like(x, 7.0)
    rc = lib.fuse_rmsnorm_unfused_static(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, hidden,
                                         ctypes.c_float(1e-6), None)
    torch.cuda.synchronize()
    assert rc == fc.FUSE_EUNSUPPORTED
    assert bool(torch.all(y == 7.0))   # nothing was launched
