"""Parity of RMSNorm (fused / four-kernel unfused) against the CPU oracle through the C ABI.

Bar: per element |y - ref| <= 1e-5 |ref| + 1e-30 (fp32 accumulation on the GPU, double in the
oracle; y is a row scalar times x times w, so the error is relative per element)."""
import numpy as np
import pytest

import epilogue_chains_gb300 as fc
import oracle
from epilogue_chains_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _close(y, ref, rtol=1e-5):
    err = np.abs(y.astype(np.float64) - ref.astype(np.float64))
    bad = err > rtol * np.abs(ref.astype(np.float64)) + 1e-30
    assert not bad.any(), (int(bad.sum()), float((err / (np.abs(ref) + 1e-30)).max()))


def _run(x, w, eps, mode, x_off=0, y_off=0):
    import torch
    rows, H = x.shape
    xb = torch.empty(rows * H + 8, device="cuda")
    yb = torch.full((rows * H + 8,), float("nan"), device="cuda")
    xb[x_off:x_off + rows * H].copy_(torch.from_numpy(x.reshape(-1)))
    xt = xb[x_off:x_off + rows * H].view(rows, H)
    yt = yb[y_off:y_off + rows * H].view(rows, H)
    fc.fuse_rmsnorm(xt, torch.from_numpy(w).cuda(), yt, eps, mode)
    torch.cuda.synchronize()
    assert fc.fuse_check() == fc.FUSE_OK
    guard = torch.cat([yb[:y_off], yb[y_off + rows * H:]]).cpu().numpy()
    assert np.all(np.isnan(guard))
    return yt.cpu().numpy()


@pytest.mark.parametrize("mode", [fc.FUSE_FUSED, fc.FUSE_UNFUSED])
def test_full_size(cuda_device, mode):
    x, w = wl.rmsnorm_input()
    _close(_run(x, w, wl.RMS_EPS, mode), oracle.rmsnorm(x, w, wl.RMS_EPS))


@pytest.mark.parametrize("shape", [(1, 1), (3, 3), (5, 4), (7, 64), (2, 4097), (4, 12288),
                                   (3, 16384), (1, 1000), (33, 508), (2, 513)])
@pytest.mark.parametrize("mode", [fc.FUSE_FUSED, fc.FUSE_UNFUSED])
def test_shapes(cuda_device, shape, mode):
    x, w = wl.rmsnorm_input(*shape, salt=shape[1])
    _close(_run(x, w, 1e-6, mode), oracle.rmsnorm(x, w, 1e-6))


@pytest.mark.parametrize("offs", [(1, 1), (0, 2)])
def test_misaligned_rows_use_elementwise_path(cuda_device, offs):
    x, w = wl.rmsnorm_input(6, 4096, salt=3)
    for mode in (fc.FUSE_FUSED, fc.FUSE_UNFUSED):
        _close(_run(x, w, 1e-6, mode, *offs), oracle.rmsnorm(x, w, 1e-6))


def test_unfused_wide_rows(cuda_device):
    x, w = wl.rmsnorm_input(3, 65536, salt=4)
    _close(_run(x, w, 1e-6, fc.FUSE_UNFUSED), oracle.rmsnorm(x, w, 1e-6))


def test_large_eps_and_zero_rows(cuda_device):
    x, w = wl.rmsnorm_input(8, 256, salt=5)
    x[3] = 0.0
    for mode in (fc.FUSE_FUSED, fc.FUSE_UNFUSED):
        y = _run(x, w, 0.5, mode)
        _close(y, oracle.rmsnorm(x, w, 0.5))
        assert np.all(y[3] == 0)


def test_fused_matches_unfused(cuda_device):
    x, w = wl.rmsnorm_input(64, 4096, salt=6)
    _close(_run(x, w, 1e-6, fc.FUSE_FUSED), _run(x, w, 1e-6, fc.FUSE_UNFUSED))
