"""Parity of residual add + RMSNorm (fused one pass, unfused five kernels) against the CPU oracle,
through the C ABI.  h = x + r is one fp32 rounding on both sides: bit-exact.  y accumulates in
fp32 on the GPU and in double in the oracle: 1e-5 relative per element, as RMSNorm."""
import numpy as np
import pytest

import epilogue_chains_gb300 as fc
import oracle
from epilogue_chains_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
MODES = [fc.FUSE_FUSED, fc.FUSE_UNFUSED]


def _close(y, ref, rtol=1e-5):
    err = np.abs(y.astype(np.float64) - ref.astype(np.float64))
    bad = err > rtol * np.abs(ref.astype(np.float64)) + 1e-30
    assert not bad.any(), (int(bad.sum()), float((err / (np.abs(ref) + 1e-30)).max()))


def _run(x, r, w, eps, mode, off=0, inplace=None):
    """inplace: None (separate h), "x" or "r" (h written over that input)."""
    import torch
    rows, H = x.shape
    n = rows * H
    bufs = {k: torch.full((n + 8,), float("nan"), device="cuda") for k in ("x", "r", "h", "y")}
    bufs["x"][off:off + n].copy_(torch.from_numpy(x.reshape(-1)))
    bufs["r"][off:off + n].copy_(torch.from_numpy(r.reshape(-1)))
    v = {k: b[off:off + n].view(rows, H) for k, b in bufs.items()}
    h = v[inplace] if inplace else v["h"]
    fc.fuse_add_rmsnorm(v["x"], v["r"], torch.from_numpy(w).cuda(), h, v["y"], eps, mode)
    torch.cuda.synchronize()
    assert fc.fuse_check() == fc.FUSE_OK
    for k, b in bufs.items():
        guard = torch.cat([b[:off], b[off + n:]]).cpu().numpy()
        assert np.all(np.isnan(guard)), f"write outside {k}"
    return h.cpu().numpy(), v["y"].cpu().numpy()


def _check(x, r, w, eps, mode, **kw):
    h, y = _run(x, r, w, eps, mode, **kw)
    hr, yr = oracle.add_rmsnorm(x, r, w, eps)
    assert np.array_equal(h.view(np.uint32), hr.view(np.uint32))
    _close(y, yr)


@pytest.mark.parametrize("mode", MODES)
def test_full_size(cuda_device, mode):
    """[2048, 4096] as benchmarked, every element."""
    _check(*wl.add_rmsnorm_input(), wl.RMS_EPS, mode)


@pytest.mark.parametrize("shape", [(1, 4), (3, 1024), (7, 4100), (5, 8192), (2, 16384), (3, 24000),
                                   (300, 512), (1000, 64)])
@pytest.mark.parametrize("mode", MODES)
def test_shapes(cuda_device, shape, mode):
    """Row lengths on every register tier (vector and element-wise kernels), many rows per CTA,
    beyond the fused limit (16384 -> unsupported fused, fine unfused)."""
    x, r, w = wl.add_rmsnorm_input(*shape, salt=shape[1])
    if mode == fc.FUSE_FUSED and shape[1] > 16384:
        with pytest.raises(fc.FuseError):
            _run(x, r, w, wl.RMS_EPS, mode)
        return
    _check(x, r, w, wl.RMS_EPS, mode)


@pytest.mark.parametrize("where", ["x", "r"])
@pytest.mark.parametrize("mode", MODES)
def test_in_place_residual(cuda_device, where, mode):
    x, r, w = wl.add_rmsnorm_input(64, 4096, salt=3)
    _check(x, r, w, wl.RMS_EPS, mode, inplace=where)


@pytest.mark.parametrize("off", [1, 2, 3])
@pytest.mark.parametrize("mode", MODES)
def test_misaligned_pointers_use_elementwise_path(cuda_device, off, mode):
    x, r, w = wl.add_rmsnorm_input(9, 1000, salt=4)
    _check(x, r, w, wl.RMS_EPS, mode, off=off)


def test_fused_equals_unfused_h_and_close_y(cuda_device):
    x, r, w = wl.add_rmsnorm_input(128, 4096, salt=5)
    hf, yf = _run(x, r, w, wl.RMS_EPS, fc.FUSE_FUSED)
    hu, yu = _run(x, r, w, wl.RMS_EPS, fc.FUSE_UNFUSED)
    assert np.array_equal(hf.view(np.uint32), hu.view(np.uint32))
    _close(yf, yu, 2e-5)


def test_rejects_aliasing_and_missing_workspace(cuda_device):
    import torch
    x = torch.zeros(4, 64, device="cuda")
    r, w, h, y = torch.zeros_like(x), torch.ones(64, device="cuda"), torch.zeros_like(x), torch.zeros_like(x)
    with pytest.raises(fc.FuseError):
        fc.fuse_add_rmsnorm(x, r, w, h, h, 1e-6)          # y == h
    with pytest.raises(fc.FuseError):
        fc.fuse_add_rmsnorm(x, r, w, h, x, 1e-6)          # y == x
    lib = fc._load()
    assert lib.fuse_add_rmsnorm(x.data_ptr(), r.data_ptr(), w.data_ptr(), h.data_ptr(), y.data_ptr(),
                                4, 64, 1e-6, fc.FUSE_UNFUSED, None, 0, None) == fc.FUSE_EWORKSPACE
