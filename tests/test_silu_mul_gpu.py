"""Parity of SiLU(gate) * up (fused one kernel, unfused two kernels) against the CPU oracle,
through the C ABI.

The GPU evaluates SiLU in fp32 with the special-function unit's exp2 and reciprocal (relative
error about 2^-21 before the final rounding); the oracle in double, rounding once (fused) or at
the stored SiLU tensor too (unfused).  Bars: bf16/fp16 storage within 1 ulp of the oracle fused
(2 ulps unfused: the stored SiLU can round one ulp apart and the product carries it), with
off-by-one elements rare (< 2 %); fp32 within 4e-6 relative."""
import numpy as np
import pytest

import epilogue_chains_gb300 as fc
import oracle
from epilogue_chains_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
TDT = {"f32": "float32", "f16": "float16", "bf16": "bfloat16"}


def _dev(a, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16 if dtype != "f32" else np.float32)).cuda()
    return t if dtype == "f32" else t.view(getattr(torch, TDT[dtype]))


def _host(t, dtype):
    import torch
    c = t.cpu()
    return c.numpy() if dtype == "f32" else c.view(torch.int16).numpy().view(np.uint16)


def _ulps(a, b, dtype):
    """Distance in representable steps between two arrays of uint16 patterns (same-sign aware)."""
    def key(v):
        v = v.astype(np.int32)
        return np.where(v & 0x8000, -(v & 0x7FFF), v)
    return np.abs(key(a) - key(b))


def _compare(y, ref, dtype, ulps):
    if dtype == "f32":
        err = np.abs(y.astype(np.float64) - ref.astype(np.float64))
        assert np.all(err <= 4e-6 * np.abs(ref.astype(np.float64)) + 1e-37), float(err.max())
        return
    d = _ulps(y, ref, dtype)
    assert d.max() <= ulps, int(d.max())
    assert np.count_nonzero(d) <= 0.02 * d.size + 1, int(np.count_nonzero(d))


def _run_merged(gu_host, dtype, mode, y_off=0):
    import torch
    rows, ld = gu_host.shape
    cols = ld // 2
    gu = _dev(gu_host, dtype)
    ybuf = torch.full((rows * cols + 16,), float("nan"), dtype=gu.dtype, device="cuda")
    y = ybuf[y_off:y_off + rows * cols].view(rows, cols)
    fc.fuse_silu_mul(gu[:, :cols], gu[:, cols:], y, mode)
    torch.cuda.synchronize()
    assert fc.fuse_check() == fc.FUSE_OK
    guard = torch.cat([ybuf[:y_off], ybuf[y_off + rows * cols:]]).float().cpu().numpy()
    assert np.all(np.isnan(guard)), "write outside y"
    return _host(y, dtype)


@pytest.mark.parametrize("mode", [fc.FUSE_FUSED, fc.FUSE_UNFUSED])
def test_full_size_bf16(cuda_device, mode):
    """[2048, 14336] bf16 from one merged gate/up tensor, as benchmarked, every element."""
    gu = wl.silu_input()
    y = _run_merged(gu, "bf16", mode)
    _compare(y, oracle.silu_mul_merged(gu, "bf16", unfused=mode == fc.FUSE_UNFUSED), "bf16",
             1 if mode == fc.FUSE_FUSED else 2)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shape", [(1, 16), (3, 48), (17, 1000), (64, 4096), (5, 7)])
@pytest.mark.parametrize("mode", [fc.FUSE_FUSED, fc.FUSE_UNFUSED])
def test_shapes_and_types(cuda_device, dtype, shape, mode):
    """Vector path (cols a multiple of 32 bytes) and element-wise path (ragged cols)."""
    gu = wl.silu_input(*shape, dtype=dtype, salt=shape[1], scale=3.0)
    y = _run_merged(gu, dtype, mode)
    _compare(y, oracle.silu_mul_merged(gu, dtype, unfused=mode == fc.FUSE_UNFUSED), dtype,
             1 if mode == fc.FUSE_FUSED else 2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_separate_dense_tensors_and_misaligned_output(cuda_device, dtype):
    import torch
    gu = wl.silu_input(33, 512, dtype=dtype, salt=9, scale=4.0)
    g, u = np.ascontiguousarray(gu[:, :512]), np.ascontiguousarray(gu[:, 512:])
    gd, ud = _dev(g, dtype), _dev(u, dtype)
    y = torch.empty_like(gd)
    fc.fuse_silu_mul(gd, ud, y)
    torch.cuda.synchronize()
    _compare(_host(y, dtype), oracle.silu_mul(g, u, dtype), dtype, 1)
    # output one element off a 32-byte boundary: element-wise kernel
    assert np.array_equal(_run_merged(gu, dtype, fc.FUSE_FUSED, y_off=1),
                          _run_merged(gu, dtype, fc.FUSE_FUSED))


def test_tails_of_silu(cuda_device):
    """Far negative gates give -0 / tiny values, far positive gates pass through (SiLU(v) -> v),
    zero gives zero; up = 1."""
    vals = np.array([-120.0, -90.0, -40.0, -20.0, -8.0, -1e-3, 0.0, 1e-3, 8.0, 20.0, 40.0, 90.0,
                     -3.0, 3.0, -0.5, 0.5], np.float32)
    g = np.tile(vals, (2, 2))
    u = np.ones_like(g)
    import torch
    gd, ud = _dev(g, "f32"), _dev(u, "f32")
    y = torch.empty_like(gd)
    fc.fuse_silu_mul(gd, ud, y)
    torch.cuda.synchronize()
    ref = oracle.silu_mul(g, u, "f32")
    yy = y.cpu().numpy()
    assert np.all(np.abs(yy - ref) <= 4e-6 * np.abs(ref) + 1e-37), np.max(np.abs(yy - ref))
    assert np.all(yy[g >= 20] == g[g >= 20])


def test_in_place_over_dense_gate(cuda_device):
    import torch
    gu = wl.silu_input(16, 256, dtype="bf16", salt=10)
    g, u = np.ascontiguousarray(gu[:, :256]), np.ascontiguousarray(gu[:, 256:])
    for mode in (fc.FUSE_FUSED, fc.FUSE_UNFUSED):
        gd, ud = _dev(g, "bf16"), _dev(u, "bf16")
        fc.fuse_silu_mul(gd, ud, gd, mode)
        torch.cuda.synchronize()
        _compare(_host(gd, "bf16"), oracle.silu_mul(g, u, "bf16", unfused=mode == fc.FUSE_UNFUSED),
                 "bf16", 1 if mode == fc.FUSE_FUSED else 2)


def test_rejects_overlap_with_up(cuda_device):
    import torch
    gu = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    lib = fc._load()
    g, u = gu.data_ptr(), gu.data_ptr() + 64
    assert lib.fuse_silu_mul(g, u, 64, u, 4, 32, fc.FUSE_BF16, fc.FUSE_FUSED,
                             None) == fc.FUSE_EINVAL                                 # y over up
    assert lib.fuse_silu_mul(g, u, 64, g, 4, 32, fc.FUSE_BF16, fc.FUSE_FUSED,
                             None) == fc.FUSE_EINVAL                                 # y over strided gate
    assert lib.fuse_silu_mul(gu.data_ptr(), gu.data_ptr() + 64, 16, gu.data_ptr() + 4096, 4, 32,
                             fc.FUSE_BF16, fc.FUSE_FUSED, None) == fc.FUSE_EINVAL   # ld < cols
