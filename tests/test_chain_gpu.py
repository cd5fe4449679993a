"""Parity of the pointwise chain (fused / unfused / fat) against the CPU oracle, through the C ABI.

The chain rounds twice per stage in fp32 on both sides, so the bar is bit-exact.  The 8-stage
affine chain is also checked against the closed form A^K x + B (A^K - 1)/(A - 1) at the pages'
own metric, max|d|/max|ref| <= 1e-6.
"""
import numpy as np
import pytest

import epilogue_chains_gb300 as fc
import oracle
from epilogue_chains_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MODES = [fc.FUSE_FUSED, fc.FUSE_UNFUSED, fc.FUSE_FAT]


def _stages(relu, a, b):
    return [(fc.FUSE_OP_AFFINE_RELU if r else fc.FUSE_OP_AFFINE, float(x), float(y))
            for r, x, y in zip(relu, a, b)]


def _run(stages, x_host, mode, dtype="f32", x_off=0, y_off=0):
    import torch
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    n = x_host.size
    xb = torch.empty(n + 8, dtype=tdt, device="cuda")
    yb = torch.full((n + 8,), float("nan"), dtype=tdt, device="cuda")
    xh = torch.from_numpy(x_host.view(np.int16) if dtype != "f32" else x_host)
    xb[x_off:x_off + n].copy_(xh.view(tdt) if dtype != "f32" else xh)
    fc.fuse_chain_run(stages, xb[x_off:x_off + n], yb[y_off:y_off + n], mode)
    torch.cuda.synchronize()
    assert fc.fuse_check() == fc.FUSE_OK
    out = yb[y_off:y_off + n].cpu()
    guard = torch.cat([yb[:y_off], yb[y_off + n:]]).float().cpu().numpy()
    assert np.all(np.isnan(guard)), "write outside y"
    return out.numpy() if dtype == "f32" else out.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("mode", MODES)
def test_affine_chain_config0(cuda_device, mode):
    relu, a, b, x = wl.affine_chain()
    y = _run(_stages(relu, a, b), x, mode)
    ref = oracle.chain(relu, a, b, x)
    assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))
    cf = oracle.affine_closed_form(x, wl.AFFINE_K, wl.AFFINE_A, wl.AFFINE_B)
    assert np.max(np.abs(y - cf)) / np.max(np.abs(cf)) <= 1e-6


@pytest.mark.parametrize("K", wl.CHAIN_KS)
@pytest.mark.parametrize("mode", MODES)
def test_pointwise_chain_ragged(cuda_device, K, mode):
    relu, a, b = wl.chain_stages(K)
    x = wl.chain_input(3 * 65536 + 13, salt=K)          # several waves and a ragged tail
    y = _run(_stages(relu, a, b), x, mode)
    assert np.array_equal(y.view(np.uint32), oracle.chain(relu, a, b, x).view(np.uint32))


@pytest.mark.parametrize("K", wl.CHAIN_KS)
def test_pointwise_chain_full_size_all_modes(cuda_device, K):
    """N = 16,777,216 as benchmarked, every mode, every element against the oracle."""
    import torch
    relu, a, b = wl.chain_stages(K)
    x = wl.chain_input(wl.CHAIN_N, device="cuda", salt=K)
    ref = oracle.chain(relu, a, b, x.cpu().numpy())
    for mode in MODES:
        y = torch.empty_like(x)
        fc.fuse_chain_run(_stages(relu, a, b), x, y, mode)
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy().view(np.uint32), ref.view(np.uint32)), mode


@pytest.mark.parametrize("n", [1, 3, 4, 5, 7, 8, 255, 4097])
@pytest.mark.parametrize("mode", MODES)
def test_small_and_odd_sizes(cuda_device, n, mode):
    relu, a, b = wl.chain_stages(6)
    x = wl.chain_input(n, salt=100 + n)
    y = _run(_stages(relu, a, b), x, mode)
    assert np.array_equal(y.view(np.uint32), oracle.chain(relu, a, b, x).view(np.uint32))


@pytest.mark.parametrize("offs", [(1, 1), (3, 3), (1, 2), (0, 3), (2, 0)])
@pytest.mark.parametrize("mode", MODES)
def test_misaligned_pointers(cuda_device, offs, mode):
    """Shared misalignment uses a scalar head; mismatched alignment the element-wise path."""
    relu, a, b = wl.chain_stages(4)
    x = wl.chain_input(10007, salt=7)
    y = _run(_stages(relu, a, b), x, mode, x_off=offs[0], y_off=offs[1])
    assert np.array_equal(y.view(np.uint32), oracle.chain(relu, a, b, x).view(np.uint32))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("mode", MODES)
def test_half_storage_types(cuda_device, dtype, mode):
    relu, a, b = wl.chain_stages(8)
    x32 = wl.chain_input(70001, salt=9)
    xs = x32.astype(np.float16).view(np.uint16) if dtype == "f16" else wl.bf16_bits_from_f32(x32)
    y = _run(_stages(relu, a, b), xs, mode, dtype=dtype)
    if mode == fc.FUSE_UNFUSED:
        # every stage stores its output in the storage type: the oracle applied stage by stage
        ref = xs
        for s in range(len(a)):
            ref = oracle.chain(relu[s:s + 1], a[s:s + 1], b[s:s + 1], ref, dtype)
    else:
        ref = oracle.chain(relu, a, b, xs, dtype)
    assert np.array_equal(y, ref)


@pytest.mark.parametrize("K", [1, 32])
def test_stage_count_limits(cuda_device, K):
    g = np.random.default_rng(K)
    relu = np.arange(K) % 2 == 0
    a = g.uniform(0.95, 1.05, K).astype(np.float32)
    b = g.uniform(-0.05, 0.05, K).astype(np.float32)
    x = wl.chain_input(5000, salt=K)
    for mode in MODES:
        y = _run(_stages(relu, a, b), x, mode)
        assert np.array_equal(y.view(np.uint32), oracle.chain(relu, a, b, x).view(np.uint32))


def test_in_place(cuda_device):
    import torch
    relu, a, b = wl.chain_stages(8)
    x = wl.chain_input(123457, salt=11)
    ref = oracle.chain(relu, a, b, x)
    for mode in MODES:
        t = torch.from_numpy(x.copy()).cuda()
        fc.fuse_chain_run(_stages(relu, a, b), t, t, mode)
        torch.cuda.synchronize()
        assert np.array_equal(t.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_partial_overlap_rejected(cuda_device):
    import torch
    t = torch.zeros(1000, device="cuda")
    with pytest.raises(fc.FuseError):
        fc.fuse_chain_run([(0, 1.0, 0.0)], t[:900], t[10:910])


def test_fat_probe_register_report(cuda_device):
    """[C05] §6.2: the thin fused kernel keeps occupancy, the fat one collapses it."""
    recs = [fc.fuse_kernel_report(i) for i in range(fc.fuse_kernel_count())]
    fused = next(r for r in recs if r["name"].startswith("chain_fused_kernel<f32>"))
    fat = next(r for r in recs if r["name"].startswith("chain_fat_kernel<f32>"))
    assert fat["regs_per_thread"] >= 192          # 4 elements x 48 temporaries stay live
    assert fat["blocks_per_sm"] == 1
    assert fused["blocks_per_sm"] >= 6
    assert fused["local_bytes_per_thread"] == 0


@pytest.mark.parametrize("n,slices,pinned,mode", [(1, 1, True, fc.FUSE_FUSED), (100_003, 3, True, fc.FUSE_FUSED),
                                                  (1 << 20, 8, True, fc.FUSE_UNFUSED),
                                                  (65_537, 64, False, fc.FUSE_FUSED),
                                                  (4096, 5, True, fc.FUSE_FAT)])
def test_host_buffer_entry_point(cuda_device, n, slices, pinned, mode):
    """fuse_chain_run_host: x from host memory, y back to host memory, through the caller's
    device scratch, in slices whose copies overlap the kernels: bit-exact with the oracle (the
    chain is element-wise, so slicing changes nothing), for pinned and pageable host memory."""
    import torch
    relu, a, b = wl.chain_stages(6)
    st = _stages(relu, a, b)
    x = wl.chain_input(n, salt=21)
    xh = torch.from_numpy(x)
    yh = torch.full((n,), float("nan"))
    if pinned:
        xh, yh = xh.pin_memory(), yh.pin_memory()
    xd = torch.empty(n, device="cuda")
    yd = torch.empty(n, device="cuda")
    s = torch.cuda.Stream()
    fc.fuse_chain_run_host(st, xh, yh, xd, yd, mode, slices, stream=s)
    s.synchronize()
    assert fc.fuse_check() == fc.FUSE_OK
    assert np.array_equal(yh.numpy().view(np.uint32), oracle.chain(relu, a, b, x).view(np.uint32))


def test_host_buffer_entry_point_is_stream_ordered_and_in_place(cuda_device):
    """Work queued on the stream before the call (a kernel writing the host-visible input through
    a device copy) is finished before the copies start; x_dev may be y_dev; two calls in a row on
    one stream give the chain applied twice."""
    import torch
    relu, a, b = wl.chain_stages(3)
    st = _stages(relu, a, b)
    n = 300_001
    x = wl.chain_input(n, salt=22)
    xh = torch.from_numpy(x).pin_memory()
    mid = torch.empty(n).pin_memory()
    out = torch.empty(n).pin_memory()
    buf = torch.empty(n, device="cuda")
    s = torch.cuda.Stream()
    fc.fuse_chain_run_host(st, xh, mid, buf, buf, fc.FUSE_FUSED, 4, stream=s)
    fc.fuse_chain_run_host(st, mid, out, buf, buf, fc.FUSE_FUSED, 7, stream=s)
    s.synchronize()
    once = oracle.chain(relu, a, b, x)
    assert np.array_equal(mid.numpy().view(np.uint32), once.view(np.uint32))
    assert np.array_equal(out.numpy().view(np.uint32), oracle.chain(relu, a, b, once).view(np.uint32))
    lib = fc._load()
    arr = fc._stages(st)
    assert lib.fuse_chain_run_host(arr, 3, xh.data_ptr(), out.data_ptr(), n, fc.FUSE_F32, fc.FUSE_FUSED,
                                   buf.data_ptr(), buf.data_ptr(), 0, s.cuda_stream) == fc.FUSE_EINVAL
    assert lib.fuse_chain_run_host(arr, 3, xh.data_ptr(), out.data_ptr(), n, fc.FUSE_F32, fc.FUSE_FUSED,
                                   buf.data_ptr(), buf.data_ptr() + 4, 2, s.cuda_stream) == fc.FUSE_EINVAL
    assert lib.fuse_chain_run_host(arr, 3, None, out.data_ptr(), n, fc.FUSE_F32, fc.FUSE_FUSED,
                                   buf.data_ptr(), buf.data_ptr(), 2, s.cuda_stream) == fc.FUSE_EINVAL
