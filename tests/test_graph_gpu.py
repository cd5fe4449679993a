"""CUDA-graph capture of the library's calls ("AIGC fundamentals | operator fusion and CUDA Graph"
§3.4, §6.4): a captured plan launches the same kernels as the eager call, so its replay must give
the oracle's result bit for bit where the eager call does, and the capture itself runs nothing."""
import numpy as np
import pytest

import epilogue_chains_gb300 as fc
import oracle
from epilogue_chains_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _stages(relu, a, b):
    return [(fc.FUSE_OP_AFFINE_RELU if r else fc.FUSE_OP_AFFINE, float(x), float(y))
            for r, x, y in zip(relu, a, b)]


def _capture(stream, issue):
    import torch
    with torch.cuda.stream(stream):
        fc.fuse_graph_begin(stream)
        try:
            issue()
        finally:
            g = fc.fuse_graph_end(stream)
    return g


def _replay(g, stream):
    import torch
    fc.fuse_graph_launch(g, stream)
    stream.synchronize()
    assert fc.fuse_check(stream) == fc.FUSE_OK
    torch.cuda.synchronize()


@pytest.mark.parametrize("mode,kernels", [(fc.FUSE_UNFUSED, 8), (fc.FUSE_FUSED, 1)])
def test_affine_chain_graph_replays_bit_exact(cuda_device, mode, kernels):
    """The 8-stage affine chain on 4096 elements: capture once, replay on three inputs written in
    place into the captured buffer."""
    import torch
    relu, a, b, x0 = wl.affine_chain()
    st = _stages(relu, a, b)
    s = torch.cuda.Stream()
    x = torch.from_numpy(x0).cuda()
    y = torch.full_like(x, float("nan"))
    torch.cuda.synchronize()
    g = _capture(s, lambda: fc.fuse_chain_run(st, x, y, mode, stream=s))
    try:
        assert fc.fuse_graph_kernel_count(g) == kernels
        assert torch.isnan(y).all(), "capturing must not run the kernels"
        for salt in range(3):
            xh = x0 if salt == 0 else wl.chain_input(x0.size, salt=50 + salt)
            x.copy_(torch.from_numpy(xh))
            torch.cuda.synchronize()
            _replay(g, s)
            ref = oracle.chain(relu, a, b, xh)
            assert np.array_equal(y.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    finally:
        fc.fuse_graph_destroy(g)


@pytest.mark.parametrize("K", [2, 8])
def test_pointwise_chain_graph_ragged(cuda_device, K):
    import torch
    relu, a, b = wl.chain_stages(K)
    xh = wl.chain_input(65536 * 3 + 5, salt=60 + K)
    s = torch.cuda.Stream()
    x = torch.from_numpy(xh).cuda()
    y = torch.full_like(x, float("nan"))
    torch.cuda.synchronize()
    g = _capture(s, lambda: fc.fuse_chain_run(_stages(relu, a, b), x, y, fc.FUSE_UNFUSED, stream=s))
    try:
        assert fc.fuse_graph_kernel_count(g) == K
        _replay(g, s)
        assert np.array_equal(y.cpu().numpy().view(np.uint32),
                              oracle.chain(relu, a, b, xh).view(np.uint32))
    finally:
        fc.fuse_graph_destroy(g)


@pytest.mark.parametrize("plan,mask,kernels", [("[1,1,1,1]", 7, 4), ("[2,2]", 2, 2), ("[4]", 0, 1)])
def test_decode_gemm_plan_graph(cuda_device, plan, mask, kernels):
    """M = 16, N = K = 4096, the launch-bound decode shape, every element against the oracle at
    the tolerance of the eager parity test (the replay runs the same kernels, so it must also equal
    the eager result exactly)."""
    import torch
    A, B, bias, R = wl.gemm_input(16)
    dev = [torch.from_numpy(np.ascontiguousarray(t).view(np.int16)).cuda().view(torch.float16)
           for t in (A, B, bias, R)]
    Ye = torch.empty(16, 4096, dtype=torch.float16, device="cuda")
    fc.fuse_gemm_epilogue(*dev, Ye, cut_mask=mask)
    Yg = torch.full((16, 4096), float("nan"), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = _capture(s, lambda: fc.fuse_gemm_epilogue(*dev, Yg, cut_mask=mask, stream=s))
    try:
        assert fc.fuse_graph_kernel_count(g) == kernels
        for _ in range(2):
            _replay(g, s)
        assert torch.equal(Ye.view(torch.int16), Yg.view(torch.int16))
    finally:
        fc.fuse_graph_destroy(g)
    ref = oracle.gemm_epilogue(A, B, bias, R, mask).view(np.float16).astype(np.float64)
    y = Yg.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(y - ref) <= 2e-2 * (np.abs(ref) + np.sqrt(np.mean(ref ** 2))))


def test_rmsnorm_and_softmax_unfused_graphs(cuda_device):
    import torch
    x_h, w_h = wl.rmsnorm_input(rows=64, hidden=4096, salt=3)
    x, w = torch.from_numpy(x_h).cuda(), torch.from_numpy(w_h).cuda()
    y = torch.full_like(x, float("nan"))
    ws = torch.empty(fc.fuse_rmsnorm_workspace_bytes(64, 4096, fc.FUSE_UNFUSED), dtype=torch.uint8,
                     device="cuda")
    sb = wl.softmax_input(2, 256, salt=4)
    sm = torch.from_numpy(sb.view(np.int16)).cuda().view(torch.bfloat16)
    p = torch.full_like(sm, float("nan"))
    sws = torch.empty(fc.fuse_causal_softmax_workspace_bytes(2, 256, fc.FUSE_UNFUSED),
                      dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()

    def issue():
        fc.fuse_rmsnorm(x, w, y, wl.RMS_EPS, fc.FUSE_UNFUSED, workspace=ws, stream=s)
        fc.fuse_causal_softmax(sm, p, wl.SM_SCALE, 0, fc.FUSE_UNFUSED, workspace=sws, stream=s)
    g = _capture(s, issue)
    try:
        assert fc.fuse_graph_kernel_count(g) == 4 + 5
        _replay(g, s)
    finally:
        fc.fuse_graph_destroy(g)
    ref = oracle.rmsnorm(x_h, w_h, wl.RMS_EPS)
    yy = y.cpu().numpy()
    assert np.all(np.abs(yy - ref) <= 1e-5 * np.abs(ref) + 1e-30)
    pref = oracle.causal_softmax(sb, wl.SM_SCALE, unfused=True)
    pp = p.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.abs(pp.astype(np.int32) - pref.astype(np.int32)).max() <= 2


def test_graph_argument_errors(cuda_device):
    import torch
    lib = fc._load()
    assert lib.fuse_graph_begin(None) == fc.FUSE_EINVAL          # legacy stream: not capturable
    assert lib.fuse_graph_launch(None, None) == fc.FUSE_EINVAL
    assert lib.fuse_graph_kernel_count(None) == fc.FUSE_EINVAL
    lib.fuse_graph_destroy(None)
    s = torch.cuda.Stream()
    with pytest.raises(fc.FuseError):                             # no capture in progress
        fc.fuse_graph_end(s)
    g = _capture(s, lambda: None)                                 # an empty capture is valid
    assert fc.fuse_graph_kernel_count(g) == 0
    fc.fuse_graph_launch(g, s)
    s.synchronize()
    fc.fuse_graph_destroy(g)
