"""Seeded random sweeps of every entry point against the CPU oracle, through the C ABI.

The targeted tests fix their sizes by hand; here each call draws its arguments (sizes, pointer
offsets, dtypes, stage counts, skip tiles, cut masks, scales) from a seeded generator, so the
combinations between the hand-picked cases are exercised too.  Every case uses the same bar as
its row's own test: bit-exact for the pointwise chain (stage by stage in the storage type for
the unfused 16-bit form, which stores every intermediate) and the residual sum, 1e-5 relative for
RMSNorm, <= 1 bf16 ulp (fused) / 2 ulps (unfused, four-rounding oracle) for the causal softmax,
the fp16 error model of the GEMM test, 1-2 storage ulps for SiLU*up, and the bf16 bound of the
attention test."""
import numpy as np
import pytest

import epilogue_chains_gb300 as fc
import oracle
from epilogue_chains_gb300 import workloads as wl

import test_add_rmsnorm_gpu as T_add
import test_attention_gpu as T_att
import test_chain_gpu as T_chain
import test_gemm_gpu as T_gemm
import test_rmsnorm_gpu as T_rms
import test_silu_mul_gpu as T_silu
import test_softmax_gpu as T_sm

pytestmark = pytest.mark.gpu
SEED = wl.RNG_SEED + 9000


def _rng(case, row):
    return np.random.default_rng([SEED, row, case])


def _log_uniform(g, lo, hi):
    return int(round(np.exp(g.uniform(np.log(lo), np.log(hi)))))


@pytest.mark.parametrize("case", range(48))
def test_chain(cuda_device, case):
    g = _rng(case, 1)
    dtype = ["f32", "f16", "bf16"][case % 3]
    mode = [fc.FUSE_FUSED, fc.FUSE_UNFUSED, fc.FUSE_FAT][(case // 3) % 3]
    n = _log_uniform(g, 1, 1 << 21)
    K = int(g.integers(1, 33))
    relu = g.integers(0, 2, K).astype(np.int32)
    a = g.uniform(0.9, 1.1, K).astype(np.float32)
    b = g.uniform(-0.1, 0.1, K).astype(np.float32)
    x = g.standard_normal(n).astype(np.float32)
    if dtype == "bf16":
        x = wl.bf16_bits_from_f32(x)
    elif dtype == "f16":
        x = wl.f16_bits_from_f64(x.astype(np.float64))
    y = T_chain._run(T_chain._stages(relu, a, b), x, mode, dtype,
                     x_off=int(g.integers(0, 8)), y_off=int(g.integers(0, 8)))
    if mode == fc.FUSE_UNFUSED and dtype != "f32":
        # every stage stores its output in the storage type: the oracle applied stage by stage
        ref = x
        for s in range(K):
            ref = oracle.chain(relu[s:s + 1], a[s:s + 1], b[s:s + 1], ref, dtype)
    else:
        ref = oracle.chain(relu, a, b, x, dtype)
    wide = np.uint32 if dtype == "f32" else np.uint16
    assert np.array_equal(y.view(wide), ref.view(wide)), (dtype, mode, n, K)


@pytest.mark.parametrize("case", range(24))
def test_rmsnorm(cuda_device, case):
    g = _rng(case, 2)
    mode = [fc.FUSE_FUSED, fc.FUSE_UNFUSED][case % 2]
    rows = int(g.integers(1, 301))
    hidden = _log_uniform(g, 1, 16384 if mode == fc.FUSE_FUSED else 65536)
    eps = float([1e-6, 1e-3, 1.0][int(g.integers(0, 3))])
    x = (g.standard_normal((rows, hidden)) * g.uniform(0.01, 10)).astype(np.float32)
    w = (1.0 + 0.02 * g.standard_normal(hidden)).astype(np.float32)
    y = T_rms._run(x, w, eps, mode, x_off=int(g.integers(0, 4)), y_off=int(g.integers(0, 4)))
    T_rms._close(y, oracle.rmsnorm(x, w, eps))


@pytest.mark.parametrize("case", range(16))
def test_add_rmsnorm(cuda_device, case):
    g = _rng(case, 3)
    mode = [fc.FUSE_FUSED, fc.FUSE_UNFUSED][case % 2]
    rows = int(g.integers(1, 201))
    hidden = _log_uniform(g, 1, 16384)
    eps = float([1e-6, 1e-3][int(g.integers(0, 2))])
    x = g.standard_normal((rows, hidden)).astype(np.float32)
    r = g.standard_normal((rows, hidden)).astype(np.float32)
    w = (1.0 + 0.02 * g.standard_normal(hidden)).astype(np.float32)
    inplace = [None, "x", "r"][int(g.integers(0, 3))]
    h, y = T_add._run(x, r, w, eps, mode, off=int(g.integers(0, 4)), inplace=inplace)
    h_ref, y_ref = oracle.add_rmsnorm(x, r, w, eps)
    assert np.array_equal(h.view(np.uint32), h_ref.view(np.uint32))
    T_add._close(y, y_ref)


@pytest.mark.parametrize("case", range(24))
def test_causal_softmax(cuda_device, case):
    g = _rng(case, 4)
    bh = int(g.integers(1, 5))
    S = _log_uniform(g, 1, 3000)
    scale = float(g.choice([1.0 / 16, 0.5, 2.0]))
    mode = fc.FUSE_UNFUSED if case % 4 == 3 else fc.FUSE_FUSED
    out = "f32" if case % 4 == 2 else "bf16"
    tile = 0 if mode == fc.FUSE_UNFUSED else int(g.choice([0, 16, 32, 64, 128, 256]))
    s = wl.softmax_input(bh, S, salt=1000 + case)
    p = T_sm._run(s, scale, tile, mode, out=out, p_off=int(g.integers(0, 8)))
    if out == "f32":
        ref = oracle.causal_softmax(s, scale, out="f32")
        iu = np.triu_indices(S, 1)
        assert np.all(p[..., iu[0], iu[1]].view(np.uint32) == 0)
        err = np.abs(p.astype(np.float64) - ref)
        assert np.all(err <= 1e-5 * np.abs(ref) + 1e-30)
    elif mode == fc.FUSE_UNFUSED:
        T_sm._check_bf16(p, oracle.causal_softmax(s, scale, unfused=True), S, 2)
    else:
        T_sm._check_bf16(p, oracle.causal_softmax(s, scale), S, 1)


@pytest.mark.parametrize("case", range(20))
def test_gemm_epilogue(cuda_device, case):
    g = _rng(case, 5)
    M = _log_uniform(g, 1, 700)
    N = 8 * _log_uniform(g, 1, 128)
    K = 8 * _log_uniform(g, 1, 160)
    mask = int(g.integers(0, 8))
    std = float(g.choice([1.0 / 64, 1.0 / 8]))
    A, B, bias, R = wl.gemm_input(M, N, K, salt=2000 + case, std=std)
    Y = T_gemm._run(A, B, bias, R, mask, ws=bool(case % 2))
    T_gemm._check(Y, oracle.gemm_epilogue(A, B, bias, R, mask), mask, A, B)


@pytest.mark.parametrize("case", range(16))
def test_silu_mul(cuda_device, case):
    g = _rng(case, 6)
    dtype = ["f32", "f16", "bf16"][case % 3]
    mode = [fc.FUSE_FUSED, fc.FUSE_UNFUSED][(case // 3) % 2]
    rows = int(g.integers(1, 129))
    cols = _log_uniform(g, 1, 6000)
    gu = wl.silu_input(rows, cols, dtype, salt=3000 + case, scale=float(g.choice([1.0, 4.0])))
    y = T_silu._run_merged(gu, dtype, mode, y_off=int(g.integers(0, 8)))
    ref = oracle.silu_mul_merged(gu, dtype, unfused=mode == fc.FUSE_UNFUSED)
    T_silu._compare(y, ref, dtype, 1 if mode == fc.FUSE_FUSED else 2)


@pytest.mark.parametrize("case", range(12))
def test_attention(cuda_device, case):
    g = _rng(case, 7)
    D = [64, 128, 256][case % 3]
    bh = int(g.integers(1, 5))
    S = 128 * int(g.integers(1, 9))
    q, k, v = wl.attention_input(bh, S, D, salt=4000 + case)
    scale = float(g.choice([1.0 / np.sqrt(D), 0.5 / np.sqrt(D), 2.0 / np.sqrt(D)]))
    o = T_att._run(q, k, v, scale)
    T_att._check(o, oracle.attention(q, k, v, scale), v)
    assert np.array_equal(o[:, 0], v[:, 0])
