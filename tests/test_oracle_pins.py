"""Pins of the CPU oracle against facts fixed outside it: values printed on the pages, closed
forms, textbook constants, invariants of the definitions, and brute force on tiny inputs through
an independent arithmetic engine (numpy fp32/fp16 scalars, Python fractions).

None of these tests touches a GPU or the CUDA library.
"""
from fractions import Fraction
import math

import numpy as np
import pytest

import oracle
from conftest import read_golden
from epilogue_chains_gb300 import workloads as wl


# ============================================================== storage-type conversions
def test_half_decode_exhaustive():
    """Every fp16 bit pattern decodes to numpy's value."""
    ref = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.half_value(h) for h in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decode_exhaustive():
    import torch
    ref = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_value(h) for h in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_half_rounding_matches_numpy_including_ties():
    g = np.random.default_rng(7)
    vals = list(g.standard_normal(3000) * np.exp(g.uniform(-20, 11, 3000)))
    # exact midpoints between neighbouring finite fp16 values (ties -> even), subnormals too
    for h in g.integers(0, 0x7BFF, 2000):
        lo = np.uint16(h).view(np.float16).astype(np.float64)
        hi = np.uint16(h + 1).view(np.float16).astype(np.float64)
        vals += [(lo + hi) / 2, -(lo + hi) / 2]
    vals += [65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25, 2.0 ** -26, 0.0, -0.0]
    np.seterr(over="ignore")
    for v in vals:
        want = int(np.array(v, dtype=np.float64).astype(np.float16).view(np.uint16))
        assert oracle.half_bits(v) == want, v


def test_bf16_rounding_matches_torch_including_ties():
    import torch
    g = np.random.default_rng(8)
    f = (g.standard_normal(4000) * np.exp(g.uniform(-30, 30, 4000))).astype(np.float32)
    bits = f.view(np.uint32)
    ties = ((bits & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)  # exact halfway
    f = np.concatenate([f, ties, np.array([3.3895314e38, -1e-40, 1e-45], dtype=np.float32)])
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_bits(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, want)


# ============================================================== O1/O2 pointwise chain
def test_chain_reproduces_printed_v1_v3_relative_error():
    """The literal chain (multiply then add, fp32 constants) against the page's closed form V3,
    computed the way the page's numpy script computes it, gives the printed relative errors."""
    rng = np.random.default_rng(wl.RNG_SEED)
    K, A, B = 8, 1.01, 0.01
    for n_s, rel_s in read_golden("ofcg_v1_v3_relerr.txt"):
        n = int(n_s)
        x = rng.standard_normal(n).astype(np.float32)
        v1 = oracle.chain(np.zeros(K), np.full(K, A), np.full(K, B), x)
        Ak = A ** K
        Bk = B * (Ak - 1.0) / (A - 1.0)
        v3 = np.empty_like(x)
        np.multiply(x, Ak, out=v3)
        np.add(v3, Bk, out=v3)
        rel = float(np.max(np.abs(v1 - v3)) / np.max(np.abs(v1)))
        assert f"{rel:.2e}" == rel_s, (n, rel, rel_s)


def test_affine_closed_form_constants():
    """A^8 and B (A^8 - 1)/(A - 1) for A = fl32(1.01), B = fl32(0.01): about 1.0828566 and
    0.0828567 (1.01^8 = 1.0828567 in double; the fp32 constant is 9.5e-9 smaller)."""
    y = oracle.affine_closed_form(np.array([0.0, 1.0], dtype=np.float32), 8, 1.01, 0.01)
    A = float(np.float32(1.01))
    B = float(np.float32(0.01))
    assert abs(y[0] - 0.0828567) < 5e-8
    assert abs((y[1] - y[0]) - 1.0828566) < 5e-8
    # the same numbers from the geometric series sum_{k<8} A^k, summed term by term
    series = sum(Fraction(A) ** k for k in range(8))
    assert abs(y[0] - float(Fraction(B) * series)) < 1e-15
    assert abs((y[1] - y[0]) - float(Fraction(A) ** 8)) < 1e-15


def test_chain_config0_within_1e6_of_closed_form():
    relu, a, b, x = wl.affine_chain()
    lit = oracle.chain(relu, a, b, x)
    cf = oracle.affine_closed_form(x, wl.AFFINE_K, wl.AFFINE_A, wl.AFFINE_B)
    assert np.max(np.abs(lit - cf)) / np.max(np.abs(cf)) <= 1e-6


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_chain_identity_stages(dtype):
    x = wl.chain_input(1000, salt=3)
    if dtype == "f16":
        x = x.astype(np.float16).view(np.uint16)
    elif dtype == "bf16":
        x = wl.bf16_bits_from_f32(x)
    K = 5
    y = oracle.chain(np.zeros(K), np.ones(K), np.zeros(K), x, dtype)
    assert np.array_equal(y, x)


def test_chain_power_of_two_scaling_is_exact():
    x = wl.chain_input(1000, salt=4)
    y = oracle.chain(np.zeros(3), [2.0, 0.5, 4.0], [0.0] * 3, x)
    assert np.array_equal(y, x * np.float32(4.0))


def test_chain_zero_coefficient_forgets_input():
    x = wl.chain_input(64, salt=5)
    y = oracle.chain([0, 0, 1], [1.3, 0.7, 0.0], [0.2, -0.1, -0.25], x)
    assert np.all(y.view(np.uint32) == 0)      # ReLU(0*v - 0.25) = +0 on even stage 2
    y = oracle.chain([0, 0], [1.3, 0.0], [0.2, -0.25], x)
    assert np.all(y == np.float32(-0.25))


def test_chain_relu_on_even_stages_only():
    relu, a, b = wl.chain_stages(3)
    assert list(relu) == [1, 0, 1]
    x = wl.chain_input(4096, salt=6)
    assert np.all(oracle.chain(relu, a, b, x) >= 0)          # last stage (s = 2) is even
    # stage 1 (odd) has no ReLU: an affine odd stage that shifts down leaves negatives
    y = oracle.chain([1, 0], [1.0, 1.0], [0.0, -1.0], x)
    assert y.min() < 0 and np.all(y >= -1.0)


def test_chain_composition_and_order():
    """chain(s_0..s_{K-1}) == chain(s_k..s_{K-1}) o chain(s_0..s_{k-1}), bit for bit."""
    relu, a, b = wl.chain_stages(8)
    x = wl.chain_input(2048, salt=7)
    full = oracle.chain(relu, a, b, x)
    for k in range(1, 8):
        head = oracle.chain(relu[:k], a[:k], b[:k], x)
        both = oracle.chain(relu[k:], a[k:], b[k:], head)
        assert np.array_equal(full, both)
    rev = oracle.chain(relu[::-1], a[::-1], b[::-1], x)
    assert not np.array_equal(full, rev)


def test_chain_brute_force_numpy_fp32_scalars():
    """Tiny inputs through numpy's own fp32 scalar arithmetic (an independent engine)."""
    g = np.random.default_rng(11)
    for K in range(1, 9):
        relu = g.integers(0, 2, K)
        a = g.uniform(-1.5, 1.5, K).astype(np.float32)
        b = g.uniform(-0.5, 0.5, K).astype(np.float32)
        x = g.standard_normal(16).astype(np.float32)
        want = []
        for xi in x:
            v = np.float32(xi)
            for s in range(K):
                t = np.float32(np.float32(a[s] * v) + b[s])
                v = t if (not relu[s] or t > 0) else np.float32(0.0)
            want.append(v)
        got = oracle.chain(relu, a, b, x)
        assert np.array_equal(got.view(np.uint32), np.array(want, np.float32).view(np.uint32))


def test_chain_two_roundings_not_fused_multiply_add():
    """a*v + b rounds twice: pick operands where a single (FMA) rounding differs."""
    g = np.random.default_rng(12)
    found = 0
    for _ in range(2000):
        a, v, b = (np.float32(g.uniform(0.5, 2.0)), np.float32(g.uniform(0.5, 2.0)),
                   np.float32(g.uniform(-2, 2)))
        two = np.float32(np.float32(a * v) + b)
        exact = Fraction(float(a)) * Fraction(float(v)) + Fraction(float(b))
        one = np.float32(float(exact))   # exact value is a double here (<= 49 significant bits)
        if one != two:
            found += 1
            got = oracle.chain([0], [a], [b], np.array([v], np.float32))[0]
            assert got == two
    assert found > 10


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_chain_storage_types_round_once(dtype):
    relu, a, b = wl.chain_stages(4)
    x32 = wl.chain_input(4096, salt=9)
    if dtype == "f16":
        xs = x32.astype(np.float16)
        dec = xs.astype(np.float32)
        xs = xs.view(np.uint16)
        want = oracle.chain(relu, a, b, dec).astype(np.float16).view(np.uint16)
    else:
        import torch
        xs = wl.bf16_bits_from_f32(x32)
        dec = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).float().numpy()
        want = wl.bf16_bits_from_f32(oracle.chain(relu, a, b, dec))
    got = oracle.chain(relu, a, b, xs, dtype)
    assert np.array_equal(got, want)


# ============================================================== O3 RMSNorm
def _ulp32(v):
    return np.spacing(np.abs(np.float32(v)))


@pytest.mark.parametrize("c", [0.5, 3.0, -2.0, 1e-3, 7.25])
def test_rmsnorm_constant_row_closed_form(c):
    H, eps = 64, 1e-6
    x = np.full((2, H), c, np.float32)
    y = oracle.rmsnorm(x, np.ones(H, np.float32), eps)
    cf = float(np.float32(c)) / math.sqrt(float(np.float32(c)) ** 2 + eps)
    assert np.all(np.abs(y - np.float32(cf)) <= _ulp32(cf))


def test_rmsnorm_unit_rows_and_weight_per_column():
    H, eps = 48, 1e-6
    g = np.random.default_rng(13)
    x = np.where(g.random((3, H)) < 0.5, -1.0, 1.0).astype(np.float32)
    w = g.uniform(0.5, 1.5, H).astype(np.float32)
    y = oracle.rmsnorm(x, w, eps)
    want = (x.astype(np.float64) * w.astype(np.float64) / math.sqrt(1.0 + eps)).astype(np.float32)
    assert np.all(np.abs(y - want) <= _ulp32(want))


def test_rmsnorm_eps_inside_the_square_root():
    """With w = 1: mean_j y_j^2 = ms / (ms + eps).  A large eps makes the placement visible."""
    x, _ = wl.rmsnorm_input(4, 256)
    for eps in (0.5, 2.0):
        y = oracle.rmsnorm(x, np.ones(256, np.float32), eps).astype(np.float64)
        ms = np.mean(x.astype(np.float64) ** 2, axis=1)
        assert np.allclose(np.mean(y ** 2, axis=1), ms / (ms + eps), rtol=1e-6)


def test_rmsnorm_permutation_equivariance():
    x, w = wl.rmsnorm_input(5, 96)
    y = oracle.rmsnorm(x, w, 1e-6)
    g = np.random.default_rng(14)
    pc, pr = g.permutation(96), g.permutation(5)
    assert np.array_equal(oracle.rmsnorm(x[:, pc], w[pc], 1e-6), y[:, pc])
    assert np.array_equal(oracle.rmsnorm(x[pr], w, 1e-6), y[pr])


def test_rmsnorm_scale_invariance_without_eps():
    x, w = wl.rmsnorm_input(3, 128)
    y = oracle.rmsnorm(x, w, 0.0)
    assert np.array_equal(oracle.rmsnorm(x * np.float32(8.0), w, 0.0), y)


def test_rmsnorm_brute_force_tiny():
    x = np.array([[1, 2, 3, 4, 5], [-1, 0.5, 0.25, 2, -3], [0, 0, 0, 0, 1e-3]], np.float32)
    w = np.array([1, 0.5, 2, -1, 0.25], np.float32)
    eps = 1e-6
    y = oracle.rmsnorm(x, w, eps)
    for i in range(3):
        ms = math.fsum(float(v) ** 2 for v in x[i]) / 5
        for j in range(5):
            want = np.float32(float(x[i, j]) / math.sqrt(ms + eps) * float(w[j]))
            assert abs(y[i, j] - want) <= _ulp32(want)


# ============================================================== O4 causal softmax
def _bf16_round_fraction(q: Fraction) -> int:
    """bf16 bits of a positive rational, nearest-even, by integer arithmetic."""
    e = math.floor(math.log2(q))
    while Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    quantum = Fraction(2) ** (e - 7)
    m = q / quantum
    fl = math.floor(m)
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = fl * quantum
    return int(np.array(float(val), np.float32).view(np.uint32) >> 16)


def test_softmax_first_row_and_mask_are_exact():
    s = wl.softmax_input(2, 32)
    p = oracle.causal_softmax(s, wl.SM_SCALE)
    assert np.all(p[:, 0, 0] == 0x3F80)                      # 1.0
    iu = np.triu_indices(32, 1)
    assert np.all(p[:, iu[0], iu[1]] == 0)                   # masked outputs are +0 exactly


def test_softmax_constant_rows_give_one_over_i_plus_one():
    S = 40
    s = np.full((1, S, S), 0x3FC0, np.uint16)                # every score = 1.5
    p = oracle.causal_softmax(s, wl.SM_SCALE)
    for i in range(S):
        assert np.all(p[0, i, : i + 1] == _bf16_round_fraction(Fraction(1, i + 1)))
    pf = oracle.causal_softmax(s, wl.SM_SCALE, out="f32")
    for i in range(S):
        assert np.all(np.abs(pf[0, i, : i + 1] - np.float32(1.0 / (i + 1))) <= _ulp32(1.0 / (i + 1)))


def test_softmax_nonzero_count_is_causal_triangle():
    S = 64
    p = oracle.causal_softmax(wl.softmax_input(3, S), wl.SM_SCALE)
    for bh in range(3):
        assert int(np.count_nonzero(p[bh])) == S * (S + 1) // 2


def test_softmax_rows_sum_to_one_fp32():
    p = oracle.causal_softmax(wl.softmax_input(2, 96), wl.SM_SCALE, out="f32")
    assert np.allclose(p.astype(np.float64).sum(-1), 1.0, atol=2e-6)


def test_softmax_ignores_masked_region_and_uses_lower_triangle():
    S = 24
    s = wl.softmax_input(1, S)
    p = oracle.causal_softmax(s, wl.SM_SCALE)
    s2 = s.copy()
    iu = np.triu_indices(S, 1)
    s2[0][iu] = 0x4700                                       # 32768.0 where j > i
    assert np.array_equal(oracle.causal_softmax(s2, wl.SM_SCALE), p)
    s3 = s.copy()
    s3[0, S - 1, 0] = 0x4700                                  # a kept entry does change the row
    assert not np.array_equal(oracle.causal_softmax(s3, wl.SM_SCALE)[0, S - 1], p[0, S - 1])


def test_softmax_shift_and_scale_invariance():
    S = 32
    g = np.random.default_rng(15)
    vals = g.integers(-16, 17, (2, S, S)) / 4.0                # multiples of 1/4: exact in bf16
    s = wl.bf16_bits_from_f32(vals.astype(np.float32))
    shifted = wl.bf16_bits_from_f32((vals + 1.0).astype(np.float32))
    doubled = wl.bf16_bits_from_f32((vals * 2.0).astype(np.float32))
    p = oracle.causal_softmax(s, 1.0 / 16)
    assert np.array_equal(oracle.causal_softmax(shifted, 1.0 / 16), p)
    assert np.array_equal(oracle.causal_softmax(doubled, 1.0 / 32), p)


def test_softmax_brute_force_tiny():
    S = 6
    s = wl.softmax_input(1, S, salt=5)
    vals = np.array([[oracle.bf16_value(h) for h in row] for row in s[0]])
    p = oracle.causal_softmax(s, 0.25, out="f32")
    for i in range(S):
        e = [math.exp(vals[i, j] * 0.25) for j in range(i + 1)]
        tot = math.fsum(e)
        for j in range(S):
            want = e[j] / tot if j <= i else 0.0
            assert abs(p[0, i, j] - want) <= 2e-7 * max(want, 1e-30)


def test_softmax_unfused_oracle_tracks_fused_within_4_ulp():
    s = wl.softmax_input(2, 80)
    a = oracle.causal_softmax(s, wl.SM_SCALE).astype(np.int32)
    b = oracle.causal_softmax(s, wl.SM_SCALE, unfused=True).astype(np.int32)
    assert np.max(np.abs(a - b)) <= 4                          # same sign: bit distance = ulps
    iu = np.triu_indices(80, 1)
    assert np.all(b[:, iu[0], iu[1]] == 0) and np.all(b[:, 0, 0] == 0x3F80)


def _bf16_round_signed(q: Fraction) -> Fraction:
    """Nearest-even bf16 value of a rational of normal magnitude (or zero), by integer steps."""
    if q == 0:
        return Fraction(0)
    v = Fraction(oracle.bf16_value(_bf16_round_fraction(abs(q))))
    return v if q > 0 else -v


# The reference below takes [OFCG] fusion_lab [E]'s five steps one at a time, each stored before
# the next, in an arithmetic of its own (numpy fp32 scalars for the fp32 steps, exact fractions
# for the sum and the division, integer nearest-even rounding to bf16).  `mutation` drops or moves
# one rounding point, to show that each one is seen by the comparison.
_SOFTMAX_MUTATIONS = ("no_d_round", "no_e_round", "d_exact_then_bf16", "z_in_double",
                      "z_rounded_to_bf16", "sum_of_unrounded_e", "numerator_unrounded_e")


def _unfused_softmax_reference(vals, scale, mutation=None):
    S = vals.shape[0]
    out = np.zeros((S, S), dtype=object)
    sc = np.float32(scale)
    for i in range(S):
        if mutation == "z_in_double":
            z = [Fraction(float(vals[i, j])) * Fraction(float(scale)) for j in range(i + 1)]
        else:
            z = [Fraction(float(np.float32(np.float32(vals[i, j]) * sc))) for j in range(i + 1)]
            if mutation == "z_rounded_to_bf16":
                z = [_bf16_round_signed(t) for t in z]
        m = max(z)                                                  # step 1: row max
        e, e_raw = [], []
        for j in range(i + 1):                                      # step 2: subtract, stored bf16
            if mutation in ("z_in_double", "d_exact_then_bf16"):
                d = z[j] - m
            else:
                d = Fraction(float(np.float32(np.float32(float(z[j])) - np.float32(float(m)))))
            dq = d if mutation == "no_d_round" else _bf16_round_signed(d)
            x = Fraction(math.exp(float(dq)))                       # step 3: exp, stored bf16
            e_raw.append(x)
            e.append(x if mutation == "no_e_round" else _bf16_round_signed(x))
        l = sum(e_raw if mutation == "sum_of_unrounded_e" else e, Fraction(0))   # step 4: row sum
        for j in range(i + 1):                                      # step 5: divide
            num = e_raw[j] if mutation == "numerator_unrounded_e" else e[j]
            out[i, j] = num / l
    return out


@pytest.mark.parametrize("scale", [1.0 / 16.0, 0.3])
def test_softmax_unfused_rounding_points_brute_force(scale):
    """orc_causal_softmax_unfused against the five stored steps done by hand, bit for bit, at the
    workload's scale (1/16, exact in fp32) and at 0.3 (where the fp32 steps round)."""
    BH, S = 16, 8
    s = wl.softmax_input(BH, S, salt=11)
    got = oracle.causal_softmax(s, scale, unfused=True)
    got32 = oracle.causal_softmax(s, scale, out="f32", unfused=True)
    for bh in range(BH):
        vals = np.array([[oracle.bf16_value(h) for h in row] for row in s[bh]])
        ref = _unfused_softmax_reference(vals, scale)
        for i in range(S):
            for j in range(S):
                if j > i:
                    assert got[bh, i, j] == 0 and got32[bh, i, j] == 0
                    continue
                assert got[bh, i, j] == _bf16_round_fraction(ref[i, j]), (bh, i, j)
                assert got32[bh, i, j] == np.float32(float(ref[i, j])), (bh, i, j)


def test_softmax_unfused_pin_sees_every_rounding_point():
    """Each mutation of the hand reference (one rounding dropped or moved) changes at least one
    output bit on the inputs the brute-force pin uses, so an oracle with that mistake fails it."""
    BH, S = 16, 8
    s = wl.softmax_input(BH, S, salt=11)
    seen = {m: False for m in _SOFTMAX_MUTATIONS}
    for scale in (1.0 / 16.0, 0.3):
        for bh in range(BH):
            vals = np.array([[oracle.bf16_value(h) for h in row] for row in s[bh]])
            ref = _unfused_softmax_reference(vals, scale)
            for mut in _SOFTMAX_MUTATIONS:
                if seen[mut]:
                    continue
                bad = _unfused_softmax_reference(vals, scale, mut)
                seen[mut] = any(_bf16_round_fraction(bad[i, j]) != _bf16_round_fraction(ref[i, j])
                                for i in range(S) for j in range(i + 1))
    assert all(seen.values()), seen


# ============================================================== O5 GEMM epilogue
PHI = {1.0: 0.8413447460685429, 2.0: 0.9772498680518208, -1.0: 0.15865525393145705,
       0.5: 0.6914624612740131, 3.0: 0.9986501019683699, 0.0: 0.5, -2.0: 0.022750131948179195}


def _gelu_tb(v):
    """x * Phi(x) from textbook normal-CDF values."""
    return v * PHI[v]


@pytest.mark.parametrize("v", sorted(PHI))
def test_gelu_is_the_erf_form(v):
    assert abs(oracle.gelu(v) - _gelu_tb(v)) <= 1e-15 * max(1.0, abs(v))


def _h(v):
    return int(np.array(v, np.float64).astype(np.float16).view(np.uint16))


def _hv(v):
    return float(np.array(v, np.float64).astype(np.float16))


def _f16(vals):
    return np.array(vals, np.float64).astype(np.float16).view(np.uint16)


@pytest.mark.parametrize("mask", range(8))
def test_gemm_zero_A_reduces_to_gelu_of_bias_plus_residual(mask):
    N, M, K = 7, 3, 8
    bias_v = [1.0, 2.0, -1.0, 0.5, 3.0, 0.0, -2.0]
    R_v = np.array([[0.0, 1.0, -0.5, 0.25, 2.0, -3.0, 0.125]] * M) * np.array([[1], [2], [-1]])
    Y = oracle.gemm_epilogue(np.zeros((M, K), np.uint16), _f16(np.ones((K, N))), _f16(bias_v),
                             _f16(R_v), cut_mask=mask)
    for m in range(M):
        for n in range(N):
            g = _gelu_tb(bias_v[n])
            if mask & 4:
                g = _hv(g)
            assert Y[m, n] == _h(g + R_v[m, n]), (m, n)


@pytest.mark.parametrize("shape", [(3, 5, 5), (4, 6, 4), (2, 3, 9)])
def test_gemm_selection_matrix_catches_operand_transposes(shape):
    """B[k, n] = 1 iff k == sel[n], so acc[m, n] = A[m, sel[n]]; A from textbook GELU points."""
    M, K, N = shape
    g = np.random.default_rng(16)
    pts = np.array([1.0, 2.0, -1.0, 0.5, 3.0, 0.0, -2.0])
    A_v = g.choice(pts, (M, K))
    sel = g.choice(K, N, replace=K < N)
    B_v = np.zeros((K, N))
    B_v[sel, np.arange(N)] = 1.0
    Y = oracle.gemm_epilogue(_f16(A_v), _f16(B_v), np.zeros(N, np.uint16), np.zeros((M, N), np.uint16))
    for m in range(M):
        for n in range(N):
            assert Y[m, n] == _h(_gelu_tb(A_v[m, sel[n]])), (m, n)


def test_gemm_rounding_point_after_mm():
    """acc = 1 + 2^-12 rounds to 1 at a cut after mm; bias -1 then leaves 0 or 2^-12."""
    A = _f16([[1.0, 2.0 ** -12]])
    B = _f16([[1.0], [1.0]])
    bias, R = _f16([-1.0]), _f16([[0.0]])
    for mask in range(8):
        y = oracle.gemm_epilogue(A, B, bias, R, cut_mask=mask)[0, 0]
        if mask & 1:
            assert y == 0
        else:
            assert y == _h(2.0 ** -13) and y != 0        # GELU(2^-12) ~ 2^-13 (1 + 2^-11.3)


def test_gemm_rounding_point_after_bias():
    """acc = 1, bias = 2^-11: 1 + 2^-11 ties to 1.0 at a cut after bias."""
    A, B, R = _f16([[1.0]]), _f16([[1.0]]), _f16([[0.0]])
    bias = _f16([2.0 ** -11])
    y_cut = oracle.gemm_epilogue(A, B, bias, R, cut_mask=2)[0, 0]
    y_no = oracle.gemm_epilogue(A, B, bias, R, cut_mask=0)[0, 0]
    assert y_cut == _h(_gelu_tb(1.0))
    assert y_no != y_cut


def test_gemm_rounding_point_after_gelu():
    A, B, bias = _f16([[1.0]]), _f16([[1.0]]), _f16([0.0])
    g1 = _gelu_tb(1.0)
    hits = 0
    for r in np.arange(-4, 4, 1.0 / 64):
        R = _f16([[r]])
        want_cut = _h(_hv(g1) + _hv(r))
        want_no = _h(g1 + _hv(r))
        assert oracle.gemm_epilogue(A, B, bias, R, cut_mask=4)[0, 0] == want_cut
        assert oracle.gemm_epilogue(A, B, bias, R, cut_mask=0)[0, 0] == want_no
        hits += want_cut != want_no
    assert hits > 0


def test_gemm_row_subset_matches_full():
    A, B, bias, R = wl.gemm_input(16, 48, 40)
    full = oracle.gemm_epilogue(A, B, bias, R, cut_mask=0)
    rows = np.array([15, 0, 7])
    assert np.array_equal(oracle.gemm_epilogue(A, B, bias, R, cut_mask=0, rows=rows), full[rows])


def test_gemm_brute_force_tiny_fractions():
    M, N, K = 3, 4, 5
    A, B, bias, R = wl.gemm_input(M, N, K, std=0.5)
    Y = oracle.gemm_epilogue(A, B, bias, R, cut_mask=0)
    Av, Bv = A.view(np.float16).astype(np.float64), B.view(np.float16).astype(np.float64)
    bv, Rv = bias.view(np.float16).astype(np.float64), R.view(np.float16).astype(np.float64)
    for m in range(M):
        for n in range(N):
            acc = float(sum(Fraction(Av[m, k]) * Fraction(Bv[k, n]) for k in range(K)))
            v = acc + bv[n]
            g = 0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0)))
            assert Y[m, n] == _h(g + Rv[m, n])


# ============================================================== residual add + RMSNorm
def test_add_rmsnorm_zero_residual_is_rmsnorm():
    """r = 0: h = x exactly and y is the (independently pinned) RMSNorm of x."""
    x, _, w = wl.add_rmsnorm_input(6, 256)
    h, y = oracle.add_rmsnorm(x, np.zeros_like(x), w, 1e-6)
    assert np.array_equal(h.view(np.uint32), x.view(np.uint32))
    assert np.array_equal(y, oracle.rmsnorm(x, w, 1e-6))


def test_add_rmsnorm_sum_is_one_ieee_fp32_addition():
    """h against numpy's float32 addition (IEEE round-to-nearest-even), element by element,
    including cancellation, ties and sums that overflow to inf."""
    x, r, w = wl.add_rmsnorm_input(4, 512, salt=1)
    x[0, :4] = [1.0, 3.4e38, 2.0 ** -24, -5.5]
    r[0, :4] = [2.0 ** -24, 3.4e38, 1.0, 5.5]
    h, _ = oracle.add_rmsnorm(x, r, w, 1e-6)
    assert np.array_equal(h.view(np.uint32), (x + r).view(np.uint32))
    assert h[0, 0] == np.float32(1.0) and np.isinf(h[0, 1]) and h[0, 3] == 0.0


def test_add_rmsnorm_normalises_the_sum_not_the_inputs():
    """A constant row split between x and r: h = c and y = c / sqrt(c^2 + eps) (w = 1)."""
    H, eps, c = 64, 1e-6, 3.0
    g = np.random.default_rng(15)
    parts = g.integers(-8, 8, (2, H)).astype(np.float32)
    x = parts
    r = (np.float32(c) - parts).astype(np.float32)
    h, y = oracle.add_rmsnorm(x, r, np.ones(H, np.float32), eps)
    assert np.all(h == np.float32(c))
    cf = c / math.sqrt(c * c + eps)
    assert np.all(np.abs(y - np.float32(cf)) <= _ulp32(cf))


def test_add_rmsnorm_is_symmetric_in_x_and_r():
    x, r, w = wl.add_rmsnorm_input(3, 128, salt=2)
    h1, y1 = oracle.add_rmsnorm(x, r, w, 1e-6)
    h2, y2 = oracle.add_rmsnorm(r, x, w, 1e-6)
    assert np.array_equal(h1, h2) and np.array_equal(y1, y2)


def test_add_rmsnorm_brute_force_tiny():
    x = np.array([[1, 2, 3, 4], [0.5, -1, 0.25, 8]], np.float32)
    r = np.array([[0.5, -2, 1, 0], [0.5, 1, -0.25, -4]], np.float32)
    w = np.array([1, 2, 0.5, -1], np.float32)
    h, y = oracle.add_rmsnorm(x, r, w, 0.0)
    for i in range(2):
        hs = [float(a) + float(b) for a, b in zip(x[i], r[i])]   # exact in fp32 here
        ms = math.fsum(v * v for v in hs) / 4
        for j in range(4):
            assert h[i, j] == np.float32(hs[j])
            want = np.float32(hs[j] / math.sqrt(ms) * float(w[j]))
            assert abs(y[i, j] - want) <= _ulp32(want)


# ============================================================== SiLU(gate) * up
def test_silu_values_against_the_logistic_function():
    """SiLU(v) = v * logistic(v), with scipy's logistic (expit) as the independent routine."""
    from scipy.special import expit
    for v in [-30.0, -5.0, -1.0, -1e-3, 0.0, 1e-3, 0.5, 1.0, 2.0, 7.5, 30.0]:
        assert oracle.silu(v) == pytest.approx(v * expit(v), rel=1e-14, abs=1e-300)
    assert oracle.silu(1.0) == pytest.approx(math.e / (1 + math.e), rel=1e-15)


def test_silu_odd_part_identity():
    """SiLU(v) - SiLU(-v) = v (logistic(v) + logistic(-v) = 1)."""
    for v in np.linspace(-12, 12, 97):
        assert oracle.silu(v) - oracle.silu(-v) == pytest.approx(v, abs=1e-14)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_silu_mul_with_unit_up_is_rounded_silu(dtype):
    gu = wl.silu_input(4, 64, dtype=dtype, salt=1)
    g = gu[:, :64].copy()
    one = {"f32": np.ones((4, 64), np.float32),
           "f16": np.full((4, 64), 0x3C00, np.uint16),
           "bf16": np.full((4, 64), 0x3F80, np.uint16)}[dtype]
    y = oracle.silu_mul(g, one, dtype)
    dec = (lambda a: a.astype(np.float64)) if dtype == "f32" else (
        np.vectorize(oracle.half_value) if dtype == "f16" else np.vectorize(oracle.bf16_value))
    rnd = {"f32": lambda v: float(np.float32(v)), "f16": oracle.round_half,
           "bf16": oracle.round_bf16}[dtype]
    want = np.vectorize(lambda v: rnd(oracle.silu(v)))(dec(g))
    assert np.array_equal(dec(y), want)
    # with up = 1 the unfused form rounds the same value twice: identical
    assert np.array_equal(oracle.silu_mul(g, one, dtype, unfused=True), y)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_silu_mul_power_of_two_up_scales_exactly(dtype):
    gu = wl.silu_input(3, 40, dtype=dtype, salt=2)
    g = gu[:, :40].copy()
    two = {"f32": np.full((3, 40), 2.0, np.float32), "f16": np.full((3, 40), 0x4000, np.uint16),
           "bf16": np.full((3, 40), 0x4000, np.uint16)}[dtype]
    one = {"f32": np.ones((3, 40), np.float32), "f16": np.full((3, 40), 0x3C00, np.uint16),
           "bf16": np.full((3, 40), 0x3F80, np.uint16)}[dtype]
    y1 = oracle.silu_mul(g, one, dtype)
    y2 = oracle.silu_mul(g, two, dtype)
    if dtype == "f32":
        assert np.array_equal(y2, y1 * np.float32(2))
    else:
        dec = np.vectorize(oracle.half_value if dtype == "f16" else oracle.bf16_value)
        assert np.array_equal(dec(y2), 2 * dec(y1))


def test_silu_mul_unfused_rounds_the_intermediate():
    """bf16: the unfused form is RNE(RNE(SiLU(g)) * u), the fused form RNE(SiLU(g) * u); the two
    differ on some elements, and each matches its definition written with numpy/torch roundings."""
    import torch
    gu = wl.silu_input(8, 256, salt=3)
    g, u = gu[:, :256].copy(), gu[:, 256:].copy()
    yf = oracle.silu_mul(g, u, "bf16")
    yu = oracle.silu_mul(g, u, "bf16", unfused=True)
    gd = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).double().numpy()
    ud = torch.from_numpy(u.view(np.int16)).view(torch.bfloat16).double().numpy()
    s = gd / (1.0 + np.exp(-gd))

    def to_bf16(v):   # double -> bf16 (RNE) through an exact fp32 stage where it is exact
        return np.vectorize(oracle.bf16_bits)(v).astype(np.uint16)
    assert np.array_equal(yf, to_bf16(s * ud))
    sb = np.vectorize(oracle.bf16_value)(to_bf16(s))
    assert np.array_equal(yu, to_bf16(sb * ud))
    assert np.count_nonzero(yf != yu) > 0


def test_silu_mul_merged_layout_matches_separate_arrays():
    gu = wl.silu_input(5, 96, salt=4)
    for unfused in (False, True):
        assert np.array_equal(oracle.silu_mul_merged(gu, "bf16", unfused),
                              oracle.silu_mul(gu[:, :96], gu[:, 96:], "bf16", unfused))


def test_silu_mul_brute_force_tiny_fp32():
    g = np.array([[-2.0, -0.5, 0.0, 0.5, 3.0]], np.float32)
    u = np.array([[1.5, -2.0, 7.0, 0.25, -1.0]], np.float32)
    y = oracle.silu_mul(g, u, "f32")
    for j in range(5):
        gv, uv = float(g[0, j]), float(u[0, j])
        want = np.float32(gv / (1.0 + math.exp(-gv)) * uv)
        assert y[0, j] == want


# ============================================================== causal attention (no score matrix)
def _bf16_to_f64(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).double().numpy()


def _f64_to_bf16(a):
    return np.vectorize(oracle.bf16_bits)(a).astype(np.uint16)


def test_attention_first_row_is_the_first_value_row():
    q, k, v = wl.attention_input(3, 40, 32, salt=1)
    o = oracle.attention(q, k, v, 1 / math.sqrt(32))
    assert np.array_equal(o[:, 0], v[:, 0])


def test_attention_zero_queries_average_the_visible_values():
    """q = 0: every visible key scores 0, so o_i is the mean of v_0..v_i (rounded once)."""
    _, k, v = wl.attention_input(2, 48, 16, salt=2)
    q = np.zeros_like(k)
    o = oracle.attention(q, k, v, 0.25)
    vd = _bf16_to_f64(v)
    mean = np.cumsum(vd, axis=1) / np.arange(1, 49)[None, :, None]
    assert np.array_equal(o, _f64_to_bf16(mean))


def test_attention_is_causal():
    """o_i ignores keys and values after i: changing them leaves o_0..o_i bit-identical."""
    q, k, v = wl.attention_input(2, 64, 32, salt=3)
    o = oracle.attention(q, k, v, 1 / math.sqrt(32))
    k2, v2 = k.copy(), v.copy()
    k2[:, 40:], v2[:, 40:] = v[:, 40:], k[:, 40:]
    o2 = oracle.attention(q, k2, v2, 1 / math.sqrt(32))
    assert np.array_equal(o[:, :40], o2[:, :40])
    assert not np.array_equal(o[:, 40:], o2[:, 40:])


def test_attention_sharp_query_selects_one_key():
    """With orthogonal keys and a query aligned to key j at a large scale, o_i = v_j."""
    S, D = 16, 16
    k = _f64_to_bf16(np.eye(S, D))
    v = wl.attention_input(1, S, D, salt=4)[2][0]
    sel = np.array([0, 1, 1, 3, 2, 5, 0, 7, 8, 4, 10, 11, 12, 6, 14, 15])
    q = _f64_to_bf16(np.eye(S, D)[sel])
    o = oracle.attention(q, k, v, 100.0)
    assert np.array_equal(o, v[sel])


def test_attention_against_scipy_softmax():
    """Tiny slices against scipy's softmax of the masked score matrix times v."""
    from scipy.special import softmax
    q, k, v = wl.attention_input(2, 24, 8, salt=5)
    o = oracle.attention(q, k, v, 0.3)
    qd, kd, vd = _bf16_to_f64(q), _bf16_to_f64(k), _bf16_to_f64(v)
    for b in range(2):
        s = 0.3 * qd[b] @ kd[b].T
        s[np.triu_indices(24, 1)] = -np.inf
        ref = softmax(s, axis=1) @ vd[b]
        got = _bf16_to_f64(o[b])
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-300)


def test_attention_row_subset_matches_full():
    q, k, v = wl.attention_input(2, 96, 32, salt=6)
    o = oracle.attention(q, k, v, 1 / math.sqrt(32))
    rows = np.array([0, 5, 63, 64, 95])
    assert np.array_equal(oracle.attention(q, k, v, 1 / math.sqrt(32), rows=rows), o[:, rows])
