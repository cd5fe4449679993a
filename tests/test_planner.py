"""The cost-model planner ([K4] §② time_estimate / best_plan, §③ spill penalty): the library's
host implementation against the page's printed estimates and against the oracle's plain
enumerator.  No GPU needed."""
import itertools

import numpy as np
import pytest

import epilogue_chains_gb300 as fc
from oracle import planner as op
from conftest import read_golden

# the constants the page's estimates imply (launch 5 us, 448 GB/s, 40 TFLOP/s, penalty 3, 255 regs)
K4_MODEL = dict(hbm_bytes_per_s=448e9, flops_per_s=40e12, launch_s=5e-6, spill_penalty=3.0,
                reg_limit=255)
ORACLE_ARGS = (448e9, 40e12, 5e-6, 3.0, 255)


def mlp_epilogue_stages(M, N, K):
    """[K4] §① chain_mlp_epilogue: mm -> +bias -> GELU -> +residual (live_regs reproduce the
    printed register peaks 128 / 128 / 136 / 160)."""
    return [
        dict(op=0, a=0, b=0, writes=M * N, ext_reads=M * K + K * N, flops=2 * M * N * K, live_regs=128),
        dict(op=0, a=0, b=0, writes=M * N, ext_reads=N, flops=M * N, live_regs=8),
        dict(op=0, a=0, b=0, writes=M * N, ext_reads=0, flops=8 * M * N, live_regs=0),
        dict(op=0, a=0, b=0, writes=M * N, ext_reads=M * N, flops=M * N, live_regs=24),
    ]


def heavy_stages():
    """[K4] §③: a reads n, writes n (live 200); b reads a's n, writes n (live 100); n = 2^26."""
    n = 1 << 26
    return [dict(op=0, a=0, b=0, writes=n, ext_reads=n, flops=n, live_regs=200),
            dict(op=0, a=0, b=0, writes=n, ext_reads=0, flops=n, live_regs=100)]


CASES = {"heavy": heavy_stages, "decode_16": lambda: mlp_epilogue_stages(16, 4096, 4096),
         "square_4096": lambda: mlp_epilogue_stages(4096, 4096, 4096)}


def _round(x, digits):
    return float(f"{x:.{digits}f}")


@pytest.mark.parametrize("row", read_golden("k4_time_estimates.txt"), ids=lambda r: f"{r[0]}-{r[1]}")
def test_library_reproduces_printed_estimates(row):
    case, _, mask, ms, tol, best = row
    st = CASES[case]()
    t = fc.fuse_plan_time(st, int(mask), 2, K4_MODEL) * 1e3
    assert abs(t - float(ms)) <= float(tol), (case, t)
    bmask, bsec = fc.fuse_best_plan(st, 2, K4_MODEL)
    assert (bmask == int(mask)) == (best == "yes")
    if best == "yes":
        assert bsec == pytest.approx(t * 1e-3, rel=1e-15)


@pytest.mark.parametrize("row", read_golden("k4_time_estimates.txt"), ids=lambda r: f"{r[0]}-{r[1]}")
def test_oracle_reproduces_printed_estimates(row):
    case, _, mask, ms, tol, best = row
    st = CASES[case]()
    t = op.plan_time(st, int(mask), 2, *ORACLE_ARGS) * 1e3
    assert abs(t - float(ms)) <= float(tol), (case, t)
    bmask, _ = op.best_plan(st, 2, *ORACLE_ARGS)
    assert (bmask == int(mask)) == (best == "yes")


def test_heavy_fused_is_half_the_traffic_and_half_again_slower():
    """[K4] §③: the fused plan moves half the bytes yet, spilling, takes 1.5x as long (launches
    aside): 2n*2B*3 / (4n*2B) = 1.5."""
    st = heavy_stages()
    split = op.plan_time(st, 1, 2, 448e9, 40e12, 0.0, 3.0, 255)
    fused = op.plan_time(st, 0, 2, 448e9, 40e12, 0.0, 3.0, 255)
    assert fused / split == pytest.approx(1.5, rel=1e-12)
    # without the penalty the fused plan wins by exactly 2x
    assert op.plan_time(st, 0, 2, 448e9, 40e12, 0.0, 1.0, 255) * 2 == pytest.approx(split, rel=1e-12)


def test_decode_saving_is_mostly_launches():
    """[K4] §⑥: of the 16.7 us saved at M = 16 (97.5 - 80.8, the printed values' difference), 15 us
    are the three launches not made."""
    st = mlp_epilogue_stages(16, 4096, 4096)
    saved = op.plan_time(st, 7, 2, *ORACLE_ARGS) - op.plan_time(st, 0, 2, *ORACLE_ARGS)
    assert abs(saved * 1e6 - 16.7) <= 0.1
    no_launch = (op.plan_time(st, 7, 2, 448e9, 40e12, 0.0, 3.0, 255)
                 - op.plan_time(st, 0, 2, 448e9, 40e12, 0.0, 3.0, 255))
    assert _round((saved - no_launch) * 1e6, 1) == 15.0


def test_oracle_memory_term_is_the_byte_ledger():
    """With launch = 0, flops = 0 and no spill the estimate is the ledger's bytes / bandwidth,
    the independently pinned [K4] §① byte counts."""
    st = [dict(s, flops=0) for s in mlp_epilogue_stages(4096, 4096, 4096)]
    for plan, mask, nbytes, _ in read_golden("k4_ledger_bytes.txt"):
        t = op.plan_time(st, int(mask), 2, 1.0, 1.0, 0.0, 3.0, 10 ** 6)
        assert t == int(nbytes), plan


def test_oracle_segments_enumerate_every_composition():
    """2^(n-1) masks give the 2^(n-1) distinct ways to split n stages into consecutive groups."""
    for n in range(1, 7):
        seen = set()
        for mask in range(2 ** (n - 1)):
            segs = op.segments(n, mask)
            assert segs[0][0] == 0 and segs[-1][1] == n - 1
            assert all(b[0] == a[1] + 1 for a, b in zip(segs, segs[1:]))
            seen.add(tuple(segs))
        assert len(seen) == 2 ** (n - 1)


def test_oracle_best_plan_is_the_brute_force_minimum():
    g = np.random.default_rng(11)
    for _ in range(20):
        n = int(g.integers(1, 6))
        st = [dict(writes=int(g.integers(0, 10 ** 7)), ext_reads=int(g.integers(0, 10 ** 7)),
                   flops=int(g.integers(0, 10 ** 10)), live_regs=int(g.integers(0, 200)))
              for _ in range(n)]
        times = [op.plan_time(st, m, 2, *ORACLE_ARGS) for m in range(2 ** (n - 1))]
        mask, t = op.best_plan(st, 2, *ORACLE_ARGS)
        assert t == min(times) and mask == times.index(min(times))


def test_library_matches_oracle_on_random_chains():
    g = np.random.default_rng(12)
    for trial in range(60):
        n = int(g.integers(1, 9))
        st = [dict(op=0, a=0, b=0, writes=int(g.integers(0, 10 ** 8)),
                   ext_reads=int(g.integers(0, 10 ** 8)), flops=int(g.integers(0, 10 ** 12)),
                   live_regs=int(g.integers(0, 180))) for _ in range(n)]
        model = dict(hbm_bytes_per_s=float(g.uniform(1e11, 8e12)),
                     flops_per_s=float(g.uniform(1e12, 2e15)), launch_s=float(g.uniform(0, 1e-5)),
                     spill_penalty=float(g.uniform(1, 4)), reg_limit=int(g.integers(100, 300)))
        eb = int(g.choice([1, 2, 4]))
        args = (model["hbm_bytes_per_s"], model["flops_per_s"], model["launch_s"],
                model["spill_penalty"], model["reg_limit"])
        for mask in itertools.islice(range(2 ** (n - 1)), 16):
            assert fc.fuse_plan_time(st, mask, eb, model) == pytest.approx(
                op.plan_time(st, mask, eb, *args), rel=1e-12)
        bmask, bsec = fc.fuse_best_plan(st, eb, model)
        omask, osec = op.best_plan(st, eb, *args)
        assert bsec == pytest.approx(osec, rel=1e-12)
        # equal-cost plans may be ordered differently by rounding; the chosen one must be optimal
        assert op.plan_time(st, bmask, eb, *args) == pytest.approx(osec, rel=1e-12)


def test_planner_rejects_bad_arguments():
    st = fc._stages(mlp_epilogue_stages(16, 16, 16))
    lib = fc._load()
    m = fc.fuse_cost_model(**K4_MODEL)
    import ctypes
    out = ctypes.c_double()
    assert lib.fuse_plan_time(st, 4, 8, 2, ctypes.byref(m), ctypes.byref(out)) == fc.FUSE_EINVAL
    assert lib.fuse_plan_time(st, 4, 0, 0, ctypes.byref(m), ctypes.byref(out)) == fc.FUSE_EINVAL
    bad = fc.fuse_cost_model(**dict(K4_MODEL, hbm_bytes_per_s=0.0))
    assert lib.fuse_plan_time(st, 4, 0, 2, ctypes.byref(bad), ctypes.byref(out)) == fc.FUSE_EINVAL
    bad = fc.fuse_cost_model(**dict(K4_MODEL, spill_penalty=0.5))
    assert lib.fuse_plan_time(st, 4, 0, 2, ctypes.byref(bad), ctypes.byref(out)) == fc.FUSE_EINVAL
    mask, sec = ctypes.c_uint32(), ctypes.c_double()
    assert lib.fuse_best_plan(st, 0, 2, ctypes.byref(m), ctypes.byref(mask),
                              ctypes.byref(sec)) == fc.FUSE_EINVAL
