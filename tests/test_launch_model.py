"""Launch timeline model ("AIGC fundamentals | operator fusion and CUDA Graph" §3.4, [F1]/[F2]):
the oracle's event-by-event simulation against the page's printed speed-ups, and the library's
closed form against the oracle.  No GPU needed."""
import numpy as np
import pytest

import epilogue_chains_gb300 as fc
from conftest import read_golden
from oracle import launch_model as lm

N, T_LAUNCH, T_DISP = 700, 3.0, 0.5


@pytest.mark.parametrize("row", read_golden("ofcg_graph_speedups.txt"), ids=lambda r: r[0])
def test_oracle_reproduces_printed_speedups(row):
    te, printed = float(row[0]), float(row[1])
    eager, _ = lm.simulate_eager(N, T_LAUNCH, te)
    graph, _ = lm.simulate_graph(N, T_LAUNCH, te, T_DISP)
    assert f"{eager / graph:.2f}" == f"{printed:.2f}"


def test_oracle_regimes_have_the_stated_closed_forms():
    """§3.4: host-bound (t_launch > t_exec): about N t_launch, the GPU idle for
    1 - t_exec/t_launch of it; GPU-bound: about N t_exec + t_launch."""
    e, idle = lm.simulate_eager(N, 3.0, 1.0)
    assert e == pytest.approx(N * 3.0 + 1.0) and idle == pytest.approx(e - N * 1.0)
    assert idle / e == pytest.approx(1 - 1.0 / 3.0, abs=1e-3)
    e, idle = lm.simulate_eager(N, 3.0, 5.0)
    assert e == pytest.approx(3.0 + N * 5.0) and idle == pytest.approx(3.0)
    # break-even near t_exec = t_launch - t_dispatch: the graph wins below it, loses above it
    assert lm.simulate_eager(N, 3.0, 2.4)[0] > lm.simulate_graph(N, 3.0, 2.4, 0.5)[0]
    assert lm.simulate_eager(N, 3.0, 2.6)[0] < lm.simulate_graph(N, 3.0, 2.6, 0.5)[0]


def test_oracle_brute_force_timeline_on_tiny_cases():
    """Hand-worked: 3 kernels, launch 2, exec 1 -> starts at 2, 4, 6; ends at 7; idle 2+1+1."""
    assert lm.simulate_eager(3, 2.0, 1.0) == (7.0, 4.0)
    assert lm.simulate_eager(3, 1.0, 2.0) == (7.0, 1.0)   # starts 1, 3, 5
    assert lm.simulate_eager(0, 1.0, 2.0) == (0.0, 0.0)
    assert lm.simulate_graph(3, 2.0, 1.0, 0.5) == (6.5, 2.0)


def test_library_matches_oracle():
    g = np.random.default_rng(13)
    for _ in range(200):
        n = int(g.integers(0, 2000))
        tl, te, td = (float(v) for v in g.uniform(0, 10, 3))
        e, idle = lm.simulate_eager(n, tl, te)
        gr, _ = lm.simulate_graph(n, tl, te, td)
        out = fc.fuse_launch_model(n, tl, te, td)
        assert out["eager"] == pytest.approx(e, rel=1e-9, abs=1e-9)
        assert out["eager_idle"] == pytest.approx(idle, rel=1e-6, abs=1e-6)
        assert out["graph"] == pytest.approx(gr, rel=1e-12)


def test_library_rejects_bad_arguments():
    with pytest.raises(fc.FuseError):
        fc.fuse_launch_model(-1, 1.0, 1.0, 1.0)
    with pytest.raises(fc.FuseError):
        fc.fuse_launch_model(4, -1.0, 1.0, 1.0)
