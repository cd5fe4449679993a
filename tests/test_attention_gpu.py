"""Parity of the causal attention kernel (tcgen05, no score matrix) against the CPU oracle
(plain causal softmax(scale q k^T) v in double), through the C ABI.

Bar per output element: P is rounded to bf16 before it multiplies V (relative 2^-9 per weight),
the row sum uses the unrounded weights, the scores and O accumulate in fp32 and O is rounded once
to bf16, so |O - ref| <= 2^-8 max_j<=i |v_j| + 2^-8 |ref| (per column), and the RMS error stays
at the level of the bf16 rounding of P (2^-9 of the values' RMS).  Row 0 of every slice sees only
key 0 and must equal v_0 bit for bit."""
import numpy as np
import pytest

import epilogue_chains_gb300 as fc
import oracle
from epilogue_chains_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _f(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _run(q, k, v, scale):
    import torch
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    fc.fuse_attention(_dev(q), _dev(k), _dev(v), o, scale)
    torch.cuda.synchronize()
    assert fc.fuse_check() == fc.FUSE_OK
    return o.cpu().view(torch.int16).numpy().view(np.uint16)


def _check(o, ref, v, rows=None):
    od, rd, vd = _f(o), _f(ref), _f(v)
    assert np.all(np.isfinite(od))
    S = v.shape[1]
    rows = np.arange(S) if rows is None else np.asarray(rows)
    vmax = np.maximum.accumulate(np.abs(vd), axis=1)[:, rows]          # max_j<=i |v_j| per column
    err = np.abs(od - rd)
    bound = 2.0 ** -8 * vmax + 2.0 ** -8 * np.abs(rd) + 2.0 ** -133
    bad = err > bound
    assert not bad.any(), (int(bad.sum()), float(err.max()), np.argwhere(bad)[:4].tolist())
    assert np.sqrt(np.mean(err ** 2)) <= 2.0 ** -9 * np.sqrt(np.mean(vd ** 2))


# (bh, S, D): an even number of 128-row query tiles at D = 128 / 256 runs the 2-SM kernel, an odd
# number (or D = 64) the one-CTA kernel
@pytest.mark.parametrize("shape", [(2, 256, 256), (1, 128, 64), (3, 384, 128), (2, 512, 256),
                                   (1, 384, 256), (5, 256, 128), (2, 1024, 64)])
def test_small_shapes_every_row(cuda_device, shape):
    bh, S, D = shape
    q, k, v = wl.attention_input(bh, S, D, salt=S + D)
    scale = 1.0 / np.sqrt(D)
    o = _run(q, k, v, scale)
    _check(o, oracle.attention(q, k, v, scale), v)
    assert np.array_equal(o[:, 0], v[:, 0])


@pytest.mark.parametrize("shape", [(160, 256, 128), (97, 512, 256), (12, 4096, 256), (24, 4096, 128)])
def test_more_tile_pairs_than_resident_clusters(cuda_device, shape):
    """More (slice, tile pair) items than clusters fit on the GPU (~74): each cluster walks
    several items of different lengths (at S = 4096 up to 32 key blocks each), and the counts per
    cluster are uneven.  The first, second and last rows of every 128-row tile and a few random
    rows are checked in every slice."""
    bh, S, D = shape
    q, k, v = wl.attention_input(bh, S, D, salt=7 * S + D)
    scale = 1.0 / np.sqrt(D)
    o = _run(q, k, v, scale)
    t0 = np.arange(0, S, 128)
    rows = np.unique(np.concatenate([t0, t0 + 1, t0 + 127, np.random.default_rng(S).integers(0, S, 4)]))
    _check(o[:, rows], oracle.attention(q, k, v, scale, rows=rows), v, rows)
    assert np.array_equal(o[:, 0], v[:, 0])


def test_full_size_every_row(cuda_device):
    """[128, 2048, 256] as benchmarked: every row of all 128 slices against the oracle, which
    runs on several host threads, one slice per task (about a minute on the GPU machine's cores)."""
    import concurrent.futures as cf
    import os
    q, k, v = wl.attention_input()
    o = _run(q, k, v, wl.ATT_SCALE)
    workers = max(1, min(16, (os.cpu_count() or 2) - 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        futs = {ex.submit(oracle.attention, q[b:b + 1], k[b:b + 1], v[b:b + 1], wl.ATT_SCALE): b
                for b in range(q.shape[0])}
        for f in cf.as_completed(futs):
            b = futs[f]
            _check(o[b:b + 1], f.result(), v[b:b + 1])
    assert np.array_equal(o[:, 0], v[:, 0])


def test_sharp_queries_select_exactly_one_value_row(cuda_device):
    """Keys 0..63 are the unit vectors, keys 64..127 zero; query i points at key sel(i) <= i with
    score 32 against 0 elsewhere, so O_i = v_sel(i) bit for bit."""
    S, D = 128, 64
    k = np.zeros((S, D))
    k[:64] = np.eye(64)
    g = np.random.default_rng(22)
    sel = np.array([g.integers(0, min(i, 63) + 1) for i in range(S)])
    q = np.zeros((S, D))
    q[np.arange(S), sel] = 32.0
    qb, kb = wl.bf16_bits_from_f32(q.astype(np.float32)), wl.bf16_bits_from_f32(k.astype(np.float32))
    v = wl.attention_input(1, S, D, salt=23)[2][0]
    o = _run(qb[None], kb[None], v[None], 1.0)[0]
    assert np.array_equal(o, v[sel])


@pytest.mark.parametrize("D", [64, 128, 256])
def test_growing_scores_rescale_every_block(cuda_device, D):
    """Scores that rise by 64 (natural units) per 128-key block force the O rescale in every block
    of every row; large magnitudes also exercise the far tails of exp.  D = 64 runs the one-CTA
    kernel, D = 128 and 256 the 2-SM kernel (four query tiles: two pairs)."""
    S = 512
    k = np.zeros((S, D), np.float32)
    k[:, 0] = np.arange(S) / 2.0                      # rounded to bf16 below; both sides see it
    g = np.random.default_rng(24)
    q = g.standard_normal((S, D)).astype(np.float32) * 0.1
    q[:, 0] = 1.0
    qb, kb = wl.bf16_bits_from_f32(q), wl.bf16_bits_from_f32(k)
    v = wl.attention_input(1, S, D, salt=25)[2]
    o = _run(qb[None], kb[None], v, 1.0)
    _check(o, oracle.attention(qb[None], kb[None], v, 1.0), v)


def test_large_scale_and_wide_values(cuda_device):
    q, k, v = wl.attention_input(2, 256, 128, salt=26)
    o = _run(q, k, v, 0.5)              # sharper softmax than 1/sqrt(D)
    _check(o, oracle.attention(q, k, v, 0.5), v)


def test_rejects_unsupported_and_bad_arguments(cuda_device):
    import torch
    lib = fc._load()
    t = torch.zeros(2, 256, 256, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(t)
    p = t.data_ptr()
    assert lib.fuse_attention(p, p, p, o.data_ptr(), 2, 200, 256, 0.1, None) == fc.FUSE_EUNSUPPORTED
    assert lib.fuse_attention(p, p, p, o.data_ptr(), 2, 128, 96, 0.1, None) == fc.FUSE_EUNSUPPORTED
    assert lib.fuse_attention(p + 2, p, p, o.data_ptr(), 1, 128, 256, 0.1, None) == fc.FUSE_EALIGN
    assert lib.fuse_attention(p, p, p, p, 1, 128, 256, 0.1, None) == fc.FUSE_EINVAL      # o over q
    assert lib.fuse_attention(p, p, p, o.data_ptr(), 1, 128, 256, 0.0, None) == fc.FUSE_EINVAL
    assert lib.fuse_attention(p, p, p, o.data_ptr(), 0, 128, 256, 0.1, None) == fc.FUSE_OK


def test_repeated_calls_and_graph_replays(cuda_device):
    """Back-to-back calls on one stream and the replays of one captured call give the first call's
    result bit for bit: the persistent kernel keeps no state between launches that could change
    which item a cluster runs or how.  160 slices of S = 512: 320 items on ~76 clusters."""
    import torch
    bh, S, D = 160, 512, 256
    q, k, v = wl.attention_input(bh, S, D, salt=3)
    qd, kd, vd = _dev(q), _dev(k), _dev(v)
    ref = _run(q, k, v, 1.0 / 16)
    s = torch.cuda.Stream()
    o = torch.empty_like(qd)
    for _ in range(3):
        o.fill_(float("nan"))
        fc.fuse_attention(qd, kd, vd, o, 1.0 / 16, stream=s)
        s.synchronize()
        assert fc.fuse_check() == fc.FUSE_OK
        assert np.array_equal(o.cpu().view(torch.int16).numpy().view(np.uint16), ref)
    o.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        fc.fuse_graph_begin(s)
        try:
            fc.fuse_attention(qd, kd, vd, o, 1.0 / 16, stream=s)
        finally:
            g = fc.fuse_graph_end(s)
    try:
        assert torch.isnan(o.float()).all(), "capturing must not run the kernel"
        for _ in range(3):
            o.fill_(float("nan"))
            torch.cuda.synchronize()
            fc.fuse_graph_launch(g, s)
            s.synchronize()
            assert fc.fuse_check(s) == fc.FUSE_OK
            assert np.array_equal(o.cpu().view(torch.int16).numpy().view(np.uint16), ref)
    finally:
        fc.fuse_graph_destroy(g)
