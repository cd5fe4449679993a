"""Host arithmetic of the persistent attention kernel's work lists (fuse_attention_schedule, no
GPU): every tile pair is assigned exactly once, each cluster's list keeps the global order, and
the estimated finish times of the clusters are balanced (10 per key block + 8 per pair), at least
as well as by the plain one-after-another assignment that the same-group trades start from."""
import numpy as np
import pytest

import epilogue_chains_gb300 as fc


def _key_blocks(i, bh, per_head):
    """Key blocks of item i in the documented order: groups of 16 slices, heaviest pair first."""
    g = i // (16 * per_head)
    gs = min(16, bh - 16 * g)
    r = i - 16 * per_head * g
    u = per_head - 1 - r // gs
    return 2 * u + 2


def _cost(i, bh, per_head):
    return 10 * _key_blocks(i, bh, per_head) + 8


def _greedy_max(bh, S, clusters):
    """Busiest cluster's load when every pair, in order, goes to the least loaded cluster."""
    per_head = S // 256
    load = np.zeros(clusters)
    for i in range(bh * per_head):
        load[int(np.argmin(load))] += _cost(i, bh, per_head)
    return load.max()


def _loads(bh, S, clusters):
    first, items = fc.fuse_attention_schedule(bh, S, clusters)
    per_head = S // 256
    cost = [sum(_cost(i, bh, per_head) for i in items[first[c]:first[c + 1]]) for c in range(clusters)]
    return first, items, np.array(cost, dtype=np.float64)


@pytest.mark.parametrize("bh,S,clusters", [(128, 2048, 76), (32, 2048, 76), (160, 256, 76),
                                           (97, 512, 74), (1, 512, 2), (5, 4096, 9), (16, 8192, 76)])
def test_every_item_once_in_order(bh, S, clusters):
    first, items = fc.fuse_attention_schedule(bh, S, clusters)
    n = bh * S // 256
    assert first[0] == 0 and first[-1] == n and len(first) == clusters + 1
    assert all(first[c] <= first[c + 1] for c in range(clusters))
    assert sorted(items) == list(range(n))
    for c in range(clusters):
        seg = items[first[c]:first[c + 1]]
        assert seg == sorted(seg)


def test_benchmarked_shape_is_balanced():
    """[128, 2048] on 76 clusters: the busiest cluster within 1 % of the mean (one pair after
    another: 2 %; round-robin: more than 10 %)."""
    _, _, cost = _loads(128, 2048, 76)
    assert cost.max() <= 1.01 * cost.mean()
    assert _greedy_max(128, 2048, 76) > 1.015 * cost.mean()
    n = 128 * 8
    rr = np.zeros(76)
    for i in range(n):
        rr[i % 76] += _cost(i, 128, 8)
    assert rr.max() > 1.10 * rr.mean()


@pytest.mark.parametrize("bh,S,clusters", [(128, 2048, 76), (128, 2048, 74), (32, 2048, 76),
                                           (97, 512, 74), (5, 4096, 9), (16, 8192, 76)])
def test_trades_never_unbalance(bh, S, clusters):
    """The trades only ever narrow the gap between the busiest and the idlest cluster."""
    _, _, cost = _loads(bh, S, clusters)
    assert cost.max() <= _greedy_max(bh, S, clusters)


def test_greedy_rule_on_tiny_cases():
    # two pairs of one slice (4 and 2 key blocks), two clusters: one each, heaviest to cluster 0
    first, items = fc.fuse_attention_schedule(1, 512, 2)
    assert first == [0, 1, 2] and items == [0, 1]
    # one cluster takes everything
    first, items = fc.fuse_attention_schedule(3, 256, 1)
    assert first == [0, 3] and items == [0, 1, 2]
    # 16 slices of 2 pairs on 3 clusters: the 16 heavy items (cost 48) spread first, then the light
    # ones (28) go to whichever cluster is least loaded
    _, _, cost = _loads(16, 512, 3)
    assert cost.max() - cost.min() <= 48


def test_arguments():
    for bh, S, cl in [(0, 256, 4), (2, 300, 4), (2, 128, 4), (2, 256, 0)]:
        with pytest.raises(fc.FuseError):
            fc.fuse_attention_schedule(bh, S, cl)
    with pytest.raises(fc.FuseError):
        fc.fuse_attention_schedule(2, 256, 97)          # more clusters than the lists hold
    with pytest.raises(fc.FuseError):
        fc.fuse_attention_schedule(4097, 256, 76)       # more items than the lists hold
