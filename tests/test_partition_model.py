"""CPU checks of the split-KV partition model (tests/partition_model.py), the
arithmetic the on-device partitioner runs: every (request, row group) KV
range covered exactly once, in order, by contiguous chunks; owners
nondecreasing over the work list; each busy worker within one tile plus one
overhead of its fair share; lanes cutting every lane at the same tiles;
idle workers (past the busy count) with empty ranges."""
import numpy as np
import pytest

from partition_model import MIN_UNITS, OVERHEAD, TILE, ceil_div, partition


def case(rng, B, H, q_fixed=None, max_len=5000):
    q = np.full(B, q_fixed) if q_fixed else rng.integers(1, 9, size=B)
    L = rng.integers(1, max_len, size=B)
    L = np.maximum(L, q)
    qs = np.concatenate([[0], np.cumsum(q)])[:-1]
    return L, q, qs, H


@pytest.mark.parametrize("seed", range(60))
def test_partition_invariants(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 200))
    H = int(rng.choice([16, 32, 64, 128]))
    q_fixed = int(rng.choice([0, 1, 2, 4])) or None
    L, q, qs, H = case(rng, B, H, q_fixed, max_len=int(rng.choice([100, 3000, 40000])))
    n = int(rng.choice([2, 17, 76, 148]))
    items, wb, info = partition(L, q, qs, H, n, L - q)
    # coverage: every group of every request, its KV range in contiguous order
    want = {(b, g): int(L[b]) for b in range(B) for g in range(ceil_div(int(q[b]) * H, 128))}
    seen = {}
    for (b, g, k0, k1, slot, *_rest) in items:
        assert k0 < k1 and k0 % TILE == 0
        assert seen.get((b, g), 0) == k0, (b, g)
        seen[(b, g)] = k1
    assert seen == want
    # owners nondecreasing and ranges consistent
    owners = info["owners"]
    assert all(a <= b for a, b in zip(owners, owners[1:]))
    assert wb[0] == 0 and wb[-1] == len(items) and all(a <= b for a, b in zip(wb, wb[1:]))
    for w in range(n):
        for i in range(wb[w], wb[w + 1]):
            assert owners[i] == w
    # idle workers past the busy count have nothing
    n_eff = info["n_eff"]
    assert n_eff == max(1, min(n, info["W"] // MIN_UNITS))
    busy = info["lanes"] * (n_eff // info["lanes"])
    for w in range(busy, n):
        assert wb[w] == wb[w + 1]
    # balance: a worker's units (tiles of its items + one overhead per item)
    # exceed the fair share by at most one overhead and one tile per boundary
    share = info["W"] / max(1, busy)
    for w in range(busy):
        units = sum(OVERHEAD + ceil_div(k1 - k0, TILE) for (_, _, k0, k1, *_r) in items[wb[w]:wb[w + 1]])
        n_items_w = wb[w + 1] - wb[w]
        assert units <= share + 2 * (OVERHEAD + 1) + OVERHEAD * max(0, n_items_w - 1) + 1, (w, units, share)
    # split groups: slots and combine entries numbered densely
    slots = sorted(s for (_, _, _, _, s, *_r) in items if s >= 0)
    assert slots == list(range(len(slots)))


def test_lanes_cut_every_lane_at_the_same_tiles():
    rng = np.random.default_rng(5)
    L, q, qs, H = case(rng, 32, 128, q_fixed=4, max_len=16000)
    items, wb, info = partition(L, q, qs, H, 76, L - q)
    assert info["lanes"] == 4
    cuts = {}
    for (b, g, k0, k1, *_r) in items:
        cuts.setdefault(g, []).append((b, k0, k1))
    assert cuts[0] == [(b, k0, k1) for (b, k0, k1) in cuts[1]] == cuts[2] == cuts[3]


def test_small_problem_uses_few_workers_and_no_splits():
    """Two short requests (the tiny workload) give about two units of work per
    item: two busy workers, nothing split, so no combine pass."""
    L = np.array([37, 64]); q = np.array([1, 1]); qs = np.array([0, 1])
    items, wb, info = partition(L, q, qs, 16, 76, L - q)
    assert info["n_eff"] == 2
    assert all(s == -1 for (_, _, _, _, s, *_r) in items)
    assert len(items) == 2
