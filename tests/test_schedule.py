"""CPU tests of the decode scheduler's partition (kvarn_partition_units).

A decode call spreads its (sequence, KV head) blocks over CTAs as ranges of scheduling
units; the exact part and the seal of a block (its head) must go whole to one CTA, the
one that does that work. The partition is pinned against an exhaustive dynamic program
over every valid cut set on small lines, and its invariants are checked on lines of the
decode workloads' shapes.
"""
import functools
import random

import pytest

from quantized_kv_cache_seal_gb300 import kvarn as K


def _allowed(units, head):
    """Cut positions strictly inside (0, total) that fall inside no head."""
    begin = [0]
    for u in units:
        begin.append(begin[-1] + u)
    total = begin[-1]
    banned = set()
    for b, h in zip(begin, head):
        banned.update(range(b + 1, b + h))
    return [x for x in range(1, total) if x not in banned], begin, total


def _check_valid(units, head, cuts, max_ctas, max_span):
    allowed, begin, total = _allowed(units, head)
    assert cuts[0] == 0 and cuts[-1] == total
    n = len(cuts) - 1
    assert 1 <= n <= max_ctas
    assert all(a < b for a, b in zip(cuts, cuts[1:])), "empty range"
    assert all(c in allowed for c in cuts[1:-1]), "cut inside a head"
    for k in range(len(units)):
        a, z = begin[k], begin[k + 1] - 1
        ca = max(i for i in range(n) if cuts[i] <= a)
        cz = max(i for i in range(n) if cuts[i] <= z)
        assert cz - ca + 1 <= max_span, f"block {k} spans {cz - ca + 1} CTAs"
    return max(b - a for a, b in zip(cuts, cuts[1:]))


def _optimal(units, head, max_ctas):
    """Smallest largest range over every valid cut set of at most max_ctas ranges
    (dynamic program over the allowed cut positions)."""
    allowed, _, total = _allowed(units, head)
    pts = [0] + allowed + [total]

    @functools.lru_cache(maxsize=None)
    def best(i, c):  # ranges covering pts[i] .. total with at most c ranges
        if pts[i] == total:
            return 0
        if c == 0:
            return float("inf")
        out = float("inf")
        for j in range(i + 1, len(pts)):
            out = min(out, max(pts[j] - pts[i], best(j, c - 1)))
        return out

    return best(0, max_ctas)


@pytest.mark.parametrize("seed", range(40))
def test_partition_matches_exhaustive_optimum(seed):
    rng = random.Random(seed)
    nb = rng.randint(1, 6)
    units = [rng.randint(1, 9) for _ in range(nb)]
    head = [rng.randint(1, u) for u in units]
    max_ctas = rng.randint(1, 8)
    cuts = K.kvarn_partition_units(units, head, max_ctas, 64, 1)
    got = _check_valid(units, head, cuts, max_ctas, 64)
    assert got == _optimal(units, head, max_ctas), (units, head, max_ctas, cuts)


def test_min_load_limits_the_number_of_ctas():
    cuts = K.kvarn_partition_units([100] * 4, [2] * 4, 152, 32, 24)
    assert max(b - a for a, b in zip(cuts, cuts[1:])) == 24
    assert len(cuts) - 1 == -(-400 // 24)


def test_headline_shape_is_even_and_seal_heads_stay_whole():
    # 16 sequences x 8 KV heads at ~32k: 8 exact units + 254 groups; one sequence seals
    # (head 8 + 140) in this call
    units, head = [], []
    for s in range(16):
        for h in range(8):
            seal = 140 if s == 5 else 0
            units.append(8 + seal + 254)
            head.append(8 + seal)
    cuts = K.kvarn_partition_units(units, head, 152, 32, 24)
    largest = _check_valid(units, head, cuts, 152, 32)
    total = sum(units)
    assert largest <= -(-total // 152) + max(head)
    # every seal head lies inside one CTA's range
    begin = 0
    for u, hd in zip(units, head):
        ca = max(i for i in range(len(cuts) - 1) if cuts[i] <= begin)
        assert cuts[ca + 1] >= begin + hd
        begin += u


def test_span_limit_binds_on_one_long_block():
    # one block of 10000 units over up to 152 CTAs: at most 32 of them may share it
    cuts = K.kvarn_partition_units([10000], [4], 152, 32, 24)
    assert len(cuts) - 1 <= 32
    _check_valid([10000], [4], cuts, 152, 32)


@pytest.mark.parametrize("units,head,max_ctas,max_span,min_load", [
    ([], [], 4, 32, 1),          # no block
    ([5], [6], 4, 32, 1),        # head longer than its block
    ([5], [0], 4, 32, 1),        # empty head
    ([0], [0], 4, 32, 1),        # empty block
    ([5], [1], 0, 32, 1),        # no CTA
    ([5], [1], 4, 0, 1),         # no span
])
def test_partition_rejects_bad_arguments(units, head, max_ctas, max_span, min_load):
    with pytest.raises(K.KVarNError) as e:
        K.kvarn_partition_units(units, head, max_ctas, max_span, min_load)
    assert e.value.status == 1


def _cost(begin, a, b, item_cost):
    """Units of range [a, b) plus item_cost for every block it touches beyond its first two."""
    blocks = sum(1 for k in range(len(begin) - 1) if begin[k] < b and begin[k + 1] > a)
    return (b - a) + item_cost * max(0, blocks - 2)


def _optimal_cost(units, head, max_ctas, item_cost):
    """Smallest largest range cost over every valid cut set of at most max_ctas ranges."""
    allowed, begin, total = _allowed(units, head)
    pts = [0] + allowed + [total]

    @functools.lru_cache(maxsize=None)
    def best(i, c):
        if pts[i] == total:
            return 0
        if c == 0:
            return float("inf")
        return min(max(_cost(begin, pts[i], pts[j], item_cost), best(j, c - 1)) for j in range(i + 1, len(pts)))

    return best(0, max_ctas)


@pytest.mark.parametrize("seed", range(60))
def test_partition_with_block_cost_matches_exhaustive_optimum(seed):
    """With a cost per block beyond a range's second (the decode CTA's on-demand query
    tables), the greedy fill at the bisected bound is still the exhaustive optimum."""
    rng = random.Random(1000 + seed)
    nb = rng.randint(1, 9)
    units = [rng.randint(1, 7) for _ in range(nb)]
    head = [rng.randint(1, u) for u in units]
    max_ctas = rng.randint(1, 5)
    item_cost = rng.randint(1, 6)
    cuts = K.kvarn_partition_units(units, head, max_ctas, 64, 1, item_cost)
    _check_valid(units, head, cuts, max_ctas, 64)
    _, begin, _ = _allowed(units, head)
    got = max(_cost(begin, a, b, item_cost) for a, b in zip(cuts, cuts[1:]))
    assert got == _optimal_cost(units, head, max_ctas, item_cost), (units, head, max_ctas, item_cost, cuts)
