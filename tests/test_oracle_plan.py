"""Pins of the oracle's split plans: hand-computed examples, coverage
invariants and the defining batch-invariance property.  CPU only."""

import random

import pytest

from oracle import plan as P

FMA = P.VARIANT_CONSTANTS["fma"]


def test_invariant_hand_examples():
    # tile 64, >= 16 tiles per split, <= 64 splits (the FMA variant's constants)
    T, mn, mx = FMA
    assert (T, mn, mx) == (64, 16, 64)
    cases = {
        0: [0, 0],                    # empty row: one empty split
        1: [0, 1],
        64: [0, 1],
        1024: [0, 16],                # 16 tiles: exactly one minimum split
        1025: [0, 16, 17],            # 17 tiles: a full split and a 1-tile tail
        4096: list(range(0, 65, 16)), # 64 tiles -> 4 splits of 16
        # 2048 tiles: tps = max(16, ceil(2048 / 64)) = 32 -> 64 splits of 32
        131072: list(range(0, 2049, 32)),
        # 2049 tiles: tps = ceil(2049 / 64) = 33 -> 63 splits of 33 + 2 tiles
        131073: list(range(0, 2049, 33)) + [2049],
    }
    for L, want in cases.items():
        assert P.plan_invariant([L], T, mn, mx) == [want], L


def test_invariant_hand_examples_tensor_core_variant():
    # tile 64, >= 8 tiles per split, <= 32 splits (the MLA variant's constants)
    T, mn, mx = P.VARIANT_CONSTANTS["mla"]
    assert (T, mn, mx) == (64, 8, 32)
    assert P.plan_invariant([2048], T, mn, mx) == [[0, 8, 16, 24, 32]]
    assert P.plan_invariant([513], T, mn, mx) == [[0, 8, 9]]
    assert P.plan_invariant([256], T, mn, mx) == [[0, 4]]


def test_invariant_coverage_and_limits():
    T, mn, mx = FMA
    for L in list(range(0, 3000)) + [131071, 131072, 131073, 1 << 20, 1 << 24]:
        (cuts,) = P.plan_invariant([L], T, mn, mx)
        n_tiles = -(-L // T)
        assert cuts[0] == 0 and cuts[-1] == n_tiles
        n = len(cuts) - 1
        assert 1 <= n <= mx
        sizes = [b - a for a, b in zip(cuts[:-1], cuts[1:])]
        if L == 0:
            assert sizes == [0]
            continue
        assert all(s > 0 for s in sizes)
        tps = sizes[0]
        assert tps >= mn or n == 1
        assert all(s == tps for s in sizes[:-1]) and sizes[-1] <= tps


def test_invariant_plan_of_a_row_does_not_depend_on_its_batch():
    # the defining property: a row's splits are a function of its own length
    rng = random.Random(0)
    T, mn, mx = FMA
    target = 4096
    solo = P.plan_invariant([target], T, mn, mx)[0]
    for B in (1, 2, 7, 64, 256):
        lens = [int(2 ** (17 * rng.random())) for _ in range(B)]
        pos = rng.randrange(B)
        lens[pos] = target
        assert P.plan_invariant(lens, T, mn, mx)[pos] == solo


def test_balanced_hand_example():
    # 3 rows of 10, 1, 20 tiles (tile 1), overhead 2, 4 parts:
    # total = 12 + 3 + 22 = 37, payload = ceil(37 / 4) + 2 = 12.
    # part 0: row 0 (10 + 2 = 12) fills it exactly.
    # part 1: row 1 (1 + 2) leaves room 9; row 2 takes 9 - 2 = 7 tiles, cut at 7.
    # part 2: row 2's remaining 13 + 2 > 12: takes 10 tiles, cut at 17.
    # part 3: remaining 3 + 2 fits.
    got = P.plan_balanced([10, 1, 20], 1, 64, 4, 2)
    assert got == [[0, 10], [0, 1], [0, 7, 17, 20]]


def test_balanced_quota_raised_for_the_longest_row():
    # one row of 4096 tiles (tile 1), 152 parts, overhead 2, 64 splits at most:
    # the page's quota is ceil(4098 / 152) + 2 = 29, which would need 152
    # pieces; raised to ceil(4096 / 63) + 2 = 68, full parts of 66 tiles cut
    # the row into 63 pieces, the last one 4 tiles -- no overloaded split.
    got = P.plan_balanced([4096], 1, 64, 152, 2)[0]
    assert got == list(range(0, 4093, 66)) + [4096]
    assert max(b - a for a, b in zip(got[:-1], got[1:])) == 66
    # when the quota already fits the longest row it is the page's own:
    # total = 100 * (40 + 2) = 4200, 7 parts -> 600 + 2 = 602 (>= 40 / 63 + 2);
    # 14 rows fill 588 of the first part, row 14 takes 14 - 2 = 12 tiles there
    many = P.plan_balanced([40] * 100, 1, 64, 7, 2)
    assert many[13] == [0, 40] and many[14] == [0, 12, 40]


def test_balanced_coverage_and_split_cap():
    rng = random.Random(1)
    for _ in range(200):
        B = rng.randint(1, 40)
        lens = [rng.choice([0, 1, rng.randint(1, 200000)]) for _ in range(B)]
        parts = rng.randint(1, 300)
        mx = rng.choice([1, 2, 8, 64])
        bounds = P.plan_balanced(lens, 64, mx, parts, 2)
        for L, cuts in zip(lens, bounds):
            n_tiles = -(-L // 64)
            assert cuts[0] == 0 and cuts[-1] == n_tiles
            assert 1 <= len(cuts) - 1 <= mx
            assert all(b > a for a, b in zip(cuts[:-1], cuts[1:])) or n_tiles == 0


def test_balanced_split_depends_on_batchmates():
    # the counter-example the page describes: the same row is cut
    # differently when its batchmates change
    solo = P.plan_balanced([4096 // 64], 1, 64, 100, 2)[0]
    mixed = P.plan_balanced([4096 // 64] + [2000] * 50, 1, 64, 100, 2)[0]
    assert solo != mixed


def test_work_list_order():
    # sizes: row 0 split 0: 1 tile; row 1: 2, 1, 1 tiles; row 2: empty.
    # Largest first, batch order within a size.
    bounds = [[0, 1], [0, 2, 3, 4], [0, 0]]
    assert P.work_list(bounds, 64) == [64, 0, 65, 66, 128]
    assert [P.work_key(bounds, 64, w) for w in P.work_list(bounds, 64)] == [2, 1, 1, 1, 0]
    # keys cap at 255
    assert P.work_list([[0, 300], [0, 400]], 8) == [0, 8]
