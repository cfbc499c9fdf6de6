"""Pins of the oracle's greedy token-capacity packer (first-fit decreasing).

Checked against things other than the packer itself: a placement worked out by
hand, the sum-of-sizes lower bound, the published worst-case bound of first-fit
decreasing against the optimum found by exhaustive search on small inputs, and
closed forms for inputs where the optimum is known.
"""
import itertools
import math
import random

import pytest

from oracle import lora_oracle as O


def check_valid(lengths, capacity, batch, row, n):
    sizes = [O.padded_rows(x) for x in lengths]
    assert len(batch) == len(row) == len(lengths)
    assert all(0 <= b < n for b in batch)
    assert set(batch) == set(range(n))            # no empty microbatch
    for b in range(n):
        members = sorted((row[i], sizes[i]) for i in range(len(lengths)) if batch[i] == b)
        pos = 0
        for r, s in members:                      # samples tile the microbatch from row 0, no gaps or overlap
            assert r == pos and r % 128 == 0
            pos += s
        assert pos <= capacity


def test_hand_worked_placement():
    # capacity 1024 rows.  Padded sizes: 700->768, 600->640, 300->384, 260->384, 200->256, 100->128, 90->128.
    # Longest first: 768 opens #0 (256 left); 640 opens #1 (384 left); 384 (sample 2) fits #1 (0 left);
    # 384 (sample 3) fits neither and opens #2 (640 left); 256 fits #0 (0 left); 128 (sample 5) fits #2 at
    # row 384; 128 (sample 6) fits #2 at row 512.  Three microbatches = ceil(2688 / 1024): optimal.
    lengths = [700, 600, 300, 260, 200, 100, 90]
    batch, row, n = O.greedy_pack(lengths, 1024)
    assert n == 3
    assert batch == [0, 1, 1, 2, 0, 2, 2]
    assert row == [0, 0, 640, 0, 768, 384, 512]


def test_padding_to_tiles():
    assert [O.padded_rows(x) for x in (1, 127, 128, 129, 256, 257)] == [128, 128, 128, 256, 256, 384]


def test_rejects():
    with pytest.raises(ValueError):
        O.greedy_pack([10], 100)            # capacity not a multiple of 128
    with pytest.raises(ValueError):
        O.greedy_pack([300], 256)           # sample longer than a microbatch
    with pytest.raises(ValueError):
        O.greedy_pack([0], 256)


def brute_force_optimum(sizes, capacity):
    """Fewest bins by exhaustive search (small inputs only)."""
    best = len(sizes)
    sizes = sorted(sizes, reverse=True)

    def place(i, bins):
        nonlocal best
        if len(bins) >= best:
            return
        if i == len(sizes):
            best = len(bins)
            return
        tried = set()
        for b in range(len(bins)):
            if bins[b] + sizes[i] <= capacity and bins[b] not in tried:
                tried.add(bins[b])
                bins[b] += sizes[i]
                place(i + 1, bins)
                bins[b] -= sizes[i]
        bins.append(sizes[i])
        place(i + 1, bins)
        bins.pop()

    place(0, [])
    return best


@pytest.mark.parametrize("seed", range(40))
def test_within_ffd_worst_case_bound_of_optimum(seed):
    # Dosa (2007): FFD(I) <= 11/9 OPT(I) + 6/9 for every instance, and never below the optimum.
    rng = random.Random(seed)
    capacity = 128 * rng.choice([4, 6, 8, 10])
    lengths = [rng.randint(1, capacity) for _ in range(rng.randint(1, 8))]
    batch, row, n = O.greedy_pack(lengths, capacity)
    check_valid(lengths, capacity, batch, row, n)
    opt = brute_force_optimum([O.padded_rows(x) for x in lengths], capacity)
    assert opt <= n <= 11 * opt / 9 + 6 / 9 + 1e-9


@pytest.mark.parametrize("seed", range(10))
def test_lognormal_samples_valid_and_above_lower_bound(seed):
    rng = random.Random(100 + seed)
    lengths = [int(min(2048, max(64, round(rng.lognormvariate(6.2, 0.6))))) for _ in range(200)]
    capacity = 16384
    batch, row, n = O.greedy_pack(lengths, capacity)
    check_valid(lengths, capacity, batch, row, n)
    total = sum(O.padded_rows(x) for x in lengths)
    assert n >= math.ceil(total / capacity)
    # first fit leaves at most one microbatch at most half full: the items of a later such microbatch
    # would each have fitted into an earlier one when they were placed
    fills = [0] * n
    for i, b in enumerate(batch):
        fills[b] += O.padded_rows(lengths[i])
    assert sum(1 for f in fills if f <= capacity // 2) <= 1


def test_closed_forms():
    # every sample above half the capacity: one per microbatch
    assert O.greedy_pack([600, 700, 520, 1000], 1024)[2] == 4
    # equal sizes s: ceil(n / floor(C / s)) microbatches
    for s_tiles, cap_tiles, count in itertools.product((1, 2, 3), (4, 7, 8), (1, 5, 13)):
        n = O.greedy_pack([128 * s_tiles] * count, 128 * cap_tiles)[2]
        assert n == math.ceil(count / (cap_tiles // s_tiles))
