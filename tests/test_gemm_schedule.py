"""The CTA-pair GEMM's tile schedule (host logic, no GPU): whole tiles, and stream-K split tiles that fill
a mostly idle last wave.

The kernel trusts four properties of the schedule it walks: every (tile, K stage) unit is covered exactly
once; a split tile's run at stage 0 sits on some pair c and the rest of the tile is held by the first runs
of pairs c+1 .. c+j, j <= 2 (the kernel reads their partial slots and finds them with the same unit
arithmetic); no pair has more than one run that starts inside a tile (one partial slot per pair); and split
runs come before whole tiles in every pair's order.  These tests check them on the library's own schedule
(lora_debug_gemm_runs), together with the balance the split is for.
"""
import itertools

import pytest

from lora_fine_tuning_gb300 import native

MAX_SPLIT_PARTS = 2   # other runs a split tile's stage-0 run adds (the kernel's partial-slot lookahead)


def tiles_of(M, N, bn):
    return -(-M // 256) * -(-N // bn)


def check_schedule(M, N, bn, stages, max_pairs, allow=True, single_acc=False):
    pairs, split, runs = native.gemm_runs(M, N, bn, stages, max_pairs, allow, single_acc)
    T = tiles_of(M, N, bn)
    assert 1 <= pairs <= max_pairs
    # every unit exactly once, runs non-empty and inside their tile
    seen = {}
    for pair, tile, kb0, kb1 in runs:
        assert 0 <= pair < pairs and 0 <= tile < T and 0 <= kb0 < kb1 <= stages
        for kb in range(kb0, kb1):
            assert (tile, kb) not in seen, f"unit {(tile, kb)} twice"
            seen[(tile, kb)] = pair
    assert len(seen) == T * stages
    by_pair = {c: [r for r in runs if r[0] == c] for c in range(pairs)}
    # per pair: at most one run starting inside a tile, and it is the pair's first; split runs first
    for c, rs in by_pair.items():
        inner = [i for i, r in enumerate(rs) if r[2] > 0]
        assert inner in ([], [0]), f"pair {c}: runs starting inside a tile at {inner}"
        whole = [r[2] == 0 and r[3] == stages and r[1] >= split for r in rs]
        assert all(whole[i] <= whole[i + 1] for i in range(len(whole) - 1)), f"pair {c}: whole tile before a split run"
    # split tiles: one stage-0 run on pair c, the rest on the first runs of pairs c+1 .. c+j, j <= 2,
    # which are exactly the pairs whose unit range starts inside the tile (the kernel's lookup)
    U = split * stages
    for t in range(T):
        parts = sorted((r for r in runs if r[1] == t), key=lambda r: r[2])
        if len(parts) == 1:
            assert parts[0][2:] == (0, stages)
            continue
        assert t < split
        c = parts[0][0]
        assert parts[0][2] == 0
        others = [r[0] for r in parts[1:]]
        assert others == list(range(c + 1, c + 1 + len(others)))
        assert len(others) <= MAX_SPLIT_PARTS
        lookup = [cc for cc in range(c + 1, pairs) if U * cc // pairs < (t + 1) * stages]
        assert lookup == others
        for cc in others:
            assert by_pair[cc][0][1] == t
    return pairs, split, runs


def work_per_pair(runs, pairs):
    w = [0] * pairs
    for pair, _, kb0, kb1 in runs:
        w[pair] += kb1 - kb0
    return w


# (M, N, stages, single accumulator set, split tiles expected): the rule splits where a last wave leaves
# most of the 76 pairs idle, as measured on GB300 (split / whole-tile microseconds in the comments)
CASES = [
    (1024, 4096, 64, False, 0),        # 64 tiles in one wave, 12 pairs idle: splitting lost (35 / 25)
    (1216, 4096, 64, False, 80),       # 80 tiles: 4 in a second wave (34 / 42)
    (1216, 4096, 64, True, 80),        # the backward too (35 / 43)
    (2048, 4096, 64, False, 0),        # 128 tiles: 52 of 76 in the second wave (48 / 44)
    (4096, 4096, 64, False, 104),      # 256 tiles: 3 waves + 28 (86 / 91)
    (4096, 4096, 64, True, 0),         # backward, one accumulator set (99 / 95)
    (4864, 4096, 64, False, 0),        # 304 tiles: exactly 4 waves
    (16384, 4096, 64, False, 112),     # 1024 tiles: 13 waves + 36 (318 / 326)
    (32768, 4096, 64, False, 0),       # 2048 tiles: + 72 (643 / 630)
    (8192, 14336, 64, False, 0),       # the 8B up-proj forward: 1792 tiles, + 44
    (8192, 4096, 224, True, 0),        # its backward: 512 tiles of 224 stages, + 56
    (256, 256, 16, False, 0),          # one tile of 16 stages: too shallow to split
    (256, 256, 32, False, 1),          # one tile of 32 stages: split in two
    (256, 4096, 64, True, 16),         # 16 tiles: each split in two (28 / 29)
    (8192, 1024, 64, False, 0),        # 128 tiles
    (300, 512, 9, False, 0),           # ragged, few stages
    (300, 512, 40, False, 4),          # ragged: four tiles, each split in two
    (2560, 4096, 16, False, 0),        # 160 tiles (two waves + 8) of 16 stages: splitting lost (29 / 25)
    (2560, 4096, 32, False, 84),       # the same at 32 stages
    (16384, 28672, 128, False, 0),     # the 70B up-proj forward: 7168 tiles + 24, 128 stages (4619 / 4607)
    (4096, 4096, 128, False, 0),       # 256 tiles + 28 at 128 stages: the staggered runs cost more
]


@pytest.mark.parametrize("M,N,stages,single,expect", CASES)
def test_schedule_rule_properties_and_balance(M, N, stages, single, expect):
    pairs, split, runs = check_schedule(M, N, 256, stages, 76, single_acc=single)
    assert split == expect
    T = tiles_of(M, N, 256)
    w = work_per_pair(runs, pairs)
    if split:
        # the units are spread evenly: no pair has more than one unit beyond any other
        assert max(w) - min(w) <= 1
        assert max(w) < -(-T // 76) * stages   # less than the whole-tile schedule's busiest pair
    else:
        assert pairs == min(T, 76)
        assert max(w) == -(-T // pairs) * stages


def test_no_split_when_not_allowed_or_few_stages():
    pairs, split, runs = check_schedule(4096, 4096, 256, 64, 76, allow=False)
    assert split == 0 and pairs == 76
    assert all(kb0 == 0 and kb1 == 64 for _, _, kb0, kb1 in runs)
    assert [t for c, t, _, _ in runs if c == 5] == list(range(5, 256, 76))
    pairs, split, _ = check_schedule(4096, 4096, 256, 31, 76)   # fewer than 32 stages: whole tiles
    assert split == 0


def test_exhaustive_small_grids():
    """Every tile count up to 3 waves of small grids, and stage counts around the split limits."""
    for max_pairs, stages, single in itertools.product((1, 2, 3, 7, 16, 76), (16, 32, 33, 64, 65), (False, True)):
        for n_tiles in range(1, 3 * max_pairs + 2):
            check_schedule(256 * n_tiles, 256, 256, stages, max_pairs, single_acc=single)


def test_rejects_bad_arguments():
    lib = native.lib()
    import ctypes
    p, s, n = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
    assert lib.lora_debug_gemm_runs(0, 256, 256, 8, 76, 1, 0, ctypes.byref(p), ctypes.byref(s), None, 0,
                                    ctypes.byref(n)) == 1
    assert lib.lora_debug_gemm_runs(256, 256, 256, 8, 76, 1, 0, None, ctypes.byref(s), None, 0,
                                    ctypes.byref(n)) == 1
    assert lib.lora_debug_gemm_runs(256, 256, 256, 8, 76, 1, 0, ctypes.byref(p), ctypes.byref(s), None, 4,
                                    ctypes.byref(n)) == 1
