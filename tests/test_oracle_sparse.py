"""Pins of the oracle's sparse row-list builder: hand-worked lists, brute
force over every subset on tiny inputs, and invariants."""
import itertools

import numpy as np

import oracle
import synth


def test_hand_worked_list():
    # positions 0..9; sinks 2, recent 3 -> middle 2..6; top-2 by score: 5 (0.9), 3 (0.7)
    score = np.array([[0.0, 0.0, 0.1, 0.7, 0.2, 0.9, 0.3, 0.0, 0.0, 0.0]], np.float32)
    got = oracle.select_rows(score, sinks=2, recent=3, k=2, list_len=9)
    assert got.tolist() == [[0, 1, 3, 5, 7, 8, 9, -1, -1]]


def test_ties_go_to_the_smaller_position_and_nan_ranks_last():
    score = np.array([[5.0, 1.0, np.nan, 1.0, 1.0, 0.5, 9.0]], np.float32)
    # sinks 1, recent 1 -> middle 1..5 = [1.0, nan, 1.0, 1.0, 0.5]; top-2 -> positions 1, 3
    assert oracle.select_rows(score, 1, 1, 2, 6).tolist() == [[0, 1, 3, 6, -1, -1]]
    # top-4 -> 1, 3, 4 (the ones), then 5 (0.5); the NaN stays out
    assert oracle.select_rows(score, 1, 1, 4, 6).tolist() == [[0, 1, 3, 4, 5, 6]]
    # top-5 needs the NaN
    assert oracle.select_rows(score, 1, 1, 5, 7).tolist() == [[0, 1, 2, 3, 4, 5, 6]]


def test_signed_zeros_tie_and_go_to_the_smaller_position():
    # -0.0 and +0.0 are equal numbers: middle 1..2 = [-0.0, +0.0], top-1 -> position 1
    score = np.array([[9.0, -0.0, 0.0, 9.0]], np.float32)
    assert oracle.select_rows(score, 1, 1, 1, 3).tolist() == [[0, 1, 3]]
    score = np.array([[9.0, 0.0, -0.0, 9.0]], np.float32)
    assert oracle.select_rows(score, 1, 1, 1, 3).tolist() == [[0, 1, 3]]
    # four zeros of mixed sign below a 1.0: top-3 -> the 1.0 and the first two zeros
    score = np.array([[0.0, -0.0, 0.0, 1.0, -0.0, 0.0, 0.0]], np.float32)
    assert oracle.select_rows(score, 0, 0, 3, 3).tolist() == [[0, 1, 3]]


def test_short_slices_list_every_position():
    score = np.zeros((3, 8), np.float32)
    got = oracle.select_rows(score, sinks=4, recent=4, k=2, list_len=10, n_len=np.array([3, 8, 0]))
    assert got[0].tolist() == [0, 1, 2] + [-1] * 7
    assert got[1].tolist() == list(range(8)) + [-1, -1]      # no middle positions
    assert got[2].tolist() == [-1] * 10


def test_row_map_translates_positions():
    score = np.array([[0.0, 3.0, 1.0, 2.0, 0.0]], np.float32)
    row_map = np.array([[40, 41, 17, 99, 5]], np.int32)
    # sinks 1, recent 1 -> middle 1..3, top-1 = position 1
    assert oracle.select_rows(score, 1, 1, 1, 4, row_map=row_map).tolist() == [[40, 41, 5, -1]]


def test_brute_force_over_all_subsets():
    g = synth.rng(77)
    for trial in range(40):
        n = int(g.integers(1, 12))
        sinks, recent, k = int(g.integers(0, 3)), int(g.integers(0, 3)), int(g.integers(0, 5))
        # small integer scores force ties
        score = g.integers(-2, 3, size=(1, n)).astype(np.float32)
        got = oracle.select_rows(score, sinks, recent, k, n)[0]
        lo = min(sinks, n)
        hi = max(lo, n - recent)
        middle = list(range(lo, hi))
        if len(middle) <= k:
            best = middle
        else:
            # the subset of size k with the largest score sum, ties -> lexicographically smallest positions
            best = None
            for sub in itertools.combinations(middle, k):
                key = (-sum(float(score[0, p]) for p in sub), sub)
                if best is None or key < best[0]:
                    best = (key, sub)
            best = list(best[1])
        want = list(range(lo)) + best + list(range(hi, n))
        assert got[:len(want)].tolist() == want and (got[len(want):] == -1).all(), (trial, score, got, want)


def test_invariants_at_the_sparse_workload_size():
    g = synth.rng(78)
    n = 262144
    score = g.standard_normal((1, n)).astype(np.float32)
    got = oracle.select_rows(score, sinks=4, recent=512, k=1532, list_len=2048)[0]
    assert (np.diff(got) > 0).all() and got.size == 2048
    assert got[:4].tolist() == [0, 1, 2, 3] and got[-512:].tolist() == list(range(n - 512, n))
    mid = got[4:-512]
    # every chosen middle score is >= every unchosen middle score
    chosen = np.zeros(n, bool)
    chosen[mid] = True
    inner = np.arange(4, n - 512)
    assert score[0, inner][chosen[inner]].min() >= score[0, inner][~chosen[inner]].max()
