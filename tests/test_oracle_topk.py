"""Pins of the oracle's top-k drifting clusters and position compaction."""
import itertools

import numpy as np

from oracle import topk_drift


def test_hand_worked():
    D = np.array([0.1, 0.5, 0.2, 0.9, 0.0, 0.3], np.float32)
    a = np.array([0, 1, 0, 2, 1, 3])
    counts = np.array([2, 2, 1, 1, 0])
    # means: c0 0.15, c1 0.25, c2 0.9, c3 0.3, c4 empty
    sel, sc, pos, npos, mask, _ = topk_drift(D, a, counts, 2)
    assert list(sel) == [2, 3]
    assert np.allclose(sc, [0.9, 0.3])
    assert npos == 2 and list(pos[:2]) == [3, 5] and np.all(pos[2:] == -1)
    assert list(mask) == [0, 0, 0, 1, 0, 1]


def test_brute_force_best_subset():
    rng = np.random.default_rng(0)
    for trial in range(30):
        N, C = 40, 6
        a = rng.integers(0, C, N)
        counts = np.bincount(a, minlength=C)
        D = rng.random(N).astype(np.float32)
        k = int(rng.integers(1, C + 1))
        sel, _, _, npos, mask, _ = topk_drift(D, a, counts, k)
        live = [c for c in range(C) if counts[c]]
        mean = {c: sum(float(D[i]) for i in range(N) if a[i] == c) / counts[c] for c in live}
        kk = min(k, len(live))
        best = max(itertools.combinations(live, kk), key=lambda s: sum(mean[c] for c in s))
        assert set(sel[:kk]) == set(best)
        assert np.all(sel[kk:] == -1)
        assert npos == sum(counts[c] for c in best) == mask.sum()


def test_k_equals_c_and_all_zero_drift():
    a = np.array([3, 0, 3, 1])
    counts = np.array([1, 1, 0, 2])
    sel, sc, pos, npos, _, _ = topk_drift(np.zeros(4, np.float32), a, counts, 4)
    assert list(sel) == [0, 1, 3, -1]            # ties by index; empty c2 padded
    assert sc[3] == -np.inf and npos == 4 and list(pos) == [0, 1, 2, 3]


def test_ties_go_to_lower_cluster():
    D = np.array([1.0, 1.0, 1.0], np.float32)
    sel, *_ = topk_drift(D, np.array([2, 1, 0]), np.array([1, 1, 1]), 2)
    assert list(sel) == [0, 1]
