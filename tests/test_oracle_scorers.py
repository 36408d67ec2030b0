"""Pins of the ablation drift signals (oracle): closed forms, library
routines (scipy's entropy and cosine distance), and agreement of its KL with
the proxy drift's KL."""
import numpy as np
import pytest
from scipy.spatial.distance import cosine as scipy_cosine
from scipy.stats import entropy as scipy_entropy

import oracle
from oracle.scorers import SCORER_COSINE, SCORER_ENTROPY, SCORER_KL, drift_score


def _dists(rng, N, C):
    A = rng.random((N, C)) ** 3
    return A / A.sum(1, keepdims=True)


def test_entropy_closed_forms():
    C = 8
    A = np.zeros((3, C))
    A[0] = 1.0 / C                         # uniform: ln C
    A[1, 3] = 1.0                          # one-hot: 0
    A[2, :2] = [0.25, 0.75]                # two points
    D = drift_score(A, None, SCORER_ENTROPY)
    assert D[0] == pytest.approx(np.log(C), rel=1e-15)
    assert D[1] == 0.0
    assert D[2] == pytest.approx(-(0.25 * np.log(0.25) + 0.75 * np.log(0.75)), rel=1e-15)


def test_entropy_matches_scipy():
    A = _dists(np.random.default_rng(1), 50, 64)
    A[3, 5:] = 0.0                          # zero entries contribute nothing
    A[3] /= A[3].sum()
    D = drift_score(A, None, SCORER_ENTROPY)
    assert np.allclose(D, [scipy_entropy(a) for a in A], rtol=1e-12, atol=0)


def test_cosine_closed_forms():
    A = np.array([[0.5, 0.5, 0.0, 0.0], [1.0, 0.0, 0.0, 0.0], [0.2, 0.3, 0.5, 0.0]])
    P = np.array([[0.0, 0.0, 0.5, 0.5], [0.5, 0.5, 0.0, 0.0], [0.2, 0.3, 0.5, 0.0]])
    D = drift_score(A, P, SCORER_COSINE)
    assert D[0] == 1.0                          # disjoint supports
    assert D[1] == pytest.approx(1 - 1 / np.sqrt(2), rel=1e-15)
    assert abs(D[2]) < 1e-15                    # identical rows
    assert np.all(drift_score(A, None, SCORER_COSINE) == 0)    # no previous step


def test_cosine_matches_scipy_and_is_scale_free():
    rng = np.random.default_rng(2)
    A, P = _dists(rng, 40, 32), _dists(rng, 40, 32)
    D = drift_score(A, P, SCORER_COSINE)
    assert np.allclose(D, [scipy_cosine(a, p) for a, p in zip(A, P)], rtol=1e-12, atol=1e-15)
    assert np.allclose(drift_score(3 * A, P, SCORER_COSINE), D, rtol=1e-12, atol=1e-15)


def test_kl_agrees_with_the_proxy_drift_and_scipy():
    rng = np.random.default_rng(3)
    A, P = _dists(rng, 30, 16), _dists(rng, 30, 16)
    D = drift_score(A, P, SCORER_KL)
    assert np.allclose(D, oracle.kl_divergence_rows(A, P), rtol=1e-14, atol=0)
    assert np.allclose(D, [scipy_entropy(a, p) for a, p in zip(A, P)], rtol=1e-12, atol=0)
    assert np.all(drift_score(A, A, SCORER_KL) == 0)
    assert np.all(drift_score(A, None, SCORER_KL) == 0)


def test_scorers_rank_a_shifted_row_first():
    """The three signals on a planted case: rows 0..9 keep their
    distribution, row 10 moves its mass to other clusters; KL and cosine put
    row 10 first, entropy (no previous step) does not see the move."""
    rng = np.random.default_rng(4)
    A_prev = _dists(rng, 11, 16)
    A = A_prev.copy()
    A[10] = np.roll(A_prev[10], 5)
    assert np.argmax(drift_score(A, A_prev, SCORER_KL)) == 10
    assert np.argmax(drift_score(A, A_prev, SCORER_COSINE)) == 10
    H = drift_score(A, A_prev, SCORER_ENTROPY)
    assert H[10] == pytest.approx(drift_score(A_prev, None, SCORER_ENTROPY)[10], rel=1e-13)
