"""Pins of the oracle's proxy attention and KL drift."""
import math

import numpy as np
from scipy.special import softmax
from scipy.stats import entropy

from oracle import centroid_keys, kl_divergence_rows, proxy_attn_kl


def test_kl_of_identical_distributions_is_exactly_zero():
    rng = np.random.default_rng(0)
    Q = rng.standard_normal((30, 4, 8))
    Kt = rng.standard_normal((5, 2 * 8))
    A, _ = proxy_attn_kl(Q, Kt, 4, 2, 8)
    A2, D = proxy_attn_kl(Q, Kt, 4, 2, 8, A_prev=A)
    assert np.array_equal(A, A2) and np.all(D == 0.0)


def test_kl_nonnegative_and_no_prev_gives_zero():
    rng = np.random.default_rng(1)
    Q = rng.standard_normal((50, 2, 4))
    Kt = rng.standard_normal((6, 8))
    prev = rng.dirichlet(np.ones(6), size=50)
    A, D = proxy_attn_kl(Q, Kt, 2, 2, 4, A_prev=prev)
    assert np.all(D >= 0) and np.all(D > 0)
    _, D0 = proxy_attn_kl(Q, Kt, 2, 2, 4, A_prev=None)
    assert np.all(D0 == 0)
    # the same divergence through scipy's relative entropy
    assert np.allclose(D, [entropy(A[i], prev[i]) for i in range(50)], rtol=1e-12)


def test_single_cluster_has_no_drift():
    rng = np.random.default_rng(2)
    Q = rng.standard_normal((10, 2, 4))
    A, D = proxy_attn_kl(Q, rng.standard_normal((1, 8)), 2, 2, 4,
                         A_prev=np.ones((10, 1)))
    assert np.all(A == 1.0) and np.all(D == 0.0)


def test_one_head_is_plain_softmax_with_scale():
    rng = np.random.default_rng(3)
    Q = rng.standard_normal((20, 1, 16))
    Kt = rng.standard_normal((7, 16))
    A, _ = proxy_attn_kl(Q, Kt, 1, 1, 16)
    want = softmax(Q[:, 0, :] @ Kt.T / 4.0, axis=1)
    assert np.allclose(A, want, rtol=1e-13, atol=0)


def test_two_cluster_closed_form():
    # q . k scores: s0 = 2, s1 = 0 with dh = 4 (scale 1/2) -> p = sigmoid(1)
    Q = np.zeros((1, 1, 4)); Q[0, 0, 0] = 2.0
    Kt = np.array([[2.0, 0, 0, 0], [0.0, 0, 0, 0]])
    prev = np.array([[0.3, 0.7]])
    A, D = proxy_attn_kl(Q, Kt, 1, 1, 4, A_prev=prev)
    p = 1 / (1 + math.exp(-2.0))
    q = 0.3
    kl = p * math.log(p / q) + (1 - p) * math.log((1 - p) / (1 - q))
    assert math.isclose(A[0, 0], p, rel_tol=1e-14)
    assert math.isclose(D[0], kl, rel_tol=1e-12)


def test_uniform_prev_gives_log_c_minus_entropy():
    rng = np.random.default_rng(4)
    Q = rng.standard_normal((12, 3, 4))
    Kt = rng.standard_normal((9, 12))
    A, D = proxy_attn_kl(Q, Kt, 3, 3, 4, A_prev=np.full((12, 9), 1 / 9))
    H = -np.sum(A * np.log(A), axis=1)
    assert np.allclose(D, math.log(9) - H, rtol=1e-10, atol=1e-14)


def test_head_mean_and_gqa_grouping():
    # 4 query heads on 2 KV heads: heads 0,1 read keys 0..dh-1, heads 2,3 the rest
    rng = np.random.default_rng(5)
    Q = rng.standard_normal((6, 4, 3))
    Kt = rng.standard_normal((5, 6))
    A, _ = proxy_attn_kl(Q, Kt, 4, 2, 3)
    want = np.zeros((6, 5))
    for h, g in ((0, 0), (1, 0), (2, 1), (3, 1)):
        want += softmax(Q[:, h, :] @ Kt[:, 3 * g:3 * g + 3].T / math.sqrt(3), axis=1)
    assert np.allclose(A, want / 4, rtol=1e-13)
    assert np.allclose(A.sum(axis=1), 1.0, rtol=1e-14)


def test_zero_mass_terms_and_prev_floor():
    A = np.array([[0.0, 1.0]])
    assert kl_divergence_rows(A, np.array([[1.0, 0.0]]))[0] == -math.log(1e-30)
    assert kl_divergence_rows(A, np.array([[0.5, 0.5]]))[0] == math.log(2)


def test_centroid_keys_hand_worked():
    chat = np.array([[1.0, 2.0], [0.0, -1.0]])
    Wk = np.array([[1.0, 0.0, 3.0], [0.5, 1.0, -1.0]])
    assert np.array_equal(centroid_keys(chat, Wk), [[2.0, 2.0, 1.0], [-0.5, -1.0, 1.0]])
