"""Pins of the oracle's spherical k-means and k-means++ seeding."""
import math

import numpy as np

from oracle import kmeans_spherical, kmeanspp_init, normalize_rows


def _unit(deg):
    return np.array([math.cos(math.radians(deg)), math.sin(math.radians(deg))])


def test_hand_worked_circle():
    # points at 0, 10, 80, 90 degrees (radius 2); centroids start at 0 and 90
    H = np.array([2 * _unit(a) for a in (0, 10, 80, 90)])
    mu0 = np.array([_unit(0), _unit(90)])
    r = kmeans_spherical(H, mu0, iters=1)
    assert list(r["assign"]) == [0, 0, 1, 1]
    # the normalised sum of unit vectors at 0 and 10 degrees points at 5
    assert np.allclose(r["mu"][0], _unit(5), atol=1e-15)
    assert np.allclose(r["mu"][1], _unit(85), atol=1e-15)
    # rho = 2 cos 5 for every point; C_hat = rho_bar mu
    assert np.allclose(r["rho"], 2 * math.cos(math.radians(5)), atol=1e-15)
    assert np.allclose(r["chat"][0], 2 * math.cos(math.radians(5)) * _unit(5))
    # pass 0: cosines 1, cos10, cos10, 1; pass 1: four times cos 5
    assert math.isclose(r["obj"][0], 2 + 2 * math.cos(math.radians(10)))
    assert math.isclose(r["obj"][1], 4 * math.cos(math.radians(5)))
    assert np.array_equal(r["counts"], [2, 2])


def test_unit_norm_and_monotone_objective():
    rng = np.random.default_rng(0)
    H = rng.standard_normal((300, 24))
    mu0 = normalize_rows(rng.standard_normal((7, 24)))
    r = kmeans_spherical(H, mu0, iters=12)
    assert np.all(np.abs(np.linalg.norm(r["mu"], axis=1) - 1) < 1e-12)
    assert np.all(np.diff(r["obj"]) >= -1e-12)


def test_single_cluster_closed_form():
    rng = np.random.default_rng(1)
    H = rng.standard_normal((50, 8)) + 0.5
    s = [0.0] * 8
    for row in H:                                    # sum of unit rows
        n = math.sqrt(sum(v * v for v in row))
        for j in range(8):
            s[j] += row[j] / n
    n = math.sqrt(sum(v * v for v in s))
    want = np.array(s) / n
    r = kmeans_spherical(H, normalize_rows(H[:1]), iters=1)
    assert np.allclose(r["mu"][0], want, atol=1e-14)
    assert np.all(r["assign"] == 0) and r["counts"][0] == 50


def test_planted_partition_is_recovered():
    rng = np.random.default_rng(2)
    d, m, per = 64, 6, 40
    U = np.eye(d)[:m]                                # orthogonal directions
    z = np.repeat(np.arange(m), per)
    rng.shuffle(z)
    H = U[z] * 3 + rng.normal(0, 0.05, (m * per, d))
    first = [int(np.nonzero(z == c)[0][0]) for c in range(m)]
    r = kmeans_spherical(H, normalize_rows(H[first]), iters=5)
    assert np.array_equal(r["assign"], z)


def test_brute_force_assignment_and_ties():
    rng = np.random.default_rng(4)
    H = rng.standard_normal((40, 5))
    mu = normalize_rows(rng.standard_normal((4, 5)))
    mu[3] = mu[1]                                    # exact duplicate centroid
    r = kmeans_spherical(H, mu, iters=0)
    for i, h in enumerate(H):
        n = math.sqrt(sum(v * v for v in h))
        cos = [sum(h[j] * mu[c][j] for j in range(5)) / n for c in range(4)]
        best = max(cos)
        assert r["assign"][i] == min(c for c in range(4) if cos[c] >= best - 1e-12)
        assert r["assign"][i] != 3                   # ties go to the lower index


def test_empty_cluster_keeps_centroid_and_chat():
    H = np.array([[1.0, 0.1], [1.0, -0.1], [0.9, 0.0]])
    far = np.array([-1.0, 0.0])
    chat_in = np.array([[0.0, 0.0], [7.0, 7.0]])
    r = kmeans_spherical(H, np.array([[1.0, 0.0], far]), iters=3, chat_in=chat_in)
    assert np.array_equal(r["mu"][1], far)
    assert np.array_equal(r["chat"][1], [7.0, 7.0])
    assert r["counts"][1] == 0


def test_zero_row_joins_cluster_zero():
    H = np.array([[0.0, 0.0], [0.0, 1.0], [1.0, 0.0]])
    r = kmeans_spherical(H, np.array([[1.0, 0.0], [0.0, 1.0]]), iters=0)
    assert r["assign"][0] == 0 and r["rho"][0] == 0.0


def test_kmeanspp_hand_worked():
    # rows at 0, 90 and 180 degrees; first pick row floor(0.1 * 3) = 0.
    # weights after it: 1 - cos = [0, 1, 2]; prefix [0, 1, 3]
    H = np.array([_unit(0), _unit(90), _unit(180)])
    mu, idx = kmeanspp_init(H, 2, [0.1, 0.30])      # 0.9 < 1 -> row 1
    assert list(idx) == [0, 1]
    mu, idx = kmeanspp_init(H, 2, [0.1, 0.34])      # 1.02 >= 1 -> row 2
    assert list(idx) == [0, 2]
    assert np.allclose(mu[1], _unit(180))
    mu, idx = kmeanspp_init(H, 3, [0.99, 0.0, 0.0])  # first pick row 2
    assert idx[0] == 2 and len(set(idx)) == 3


def test_kmeanspp_degenerate_all_identical():
    H = np.ones((4, 3))
    mu, idx = kmeanspp_init(H, 3, [0.6, 0.5, 0.5])
    assert list(idx) == [2, 0, 1]                    # total 0: next unchosen


def test_kmeanspp_draws_follow_weights():
    # with one distant row among many near the first pick, draws land on it
    # in proportion to its share of the weight
    H = np.vstack([np.tile(_unit(0), (9, 1)), _unit(90)[None]])
    hits = 0
    us = np.linspace(0, 1, 1001)[:-1]
    for u in us:
        _, idx = kmeanspp_init(H, 2, [0.0, u])
        hits += idx[1] == 9
    assert hits == len(us)                           # all other weights are 0
