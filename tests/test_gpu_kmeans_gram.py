"""The Gram form of the k-means passes (bf16 windows of N <= 1024 rows, I >= 2):
passes 1..I-1 run on the fixed-point cosine Gram matrix inside one cluster
launch.  Checked against the oracle (assignments where the oracle's margin
exceeds 1e-5, everything else through the shared update and final passes),
against the Lloyd form of the same library on the same inputs, and on the
degenerate cases: clusters that stay empty, zero rows, ragged row blocks."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from drift_aware_kv_spherical_gb300 import polestar as ps
from drift_aware_kv_spherical_gb300 import workloads as wl
from tests._parity import KM_MARGIN, assert_close, np_, run_kmeans

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(autouse=True)
def _lib(lib):
    return lib


def _planted(B, N, d, C, seed, noise=0.3, zero_rows=()):
    rng = np.random.default_rng(seed)
    planted = oracle.normalize_rows(rng.standard_normal((C, d)))
    z = rng.integers(0, C, (B, N))
    H = (planted[z] * 4 + rng.normal(0, noise, (B, N, d))).astype(np.float32)
    for b, i in zero_rows:
        H[b, i] = 0.0
    Ht = torch.from_numpy(H).cuda().to(torch.bfloat16)
    Hn = np_(Ht)
    mu0 = np.stack([oracle.normalize_rows(Hn[b][:C] + 1e-3) for b in range(B)])
    return Ht, Hn, mu0.astype(np.float32)


def _check(g, Hn, mu0, iters):
    """Assignments where the oracle's last margin exceeds the tie band; the
    rest where every decision of the run does.  A zero row (all cosines 0)
    has margin 0 but a fixed answer, cluster 0, so it does not count as a tie."""
    checked = 0
    for b in range(Hn.shape[0]):
        o = oracle.kmeans_spherical(Hn[b], mu0[b].astype(np.float64), iters)
        zero = ~np.any(Hn[b] != 0, axis=1)
        ok = (o["margin"][-1] > KM_MARGIN) | zero
        assert np.array_equal(g["assign"][b][ok], o["assign"][ok])
        if o["margin"][:, ~zero].min() > KM_MARGIN:
            checked += 1
            assert np.array_equal(g["counts"][b], o["counts"])
            assert_close(g["mu"][b], o["mu"], what="mu")
            assert_close(g["rho"][b], o["rho"], what="rho")
            assert_close(g["chat"][b], o["chat"], what="chat")
            assert_close(g["obj"][b], o["obj"], what="objective")
    return checked


# seeds whose oracle runs keep every decision outside the 1e-5 tie band
@pytest.mark.parametrize("B,N,d,C,iters,seed", [(1, 1024, 256, 64, 6, 1091),  # 16 CTAs x 64 rows
                                                (1, 1000, 128, 32, 4, 1032),  # last CTA 40 rows
                                                (2, 530, 320, 40, 3, 570),    # C % 8 != 0
                                                (3, 64, 64, 5, 5, 69),        # 4 CTAs x 16 rows
                                                (1, 700, 192, 200, 3, 900)])  # C > 128
def test_gram_passes_against_oracle(B, N, d, C, iters, seed):
    Ht, Hn, mu0 = _planted(B, N, d, C, seed=seed)
    g = run_kmeans(Ht, torch.from_numpy(mu0).cuda(), iters)
    assert _check(g, Hn, mu0, iters) >= 1


def test_gram_cluster_left_empty_keeps_centroid_and_chat():
    """Centroid 1 points away from every row: it stays empty through every
    Gram pass, keeps its centroid and its C_hat, and its carried column of
    cosines never wins."""
    d = 64
    rng = np.random.default_rng(3)
    H = np.zeros((1, 40, d), np.float32)
    H[0, :, 0] = 1.0
    H[0, :, 1:4] = rng.normal(0, 0.05, (40, 3))
    far = np.zeros(d, np.float32)
    far[0] = -1.0
    mu0 = np.stack([np.eye(d, dtype=np.float32)[0], far, np.eye(d, dtype=np.float32)[1]])[None]
    chat0 = np.full((1, 3, d), 3.0, np.float32)
    Ht = torch.from_numpy(H).cuda().to(torch.bfloat16)
    g = run_kmeans(Ht, torch.from_numpy(mu0).cuda(), 4, chat0=torch.from_numpy(chat0).cuda())
    assert np.array_equal(g["mu"][0][1], far)
    assert np.all(g["chat"][0][1] == 3.0) and g["counts"][0][1] == 0
    o = oracle.kmeans_spherical(np_(Ht)[0], mu0[0].astype(np.float64), 4, chat0[0])
    assert np.array_equal(g["assign"][0], o["assign"])
    assert np.array_equal(g["counts"][0], o["counts"])
    assert_close(g["mu"][0], o["mu"], what="mu")


def test_gram_zero_rows_join_cluster_zero():
    Ht, Hn, mu0 = _planted(2, 300, 128, 12, seed=11, zero_rows=[(0, 5), (1, 0), (1, 299)])
    g = run_kmeans(Ht, torch.from_numpy(mu0).cuda(), 5)
    for b, i in [(0, 5), (1, 0), (1, 299)]:
        assert g["assign"][b][i] == 0 and g["rho"][b][i] == 0.0
    assert _check(g, Hn, mu0, 5) >= 1


_LLOYD = r"""
import json, sys, torch
sys.path.insert(0, sys.argv[1])
from drift_aware_kv_spherical_gb300 import workloads as wl
from tests._parity import run_kmeans
w = wl.WORKLOADS[1]
L = wl.make_layer(w, 0, "cuda")
u = wl.make_uniforms(w, 0, "cuda")
g = run_kmeans(L["H"], torch.zeros(w.B, w.C, w.d, device="cuda"), w.iters, init_u=u)
print(json.dumps({k: v.tolist() for k, v in g.items()}))
"""


def test_gram_form_matches_lloyd_form():
    """The LLaDA-8B-shaped layer (k-means++ start, 10 passes) through both
    forms of the library: labels, counts and centroids identical (the last
    update is the same kernel on the same labels); rho, C_hat and the
    objectives, which the Gram form takes from its cosines, within rounding."""
    w = wl.WORKLOADS[1]
    L = wl.make_layer(w, 0, "cuda")
    u = wl.make_uniforms(w, 0, "cuda")
    g = run_kmeans(L["H"], torch.zeros(w.B, w.C, w.d, device="cuda"), w.iters, init_u=u)
    env = dict(os.environ, PS_KMEANS_LLOYD="1")
    out = subprocess.run([sys.executable, "-c", _LLOYD, ROOT], env=env, cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    ref = {k: np.asarray(v) for k, v in json.loads(out.stdout.strip().splitlines()[-1]).items()}
    for k in ("assign", "counts", "mu"):
        assert np.array_equal(g[k], ref[k].astype(g[k].dtype)), k
    for k in ("rho", "chat", "obj"):
        assert_close(g[k], ref[k].astype(g[k].dtype), what=k)


def test_gram_trace_shape():
    """The Gram form's launches for C <= 64: set-up, the Gram GEMM (with pass
    0's cosines as extra tiles), one kernel for passes 0..I and one scan for
    the last update and C_hat."""
    Ht, _, mu0 = _planted(1, 256, 128, 16, seed=2)
    mu = torch.from_numpy(mu0).cuda()
    ws = ps.workspace(ps.OP_KMEANS, B=1, N=256, d=128, C=16)
    out = dict(assign=torch.zeros(1, 256, dtype=torch.int32, device="cuda"),
               rho=torch.zeros(1, 256, device="cuda"), chat=torch.zeros(1, 16, 128, device="cuda"),
               counts=torch.zeros(1, 16, dtype=torch.int32, device="cuda"))
    ps.ps_trace_enable(True)
    ps.ps_kmeans_spherical(Ht, mu, out["assign"], out["rho"], out["chat"], out["counts"], 6, ws=ws)
    names = [r[0] for r in ps.ps_trace_records()]
    ps.ps_trace_enable(False)
    ps.ps_check()
    assert len(names) == 4, names
    assert sum("k_km_gram" in x for x in names) == 1
    assert sum("GramClusterEpi" in x for x in names) == 1


def test_gram_centroid_emptied_mid_run_is_kept():
    """Unit rows on a circle (degrees): centroid 1 starts at 50 and takes the
    rows from 7 to 87 in pass 0; its update moves its neighbours in, which
    take all its rows in pass 1, so it is empty from then on and keeps the
    centroid formed for pass 1 (about 46.7 degrees), not the one it started
    from.  That centroid exists only inside the Gram passes: the kernel must
    form it from H when the cluster empties."""
    d = 64
    rng = np.random.default_rng(0)
    ang = np.deg2rad([0, 3, 7, 11, 14, 18, 75, 79, 83, 87, 90])
    H = np.zeros((1, len(ang), d), np.float32)
    H[0, :, 0], H[0, :, 1] = np.cos(ang), np.sin(ang)
    H[0, :, 2:] = rng.normal(0, 0.01, (len(ang), d - 2))

    def unit(a):
        v = np.zeros(d, np.float32)
        v[0], v[1] = np.cos(np.deg2rad(a)), np.sin(np.deg2rad(a))
        return v

    mu0 = np.stack([unit(-40), unit(50), unit(125)])[None]
    Ht = torch.from_numpy(H).cuda().to(torch.bfloat16)
    g = run_kmeans(Ht, torch.from_numpy(mu0).cuda(), 3)
    o = oracle.kmeans_spherical(np_(Ht)[0], mu0[0].astype(np.float64), 3)
    assert o["margin"].min() > KM_MARGIN and o["counts"][1] == 0
    assert np.array_equal(g["assign"][0], o["assign"])
    assert np.array_equal(g["counts"][0], o["counts"])
    assert_close(g["mu"][0], o["mu"], what="mu")          # mu_1 from pass 1, not mu0_1
    assert_close(g["rho"][0], o["rho"], what="rho")
    assert_close(g["obj"][0], o["obj"], what="objective")


@pytest.mark.parametrize("B,N,d,C,seed", [(2, 700, 512, 48, 10), (3, 1024, 1024, 64, 8),
                                          (3, 257, 256, 100, 6), (1, 96, 128, 96, 3)])
def test_gram_seeding_matches_oracle_kmeanspp(B, N, d, C, seed):
    """k-means++ seeded from the window's Gram matrix (one launch), then the
    Gram passes: the seeds of every draw outside the tie band are the
    oracle's (k-means++ on the unit rows in fp64), so a window whose passes
    also stay outside the band (one near-tie moves a row, hence a centroid,
    hence rows far from any tie) matches the oracle's k-means from them in
    full.  C = N (every row a seed) and C > 64 (no pass-0 tiles) included.
    The seeds give each case such a window (a 64-round draw over 1024 rows
    clears 1e-5 about one time in four)."""
    Ht, Hn, _ = _planted(B, N, d, C, seed)
    u = torch.from_numpy(np.random.default_rng(seed).random((B, C))).cuda()
    g = run_kmeans(Ht, torch.zeros(B, C, d, device="cuda"), 3, init_u=u)
    pinned = 0
    for b in range(B):
        mu0, _, m0 = oracle.kmeanspp_init(Hn[b], C, np_(u[b]), return_margin=True)
        if m0 < 1e-5 or oracle.kmeans_spherical(Hn[b], mu0, 3)["margin"].min() <= KM_MARGIN:
            continue
        pinned += 1
        assert _check({k: v[b:b + 1] for k, v in g.items()}, Hn[b:b + 1], mu0[None], 3) == 1
    assert pinned >= 1


def test_gram_seeding_trace_shape():
    """With k-means++ the Gram form launches set-up, the Gram GEMM, the
    seeding, the passes and the scan: five kernels, none per seed."""
    Ht, _, _ = _planted(1, 256, 128, 16, seed=2)
    u = torch.rand(1, 16, dtype=torch.float64, device="cuda")
    ws = ps.workspace(ps.OP_KMEANS, B=1, N=256, d=128, C=16)
    out = dict(mu=torch.zeros(1, 16, 128, device="cuda"),
               assign=torch.zeros(1, 256, dtype=torch.int32, device="cuda"),
               rho=torch.zeros(1, 256, device="cuda"), chat=torch.zeros(1, 16, 128, device="cuda"),
               counts=torch.zeros(1, 16, dtype=torch.int32, device="cuda"))
    ps.ps_trace_enable(True)
    ps.ps_kmeans_spherical(Ht, out["mu"], out["assign"], out["rho"], out["chat"], out["counts"],
                           4, init_mode=1, init_u=u, ws=ws)
    torch.cuda.synchronize()
    names = [n for n, _ in ps.ps_trace_records()]
    ps.ps_trace_enable(False)
    ps.ps_check()
    assert len(names) == 5, names
    assert sum("k_kpp_gram" in n for n in names) == 1
    assert not any("k_kpp_pick" in n or "k_kpp_weights" in n for n in names)
