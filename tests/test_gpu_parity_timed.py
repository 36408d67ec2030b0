"""Oracle parity at the shapes the bench times, through the same calls.

* Spherical k-means in Gram form at the LLaDA-8B layer (bf16, N = 1024,
  d = 4096, C = 64, 10 iterations): the form a bf16 window of at most 1024
  rows takes (Gram GEMM, the pass kernel, the closing cluster scan), compared
  with the oracle pass by pass, over a whole warm-started run (the bench's
  step), and over a whole run seeded by k-means++.
* The commit at the Dream-7B (B 8, P 32, V 152064), 32-layer loop (B 4, P 32,
  V 126464, RATIO rule) and stress (B 32, P 64, V 126464) shapes, fp32 and
  bf16 logits, every sequence of the batch.

Assignments are compared where the oracle's top-2 cosine margin exceeds 1e-5
in every pass that led to them; k-means++ draws within 1e-5 (relative) of a
prefix-sum boundary are unpinned.  Neither kind of case is skipped silently:
the tests count them and require the pinned part to be nearly everything.
"""
import numpy as np
import pytest
import torch

import oracle
from drift_aware_kv_spherical_gb300 import polestar as ps
from drift_aware_kv_spherical_gb300 import workloads as wl
from tests._parity import (BAND, CONF_RTOL, KM_MARGIN, assert_close, np_, run_commit,
                           run_kmeans)

pytestmark = pytest.mark.gpu

LLADA = 1   # LLaDA-8B-shaped layer: the Gram form's timed shape


@pytest.fixture(autouse=True)
def _lib(lib, monkeypatch):
    monkeypatch.delenv("PS_KMEANS_LLOYD", raising=False)
    return lib


@pytest.fixture(scope="module")
def llada():
    w = wl.WORKLOADS[LLADA]
    L = wl.make_layer(w, 0, "cuda")
    H0 = L["H"]
    H1 = wl.drift_rows(w, H0, 1)
    return w, H0, H1


def _compare_run(g, o, b, what):
    """Whole-run outputs of window b: exact labels and counts, centroids,
    rho, C_hat and the objective of every pass within 1e-4 / 1e-6."""
    assert np.array_equal(g["assign"][b], o["assign"]), what
    assert np.array_equal(g["counts"][b], o["counts"]), what
    assert_close(g["mu"][b], o["mu"], what=f"{what}: mu")
    assert_close(g["rho"][b], o["rho"], what=f"{what}: rho")
    assert_close(g["chat"][b], o["chat"], what=f"{what}: chat")
    assert_close(g["obj"][b], o["obj"], what=f"{what}: objective")


def test_gram_form_pass_by_pass(llada):
    """The pass kernel fed the oracle's centroids of pass t: two more updates
    (the Gram form's smallest run) from mu^(t) must give the oracle's
    passes t, t+1 and t+2 -- every pass of a 10-iteration run is covered."""
    w, H0, H1 = llada
    Hn = np_(H1)[0]
    mu_warm = oracle.kmeanspp_init(np_(H0)[0], w.C, np_(wl.make_uniforms(w))[0])[0]
    mu_warm = oracle.kmeans_spherical(np_(H0)[0], mu_warm, w.iters)["mu"]
    ref = oracle.kmeans_spherical(Hn, mu_warm, w.iters)
    checked = 0
    for t in range(w.iters - 1):
        mu_t = ref["mus"][t].astype(np.float32)
        o = oracle.kmeans_spherical(Hn, mu_t.astype(np.float64), 2)
        g = run_kmeans(H1, torch.from_numpy(mu_t)[None].cuda(), 2)
        if o["margin"].min() <= KM_MARGIN:
            ok = o["margin"][-1] > KM_MARGIN
            assert ok.mean() > 0.99
            assert np.array_equal(g["assign"][0][ok], o["assign"][ok]), f"from pass {t}"
            continue
        _compare_run(g, o, 0, f"from pass {t}")
        checked += 1
    assert checked >= w.iters - 2


def test_gram_form_warm_started_step(llada):
    """The bench's step: centroids of the previous step as the warm start,
    10 iterations on drifted hidden states."""
    w, H0, H1 = llada
    mu0 = oracle.kmeanspp_init(np_(H0)[0], w.C, np_(wl.make_uniforms(w))[0])[0]
    prev = oracle.kmeans_spherical(np_(H0)[0], mu0, w.iters)
    mu_warm = prev["mu"].astype(np.float32)
    o = oracle.kmeans_spherical(np_(H1)[0], mu_warm.astype(np.float64), w.iters,
                                prev["chat"])
    chat0 = torch.from_numpy(prev["chat"].astype(np.float32))[None].cuda()
    g = run_kmeans(H1, torch.from_numpy(mu_warm)[None].cuda(), w.iters, chat0=chat0)
    assert o["margin"].min() > KM_MARGIN, "the warm-started run has a tie-band decision"
    _compare_run(g, o, 0, "warm start")


def _clean_draws(w, Hn, tries=40):
    """Test-only k-means++ draws for which the oracle's seeding and every
    pass of the run clear the tie band: the first of the seeded draw sets
    s = 0, 1, 2, ... (generator seed 90210 + s) that does.  Returns the draws,
    the oracle's run and how many sets were passed over as unpinned."""
    for s in range(tries):
        g = torch.Generator().manual_seed(90210 + s)
        u = torch.rand((1, w.C), generator=g, dtype=torch.float64)
        mu0, _, m0 = oracle.kmeanspp_init(Hn, w.C, u.numpy()[0], return_margin=True)
        if m0 <= 1e-5:
            continue
        o = oracle.kmeans_spherical(Hn, mu0, w.iters)
        if o["margin"].min() > KM_MARGIN:
            return u, mu0, o, s
    pytest.fail(f"no clean draw set in {tries}")


def test_gram_form_kmeanspp_run(llada):
    """Window build: k-means++ seeding from the Gram matrix, then the
    passes, against the oracle's seeding and run on the same draws."""
    w, H0, _ = llada
    Hn = np_(H0)[0]
    u, mu0, o, skipped = _clean_draws(w, Hn)
    g = run_kmeans(H0, torch.zeros(1, w.C, w.d, device="cuda"), w.iters, init_u=u.cuda())
    _compare_run(g, o, 0, f"k-means++ (draw set {skipped})")
    # the seeds themselves: a zero-iteration call returns them
    g0 = run_kmeans(H0, torch.zeros(1, w.C, w.d, device="cuda"), 0, init_u=u.cuda())
    assert_close(g0["mu"][0], mu0, rtol=0, atol=2e-6, what="k-means++ centres")
    print(f"draw sets passed over as unpinned: {skipped}")


# ---------------------------------------------------------------- commit
COMMIT_SHAPES = [(2, 0), (3, 2), (4, 0)]   # (workload, rule): Dream-7B, loop, stress


def _commit_inputs(w, seed):
    rng = np.random.default_rng(seed)
    B, P = w.B, w.P
    role = np.zeros(P, np.uint8)
    role[P // 2:] = 1                 # a suffix half, gated by the position mask
    role[-1] = 2
    und = (rng.random((B, P)) < 0.85).astype(np.uint8)
    D = rng.gamma(2.0, 0.05, (B, P)).astype(np.float32)
    cnt = rng.integers(0, 4, (B, P)).astype(np.int32)
    s = (cnt * rng.gamma(2.0, 0.05, (B, P))).astype(np.float32)
    prev = rng.gamma(2.0, 0.05, (B, P)).astype(np.float32)
    if w.mode == wl.MODE_RATIO:       # the loop's rule: D below ratio x the last D
        prev = (D / w.ratio * rng.choice([0.5, 2.0], (B, P))).astype(np.float32)
    ssel = (rng.random((B, P)) < 0.5).astype(np.uint8)
    params = oracle.CommitParams(tau_s=w.tau_s, alpha=w.alpha, ratio=w.ratio, mode=w.mode,
                                 ensure_progress=1)
    return role, und, D, s, cnt, prev, ssel, params


@pytest.mark.parametrize("widx", [2, 3, 4])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_commit_at_timed_shapes(widx, dtype):
    w = wl.WORKLOADS[widx]
    logits = wl.make_logits(w, 1, "cuda")
    if dtype == "bf16":
        logits = logits.to(torch.bfloat16)
    role, und, D, s, cnt, prev, ssel, p = _commit_inputs(w, 100 + widx)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    g = run_commit(logits, dev(role), dev(und), dev(D), w.P, dev(s), dev(cnt), dev(prev),
                   dev(ssel), ps.CommitParams(p.tau_s, p.alpha, p.ratio, p.mode,
                                              p.ensure_progress))
    Ln = np_(logits)
    unpinned = 0
    for b in range(w.B):
        o = oracle.commit_rule(Ln[b], role, und[b], D[b], s[b], cnt[b], prev[b], ssel[b], p)
        assert np.array_equal(g["token"][b], o["token"]), b
        assert_close(g["conf"][b], o["conf"], rtol=CONF_RTOL, atol=0, what=f"conf {b}")
        band = o["margin"] <= BAND
        unpinned += int(band.sum())
        if not band.any():
            assert np.array_equal(g["commit"][b], o["commit"]), b
            assert np.array_equal(g["undecided"][b], o["undecided"]), b
        assert np.array_equal(g["d_sum"][b], o["d_sum"])
        assert np.array_equal(g["d_cnt"][b], o["d_cnt"])
        assert np.array_equal(g["d_prev"][b], o["d_prev"])
    assert unpinned <= max(1, w.B * w.P // 1000)
    assert g["commit"].any() and not g["commit"].all()
