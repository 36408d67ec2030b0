"""The ablation drift signals (ps_drift_score) against the oracle: random
distributions with ragged C, the proxy's own distributions at the LLaDA-8B
layer, agreement of its KL with the proxy's fused KL, the pipeline's scorer
option, and argument errors."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from drift_aware_kv_spherical_gb300 import polestar as ps
from drift_aware_kv_spherical_gb300 import workloads as wl
from drift_aware_kv_spherical_gb300.pipeline import Pipeline
from tests._parity import RTOL, assert_close, np_

pytestmark = pytest.mark.gpu

SCORERS = [ps.SCORER_KL, ps.SCORER_COSINE, ps.SCORER_ENTROPY]
ATOL_SCORE = 2e-6  # fp32 sums of C <= 256 terms of size <= 1 (cosine: 1 - cos near 0)


@pytest.fixture(autouse=True)
def _lib(lib):
    return lib


def _dists(rng, B, N, C, zeros=False):
    A = rng.random((B, N, C)) ** 4
    if zeros:
        A[:, ::3, : C // 2] = 0.0      # rows with empty entries: skipped terms
    A /= A.sum(-1, keepdims=True)
    return A


def _run(A, P, scorer):
    At = torch.from_numpy(A.astype(np.float32)).cuda()
    Pt = None if P is None else torch.from_numpy(P.astype(np.float32)).cuda()
    D = torch.full(A.shape[:2], -7.0, device="cuda")
    ps.ps_drift_score(At, Pt, scorer, D)
    torch.cuda.synchronize()
    ps.ps_check()
    return np_(D), np_(At).astype(np.float64), None if Pt is None else np_(Pt).astype(np.float64)


@pytest.mark.parametrize("B,N,C", [(2, 300, 64), (3, 77, 37), (1, 1024, 256), (1, 5, 1)])
@pytest.mark.parametrize("scorer", SCORERS)
def test_drift_score_matches_oracle(B, N, C, scorer):
    rng = np.random.default_rng(B * 1000 + N + C + scorer)
    A, P = _dists(rng, B, N, C, zeros=C > 1), _dists(rng, B, N, C)
    D, A32, P32 = _run(A, P, scorer)
    for b in range(B):
        want = oracle.drift_score(A32[b], P32[b], scorer)
        assert_close(D[b], want, rtol=RTOL, atol=ATOL_SCORE, what=f"scorer {scorer}")
    D0, A32, _ = _run(A, None, scorer)          # no previous step
    for b in range(B):
        want = oracle.drift_score(A32[b], None, scorer)
        assert_close(D0[b], want, rtol=RTOL, atol=ATOL_SCORE, what="no prev")
    if scorer != ps.SCORER_ENTROPY:
        assert np.all(D0 == 0.0)


def test_identical_steps_score_zero_drift():
    rng = np.random.default_rng(5)
    A = _dists(rng, 1, 200, 64)
    for scorer in (ps.SCORER_KL, ps.SCORER_COSINE):
        D, _, _ = _run(A, A, scorer)
        assert np.all(D == 0.0) if scorer == ps.SCORER_KL else np.all(D <= 1e-6)


def test_kl_scorer_agrees_with_the_fused_proxy_kl():
    """LLaDA-8B layer: the proxy's fused KL and the scoring pass's KL over
    the same distributions agree to fp32 summation order; cosine and entropy
    of those distributions match the oracle row by row."""
    w = wl.WORKLOADS[1]
    L = wl.make_layer(w, 0, "cuda")
    u = wl.make_uniforms(w, 0, "cuda")
    logits = wl.make_logits(w, 0, "cuda")
    pipe = Pipeline(w, layers=1)
    pipe.step([L["H"]], [wl.make_queries(w, L["H"], L["Wq"])], [L["Wk"]], [L["Wv"]], logits,
              init_us=[u], first=True)
    H1 = wl.drift_rows(w, L["H"], 1)
    pipe.step([H1], [wl.make_queries(w, H1, L["Wq"])], [L["Wk"]], [L["Wv"]], logits)
    torch.cuda.synchronize()
    ps.ps_check()
    st = pipe.state[0]
    cur, prev = st.A[(pipe.t + 1) % 2], st.A[pipe.t % 2]
    out = {}
    for scorer in SCORERS:
        D = torch.empty(w.B, w.N, device="cuda")
        ps.ps_drift_score(cur, prev, scorer, D)
        torch.cuda.synchronize()
        out[scorer] = np_(D)[0]
    assert_close(out[ps.SCORER_KL], np_(st.D)[0], rtol=1e-4, atol=1e-6, what="fused vs pass")
    An, Pn = np_(cur)[0].astype(np.float64), np_(prev)[0].astype(np.float64)
    for scorer in SCORERS:
        assert_close(out[scorer], oracle.drift_score(An, Pn, scorer), rtol=RTOL, atol=ATOL_SCORE,
                     what=f"scorer {scorer}")
    assert (out[ps.SCORER_COSINE] > 1e-5).mean() > 0.05     # the drift is not trivially zero


@pytest.mark.parametrize("scorer", [ps.SCORER_COSINE, ps.SCORER_ENTROPY])
def test_pipeline_with_an_ablation_scorer(scorer):
    """The pipeline's scorer option: D is the chosen signal of the step's
    distributions, and the top-k and refresh follow that D."""
    w = wl.WORKLOADS[0]
    L = wl.make_layer(w, 0, "cuda")
    u = wl.make_uniforms(w, 0, "cuda")
    logits = wl.make_logits(w, 0, "cuda")
    pipe = Pipeline(w, layers=1, scorer=scorer)
    pipe.step([L["H"]], [wl.make_queries(w, L["H"], L["Wq"])], [L["Wk"]], [L["Wv"]], logits,
              init_us=[u], first=True)
    torch.cuda.synchronize()
    st = pipe.state[0]
    D_first = np_(st.D)[0]
    A0 = np_(st.A[0])[0].astype(np.float64)
    assert_close(D_first, oracle.drift_score(A0, None, scorer), rtol=RTOL, atol=ATOL_SCORE)
    H1 = wl.drift_rows(w, L["H"], 1)
    pipe.step([H1], [wl.make_queries(w, H1, L["Wq"])], [L["Wk"]], [L["Wv"]], logits)
    torch.cuda.synchronize()
    ps.ps_check()
    A1 = np_(st.A[1])[0].astype(np.float64)
    D = np_(st.D)[0]
    assert_close(D, oracle.drift_score(A1, A0, scorer), rtol=RTOL, atol=ATOL_SCORE)
    sel, _, pos, npos, pm, _ = oracle.topk_drift(D, np_(st.assign)[0], np_(st.counts)[0], w.k)
    assert np.array_equal(np_(st.posmask)[0], pm)
    assert int(np_(st.npos)[0]) == npos


def test_drift_score_rejects_bad_arguments():
    lib = ps._lib()
    A = torch.rand(1, 8, 4, device="cuda")
    D = torch.empty(1, 8, device="cuda")
    h = lib.handle()
    s = torch.cuda.current_stream().cuda_stream
    f = lib.cdll.ps_drift_score
    assert f(h, A.data_ptr(), None, 1, 8, 4, 3, D.data_ptr(), s) == ps.PS_ERR_ARG
    assert f(h, A.data_ptr(), None, 1, 8, 0, 0, D.data_ptr(), s) == ps.PS_ERR_ARG
    assert f(h, A.data_ptr(), None, 1, 8, 4097, 0, D.data_ptr(), s) == ps.PS_ERR_ARG
    assert f(h, A.data_ptr(), A.data_ptr(), 1, 8, 4, 1, A.data_ptr(), s) == ps.PS_ERR_ARG
    assert f(None, A.data_ptr(), None, 1, 8, 4, 0, D.data_ptr(), s) == ps.PS_ERR_ARG
    assert f(h, None, None, 0, 8, 4, 0, None, s) == ps.PS_OK    # B == 0: no-op
