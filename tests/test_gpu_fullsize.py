"""Parity at the workloads' full sizes, through the same calls and launch
configuration the bench uses (one layer of each workload).  Where the oracle
would take too long on the whole batch, sampled windows are compared; every
output the oracle cannot afford is checked through properties that hold at
any size (unit centroids, counts summing to N, distributions summing to 1,
selected positions consistent with the selected clusters)."""
import numpy as np
import pytest
import torch

import oracle
from drift_aware_kv_spherical_gb300 import polestar as ps
from drift_aware_kv_spherical_gb300 import workloads as wl
from drift_aware_kv_spherical_gb300.pipeline import Pipeline
from tests._parity import KM_MARGIN, assert_close, np_

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _kv_ok(g, o):
    rms = np.sqrt(np.mean(o.astype(np.float64) ** 2, axis=-1, keepdims=True))
    return np.all(np.abs(g - o) <= 2e-2 * np.abs(o) + 1e-3 * rms)


def _one_layer(widx, B=None):
    w = wl.WORKLOADS[widx]
    L = wl.make_layer(w, 0, "cuda", B=B)
    Q = wl.make_queries(w, L["H"], L["Wq"])
    return w, L, Q


def _run_step(w, L, Q, B, first_u, steps=2):
    """Build the window (k-means++), then `steps - 1` warm-started steps on
    drifted hidden states; returns the pipeline and the per-step inputs."""
    pipe = Pipeline(w if B == w.B else _with_batch(w, B), layers=1)
    Hs, Qs = [L["H"]], [Q]
    for t in range(1, steps):
        Hs.append(wl.drift_rows(w, Hs[-1], t))
        Qs.append(wl.make_queries(w, Hs[-1], L["Wq"]))
    logits = wl.make_logits(w, 0, "cuda", B=B)
    snaps = []
    for t in range(steps):
        st = pipe.state[0]
        mu_in = st.mu.clone()
        A_prev = st.A[(pipe.t + 1) % 2].clone()
        pipe.step([Hs[t]], [Qs[t]], [L["Wk"]], [L["Wv"]], logits,
                  init_us=[first_u] if t == 0 else None, first=(t == 0))
        torch.cuda.synchronize()
        ps.ps_check()
        snaps.append(dict(mu_in=mu_in, A_prev=A_prev, mu=st.mu.clone(),
                          assign=st.assign.clone(), rho=st.rho.clone(), chat=st.chat.clone(),
                          counts=st.counts.clone(), A=st.A[pipe.t % 2 ^ 1].clone(),
                          D=st.D.clone(), pos=st.pos.clone(), npos=st.npos.clone(),
                          sel=st.sel.clone(), Kc=st.Kc.clone(), codes=st.codes.clone(),
                          scales=st.scales.clone(), S=st.S.clone()))
    return pipe, Hs, Qs, snaps


def _with_batch(w, B):
    from dataclasses import replace
    return replace(w, B=B)


def _check_window(w, L, H, Q, snap, b, first_u=None):
    """Oracle comparison of one window b of one step."""
    Hn = np_(H[b])
    mu_in = np_(snap["mu_in"][b]).astype(np.float64)
    if first_u is not None:
        mu_in, _, m0 = oracle.kmeanspp_init(Hn, w.C, np_(first_u[b]), return_margin=True)
        if m0 < 1e-5:
            return "unpinned draw"
    o = oracle.kmeans_spherical(Hn, mu_in, w.iters)
    ok = o["margin"][-1] > KM_MARGIN
    assert np.array_equal(np_(snap["assign"][b])[ok], o["assign"][ok])
    if o["margin"].min() > KM_MARGIN:
        assert np.array_equal(np_(snap["counts"][b]), o["counts"])
        assert_close(np_(snap["mu"][b]), o["mu"], what="mu")
        assert_close(np_(snap["chat"][b]), o["chat"], what="chat")
    # NVFP4 from the GPU's own k-means outputs: bit-exact
    oc, os_, oS, _ = oracle.nvfp4_residual(Hn, np_(snap["mu"][b]), np_(snap["assign"][b]),
                                           np_(snap["rho"][b]))
    assert np_(snap["S"])[b] == oS
    assert np.array_equal(np_(snap["scales"][b]), os_)
    assert np.array_equal(np_(snap["codes"][b]), oc)
    # proxy + KL from the GPU's C_hat
    Kt = oracle.centroid_keys(np_(snap["chat"][b]), np_(L["Wk"]))
    prev = None if first_u is not None else np_(snap["A_prev"][b])
    oA, oD = oracle.proxy_attn_kl(np_(Q[b]), Kt, w.Hq, w.Hkv, w.dh, prev)
    assert_close(np_(snap["A"][b]), oA, what="A")
    assert_close(np_(snap["D"][b]), oD, what="D")
    # top-k from the GPU's drift: bit-exact
    sel, _, pos, npos, _, _ = oracle.topk_drift(np_(snap["D"][b]), np_(snap["assign"][b]),
                                               np_(snap["counts"][b]), w.k)
    assert np.array_equal(np_(snap["sel"][b]), sel)
    assert int(np_(snap["npos"])[b]) == npos
    assert np.array_equal(np_(snap["pos"][b]), pos)
    # refresh: sampled selected rows against the oracle product
    rows = pos[:npos]
    pick = rows[np.linspace(0, max(npos - 1, 0), min(8, npos)).astype(int)] if npos else rows
    Wk = np_(L["Wk"]).astype(np.float64)
    Kc = np_(snap["Kc"][b]).reshape(w.Ncache, -1)
    for p in pick:
        want = oracle.bf16_round(Hn[p] @ Wk)
        assert _kv_ok(Kc[p][None], want[None])
    return "checked"


@pytest.mark.parametrize("widx", [2])
def test_dream7b_gqa_batch8_full(widx):
    """Dream-7B-shaped GQA layer, B = 8, window 2048: every window checked."""
    w, L, Q = _one_layer(widx)
    u = wl.make_uniforms(w, 0, "cuda")
    pipe, Hs, Qs, snaps = _run_step(w, L, Q, w.B, u, steps=2)
    results = [_check_window(w, L, Hs[0], Qs[0], snaps[0], b, first_u=u) for b in range(w.B)]
    results += [_check_window(w, L, Hs[1], Qs[1], snaps[1], b) for b in range(w.B)]
    assert results.count("checked") >= w.B


@pytest.mark.parametrize("widx,B,sample", [(3, None, [0, 3]), (4, 4, [0, 3])])
def test_loop_and_stress_layers_sampled(widx, B, sample):
    """One layer of the 32-layer loop (B = 4, window 768) and of the stress
    workload (B = 32, window 4096, C = 256) at full size; sampled windows
    against the oracle, the rest through invariants."""
    w, L, Q = _one_layer(widx, B)
    Bn = w.B if B is None else B
    u = wl.make_uniforms(w, 0, "cuda", B=Bn)
    pipe, Hs, Qs, snaps = _run_step(w, L, Q, Bn, u, steps=2)
    for snap in snaps:
        mu = np_(snap["mu"])
        cnt = np_(snap["counts"])
        assert np.all(cnt.sum(axis=1) == w.N)
        norms = np.linalg.norm(mu, axis=2)
        assert np.all(np.abs(norms[cnt > 0] - 1) < 1e-5)
        A = np_(snap["A"])
        assert np.allclose(A.sum(axis=2), 1.0, atol=1e-5)
        assert np.all(np_(snap["D"]) >= 0)
        npos = np_(snap["npos"])
        assert np.all((npos > 0) & (npos <= w.N))
    for b in sample:
        _check_window(w, L, Hs[1], Qs[1], snaps[1], b)


def test_concurrent_step_matches_sequential():
    """The step with NVFP4 and the commit on side streams (as the bench
    captures it) gives bit-identical outputs to the single-stream step."""
    w, L, Q = _one_layer(1)
    u = wl.make_uniforms(w, 0, "cuda")
    logits = wl.make_logits(w, 0, "cuda")
    H1 = wl.drift_rows(w, L["H"], 1)
    Q1 = wl.make_queries(w, H1, L["Wq"])
    outs = []
    for concurrent in (False, True):
        pipe = Pipeline(w, layers=1)
        pipe.step([L["H"]], [Q], [L["Wk"]], [L["Wv"]], logits, init_us=[u], first=True,
                  concurrent=concurrent)
        pipe.step([H1], [Q1], [L["Wk"]], [L["Wv"]], logits, concurrent=concurrent)
        torch.cuda.synchronize()
        ps.ps_check()
        st = pipe.state[0]
        outs.append([x.clone() for x in (st.mu, st.assign, st.chat, st.codes, st.scales, st.S,
                                         st.A[0], st.A[1], st.D, st.pos, st.npos, st.Kc,
                                         st.Vc, pipe.token, pipe.conf, pipe.commit,
                                         pipe.undecided, pipe.d_sum, pipe.d_cnt)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
