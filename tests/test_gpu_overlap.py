"""Latency hiding: the drift step on a side stream behind a main forward.

The synthetic main forward fills each layer's hidden states and queries (and
finally the block's logits) on the main stream, after a device-side spin, into
buffers that hold NaN until then.  Pipeline.step_overlapped forks every
layer's drift work onto the drift stream right after that layer's forward, so
the outputs can only match the oracle if every fork waited for its layer's
inputs.  Two steps (window build, then a warm-started step) of a two-layer
tiny fp32 window are compared with the oracle stage by stage from the GPU's
own state before each step, and with the single-stream step bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from drift_aware_kv_spherical_gb300 import polestar as ps
from drift_aware_kv_spherical_gb300 import workloads as wl
from drift_aware_kv_spherical_gb300.pipeline import Pipeline
from tests._parity import BAND, CONF_RTOL, KM_MARGIN, assert_close, np_

pytestmark = pytest.mark.gpu

LAYERS = 2


@pytest.fixture(autouse=True)
def _lib(lib):
    return lib


def _inputs(w):
    Ls = [wl.make_layer(w, l, "cuda") for l in range(LAYERS)]
    H = [[L["H"], wl.drift_rows(w, L["H"], 1, l)] for l, L in enumerate(Ls)]
    Q = [[wl.make_queries(w, h, L["Wq"]) for h in H[l]] for l, L in enumerate(Ls)]
    logits = [wl.make_logits(w, t, "cuda") for t in range(2)]
    us = [wl.make_uniforms(w, l, "cuda") for l in range(LAYERS)]
    return Ls, H, Q, logits, us


def _snap(pipe):
    out = []
    for st in pipe.state:
        out.append({k: getattr(st, k).clone() for k in
                    ("mu", "assign", "rho", "chat", "counts", "codes", "scales", "S", "D",
                     "sel", "pos", "npos", "Kc", "Vc")})
        out[-1]["A"] = [a.clone() for a in st.A]
    out.append({k: getattr(pipe, k).clone() for k in
                ("token", "conf", "commit", "undecided", "d_sum", "d_cnt", "d_prev")})
    return out


def _kv_check(g, o):
    rms = np.sqrt(np.mean(o.astype(np.float64) ** 2, axis=-1, keepdims=True))
    assert np.all(np.abs(g - o) <= 1e-5 * np.abs(o) + 1e-3 * rms)


def test_overlapped_step_matches_oracle_and_sequential():
    w = wl.WORKLOADS[0]
    Ls, H, Q, logits, us = _inputs(w)
    Wks, Wvs = [L["Wk"] for L in Ls], [L["Wv"] for L in Ls]
    main, drift = torch.cuda.Stream(), torch.cuda.Stream()
    Hb = [torch.full_like(H[l][0], float("nan")) for l in range(LAYERS)]
    Qb = [torch.full_like(Q[l][0], float("nan")) for l in range(LAYERS)]
    Lb = torch.full_like(logits[0], float("nan"))

    def forward_for(t):
        def forward(l, s):
            with torch.cuda.stream(s):
                torch.cuda._sleep(2_000_000)   # a slow layer: an early fork would read NaN
                if l < LAYERS:
                    Hb[l].copy_(H[l][t])
                    Qb[l].copy_(Q[l][t])
                else:
                    Lb.copy_(logits[t])
        return forward

    pipe = Pipeline(w, layers=LAYERS)
    before, after = [], []
    for t in range(2):
        main.synchronize()
        before.append(_snap(pipe))
        pipe.step_overlapped(Hb, Qb, Wks, Wvs, Lb, main, drift, forward=forward_for(t),
                             init_us=us if t == 0 else None, first=(t == 0))
        main.synchronize()
        ps.ps_check()
        after.append(_snap(pipe))

    # the single-stream step on the same inputs: bit-identical
    seq = Pipeline(w, layers=LAYERS)
    for t in range(2):
        seq.step([H[l][t] for l in range(LAYERS)], [Q[l][t] for l in range(LAYERS)], Wks, Wvs,
                 logits[t], init_us=us if t == 0 else None, first=(t == 0))
    torch.cuda.synchronize()
    ref = _snap(seq)
    for a, b in zip(after[1], ref):
        for k in a:
            if k == "A":
                assert all(torch.equal(x, y) for x, y in zip(a[k], b[k]))
            else:
                assert torch.equal(a[k], b[k]), k

    # against the oracle, stage by stage, step 1 (warm start) of every layer
    for l in range(LAYERS):
        g0, g1 = before[1][l], after[1][l]
        Hn, Qn = np_(H[l][1])[0], np_(Q[l][1])[0]
        o = oracle.kmeans_spherical(Hn, np_(g0["mu"])[0].astype(np.float64), w.iters,
                                    np_(g0["chat"])[0])
        ok = o["margin"][-1] > KM_MARGIN
        assert np.array_equal(np_(g1["assign"])[0][ok], o["assign"][ok])
        if o["margin"].min() > KM_MARGIN:
            assert_close(np_(g1["mu"])[0], o["mu"], what="mu")
            assert_close(np_(g1["chat"])[0], o["chat"], what="chat")
        oc, osc, oS, _ = oracle.nvfp4_residual(Hn, np_(g1["mu"])[0], np_(g1["assign"])[0],
                                               np_(g1["rho"])[0])
        assert np.array_equal(np_(g1["codes"])[0], oc)
        assert np.array_equal(np_(g1["scales"])[0], osc)
        Kt = oracle.centroid_keys(np_(g1["chat"])[0], np_(Ls[l]["Wk"]))
        A_prev = np_(g0["A"][0])[0]        # step 0 wrote A[0], step 1 A[1]
        oA, oD = oracle.proxy_attn_kl(Qn, Kt, w.Hq, w.Hkv, w.dh, A_prev)
        assert_close(np_(g1["A"][1])[0], oA, what="A")
        assert_close(np_(g1["D"])[0], oD, what="D")
        sel, _, pos, npos, _, _ = oracle.topk_drift(np_(g1["D"])[0], np_(g1["assign"])[0],
                                                    np_(g1["counts"])[0], w.k)
        assert np.array_equal(np_(g1["sel"])[0], sel)
        assert int(np_(g1["npos"])[0]) == npos
        assert np.array_equal(np_(g1["pos"])[0], pos)
        Kc = np_(g1["Kc"])[0].reshape(w.Ncache, -1)
        Kc0 = np_(g0["Kc"])[0].reshape(w.Ncache, -1)
        rows = pos[:npos]
        _kv_check(Kc[rows], Hn[rows] @ np_(Ls[l]["Wk"]).astype(np.float64))
        others = np.setdiff1d(np.arange(w.N), rows)
        assert np.array_equal(Kc[others], Kc0[others])

    # the commit of step 1 on the last layer's drift and position mask
    c0, c1 = before[1][LAYERS], after[1][LAYERS]
    last = after[1][LAYERS - 1]
    role = np_(pipe.role)
    D_blk = np_(last["D"])[0][w.blk_start:w.blk_start + w.P]
    p = oracle.CommitParams(w.tau_s, w.alpha, w.ratio, w.mode, 1)
    mask = np.zeros(w.N, np.uint8)
    mask[np_(last["pos"])[0][:int(np_(last["npos"])[0])]] = 1
    oc = oracle.commit_rule(np_(logits[1])[0], role, np_(c0["undecided"])[0], D_blk,
                            np_(c0["d_sum"])[0], np_(c0["d_cnt"])[0], np_(c0["d_prev"])[0],
                            mask[w.blk_start:w.blk_start + w.P], p)
    assert np.array_equal(np_(c1["token"])[0], oc["token"])
    assert_close(np_(c1["conf"])[0], oc["conf"], rtol=CONF_RTOL, atol=0, what="conf")
    if not (oc["margin"] <= BAND).any():
        assert np.array_equal(np_(c1["commit"])[0], oc["commit"])
