"""The decode loop under the refresh schedule, step by step against the oracle.

Each step is checked from the GPU's own state before it (so that a near-tie
in one step cannot cascade): the action taken equals the oracle schedule's
decision on the previous step's committed count and block state; a step
without REFRESH leaves every layer's clustering, drift and cache untouched;
a refreshing step matches the oracle's k-means (k-means++ on REINIT), proxy
drift (no previous distribution on REINIT), top-k and refresh (every row
from H on FULL, only the top-k rows otherwise); the commit of every step
matches the oracle's rule on the last layer's drift, with suffix-block tokens
gated by the last layer's position mask."""
import numpy as np
import pytest
import torch

import oracle
from oracle.schedule import ScheduleState, schedule_step
from drift_aware_kv_spherical_gb300 import polestar as ps
from drift_aware_kv_spherical_gb300 import workloads as wl
from drift_aware_kv_spherical_gb300.pipeline import Pipeline
from tests._parity import BAND, KM_MARGIN, assert_close, np_

pytestmark = pytest.mark.gpu

TAU_UPD, FULL_PERIOD, TAU_S, STEPS, LAYERS = 4, 2, 0.95, 24, 2


@pytest.fixture(autouse=True)
def _lib(lib):
    return lib


def _kv_check(g, o):
    rms = np.sqrt(np.mean(o.astype(np.float64) ** 2, axis=-1, keepdims=True))
    assert np.all(np.abs(g - o) <= 1e-5 * np.abs(o) + 1e-3 * rms)


class _Inputs:
    """Per-step inputs of the tiny fp32 workload: window `block_start // P`
    has its own seeded layers; step t drifts them once more."""

    def __init__(self, w, pipe):
        self.w, self.pipe, self.snap = w, pipe, []
        self.layers = {}

    def layer(self, l, widx):
        key = (l, widx)
        if key not in self.layers:
            L = wl.make_layer(self.w, l + 10 * widx, "cuda")
            self.layers[key] = (L, wl.make_uniforms(self.w, l + 10 * widx, "cuda"))
        return self.layers[key]

    def __call__(self, t, block_start):
        w, pipe = self.w, self.pipe
        widx = block_start // w.P
        Hs, Qs, Wks, Wvs, us = [], [], [], [], []
        for l in range(pipe.layers):
            L, u = self.layer(l, widx)
            H = wl.drift_rows(w, L["H"], t + 1, l)
            Hs.append(H)
            Qs.append(wl.make_queries(w, H, L["Wq"]))
            Wks.append(L["Wk"])
            Wvs.append(L["Wv"])
            us.append(u)
        logits = wl.make_logits(w, t, "cuda")
        torch.cuda.synchronize()
        self.snap.append(dict(pre=_state(pipe), Hs=Hs, Qs=Qs, Wks=Wks, Wvs=Wvs, us=us,
                              logits=logits))
        return Hs, Qs, Wks, Wvs, logits, us


def _state(pipe):
    layers = []
    for st in pipe.state:
        layers.append({k: np_(getattr(st, k)).copy()
                       for k in ("mu", "assign", "counts", "chat", "D", "posmask", "Kc", "Vc")})
        layers[-1]["A_cur"] = np_(st.A[(pipe.t + 1) % 2]).copy()   # written by the last refresh
    return dict(t=pipe.t, layers=layers,
                **{k: np_(getattr(pipe, k)).copy()
                   for k in ("undecided", "d_sum", "d_cnt", "d_prev", "commit")})


def _check_layer(w, pre, post, H, Q, Wk, Wv, u, act):
    Hn, Qn = np_(H[0]).astype(np.float64), np_(Q[0])
    # k-means from the GPU's previous centroids, or k-means++ on REINIT
    pinned = True
    if act & ps.SCHED_REINIT:  # a seeding draw inside the tie band leaves the clustering unpinned
        mu0, _, m0 = oracle.kmeanspp_init(Hn, w.C, np_(u[0]), return_margin=True)
        pinned = m0 > 1e-5
    else:
        mu0 = pre["mu"][0].astype(np.float64)
    if pinned:
        o = oracle.kmeans_spherical(Hn, mu0, w.iters)
        ok = o["margin"][-1] > KM_MARGIN
        assert ok.mean() > 0.9
        assert np.array_equal(post["assign"][0][ok], o["assign"][ok])
    # proxy drift from the GPU's centroid summaries and previous distribution
    Kt = oracle.centroid_keys(post["chat"][0], np_(Wk))
    A_prev = None if act & ps.SCHED_REINIT else pre["A_cur"][0]
    oA, oD = oracle.proxy_attn_kl(Qn, Kt, w.Hq, w.Hkv, w.dh, A_prev)
    assert_close(post["A_cur"][0], oA, what="A")
    assert_close(post["D"][0], oD, what="D")
    # top-k of the GPU's drift, then the refresh
    _, _, pos, npos, pm, _ = oracle.topk_drift(post["D"][0], post["assign"][0],
                                               post["counts"][0], w.k)
    assert np.array_equal(post["posmask"][0], pm)
    Kpre = pre["Kc"][0].reshape(w.Ncache, -1)
    Vpre = pre["Vc"][0].reshape(w.Ncache, -1)
    if act & ps.SCHED_FULL:
        pos, npos = np.arange(w.N), w.N
    oK, oV = oracle.refresh_kv(Hn, pos, npos, np_(Wk), np_(Wv), Kpre, Vpre, 0, False)
    gK, gV = post["Kc"][0].reshape(w.Ncache, -1), post["Vc"][0].reshape(w.Ncache, -1)
    touched = np.zeros(w.Ncache, bool)
    touched[pos[:npos]] = True
    assert np.array_equal(gK[~touched], Kpre[~touched])
    assert np.array_equal(gV[~touched], Vpre[~touched])
    _kv_check(gK[touched], oK[touched])
    _kv_check(gV[touched], oV[touched])
    return int(touched.sum()), int(pinned)


def test_decode_loop_follows_the_schedule():
    w = wl.WORKLOADS[0]
    role = torch.zeros(w.P, dtype=torch.uint8)
    role[12:] = wl.ROLE_SUFFIX                        # 12 current-block, 4 suffix tokens
    pipe = Pipeline(w, layers=LAYERS, role=role)
    pipe.params = ps.CommitParams(TAU_S, w.alpha, w.ratio, w.mode, 1)
    sched = ps.Schedule(TAU_UPD, FULL_PERIOD, w.P)
    inputs = _Inputs(w, pipe)
    acts = pipe.decode(sched, inputs, STEPS)
    torch.cuda.synchronize()
    ps.ps_check()
    post_final = _state(pipe)
    role_n = np_(role)
    p = oracle.CommitParams(tau_s=TAU_S, alpha=w.alpha, ratio=w.ratio, mode=w.mode,
                            ensure_progress=1)
    o_sched = ScheduleState()
    expect = ps.SCHED_REFRESH | ps.SCHED_FULL | ps.SCHED_REINIT
    seen = {0: 0, ps.SCHED_REFRESH: 0, ps.SCHED_FULL: 0, ps.SCHED_SLIDE: 0}
    suffix_checked = refreshed_rows = pinned_km = 0
    for t in range(STEPS):
        s = inputs.snap[t]
        pre = s["pre"]
        post = inputs.snap[t + 1]["pre"] if t + 1 < STEPS else post_final
        act = acts[t]
        assert act == expect, (t, act, expect)
        for f in seen:
            seen[f] += int(act == 0) if f == 0 else int(bool(act & f))
        for l in range(LAYERS):
            a, b = pre["layers"][l], post["layers"][l]
            if act & ps.SCHED_REFRESH:
                n, pin = _check_layer(w, a, b, s["Hs"][l], s["Qs"][l], s["Wks"][l],
                                      s["Wvs"][l], s["us"][l], act)
                refreshed_rows += n
                pinned_km += pin
            else:                                     # the cache is reused as it stands
                for k in a:
                    assert np.array_equal(a[k], b[k]), (t, l, k)
        # the commit: state reset on SLIDE, the last layer's drift and mask
        und, dsum, dcnt, dprev = (pre[k][0] for k in ("undecided", "d_sum", "d_cnt", "d_prev"))
        if act & ps.SCHED_SLIDE:
            und, dsum = np.ones_like(und), np.zeros_like(dsum)
            dcnt, dprev = np.zeros_like(dcnt), np.zeros_like(dprev)
        last = post["layers"][-1]
        blk = slice(w.blk_start, w.blk_start + w.P)
        r = oracle.commit_rule(np_(s["logits"][0]), role_n, und, last["D"][0][blk], dsum, dcnt,
                               dprev, last["posmask"][0][blk], p)
        ok = r["margin"] > BAND
        assert ok.all()
        assert np.array_equal(post["commit"][0], r["commit"].astype(np.uint8))
        assert np.array_equal(post["undecided"][0], np.asarray(r["undecided"], np.uint8))
        assert_close(post["d_sum"][0], r["d_sum"], what="d_sum")
        assert np.array_equal(post["d_cnt"][0], r["d_cnt"])
        sfx = (role_n == wl.ROLE_SUFFIX) & (und == 1) & (r["conf"] >= TAU_S)
        suffix_checked += int(sfx.sum())
        # the schedule's decision for the next step, from this step's outcome
        committed = int(r["commit"].sum())
        done = not bool(((np.asarray(r["undecided"]) == 1) & (role_n == wl.ROLE_CURRENT)).any())
        expect = schedule_step(TAU_UPD, FULL_PERIOD, w.P, o_sched, committed, done)
    assert all(v > 0 for v in seen.values()), seen  # every kind of step was exercised
    assert suffix_checked > 0 and refreshed_rows > 0 and pinned_km >= 8
    assert sched.state.block_start == o_sched.block_start > 0


def test_full_step_refreshes_every_row_of_an_offloaded_layer():
    """LLaDA-8B-shaped layer in offload mode: a FULL step refreshes every row
    from H (not from the store's reconstruction), sampled against the oracle;
    the next top-k step refreshes only the top-k rows."""
    w = wl.WORKLOADS[1]
    L = wl.make_layer(w, 0, "cuda")
    Q = wl.make_queries(w, L["H"], L["Wq"])
    u = wl.make_uniforms(w, 0, "cuda")
    logits = wl.make_logits(w, 0, "cuda")
    pipe = Pipeline(w, layers=1, offload=True)
    full = ps.SCHED_REFRESH | ps.SCHED_FULL | ps.SCHED_REINIT
    pipe.decode_step(full, [L["H"]], [Q], [L["Wk"]], [L["Wv"]], logits, init_us=[u])
    torch.cuda.synchronize()
    ps.ps_check()
    st = pipe.state[0]
    K1 = np_(st.Kc[0]).reshape(w.N, -1)
    Hn, Wkn = np_(L["H"][0]).astype(np.float64), np_(L["Wk"]).astype(np.float64)
    for i in range(0, w.N, 97):
        ref = oracle.bf16_round(Hn[i] @ Wkn)
        rms = np.sqrt(np.mean(ref.astype(np.float64) ** 2))
        assert np.all(np.abs(K1[i] - ref) <= 2e-2 * np.abs(ref) + 1e-3 * rms), i
    H1 = wl.drift_rows(w, L["H"], 1)
    pipe.decode_step(ps.SCHED_REFRESH, [H1], [wl.make_queries(w, H1, L["Wq"])], [L["Wk"]],
                     [L["Wv"]], logits)
    torch.cuda.synchronize()
    ps.ps_check()
    K2 = np_(st.Kc[0]).reshape(w.N, -1)
    touched = np.zeros(w.N, bool)
    touched[np_(st.pos[0])[: int(np_(st.npos)[0])]] = True
    assert 0 < touched.sum() < w.N
    assert np.array_equal(K2[~touched], K1[~touched])


@pytest.mark.parametrize("widx,steps", [(0, 20), (1, 12)])
def test_graph_decode_matches_eager(widx, steps):
    """The decode loop through CUDA graphs (one per action kind and
    distribution parity, captured on first use) gives the eager loop's
    actions and every output bit for bit: the same kernels in the same order."""
    w = wl.WORKLOADS[widx]
    layers = min(2, w.layers) if widx == 0 else 1
    cache = {}

    def inputs(t, block_start):
        widx_ = block_start // w.P
        Hs, Qs, Wks, Wvs, us = [], [], [], [], []
        for l in range(layers):
            if (l, widx_) not in cache:
                cache[(l, widx_)] = (wl.make_layer(w, l + 10 * widx_, "cuda"),
                                     wl.make_uniforms(w, l + 10 * widx_, "cuda"))
            L, u = cache[(l, widx_)]
            H = wl.drift_rows(w, L["H"], t + 1, l)
            Hs.append(H)
            Qs.append(wl.make_queries(w, H, L["Wq"]))
            us.append(u)
        Ws = [cache[(l, 0)][0] for l in range(layers)]    # one set of weights for every window
        logits = wl.make_logits(w, t, "cuda").to(wl.torch_dtype(w))
        return Hs, Qs, [x["Wk"] for x in Ws], [x["Wv"] for x in Ws], logits, us

    outs = []
    for graphs in (False, True):
        pipe = Pipeline(w, layers=layers)
        pipe.params = ps.CommitParams(TAU_S, w.alpha, w.ratio, w.mode, 1)
        acts = pipe.decode(ps.Schedule(TAU_UPD, FULL_PERIOD, w.P), inputs, steps, graphs=graphs)
        torch.cuda.synchronize()
        ps.ps_check()
        st = [(x.mu, x.assign, x.D, x.A[0], x.A[1], x.Kc, x.Vc, x.posmask) for x in pipe.state]
        outs.append((acts, [t.clone() for layer in st for t in layer],
                     [t.clone() for t in (pipe.undecided, pipe.d_sum, pipe.d_cnt, pipe.token)]))
    (a0, s0, c0), (a1, s1, c1) = outs
    assert a0 == a1
    assert len(set(a0)) >= 3                                  # several kinds of step replayed
    for x, y in zip(s0 + c0, s1 + c1):
        assert torch.equal(x, y)


@pytest.mark.parametrize("B,P", [(1, 16), (4, 32), (32, 64), (3, 1000)])
def test_block_progress_matches_oracle(B, P):
    g = torch.Generator(device="cuda").manual_seed(B * 1000 + P)
    role = torch.randint(0, 3, (P,), device="cuda", generator=g, dtype=torch.uint8)
    out = ps.HostStore(16)
    view = out.view()[:8].view("int32")
    dev_out = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    for density in (0.0, 0.02, 0.5):
        commit = (torch.rand(B, P, device="cuda", generator=g) < density).to(torch.uint8)
        undecided = (torch.rand(B, P, device="cuda", generator=g) < density).to(torch.uint8)
        ps.ps_block_progress(commit, undecided, role, out)
        ps.ps_block_progress(commit, undecided, role, dev_out)
        torch.cuda.synchronize()
        ps.ps_check()
        want = oracle.block_progress(np_(commit).tolist(), np_(undecided).tolist(),
                                     np_(role).tolist())
        assert (int(view[0]), bool(view[1])) == want
        assert (int(dev_out[0]), bool(dev_out[1])) == want
