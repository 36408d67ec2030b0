"""Parity at the C ABI's largest sizes (include/polestar.h): d = 8192 and
C = 256 for k-means (bf16 on the tensor cores, fp32 on CUDA cores), dh = 256
with C = 256 for the proxy, d = 8192 for the K/V refresh, P = 1024 positions
for the commit.  Windows are short so the oracle stays quick."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from drift_aware_kv_spherical_gb300 import polestar as ps
from drift_aware_kv_spherical_gb300 import workloads as wl
from tests._parity import (BAND, CONF_RTOL, KM_MARGIN, assert_close, np_, run_commit,
                           run_kmeans, run_proxy)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_kmeans_largest_d_and_c(dt):
    rng = np.random.default_rng(8192 + (dt == "f32"))
    B, N, d, C, iters = 1, 640, 8192, 256, 2
    planted = oracle.normalize_rows(rng.standard_normal((C, d)))
    z = np.arange(N) % C
    H = (planted[z] * 40 + rng.normal(0, 0.3, (N, d)))[None].astype(np.float32)
    Ht = torch.from_numpy(H).cuda()
    if dt == "bf16":
        Ht = Ht.to(torch.bfloat16)
    Hn = np_(Ht)
    mu0 = oracle.normalize_rows(Hn[0][:C])[None].astype(np.float32)
    g = run_kmeans(Ht, torch.from_numpy(mu0).cuda(), iters)
    o = oracle.kmeans_spherical(Hn[0], mu0[0].astype(np.float64), iters)
    ok = o["margin"][-1] > KM_MARGIN
    assert ok.mean() > 0.99
    assert np.array_equal(g["assign"][0][ok], o["assign"][ok])
    if o["margin"].min() > KM_MARGIN:
        assert np.array_equal(g["counts"][0], o["counts"])
        assert_close(g["mu"][0], o["mu"], what="mu")
        assert_close(g["chat"][0], o["chat"], what="chat")
        assert_close(g["obj"][0], o["obj"], what="objective")


def test_proxy_largest_dh_and_c():
    rng = np.random.default_rng(256)
    B, N, Hq, Hkv, dh, C, d = 1, 200, 4, 2, 256, 256, 256
    Q = torch.from_numpy(rng.standard_normal((B, N, Hq, dh)).astype(np.float32))
    Q = Q.to(torch.bfloat16).cuda()
    chat = torch.from_numpy(rng.standard_normal((B, C, d)).astype(np.float32)).cuda()
    Wk = torch.from_numpy((rng.standard_normal((d, Hkv * dh)) * 0.05).astype(np.float32))
    Wk = Wk.to(torch.bfloat16).cuda()
    prev = torch.softmax(torch.randn(B, N, C, device="cuda"), dim=2)
    A, D = run_proxy(Q, chat, Wk, Hkv, A_prev=prev)
    w = dataclasses.replace(wl.WORKLOADS[0], Hq=Hq, Hkv=Hkv, dh=dh)
    Kt = oracle.centroid_keys(np_(chat)[0], np_(Wk))
    oA, oD = oracle.proxy_attn_kl(np_(Q)[0], Kt, w.Hq, w.Hkv, w.dh, np_(prev)[0])
    assert_close(np_(A)[0], oA, what="A")
    assert_close(np_(D)[0], oD, what="D")


def test_refresh_largest_d():
    rng = np.random.default_rng(8193)
    B, N, d, Hkv, dh = 1, 96, 8192, 2, 128
    H = torch.from_numpy(rng.standard_normal((B, N, d)).astype(np.float32)).cuda().to(torch.bfloat16)
    Wk = torch.from_numpy((rng.standard_normal((d, Hkv * dh)) * 0.02).astype(np.float32)).cuda().to(torch.bfloat16)
    Wv = torch.from_numpy((rng.standard_normal((d, Hkv * dh)) * 0.02).astype(np.float32)).cuda().to(torch.bfloat16)
    sel = np.sort(rng.choice(N, 40, replace=False)).astype(np.int32)
    pos = torch.full((B, N), -1, dtype=torch.int32)
    pos[0, :40] = torch.from_numpy(sel)
    pos = pos.cuda()
    npos = torch.tensor([40], dtype=torch.int32, device="cuda")
    Kc = torch.zeros(B, N, Hkv, dh, device="cuda", dtype=torch.bfloat16)
    Vc = torch.zeros_like(Kc)
    ws = ps.workspace(ps.OP_REFRESH, B=B, N=N, d=d, Hkv=Hkv, dh=dh)
    ps.ps_refresh_kv(H, pos, npos, Wk, Wv, Kc, Vc, Hkv, dh, ws=ws)
    torch.cuda.synchronize()
    ps.ps_check()
    Hn = np_(H)[0].astype(np.float64)
    for Wt, cache in ((Wk, Kc), (Wv, Vc)):
        want = oracle.bf16_round(Hn[sel] @ np_(Wt).astype(np.float64))
        got = np_(cache)[0].reshape(N, -1)[sel]
        rms = np.sqrt(np.mean(want ** 2, axis=-1, keepdims=True))
        assert np.all(np.abs(got - want) <= 2e-2 * np.abs(want) + 1e-3 * rms)
        untouched = np.setdiff1d(np.arange(N), sel)
        assert np.all(np_(cache)[0].reshape(N, -1)[untouched] == 0)


def test_commit_largest_p():
    rng = np.random.default_rng(1024)
    B, P, V = 2, 1024, 4096
    Ln = rng.normal(0, 3, (B, P, V)).astype(np.float32)
    peak = rng.random((B, P)) < 0.5
    idx = rng.integers(0, V, (B, P))
    bb, pp = np.nonzero(peak)
    Ln[bb, pp, idx[bb, pp]] += 25.0
    logits = torch.from_numpy(Ln).cuda()
    role = np.zeros(P, np.uint8)
    role[P // 2:] = 1
    und = np.ones((B, P), np.uint8)
    D = rng.gamma(2.0, 0.05, (B, P)).astype(np.float32)
    cnt = rng.integers(0, 4, (B, P)).astype(np.int32)
    s = (cnt * rng.gamma(2.0, 0.05, (B, P))).astype(np.float32)
    prev = rng.gamma(2.0, 0.05, (B, P)).astype(np.float32)
    ssel = (rng.random((B, P)) < 0.5).astype(np.uint8)
    p = oracle.CommitParams(tau_s=0.9, alpha=1.0, ratio=0.1, mode=0, ensure_progress=1)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    g = run_commit(logits, dev(role), dev(und), dev(D), P, dev(s), dev(cnt), dev(prev),
                   dev(ssel), ps.CommitParams(p.tau_s, p.alpha, p.ratio, p.mode,
                                              p.ensure_progress))
    for b in range(B):
        o = oracle.commit_rule(Ln[b], role, und[b], D[b], s[b], cnt[b], prev[b], ssel[b], p)
        assert np.array_equal(g["token"][b], o["token"])
        assert_close(g["conf"][b], o["conf"], rtol=CONF_RTOL, atol=0, what="conf")
        if not (o["margin"] <= BAND).any():
            assert np.array_equal(g["commit"][b], o["commit"])
            assert np.array_equal(g["undecided"][b], o["undecided"])
        assert np.array_equal(g["d_sum"][b], o["d_sum"])
        assert np.array_equal(g["d_cnt"][b], o["d_cnt"])
