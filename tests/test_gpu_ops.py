"""GPU parity of every libpolestar call against the CPU oracle.

Each test feeds both sides identical seeded inputs (oracle-produced where a
call consumes an earlier stage's output) and compares element by element with
the path's criteria: integer outputs bit-exact, k-means assignments exact
where the oracle's top-2 margin exceeds 1e-5, fp32 outputs within 1e-4
relative / 1e-6 absolute, bf16 K/V within 2e-2 relative.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
from drift_aware_kv_spherical_gb300 import polestar as ps
from drift_aware_kv_spherical_gb300 import workloads as wl
from tests._parity import (ATOL, BAND, CONF_RTOL, KM_MARGIN, KV_RTOL, RTOL, Guarded,
                           assert_close, np_, run_commit, run_kmeans, run_nvfp4,
                           run_proxy, run_topk)

pytestmark = pytest.mark.gpu

SMALL = [0, 1]   # tiny fp32 layer; LLaDA-8B-shaped bf16 layer (full size)


@pytest.fixture(autouse=True)
def _lib(lib):
    return lib


def _layer(widx, device="cuda"):
    w = wl.WORKLOADS[widx]
    L = wl.make_layer(w, 0, device)
    return w, L


def _oracle_km(Hn, mu0, iters, chat0=None):
    return [oracle.kmeans_spherical(Hn[b], mu0[b], iters,
                                    None if chat0 is None else chat0[b])
            for b in range(Hn.shape[0])]


# ---------------------------------------------------------------- k-means
@pytest.mark.parametrize("widx", SMALL)
def test_kmeanspp_seeding(widx):
    w, L = _layer(widx)
    u = wl.make_uniforms(w, 0, "cuda")
    g = run_kmeans(L["H"], torch.zeros(w.B, w.C, w.d, device="cuda"), 0, init_u=u)
    Hn, un = np_(L["H"]), np_(u)
    for b in range(w.B):
        mu, idx, margin = oracle.kmeanspp_init(Hn[b], w.C, un[b], return_margin=True)
        if margin < 1e-5:
            pytest.skip(f"draw within {margin:.1e} of a boundary (unpinned)")
        assert_close(g["mu"][b], mu, rtol=0, atol=2e-6, what="kmeans++ centres")


@pytest.mark.parametrize("widx", SMALL)
def test_kmeans_each_pass(widx):
    """Every pass, fed the oracle's centroids: assignments, rho, counts,
    C_hat and objective; then one update from them."""
    w, L = _layer(widx)
    H = L["H"]
    Hn = np_(H)
    u = np_(wl.make_uniforms(w, 0, "cuda"))
    mu0 = np.stack([oracle.kmeanspp_init(Hn[b], w.C, u[b])[0] for b in range(w.B)])
    ref = _oracle_km(Hn, mu0, w.iters)
    for t in range(w.iters + 1):
        mu_t = np.stack([ref[b]["mus"][t] for b in range(w.B)]).astype(np.float32)
        mu_dev = torch.from_numpy(mu_t).cuda()
        g = run_kmeans(H, mu_dev, 0)
        o = _oracle_km(Hn, mu_t.astype(np.float64), 0)
        for b in range(w.B):
            ok = o[b]["margin"][0] > KM_MARGIN
            assert ok.mean() > 0.99
            assert np.array_equal(g["assign"][b][ok], o[b]["assign"][ok]), f"pass {t}"
            if ok.all():
                assert np.array_equal(g["counts"][b], o[b]["counts"])
                assert_close(g["rho"][b], o[b]["rho"], what="rho")
                assert_close(g["chat"][b], o[b]["chat"], what="chat")
                assert_close(g["obj"][b][0], o[b]["obj"][0], what="objective")
        if t < w.iters:
            g1 = run_kmeans(H, mu_dev, 1)
            o1 = _oracle_km(Hn, mu_t.astype(np.float64), 1)
            for b in range(w.B):
                if (o1[b]["margin"] > KM_MARGIN).all():
                    assert_close(g1["mu"][b], o1[b]["mu"], what=f"update {t}")
                    assert np.allclose(np.linalg.norm(g1["mu"][b], axis=1), 1, atol=1e-5)


@pytest.mark.parametrize("widx", SMALL)
def test_kmeans_whole_run(widx):
    w, L = _layer(widx)
    u = wl.make_uniforms(w, 0, "cuda")
    g = run_kmeans(L["H"], torch.zeros(w.B, w.C, w.d, device="cuda"), w.iters, init_u=u)
    Hn, un = np_(L["H"]), np_(u)
    for b in range(w.B):
        mu0, _, m0 = oracle.kmeanspp_init(Hn[b], w.C, un[b], return_margin=True)
        o = oracle.kmeans_spherical(Hn[b], mu0, w.iters)
        if m0 < 1e-5 or o["margin"].min() <= KM_MARGIN:
            pytest.skip("a decision inside the tie band (unpinned)")
        assert np.array_equal(g["assign"][b], o["assign"])
        assert np.array_equal(g["counts"][b], o["counts"])
        assert_close(g["mu"][b], o["mu"], what="mu")
        assert_close(g["rho"][b], o["rho"], what="rho")
        assert_close(g["chat"][b], o["chat"], what="chat")
        assert_close(g["obj"][b], o["obj"], what="objective")
        assert np.all(np.diff(g["obj"][b]) >= -1e-4 * abs(g["obj"][b][-1]))


def test_kmeans_ragged_and_degenerate():
    rng = np.random.default_rng(5)
    # N = 17 rows (ragged tile), C = 3, d = 48 (not a multiple of 32), one zero row
    H = rng.standard_normal((2, 17, 48)).astype(np.float32)
    H[1, 4] = 0.0
    mu0 = oracle.normalize_rows(rng.standard_normal((3, 48)))
    mu0b = np.stack([mu0, mu0[::-1].copy()]).astype(np.float32)
    g = run_kmeans(torch.from_numpy(H).cuda(), torch.from_numpy(mu0b).cuda(), 4)
    for b in range(2):
        o = oracle.kmeans_spherical(H[b], mu0b[b].astype(np.float64), 4)
        if o["margin"].min() > KM_MARGIN:
            assert np.array_equal(g["assign"][b], o["assign"])
            assert_close(g["mu"][b], o["mu"], what="mu")
            assert_close(g["chat"][b], o["chat"], what="chat")
    assert g["assign"][1][4] == 0 and g["rho"][1][4] == 0.0
    # C = 1: the normalised mean direction
    g1 = run_kmeans(torch.from_numpy(H[:1]).cuda(), torch.from_numpy(mu0b[:1, :1]).cuda(), 1)
    o1 = oracle.kmeans_spherical(H[0], mu0b[0, :1].astype(np.float64), 1)
    assert_close(g1["mu"][0], o1["mu"], what="C=1")


@pytest.mark.parametrize("B,N,d,C,iters,dt", [(3, 177, 80, 24, 3, "bf16"),
                                               (2, 300, 256, 128, 2, "bf16"),
                                               (1, 129, 64, 64, 1, "bf16"),
                                               (1, 301, 1552, 20, 2, "bf16"),
                                               (1, 333, 320, 150, 2, "bf16"),
                                               (1, 200, 1040, 5, 2, "f32")])
def test_kmeans_ragged_tiles(B, N, d, C, iters, dt):
    """bf16 windows on the tensor-core path: row tiles straddling windows,
    C not a power of two, a partial 64-wide K block, iters >= 1; d-chunks
    reduced in a thread-block cluster (2 and 4 chunks) and, for C = 150 > 128,
    through global memory (5 chunks).  The 1552- and 1040-column cases give few
    (cluster, window) pairs, so the centroid update splits d into 2 (bf16) and
    4 (f32) column slices, the last one shorter."""
    rng = np.random.default_rng(N + C)
    planted = oracle.normalize_rows(rng.standard_normal((C, d)))
    z = rng.integers(0, C, (B, N))
    H = (planted[z] * 4 + rng.normal(0, 0.3, (B, N, d))).astype(np.float32)
    Ht = torch.from_numpy(H).cuda()
    if dt == "bf16":
        Ht = Ht.to(torch.bfloat16)
    Hn = np_(Ht)
    mu0 = np.stack([oracle.normalize_rows(Hn[b][:C]) for b in range(B)]).astype(np.float32)
    g = run_kmeans(Ht, torch.from_numpy(mu0).cuda(), iters)
    checked = 0
    for b in range(B):
        o = oracle.kmeans_spherical(Hn[b], mu0[b].astype(np.float64), iters)
        ok = o["margin"][-1] > KM_MARGIN
        assert np.array_equal(g["assign"][b][ok], o["assign"][ok])
        if o["margin"].min() > KM_MARGIN:
            checked += 1
            assert np.array_equal(g["counts"][b], o["counts"])
            assert_close(g["mu"][b], o["mu"], what="mu")
            assert_close(g["rho"][b], o["rho"], what="rho")
            assert_close(g["chat"][b], o["chat"], what="chat")
            assert_close(g["obj"][b], o["obj"], what="objective")
    assert checked >= 1


def test_kmeans_empty_cluster_keeps_centroid_and_chat():
    H = np.tile(np.array([[1.0, 0.1] + [0.0] * 14], np.float32), (5, 1))[None]
    far = np.zeros(16, np.float32); far[0] = -1.0
    mu0 = np.stack([np.eye(16, dtype=np.float32)[0], far])[None]
    chat0 = np.full((1, 2, 16), 3.0, np.float32)
    g = run_kmeans(torch.from_numpy(H).cuda(), torch.from_numpy(mu0).cuda(), 2,
                   chat0=torch.from_numpy(chat0).cuda())
    assert np.array_equal(g["mu"][0][1], far)
    assert np.all(g["chat"][0][1] == 3.0) and g["counts"][0][1] == 0


# ---------------------------------------------------------------- NVFP4
@pytest.mark.parametrize("widx", SMALL)
def test_nvfp4_oracle_fed(widx):
    w, L = _layer(widx)
    H = L["H"]
    Hn = np_(H)
    rng = np.random.default_rng(widx)
    mu = oracle.normalize_rows(rng.standard_normal((w.C, w.d)))
    ref = oracle.kmeans_spherical(Hn[0], mu, 2)
    mu32 = np.broadcast_to(ref["mu"].astype(np.float32), (w.B, w.C, w.d)).copy()
    a = np.broadcast_to(ref["assign"].astype(np.int32), (w.B, w.N)).copy()
    rho = np.broadcast_to(ref["rho"].astype(np.float32), (w.B, w.N)).copy()
    codes, scales, S = run_nvfp4(H, torch.from_numpy(mu32).cuda(),
                                 torch.from_numpy(a).cuda(), torch.from_numpy(rho).cuda())
    for b in range(w.B):
        oc, os_, oS, _ = oracle.nvfp4_residual(Hn[b], mu32[b], a[b], rho[b])
        assert S[b] == oS
        assert np.array_equal(scales[b], os_)
        assert np.array_equal(codes[b], oc)


def _e2m1_probe_values():
    """fp32 values in [-6, 6]: a strided sweep of bit patterns plus +-3 ulp
    around every rounding midpoint and grid point of E2M1."""
    pos = np.arange(0, 0x40C00001, 4099, dtype=np.uint64).astype(np.uint32).view(np.float32)
    marks = [0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, 6.0]
    near = []
    for m in marks:
        x = np.float32(m)
        for k in range(-3, 4):
            v = x
            for _ in range(abs(k)):
                v = np.nextafter(v, np.float32(np.inf if k > 0 else -np.inf), dtype=np.float32)
            near.append(v)
    near.extend([np.float32(0.0), np.float32(1e-30), np.float32(1e-45)])
    v = np.concatenate([pos, np.array(near, np.float32)])
    v = v[np.abs(v) <= 6.0]
    return np.concatenate([v, -v]).astype(np.float32)


def test_nvfp4_e2m1_conversion_sweep():
    """Every block holds a 6.0 (block scale 1) and the window amax is 2688
    (tensor scale 1), so element codes are E2M1(value) directly."""
    vals = _e2m1_probe_values()
    per_row = 256 // 16 * 15
    n_rows = math.ceil(len(vals) / per_row)
    body = np.zeros(n_rows * per_row, np.float32)
    body[:len(vals)] = vals
    body = body.reshape(n_rows, 16, 15)
    H = np.concatenate([np.full((n_rows, 16, 1), 6.0, np.float32), body], axis=2)
    H = H.reshape(n_rows, 256)
    H = np.concatenate([np.zeros((1, 256), np.float32), H])
    H[0, :16] = 0.0
    H[0, 0] = 2688.0
    codes, scales, S = run_nvfp4(torch.from_numpy(H[None]).cuda(), None, None, None)
    oc, os_, oS, _ = oracle.nvfp4_residual(H, None, None, None)
    assert S[0] == oS == 1.0
    assert np.array_equal(scales[0], os_)
    assert np.array_equal(codes[0], oc)


def test_nvfp4_e4m3_scale_sweep():
    """Block amax 6 m (S = 1) makes the block scale E4M3(m) for m over the
    whole E4M3 range, its midpoints and random values."""
    grid = oracle.e4m3_decode(np.arange(127)).astype(np.float64)
    mids = (grid[:-1] + grid[1:]) / 2
    rng = np.random.default_rng(3)
    ms = np.concatenate([grid, mids, rng.uniform(0, 448, 2000),
                         np.ldexp(rng.uniform(1, 2, 500), rng.integers(-12, 0, 500))])
    ms = ms.astype(np.float32)
    nb = len(ms)
    rows = math.ceil(nb / 16)
    H = np.zeros((rows * 16, 16), np.float32)
    H[:nb, 0] = (np.float32(6.0) * ms).astype(np.float32)
    H[:nb, 1] = -ms
    H = H.reshape(rows, 256)
    H = np.concatenate([np.zeros((1, 256), np.float32), H])
    H[0, 0] = 2688.0
    codes, scales, S = run_nvfp4(torch.from_numpy(H[None]).cuda(), None, None, None)
    oc, os_, oS, _ = oracle.nvfp4_residual(H, None, None, None)
    assert S[0] == oS == 1.0
    assert np.array_equal(scales[0], os_)
    assert np.array_equal(codes[0], oc)


def test_nvfp4_codes_at_boundaries_after_division():
    """Blocks with scale s (E4M3 values that are not powers of two, S = 1)
    whose elements are fl(m s) for m within a few ulp of every E2M1 midpoint
    and grid point: the quotient r / s lands on or next to a rounding
    boundary, where the kernel's reciprocal product must give way to the
    IEEE division; every code against the oracle."""
    marks = [0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0]
    ms = []
    for mk in marks:
        x = np.float32(mk)
        for k in range(-2, 3):
            v = x
            for _ in range(abs(k)):
                v = np.nextafter(v, np.float32(np.inf if k > 0 else -np.inf), dtype=np.float32)
            ms.append(v)
    ms = np.array(ms, np.float32)               # 65 multipliers, 15 a block
    scales_e4 = oracle.e4m3_decode(np.arange(1, 127)).astype(np.float32)
    blocks = []
    for sv in scales_e4:
        for j in range(0, len(ms), 15):
            blk = np.zeros(16, np.float32)
            blk[0] = np.float32(6.0) * sv           # block max: scale code E4M3(s) = s
            part = (ms[j:j + 15] * sv).astype(np.float32)
            part[1::2] *= -1
            blk[1:1 + len(part)] = part
            blocks.append(blk)
    body = np.stack(blocks)
    per_row = 256 // 16
    rows = math.ceil(len(body) / per_row)
    H = np.zeros((rows * per_row, 16), np.float32)
    H[:len(body)] = body
    H = H.reshape(rows, 256)
    H = np.concatenate([np.zeros((1, 256), np.float32), H])
    H[0, 0] = 2688.0                            # the window amax: S = 1
    codes, scales, S = run_nvfp4(torch.from_numpy(H[None]).cuda(), None, None, None)
    oc, os_, oS, _ = oracle.nvfp4_residual(H, None, None, None)
    assert S[0] == oS == 1.0
    assert np.array_equal(scales[0], os_)
    assert np.array_equal(codes[0], oc)


def test_nvfp4_zero_and_bf16_input():
    z = torch.zeros(2, 3, 32, device="cuda", dtype=torch.bfloat16)
    codes, scales, S = run_nvfp4(z, None, None, None)
    assert np.all(S == 1.0) and not codes.any() and not scales.any()
    h = torch.randn(2, 5, 64, device="cuda").to(torch.bfloat16)
    codes, scales, S = run_nvfp4(h, None, None, None)
    hn = np_(h)
    for b in range(2):
        oc, os_, oS, _ = oracle.nvfp4_residual(hn[b], None, None, None)
        assert S[b] == oS and np.array_equal(codes[b], oc) and np.array_equal(scales[b], os_)


# ---------------------------------------------------------------- proxy + KL
def _proxy_inputs(widx, B=None, N=None):
    w = wl.WORKLOADS[widx]
    L = wl.make_layer(w, 0, "cuda", B=B)
    H = L["H"][:, :N] if N else L["H"]
    Q = wl.make_queries(w, H, L["Wq"])
    Hn = np_(H)
    u = np_(wl.make_uniforms(w, 0, "cuda", B=H.shape[0]))
    chat = np.stack([oracle.kmeans_spherical(
        Hn[b], oracle.kmeanspp_init(Hn[b], w.C, u[b])[0], 2)["chat"]
        for b in range(H.shape[0])]).astype(np.float32)
    return w, L, H, Q, torch.from_numpy(chat).cuda()


def _oracle_proxy(w, Qn, chat, Wkn, A_prev=None):
    outs = []
    for b in range(Qn.shape[0]):
        Kt = oracle.centroid_keys(chat[b], Wkn)
        outs.append(oracle.proxy_attn_kl(Qn[b], Kt, w.Hq, w.Hkv, w.dh,
                                         None if A_prev is None else A_prev[b]))
    return np.stack([o[0] for o in outs]), np.stack([o[1] for o in outs])


@pytest.mark.parametrize("widx", SMALL)
def test_proxy_attn_kl(widx):
    w, L, H, Q, chat = _proxy_inputs(widx)
    Qn, Wkn, chatn = np_(Q), np_(L["Wk"]), np_(chat)
    A0, D0 = run_proxy(Q, chat, L["Wk"], w.Hkv)
    oA0, _ = _oracle_proxy(w, Qn, chatn, Wkn)
    assert_close(np_(A0), oA0, what="A (no prev)")
    assert np.all(np_(D0) == 0.0)
    # next step: drifted hidden states -> new queries; previous = oracle A
    H1 = wl.drift_rows(w, H, 1)
    Q1 = wl.make_queries(w, H1, L["Wq"])
    prev = torch.from_numpy(oA0.astype(np.float32)).cuda()
    A1, D1 = run_proxy(Q1, chat, L["Wk"], w.Hkv, A_prev=prev)
    oA1, oD1 = _oracle_proxy(w, np_(Q1), chatn, Wkn, np_(prev))
    assert_close(np_(A1), oA1, what="A")
    assert_close(np_(D1), oD1, what="D")
    assert (oD1 > 1e-6).mean() > 0.05       # the drift is not trivially zero


def test_proxy_kl_of_identical_step_is_exactly_zero():
    w, L, H, Q, chat = _proxy_inputs(1, N=256)
    A, _ = run_proxy(Q, chat, L["Wk"], w.Hkv)
    A2, D2 = run_proxy(Q, chat, L["Wk"], w.Hkv, A_prev=A)
    assert torch.equal(A, A2)
    assert bool((D2 == 0).all())


def test_proxy_gqa_and_ragged():
    # Dream-7B head layout (28 query heads on 4 KV heads), 2 windows of 177
    # rows (ragged against the 16-row tiles)
    w, L, H, Q, chat = _proxy_inputs(2, B=2, N=177)
    prev = torch.softmax(torch.randn(2, 177, w.C, device="cuda"), dim=2)
    A, D = run_proxy(Q, chat, L["Wk"], w.Hkv, A_prev=prev)
    oA, oD = _oracle_proxy(w, np_(Q), np_(chat), np_(L["Wk"]), np_(prev))
    assert_close(np_(A), oA, what="A")
    assert_close(np_(D), oD, what="D")


def test_proxy_one_head_slice_many_windows():
    """160 windows of 70 rows give 160 row tiles, so every tile keeps all its
    heads in one CTA (no head-slice cluster); bf16, GQA 4 on 2."""
    rng = np.random.default_rng(11)
    B, N, Hq, Hkv, dh, C, d = 160, 70, 4, 2, 64, 40, 128
    Q = torch.from_numpy(rng.standard_normal((B, N, Hq, dh)).astype(np.float32))
    Q = Q.to(torch.bfloat16).cuda()
    chat = torch.from_numpy(rng.standard_normal((B, C, d)).astype(np.float32)).cuda()
    Wk = torch.from_numpy((rng.standard_normal((d, Hkv * dh)) * 0.1).astype(np.float32))
    Wk = Wk.to(torch.bfloat16).cuda()
    prev = torch.softmax(torch.randn(B, N, C, device="cuda"), dim=2)
    A, D = run_proxy(Q, chat, Wk, Hkv, A_prev=prev)
    w = dataclasses.replace(wl.WORKLOADS[0], Hq=Hq, Hkv=Hkv, dh=dh)
    oA, oD = _oracle_proxy(w, np_(Q), np_(chat), np_(Wk), np_(prev))
    assert_close(np_(A), oA, what="A")
    assert_close(np_(D), oD, what="D")


@pytest.mark.parametrize("B,N,Hq,Hkv,C", [(2, 150, 8, 2, 200), (2, 150, 2, 2, 256),
                                          (160, 70, 4, 2, 160), (3, 200, 6, 3, 100)])
def test_proxy_wide_c(B, N, Hq, Hkv, C):
    """C above 128 on the tensor cores: a row's columns split over four
    epilogue warps (C = 100: two), with 8 and 2 head slices in a cluster (the
    2-slice case reads the previous distributions in place: they do not fit
    the shared memory left over) and with one slice per tile (160 windows)."""
    rng = np.random.default_rng(B * 1000 + C)
    dh, d = 64, 128
    Q = torch.from_numpy(rng.standard_normal((B, N, Hq, dh)).astype(np.float32))
    Q = Q.to(torch.bfloat16).cuda()
    chat = torch.from_numpy(rng.standard_normal((B, C, d)).astype(np.float32)).cuda()
    Wk = torch.from_numpy((rng.standard_normal((d, Hkv * dh)) * 0.1).astype(np.float32))
    Wk = Wk.to(torch.bfloat16).cuda()
    prev = torch.softmax(torch.randn(B, N, C, device="cuda"), dim=2)
    A, D = run_proxy(Q, chat, Wk, Hkv, A_prev=prev)
    w = dataclasses.replace(wl.WORKLOADS[0], Hq=Hq, Hkv=Hkv, dh=dh)
    oA, oD = _oracle_proxy(w, np_(Q), np_(chat), np_(Wk), np_(prev))
    assert_close(np_(A), oA, what="A")
    assert_close(np_(D), oD, what="D")


def test_proxy_single_cluster():
    rng = np.random.default_rng(0)
    Q = torch.from_numpy(rng.standard_normal((1, 9, 2, 16)).astype(np.float32)).cuda()
    chat = torch.from_numpy(rng.standard_normal((1, 1, 32)).astype(np.float32)).cuda()
    Wk = torch.from_numpy(rng.standard_normal((32, 32)).astype(np.float32)).cuda()
    A, D = run_proxy(Q, chat, Wk, 2, A_prev=torch.ones(1, 9, 1, device="cuda"))
    assert bool((A == 1).all()) and bool((D == 0).all())


# ---------------------------------------------------------------- top-k
def _oracle_topk(Dn, an, cn, k):
    return [oracle.topk_drift(Dn[b], an[b], cn[b], k) for b in range(Dn.shape[0])]


@pytest.mark.parametrize("case", ["random", "zeros", "k_eq_c", "empty_clusters",
                                  "wide_range", "big_total", "ties", "denormal"])
def test_topk_drift(case):
    """The kernel forms most cluster sums as exact integer totals and runs the
    sequential fp64 sum only where that could differ; the last four cases put
    clusters on both sides of that line (members 2^-60 apart, a total of
    2^53 units of the smallest member, equal means, subnormal drifts)."""
    rng = np.random.default_rng(sum(map(ord, case)))
    B, N, C, k = 3, 1000, 64, 8
    a = rng.integers(0, C, (B, N)).astype(np.int32)
    if case == "empty_clusters":
        a = (a // 4) * 4                           # only every 4th cluster used
    D = rng.gamma(2.0, 1e-3, (B, N)).astype(np.float32)
    if case == "zeros":
        D[:] = 0
    if case == "k_eq_c":
        k = C
    if case == "wide_range":                       # every 7th row tiny
        D[:, ::7] = (D[:, ::7] * 2.0 ** -60).astype(np.float32)
    if case == "big_total":                        # 1.0 and 2^-29 in one cluster
        for b in range(B):
            rows = np.nonzero(a[b] == 5)[0]
            D[b, rows] = 1.0
            D[b, rows[0]] = np.float32(2.0 ** -29)
    if case == "ties":                             # equal means in many clusters
        D = (np.round(D * 1e3) / 1e3).astype(np.float32)
        D[:, :] = np.float32(0.25) * (a % 3 == 0) + D * (a % 3 != 0)
    if case == "denormal":
        D = (D * np.float32(1e-36)).astype(np.float32)
        D[:, ::3] = np.float32(1e-45) * rng.integers(0, 50, (B, (N + 2) // 3))
    counts = np.stack([np.bincount(a[b], minlength=C) for b in range(B)]).astype(np.int32)
    sel, sc, pos, npos, mask, _, _ = run_topk(torch.from_numpy(D).cuda(),
                                              torch.from_numpy(a).cuda(),
                                              torch.from_numpy(counts).cuda(), k)
    for b, o in enumerate(_oracle_topk(D, a, counts, k)):
        assert np.array_equal(sel[b], o[0])
        assert np.array_equal(sc[b], o[1])
        assert npos[b] == o[3]
        assert np.array_equal(pos[b], o[2])
        assert np.array_equal(mask[b], o[4])


# ---------------------------------------------------------------- refresh
def _kv_check(g, o, bf16):
    rms = np.sqrt(np.mean(o.astype(np.float64) ** 2, axis=-1, keepdims=True))
    tol = (KV_RTOL if bf16 else 1e-5) * np.abs(o) + 1e-3 * rms
    assert np.all(np.abs(g - o) <= tol)


@pytest.mark.parametrize("widx", [0, 1, 2])
@pytest.mark.parametrize("off", [0, 5])
def test_refresh_kv(widx, off):
    w, L = _layer(widx)
    H = L["H"]
    B, N = w.B, w.N
    rng = np.random.default_rng(widx + off)
    a = rng.integers(0, w.C, (B, N)).astype(np.int32)
    D = rng.random((B, N)).astype(np.float32)
    counts = np.stack([np.bincount(a[b], minlength=w.C) for b in range(B)]).astype(np.int32)
    *_, pos_t, npos_t = run_topk(torch.from_numpy(D).cuda(), torch.from_numpy(a).cuda(),
                                 torch.from_numpy(counts).cuda(), w.k)
    dt = wl.torch_dtype(w)
    Ncache = N + off + 3
    Kc0 = torch.randn(B, Ncache, w.Hkv, w.dh, device="cuda").to(dt)
    Vc0 = torch.randn(B, Ncache, w.Hkv, w.dh, device="cuda").to(dt)
    Kc, Vc = Kc0.clone(), Vc0.clone()
    ws = ps.workspace(ps.OP_REFRESH, B=B, N=N, d=w.d, Hkv=w.Hkv, dh=w.dh)
    ps.ps_refresh_kv(H, pos_t, npos_t, L["Wk"], L["Wv"], Kc, Vc, w.Hkv, w.dh, cache_off=off,
                     ws=ws)
    torch.cuda.synchronize()
    ps.ps_check()
    pos, npos = np_(pos_t), np_(npos_t)
    Hn, Wkn, Wvn = np_(H), np_(L["Wk"]), np_(L["Wv"])
    for b in range(B):
        oK, oV = oracle.refresh_kv(Hn[b], pos[b], npos[b], Wkn, Wvn,
                                   np_(Kc0[b]).reshape(Ncache, -1),
                                   np_(Vc0[b]).reshape(Ncache, -1), off, dt == torch.bfloat16)
        gK = np_(Kc[b]).reshape(Ncache, -1)
        gV = np_(Vc[b]).reshape(Ncache, -1)
        touched = np.zeros(Ncache, bool)
        touched[off + pos[b][:npos[b]]] = True
        assert np.array_equal(gK[~touched], np_(Kc0[b]).reshape(Ncache, -1)[~touched])
        assert np.array_equal(gV[~touched], np_(Vc0[b]).reshape(Ncache, -1)[~touched])
        _kv_check(gK[touched], oK[touched], dt == torch.bfloat16)
        _kv_check(gV[touched], oV[touched], dt == torch.bfloat16)


def test_refresh_empty_selection_leaves_cache():
    H = torch.randn(1, 40, 64, device="cuda").to(torch.bfloat16)
    W = torch.randn(64, 32, device="cuda").to(torch.bfloat16)
    Kc = torch.randn(1, 40, 2, 16, device="cuda").to(torch.bfloat16)
    Vc = Kc.clone()
    K0 = Kc.clone()
    pos = torch.full((1, 40), -1, dtype=torch.int32, device="cuda")
    npos = torch.zeros(1, dtype=torch.int32, device="cuda")
    ps.ps_refresh_kv(H, pos, npos, W, W, Kc, Vc, 2, 16)
    torch.cuda.synchronize()
    assert torch.equal(Kc, K0) and torch.equal(Vc, K0)
    # the tensor-core path (K/V width a multiple of 64) with nothing selected
    W = torch.randn(64, 128, device="cuda").to(torch.bfloat16)
    Kc = torch.randn(2, 40, 2, 64, device="cuda").to(torch.bfloat16)
    Vc, K0 = Kc.clone(), Kc.clone()
    pos = torch.full((2, 40), -1, dtype=torch.int32, device="cuda")
    npos = torch.zeros(2, dtype=torch.int32, device="cuda")
    H2 = torch.randn(2, 40, 64, device="cuda").to(torch.bfloat16)
    ws = ps.workspace(ps.OP_REFRESH, B=2, N=40, d=64, Hkv=2, dh=64)
    ps.ps_refresh_kv(H2, pos, npos, W, W, Kc, Vc, 2, 64, ws=ws)
    torch.cuda.synchronize()
    ps.ps_check()
    assert torch.equal(Kc, K0) and torch.equal(Vc, K0)


def test_refresh_all_rows_ragged_d():
    """Every row selected, d = 80 (a partial 64-wide K block), 3 windows of
    150 rows (ragged 128-row tiles): the textbook GEMM, bf16-rounded."""
    rng = np.random.default_rng(9)
    B, N, d, Hkv, dh = 3, 150, 80, 2, 64
    H = torch.from_numpy(rng.standard_normal((B, N, d)).astype(np.float32)).cuda().to(torch.bfloat16)
    Wk = torch.from_numpy(rng.standard_normal((d, Hkv * dh)).astype(np.float32) * 0.1).cuda().to(torch.bfloat16)
    Wv = torch.from_numpy(rng.standard_normal((d, Hkv * dh)).astype(np.float32) * 0.1).cuda().to(torch.bfloat16)
    pos = torch.arange(N, dtype=torch.int32, device="cuda").repeat(B, 1).contiguous()
    npos = torch.full((B,), N, dtype=torch.int32, device="cuda")
    Kc = torch.zeros(B, N, Hkv, dh, device="cuda", dtype=torch.bfloat16)
    Vc = torch.zeros_like(Kc)
    ws = ps.workspace(ps.OP_REFRESH, B=B, N=N, d=d, Hkv=Hkv, dh=dh)
    ps.ps_refresh_kv(H, pos, npos, Wk, Wv, Kc, Vc, Hkv, dh, ws=ws)
    torch.cuda.synchronize()
    ps.ps_check()
    Hn, Wkn, Wvn = np_(H), np_(Wk), np_(Wv)
    for b in range(B):
        _kv_check(np_(Kc[b]).reshape(N, -1), oracle.bf16_round(Hn[b] @ Wkn.astype(np.float64)), True)
        _kv_check(np_(Vc[b]).reshape(N, -1), oracle.bf16_round(Hn[b] @ Wvn.astype(np.float64)), True)


def test_refresh_many_rows_unsplit():
    """1000 of 1000 rows selected against a 2 x 4096-wide [K | V]: more rows
    than the d split takes (512 here), so chunk 0 of each cluster runs the
    whole d range and scatters from TMEM while the other chunk idles."""
    rng = np.random.default_rng(10)
    B, N, d, Hkv, dh = 1, 1000, 128, 32, 128
    H = torch.from_numpy(rng.standard_normal((B, N, d)).astype(np.float32)).cuda().to(torch.bfloat16)
    Wk = torch.from_numpy(rng.standard_normal((d, Hkv * dh)).astype(np.float32) * 0.1).cuda().to(torch.bfloat16)
    Wv = torch.from_numpy(rng.standard_normal((d, Hkv * dh)).astype(np.float32) * 0.1).cuda().to(torch.bfloat16)
    pos = torch.from_numpy(rng.permutation(N).astype(np.int32))[None].cuda().contiguous()
    npos = torch.full((B,), N, dtype=torch.int32, device="cuda")
    Kc = torch.zeros(B, N, Hkv, dh, device="cuda", dtype=torch.bfloat16)
    Vc = torch.zeros_like(Kc)
    ws = ps.workspace(ps.OP_REFRESH, B=B, N=N, d=d, Hkv=Hkv, dh=dh)
    ps.ps_refresh_kv(H, pos, npos, Wk, Wv, Kc, Vc, Hkv, dh, ws=ws)
    torch.cuda.synchronize()
    ps.ps_check()
    Hn, Wkn, Wvn = np_(H), np_(Wk), np_(Wv)
    _kv_check(np_(Kc[0]).reshape(N, -1), oracle.bf16_round(Hn[0] @ Wkn.astype(np.float64)), True)
    _kv_check(np_(Vc[0]).reshape(N, -1), oracle.bf16_round(Hn[0] @ Wvn.astype(np.float64)), True)


# ---------------------------------------------------------------- commit
def _commit_case(widx, mode, suffix, B=None, seed=0):
    w = wl.WORKLOADS[widx]
    B = w.B if B is None else B
    logits = wl.make_logits(w, 0, "cuda", B=B)
    rng = np.random.default_rng(seed)
    P = w.P
    role = np.zeros(P, np.uint8)
    if suffix:
        role[P // 2:] = 1
        role[-1] = 2
    und = (rng.random((B, P)) < 0.85).astype(np.uint8)
    D = rng.gamma(2.0, 0.05, (B, P)).astype(np.float32)
    cnt = rng.integers(0, 4, (B, P)).astype(np.int32)
    s = (cnt * rng.gamma(2.0, 0.05, (B, P))).astype(np.float32)
    prev = rng.gamma(2.0, 0.05, (B, P)).astype(np.float32)
    ssel = (rng.random((B, P)) < 0.5).astype(np.uint8) if suffix else None
    params = oracle.CommitParams(tau_s=w.tau_s, alpha=w.alpha, ratio=0.5 if mode == 2 else w.ratio,
                                 mode=mode, ensure_progress=1)
    return w, logits, role, und, D, s, cnt, prev, ssel, params


@pytest.mark.parametrize("widx", SMALL)
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("suffix", [False, True])
def test_commit(widx, mode, suffix):
    w, logits, role, und, D, s, cnt, prev, ssel, p = _commit_case(widx, mode, suffix)
    dev = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()
    g = run_commit(logits, dev(role), dev(und), dev(D), w.P, dev(s), dev(cnt), dev(prev),
                   dev(ssel), ps.CommitParams(p.tau_s, p.alpha, p.ratio, p.mode,
                                              p.ensure_progress))
    Ln = np_(logits)
    unpinned = 0
    for b in range(logits.shape[0]):
        o = oracle.commit_rule(Ln[b], role, und[b], D[b], s[b], cnt[b], prev[b],
                               None if ssel is None else ssel[b], p)
        assert np.array_equal(g["token"][b], o["token"])
        assert_close(g["conf"][b], o["conf"], rtol=CONF_RTOL, atol=0, what="conf")
        band = o["margin"] <= BAND
        unpinned += int(band.sum())
        if not band.any():
            assert np.array_equal(g["commit"][b], o["commit"])
            assert np.array_equal(g["undecided"][b], o["undecided"])
        assert np.array_equal(g["d_sum"][b], o["d_sum"])
        assert np.array_equal(g["d_cnt"][b], o["d_cnt"])
        assert np.array_equal(g["d_prev"][b], o["d_prev"])
    assert unpinned <= 1


@pytest.mark.parametrize("widx,V", [(1, None), (0, 16384 * 2 + 12)])
def test_commit_bf16_logits(widx, V):
    """bf16 logits (as an LM head emits them): the oracle's decisions on the
    bf16 values, and against the fp32 path on the same (bf16-representable)
    values the same tokens and confidences within rounding (the bf16 scan
    loads 8 logits a thread where V % 8 == 0, the fp32 one 4, so their fp32
    partial sums group differently); V with a ragged last chunk (V % 8 = 4,
    4-logit loads) included."""
    w, logits, role, und, D, s, cnt, prev, ssel, p = _commit_case(widx, 0, True, seed=3)
    if V is not None:
        logits = wl.make_logits(w, 0, "cuda", V=V)
    Lb = logits.to(torch.bfloat16)
    dev = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()
    args = (dev(role), dev(und), dev(D), w.P, dev(s), dev(cnt), dev(prev), dev(ssel),
            ps.CommitParams(p.tau_s, p.alpha, p.ratio, p.mode, p.ensure_progress))
    g = run_commit(Lb, *args)
    g32 = run_commit(Lb.float(), *args)
    assert np.array_equal(g["token"], g32["token"])
    assert_close(g["conf"], g32["conf"], rtol=CONF_RTOL, atol=0, what="conf vs fp32 path")
    Ln = np_(Lb)
    for b in range(Ln.shape[0]):
        o = oracle.commit_rule(Ln[b], role, und[b], D[b], s[b], cnt[b], prev[b], ssel[b], p)
        assert np.array_equal(g["token"][b], o["token"])
        assert_close(g["conf"][b], o["conf"], rtol=CONF_RTOL, atol=0, what="conf")
        if not (o["margin"] <= BAND).any():
            assert np.array_equal(g["commit"][b], o["commit"])
            assert np.array_equal(g["undecided"][b], o["undecided"])
            assert np.array_equal(g["d_sum"][b], o["d_sum"])


def test_commit_uniform_and_onehot_closed_forms():
    V = 4096
    L = torch.zeros(1, 2, V, device="cuda")
    L[0, 1, 1234] = 6.0
    role = torch.zeros(2, dtype=torch.uint8, device="cuda")
    z = torch.zeros(1, 2, device="cuda")
    g = run_commit(L, role, torch.ones(1, 2, dtype=torch.uint8, device="cuda"), z, 2,
                   z.clone(), torch.zeros(1, 2, dtype=torch.int32, device="cuda"),
                   z.clone(), None, ps.CommitParams(0.9, 1.0, 0.1, 0, 0))
    assert g["token"][0][0] == 0 and g["token"][0][1] == 1234
    assert abs(g["conf"][0][0] - 1 / V) <= 1e-6 / V
    want = 1 / (1 + (V - 1) * math.exp(-6.0))
    assert abs(g["conf"][0][1] - want) <= 1e-6 * want


@pytest.mark.parametrize("C,Hq,Hkv,B,N", [(256, 4, 2, 160, 70), (200, 6, 3, 160, 70),
                                           (100, 2, 2, 160, 70), (256, 8, 8, 160, 70),
                                           (200, 4, 2, 80, 250), (256, 2, 1, 78, 256),
                                           (64, 4, 4, 160, 70), (20, 2, 2, 80, 130)])
def test_proxy_row_tile_path_head_sum_in_tmem(C, Hq, Hkv, B, N):
    """At least 152 row tiles (one CTA per tile takes all its heads, the head
    sum kept in TMEM); C above 128 splits a head's columns in two halves
    joined by the softmax's rescale (C = 200: a ragged second half); two row
    tiles per window (N = 250 and 130: the second ragged) and a shared KV head
    (Hkv = 1); 64- and 32-column score tiles (C = 64, 20).  With and without a
    previous distribution, and KL of an identical step exactly 0."""
    rng = np.random.default_rng(C + Hq + N)
    dh, d = 64, 128
    Q = torch.from_numpy(rng.standard_normal((B, N, Hq, dh)).astype(np.float32) * 2)
    Q = Q.to(torch.bfloat16).cuda()
    chat = torch.from_numpy(rng.standard_normal((B, C, d)).astype(np.float32)).cuda()
    Wk = torch.from_numpy((rng.standard_normal((d, Hkv * dh)) * 0.1).astype(np.float32))
    Wk = Wk.to(torch.bfloat16).cuda()
    w = dataclasses.replace(wl.WORKLOADS[0], Hq=Hq, Hkv=Hkv, dh=dh)
    A0, D0 = run_proxy(Q, chat, Wk, Hkv)
    oA0, _ = _oracle_proxy(w, np_(Q), np_(chat), np_(Wk))
    assert_close(np_(A0), oA0, what="A (no prev)")
    assert np.all(np_(D0) == 0.0)
    prev = torch.softmax(torch.randn(B, N, C, device="cuda"), dim=2)
    A, D = run_proxy(Q, chat, Wk, Hkv, A_prev=prev)
    oA, oD = _oracle_proxy(w, np_(Q), np_(chat), np_(Wk), np_(prev))
    assert_close(np_(A), oA, what="A")
    assert_close(np_(D), oD, what="D")
    _, D2 = run_proxy(Q, chat, Wk, Hkv, A_prev=A0)
    assert bool((D2 == 0).all())
