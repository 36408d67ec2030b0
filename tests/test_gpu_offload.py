"""Offload of the quantised clusters (store grouped by cluster, in device or
mapped host memory) and the fetch with reconstruction, against the oracle:
store bytes, record order and cluster offsets bit-exact; reconstructed rows
bit-exact in bf16; rows of unselected clusters untouched."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from drift_aware_kv_spherical_gb300 import polestar as ps
from drift_aware_kv_spherical_gb300 import workloads as wl
from tests._parity import np_

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(lib):
    return lib


def _quantised(B, N, d, C, seed, empty=()):
    """GPU NVFP4 residuals of random rows (bit-exact with the oracle's)."""
    rng = np.random.default_rng(seed)
    H = torch.from_numpy(rng.standard_normal((B, N, d)).astype(np.float32)).cuda()
    mu = oracle.normalize_rows(rng.standard_normal((B * C, d))).reshape(B, C, d)
    mu = torch.from_numpy(mu.astype(np.float32)).cuda()
    choices = [c for c in range(C) if c not in empty]
    assign = torch.from_numpy(rng.choice(choices, (B, N)).astype(np.int32)).cuda()
    rho = (H * mu[torch.arange(B)[:, None], assign.long()]).sum(-1).contiguous()
    codes = torch.zeros(B, N, d // 2, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(B, N, d // 16, dtype=torch.uint8, device="cuda")
    S = torch.zeros(B, device="cuda")
    ws = ps.workspace(ps.OP_NVFP4, B=B, N=N, d=d)
    ps.ps_nvfp4_residual(H, mu, assign, rho, codes, scales, S, ws=ws)
    return H, mu, assign, rho, codes, scales, S


def _pack(codes, scales, assign, C, host):
    B, N, half = codes.shape
    rec = ps.ps_store_record_bytes(2 * half)
    store = ps.HostStore(B * N * rec) if host else torch.zeros(B * N * rec, dtype=torch.uint8,
                                                               device="cuda")
    if host:
        store.view()[:] = 0x5A
    order = torch.full((B, N), -1, dtype=torch.int32, device="cuda")
    cl_off = torch.full((B, C + 1), -1, dtype=torch.int32, device="cuda")
    ps.ps_nvfp4_pack_clusters(codes, scales, assign, C, store, order, cl_off)
    torch.cuda.synchronize()
    ps.ps_check()
    got = store.view().copy() if host else np_(store)
    return store, got.reshape(B, N, rec), np_(order), np_(cl_off)


@pytest.mark.parametrize("B,N,d,C,host", [(2, 300, 256, 12, False), (1, 257, 3584, 5, True),
                                          (3, 64, 96, 7, False), (1, 1024, 4096, 64, True)])
def test_pack_matches_oracle(B, N, d, C, host):
    _, _, assign, _, codes, scales, _ = _quantised(B, N, d, C, N + C, empty=(1,))
    _, store, order, cl_off = _pack(codes, scales, assign, C, host)
    for b in range(B):
        s_o, o_o, c_o = oracle.pack_clusters(np_(codes[b]), np_(scales[b]), np_(assign[b]), C)
        assert np.array_equal(cl_off[b], c_o)
        assert np.array_equal(order[b], o_o)
        assert np.array_equal(store[b], s_o)


@pytest.mark.parametrize("B,N,d,C,host", [(2, 300, 256, 12, False), (1, 257, 3584, 5, True),
                                          (2, 200, 8192, 9, True)])
def test_fetch_dequant_matches_oracle(B, N, d, C, host):
    H, mu, assign, rho, codes, scales, S = _quantised(B, N, d, C, 7 * N + C, empty=(2,))
    st, store, order, cl_off = _pack(codes, scales, assign, C, host)
    k = 4
    sel = torch.tensor([[3, -1, 2, 0], [C - 1, 5 % C, -1, -1]][:B] + [[1, -1, -1, -1]] * (B - 2),
                       dtype=torch.int32, device="cuda")
    Ht = torch.full((B, N, d), 7.0, dtype=torch.bfloat16, device="cuda")
    ps.ps_nvfp4_fetch_dequant(st, torch.from_numpy(order).cuda(), torch.from_numpy(cl_off).cuda(),
                              sel, mu, rho, S, Ht)
    torch.cuda.synchronize()
    ps.ps_check()
    got = np_(Ht.float())
    for b in range(B):
        want = oracle.fetch_reconstruct(store[b], order[b], cl_off[b], np_(sel[b]), np_(mu[b]),
                                        np_(rho[b]), float(np_(S)[b]), d)
        for i in range(N):
            if i in want:
                assert np.array_equal(got[b, i], oracle.bf16_round(want[i])), (b, i)
            else:
                assert np.all(got[b, i] == 7.0), (b, i)        # untouched
    assert len(want) > 0


def test_rejects_a_store_the_device_cannot_reach():
    _, _, assign, _, codes, scales, _ = _quantised(1, 32, 64, 3, 1)
    lib = ps._lib()
    plain = np.zeros(32 * ps.ps_store_record_bytes(64) + 64, dtype=np.uint8)
    addr = (plain.ctypes.data + 15) // 16 * 16                   # aligned, but not mapped
    order = torch.zeros(1, 32, dtype=torch.int32, device="cuda")
    cl_off = torch.zeros(1, 4, dtype=torch.int32, device="cuda")
    st = lib.cdll.ps_nvfp4_pack_clusters(lib.handle(), codes.data_ptr(), scales.data_ptr(),
                                         assign.data_ptr(), 1, 32, 64, 3, ctypes.c_void_p(addr),
                                         order.data_ptr(), cl_off.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert st == ps.PS_ERR_ARG
    assert ps.ps_store_record_bytes(48) == 0 and ps.ps_store_record_bytes(4096) == 2304


def test_llada_layer_offload_round_trip():
    """The LLaDA-8B-shaped layer: k-means, NVFP4, the store in host memory,
    top-k of a drift, the fetch; sampled reconstructed rows bit-exact with the
    oracle's and within the NVFP4 bound of the hidden states."""
    w = wl.WORKLOADS[1]
    L = wl.make_layer(w, 0, "cuda")
    H = L["H"]
    B, N, d, C = w.B, w.N, w.d, w.C
    u = wl.make_uniforms(w, 0, "cuda")
    mu = torch.zeros(B, C, d, device="cuda")
    assign = torch.zeros(B, N, dtype=torch.int32, device="cuda")
    rho = torch.zeros(B, N, device="cuda")
    chat = torch.zeros(B, C, d, device="cuda")
    counts = torch.zeros(B, C, dtype=torch.int32, device="cuda")
    ps.ps_kmeans_spherical(H, mu, assign, rho, chat, counts, w.iters, init_mode=1, init_u=u,
                           ws=ps.workspace(ps.OP_KMEANS, B=B, N=N, d=d, C=C))
    codes = torch.zeros(B, N, d // 2, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(B, N, d // 16, dtype=torch.uint8, device="cuda")
    S = torch.zeros(B, device="cuda")
    ps.ps_nvfp4_residual(H, mu, assign, rho, codes, scales, S,
                         ws=ps.workspace(ps.OP_NVFP4, B=B, N=N, d=d))
    st, store, order, cl_off = _pack(codes, scales, assign, C, True)
    D = torch.rand(B, N, device="cuda")
    sel = torch.zeros(B, w.k, dtype=torch.int32, device="cuda")
    ps.ps_topk_drift(D, assign, counts, w.k, sel, torch.zeros(B, w.k, device="cuda"),
                     torch.zeros(B, N, dtype=torch.int32, device="cuda"),
                     torch.zeros(B, dtype=torch.int32, device="cuda"))
    Ht = torch.zeros(B, N, d, dtype=torch.bfloat16, device="cuda")
    ps.ps_nvfp4_fetch_dequant(st, torch.from_numpy(order).cuda(), torch.from_numpy(cl_off).cuda(),
                              sel, mu, rho, S, Ht)
    torch.cuda.synchronize()
    ps.ps_check()
    want = oracle.fetch_reconstruct(store[0], order[0], cl_off[0], np_(sel[0]), np_(mu[0]),
                                    np_(rho[0]), float(np_(S)[0]), d)
    assert len(want) == int(np_(counts[0])[np_(sel[0])].sum())
    got = np_(Ht[0].float())
    Hn = np_(H[0].float())
    for i in sorted(want)[:: max(1, len(want) // 12)]:
        assert np.array_equal(got[i], oracle.bf16_round(want[i]))
        assert np.max(np.abs(want[i] - Hn[i])) <= 0.5 * np.max(np.abs(Hn[i]))  # a proxy of h


def test_offload_step_matches_oracle_refresh():
    """A pipeline step in offload mode (store in host memory, side streams as
    the bench captures them): the refreshed K rows equal the oracle's refresh
    of the oracle's reconstruction of the selected rows, sampled."""
    from drift_aware_kv_spherical_gb300.pipeline import Pipeline
    w = wl.WORKLOADS[1]
    L = wl.make_layer(w, 0, "cuda")
    Q = wl.make_queries(w, L["H"], L["Wq"])
    u = wl.make_uniforms(w, 0, "cuda")
    logits = wl.make_logits(w, 0, "cuda")
    pipe = Pipeline(w, layers=1, offload=True)
    pipe.step([L["H"]], [Q], [L["Wk"]], [L["Wv"]], logits, init_us=[u], first=True,
              concurrent=True)
    H1 = wl.drift_rows(w, L["H"], 1)
    pipe.step([H1], [wl.make_queries(w, H1, L["Wq"])], [L["Wk"]], [L["Wv"]], logits,
              concurrent=True)
    torch.cuda.synchronize()
    ps.ps_check()
    st = pipe.state[0]
    rec = ps.ps_store_record_bytes(w.d)
    store = st.store.view().reshape(w.B, w.N, rec)
    want = oracle.fetch_reconstruct(store[0], np_(st.order[0]), np_(st.cl_off[0]), np_(st.sel[0]),
                                    np_(st.mu[0]), np_(st.rho[0]), float(np_(st.S)[0]), w.d)
    pos = np_(st.pos[0])[: int(np_(st.npos)[0])]
    assert set(pos.tolist()) == set(want)
    Wk = np_(L["Wk"]).astype(np.float64)
    Kc = np_(st.Kc[0]).reshape(w.Ncache, -1)
    for p in pos[:: max(1, len(pos) // 8)]:
        ref = oracle.bf16_round(oracle.bf16_round(want[p]).astype(np.float64) @ Wk)
        rms = np.sqrt(np.mean(ref.astype(np.float64) ** 2))
        assert np.all(np.abs(Kc[p] - ref) <= 2e-2 * np.abs(ref) + 1e-3 * rms)
