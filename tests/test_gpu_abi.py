"""Argument validation through the C ABI with a real handle: every bad call
returns its status before anything is launched and leaves outputs untouched."""
import ctypes

import pytest
import torch

from drift_aware_kv_spherical_gb300 import polestar as ps

pytestmark = pytest.mark.gpu


def _lib_handle(lib):
    return lib.cdll, lib.handle()


def _km(cd, h, H, mu, out, B, N, d, C, ws=None, wsb=0, iters=1):
    assign, rho, chat, counts = out
    return cd.ps_kmeans_spherical(h, H.data_ptr(), ps.PS_BF16, B, N, d, C, iters, 0, None,
                                  mu.data_ptr(), assign.data_ptr(), rho.data_ptr(),
                                  chat.data_ptr(), counts.data_ptr(), None,
                                  ws, wsb, torch.cuda.current_stream().cuda_stream)


def test_kmeans_rejects_bad_sizes_and_small_workspace(lib):
    cd, h = _lib_handle(lib)
    B, N, d, C = 1, 64, 64, 8
    H = torch.randn(B, N, d, device="cuda").to(torch.bfloat16)
    mu = torch.randn(B, C, d, device="cuda")
    out = (torch.full((B, N), 7, dtype=torch.int32, device="cuda"),
           torch.zeros(B, N, device="cuda"), torch.zeros(B, C, d, device="cuda"),
           torch.zeros(B, C, dtype=torch.int32, device="cuda"))
    need = ps.ps_workspace_bytes(ps.OP_KMEANS, B=B, N=N, d=d, C=C)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert _km(cd, h, H, mu, out, B, N, 40, C, ws.data_ptr(), need) == ps.PS_ERR_ARG  # d % 16
    assert _km(cd, h, H, mu, out, B, N, d, N + 1, ws.data_ptr(), need) == ps.PS_ERR_ARG  # C > N
    assert _km(cd, h, H, mu, out, B, N, d, 300, ws.data_ptr(), need) == ps.PS_ERR_ARG  # C > 256
    assert _km(cd, h, H, mu, out, B, N, d, C, ws.data_ptr(), need - 1) == ps.PS_ERR_WORKSPACE
    assert _km(cd, h, H, mu, out, B, N, d, C, None, 0) == ps.PS_ERR_WORKSPACE
    assert _km(cd, h, H, mu, out, B, N, d, C, ws.data_ptr(), need, iters=-1) == ps.PS_ERR_ARG
    torch.cuda.synchronize()
    assert bool((out[0] == 7).all())                 # nothing was launched
    assert _km(cd, h, H, mu, out, 0, N, d, C) == ps.PS_OK   # B = 0 is a no-op


def test_misaligned_pointer_rejected(lib):
    cd, h = _lib_handle(lib)
    H = torch.randn(1, 4, 40, device="cuda")
    codes = torch.zeros(1, 4, 17, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(1, 4, 3, dtype=torch.uint8, device="cuda")
    S = torch.zeros(1, device="cuda")
    st = cd.ps_nvfp4_residual(h, H.data_ptr() + 4, ps.PS_F32, None, None, None, 1, 4, 32, 1,
                              codes.data_ptr(), scales.data_ptr(), S.data_ptr(), None, 0,
                              torch.cuda.current_stream().cuda_stream)
    assert st == ps.PS_ERR_ARG


def test_topk_and_commit_reject_bad_k_and_mode(lib):
    cd, h = _lib_handle(lib)
    D = torch.zeros(1, 10, device="cuda")
    a = torch.zeros(1, 10, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, 4, dtype=torch.int32, device="cuda")
    sel = torch.zeros(1, 5, dtype=torch.int32, device="cuda")
    sc = torch.zeros(1, 5, device="cuda")
    pos = torch.zeros(1, 10, dtype=torch.int32, device="cuda")
    npos = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert cd.ps_topk_drift(h, D.data_ptr(), a.data_ptr(), n.data_ptr(), 1, 10, 4, 5,
                            sel.data_ptr(), sc.data_ptr(), pos.data_ptr(), npos.data_ptr(),
                            None, None, 0, s) == ps.PS_ERR_ARG       # k > C
    L = torch.zeros(1, 2, 8, device="cuda")
    u8 = torch.zeros(1, 2, dtype=torch.uint8, device="cuda")
    f = torch.zeros(1, 2, device="cuda")
    i32 = torch.zeros(1, 2, dtype=torch.int32, device="cuda")
    bad = ps.CommitParams(0.9, 1.0, 0.1, 3, 1)
    assert cd.ps_commit(h, L.data_ptr(), 0, 1, 2, 8, u8.data_ptr(), u8.data_ptr(), f.data_ptr(),
                        2, f.data_ptr(), i32.data_ptr(), f.data_ptr(), None, 2, bad,
                        i32.data_ptr(), f.data_ptr(), u8.data_ptr(), None, 0,
                        s) == ps.PS_ERR_ARG                          # unknown mode


def test_check_reports_ok_after_work(lib):
    cd, h = _lib_handle(lib)
    assert cd.ps_check(h, torch.cuda.current_stream().cuda_stream, 1) == ps.PS_OK


def test_kernel_trace_records_every_launch(lib):
    """The diagnostic trace brackets each launch of a call with events: a
    k-means call with I = 3 on the tensor-core path (Gram form) records its
    launches in order with positive durations; disabling clears the
    records."""
    H = torch.randn(1, 300, 256, device="cuda").to(torch.bfloat16)
    mu = torch.nn.functional.normalize(torch.randn(1, 24, 256, device="cuda"), dim=2)
    a = torch.zeros(1, 300, dtype=torch.int32, device="cuda")
    rho = torch.zeros(1, 300, device="cuda")
    chat = torch.zeros(1, 24, 256, device="cuda")
    n = torch.zeros(1, 24, dtype=torch.int32, device="cuda")
    ws = ps.workspace(ps.OP_KMEANS, B=1, N=300, d=256, C=24)
    ps.ps_trace_enable(True)
    ps.ps_kmeans_spherical(H, mu, a, rho, chat, n, 3, ws=ws)
    rec = ps.ps_trace_records()
    ps.ps_check()
    names = [r[0] for r in rec]
    assert len(names) == 4
    assert "k_km_prep" in names[0]
    assert sum("k_tc_gemm" in x for x in names) == 1             # Gram GEMM + pass-0 cosines
    assert sum("k_km_gram" in x for x in names) == 1             # passes 0 .. I
    assert sum("k_cluster_scan" in x for x in names) == 1        # last update + C_hat
    assert all(ms > 0 for _, ms in rec)
    ps.ps_trace_enable(False)
    assert lib.cdll.ps_trace_count(lib.handle()) == 0
    ps.ps_kmeans_spherical(H, mu, a, rho, chat, n, 3, ws=ws)     # untraced calls record nothing
    assert lib.cdll.ps_trace_count(lib.handle()) == 0
