"""Failure detection without a GPU fault: a child process sets the test-only
flag PS_TEST_STARVE_TMA, so the tensor-core kernel's TMA producer issues no
copies.  The MMA thread's bounded wait (2 s) must give up, record
PS_ERR_TIMEOUT in the handle's status word, drain, free TMEM and return; the
host reads the status with ps_check, and the same context then runs a normal
call correctly.  Covered: the K/V refresh GEMM and the k-means assignment
whose d-chunks meet in a thread-block cluster."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import os, sys, torch
    sys.path.insert(0, sys.argv[1])
    from drift_aware_kv_spherical_gb300 import polestar as ps
    torch.manual_seed(0)
    B, N, d, Hkv, dh = 1, 64, 64, 2, 64
    H = torch.randn(B, N, d, device="cuda").to(torch.bfloat16)
    W = torch.randn(d, Hkv * dh, device="cuda").to(torch.bfloat16)
    pos = torch.arange(N, dtype=torch.int32, device="cuda")[None].contiguous()
    npos = torch.full((B,), N, dtype=torch.int32, device="cuda")
    Kc = torch.zeros(B, N, Hkv, dh, device="cuda", dtype=torch.bfloat16)
    Vc = torch.zeros_like(Kc)
    ws = ps.workspace(ps.OP_REFRESH, B=B, N=N, d=d, Hkv=Hkv, dh=dh)
    os.environ["PS_TEST_STARVE_TMA"] = "1"
    ps.ps_refresh_kv(H, pos, npos, W, W, Kc, Vc, Hkv, dh, ws=ws)
    torch.cuda.synchronize()
    try:
        ps.ps_check()
        print("STATUS ok")
    except ps.PolestarError as e:
        print("STATUS", e.status)
    del os.environ["PS_TEST_STARVE_TMA"]
    ps.ps_refresh_kv(H, pos, npos, W, W, Kc, Vc, Hkv, dh, ws=ws)
    torch.cuda.synchronize()
    ps.ps_check()
    want = (H.float()[0] @ W.float()).to(torch.bfloat16).float()
    err = (Kc[0].reshape(N, -1).float() - want).abs().max().item()
    print("AFTER", err)
    # k-means assignment with its 8 d-chunks in one thread-block cluster:
    # every CTA gives up, and all still meet at the cluster barriers
    Hk = torch.randn(1, 128, 1024, device="cuda").to(torch.bfloat16)
    mu = torch.nn.functional.normalize(torch.randn(1, 16, 1024, device="cuda"), dim=2)
    assign = torch.zeros(1, 128, dtype=torch.int32, device="cuda")
    rho = torch.zeros(1, 128, device="cuda")
    chat = torch.zeros(1, 16, 1024, device="cuda")
    counts = torch.zeros(1, 16, dtype=torch.int32, device="cuda")
    wk = ps.workspace(ps.OP_KMEANS, B=1, N=128, d=1024, C=16)
    os.environ["PS_TEST_STARVE_TMA"] = "1"
    ps.ps_kmeans_spherical(Hk, mu, assign, rho, chat, counts, 0, ws=wk)
    torch.cuda.synchronize()
    try:
        ps.ps_check()
        print("KSTATUS ok")
    except ps.PolestarError as e:
        print("KSTATUS", e.status)
    del os.environ["PS_TEST_STARVE_TMA"]
    ps.ps_kmeans_spherical(Hk, mu, assign, rho, chat, counts, 0, ws=wk)
    torch.cuda.synchronize()
    ps.ps_check()
    s = torch.nn.functional.normalize(Hk.float()[0], dim=1) @ mu[0].T
    print("KAFTER", int((s.argmax(1).int() != assign[0]).sum()))
""")


def test_starved_wait_times_out_and_context_survives(lib):
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = dict(l.split(" ", 1) for l in r.stdout.splitlines() if " " in l)
    from drift_aware_kv_spherical_gb300 import polestar as ps
    assert lines["STATUS"].strip() == str(ps.PS_ERR_TIMEOUT)
    assert float(lines["AFTER"]) < 0.1
    assert lines["KSTATUS"].strip() == str(ps.PS_ERR_TIMEOUT)
    assert int(lines["KAFTER"]) <= 2     # arg-max ties of random data aside
