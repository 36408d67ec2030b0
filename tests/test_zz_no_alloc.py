"""The workspace-free NVFP4 entry point, for callers that cannot allocate
device memory (it keeps its scratch in a fixed device array inside the
library).  It must give exactly the bits of ps_nvfp4_residual, call after
call, although every call reuses the same array.  This file is collected last
so that a run stopping at the first failure has run everything else."""
import pytest
import torch

from drift_aware_kv_spherical_gb300 import polestar as ps
from drift_aware_kv_spherical_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _inputs(widx, seed):
    w = wl.WORKLOADS[widx]
    H = wl.make_layer(w, 0, "cuda")["H"]
    g = torch.Generator(device="cuda").manual_seed(seed)
    mu = torch.randn(w.B, w.C, w.d, device="cuda", generator=g)
    mu = mu / mu.norm(dim=2, keepdim=True)
    assign = torch.randint(0, w.C, (w.B, w.N), device="cuda", generator=g,
                           dtype=torch.int32)
    rho = torch.randn(w.B, w.N, device="cuda", generator=g) * 10
    return H, mu, assign, rho


def _outputs(H):
    B, N, d = H.shape
    return (torch.zeros(B, N, d // 2, dtype=torch.uint8, device="cuda"),
            torch.zeros(B, N, d // 16, dtype=torch.uint8, device="cuda"),
            torch.zeros(B, device="cuda"))


def test_noalloc_matches_workspace_entry_point_twice_in_a_row(lib):
    for widx, seed in ((1, 11), (0, 12)):        # two calls in a row, different sizes
        H, mu, assign, rho = _inputs(widx, seed)
        B, N, d = H.shape
        ref = _outputs(H)
        ws = ps.workspace(ps.OP_NVFP4, B=B, N=N, d=d)
        ps.ps_nvfp4_residual(H, mu, assign, rho, *ref, ws=ws)
        got = _outputs(H)
        ps.ps_nvfp4_residual_noalloc(H, mu, assign, rho, *got)
        torch.cuda.synchronize()
        ps.ps_check()
        for r, g in zip(ref, got):
            assert torch.equal(r, g)


def test_noalloc_rejects_batches_beyond_its_array(lib):
    H = torch.zeros(16385, 1, 16, device="cuda")
    codes, scales, S = _outputs(H)
    with pytest.raises(ps.PolestarError) as e:
        ps.ps_nvfp4_residual_noalloc(H, None, None, None, codes, scales, S)
    assert e.value.status == ps.PS_ERR_WORKSPACE


def test_noalloc_at_its_largest_batch_matches_and_allocates_nothing(lib):
    # B = 16384 is the documented maximum: the array's every slot is in use
    g = torch.Generator(device="cuda").manual_seed(13)
    B, N, d, C = 16384, 1, 16, 3
    H = (torch.randn(B, N, d, device="cuda", generator=g) * 3).to(torch.bfloat16)
    mu = torch.randn(B, C, d, device="cuda", generator=g)
    mu = mu / mu.norm(dim=2, keepdim=True)
    assign = torch.randint(0, C, (B, N), device="cuda", generator=g, dtype=torch.int32)
    rho = torch.randn(B, N, device="cuda", generator=g)
    ref = _outputs(H)
    ws = ps.workspace(ps.OP_NVFP4, B=B, N=N, d=d)
    ps.ps_nvfp4_residual(H, mu, assign, rho, *ref, ws=ws)
    got = _outputs(H)
    ps.ps_nvfp4_residual_noalloc(H, mu, assign, rho, *got)     # warm: set-up done
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(2):
        ps.ps_nvfp4_residual_noalloc(H, mu, assign, rho, *got)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    ps.ps_check()
    for r, q in zip(ref, got):
        assert torch.equal(r, q)
