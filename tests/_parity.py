"""Shared helpers of the GPU parity tests: run a libpolestar call on device
tensors, bring results to numpy, compare against the oracle with the stated
criteria, and guard output buffers with canary bands."""

import numpy as np
import torch

from drift_aware_kv_spherical_gb300 import polestar as ps

# correctness criteria (the drift-scoring path's contract)
KM_MARGIN = 1e-5          # assignments exact where the top-2 cosine margin exceeds this
RTOL, ATOL = 1e-4, 1e-6   # KL, distributions, centroids (fp32)
KV_RTOL = 2e-2            # bf16 K/V refresh; abs floor 1e-3 * RMS(row)
CONF_RTOL = 1e-6          # token confidence
BAND = 1e-5               # commit decisions closer than this to a threshold are unpinned


def np_(t):
    return t.detach().float().cpu().numpy() if t.is_floating_point() else t.detach().cpu().numpy()


def assert_close(g, r, rtol=RTOL, atol=ATOL, what=""):
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    bad = np.abs(g - r) > atol + rtol * np.abs(r)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} differ; first at "
                             f"{tuple(i)}: gpu {g[tuple(i)]!r} oracle {r[tuple(i)]!r}")


class Guarded:
    """A device tensor living inside a larger buffer whose 4 KiB head and
    tail hold a canary pattern, to catch out-of-bounds writes."""

    PAD = 4096

    def __init__(self, shape, dtype, device="cuda", fill=0):
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.empty(nbytes + 2 * self.PAD, dtype=torch.uint8, device=device)
        self.raw.fill_(0xA5)
        self.t = self.raw[self.PAD:self.PAD + nbytes].view(dtype).view(*shape)
        self.t.fill_(fill) if dtype.is_floating_point else self.t.fill_(int(fill))

    def intact(self):
        head = self.raw[:self.PAD]
        tail = self.raw[-self.PAD:]
        return bool((head == 0xA5).all()) and bool((tail == 0xA5).all())


def run_kmeans(H, mu0, iters, init_u=None, chat0=None):
    B, N, d = H.shape
    C = mu0.shape[1]
    dev = H.device
    out = dict(mu=mu0.clone().contiguous(),
               assign=torch.full((B, N), -7, dtype=torch.int32, device=dev),
               rho=torch.zeros(B, N, device=dev),
               chat=(chat0.clone() if chat0 is not None
                     else torch.zeros(B, C, d, device=dev)),
               counts=torch.zeros(B, C, dtype=torch.int32, device=dev),
               obj=torch.zeros(B, iters + 1, device=dev))
    ws = ps.workspace(ps.OP_KMEANS, B=B, N=N, d=d, C=C)
    ps.ps_kmeans_spherical(H, out["mu"], out["assign"], out["rho"], out["chat"],
                           out["counts"], iters, init_mode=1 if init_u is not None else 0,
                           init_u=init_u, objective=out["obj"], ws=ws)
    torch.cuda.synchronize()
    ps.ps_check()
    return {k: np_(v) for k, v in out.items()}


def run_nvfp4(H, mu, assign, rho):
    B, N, d = H.shape
    dev = H.device
    codes = Guarded((B, N, d // 2), torch.uint8, dev, fill=0x77)
    scales = Guarded((B, N, d // 16), torch.uint8, dev, fill=0x77)
    S = Guarded((B,), torch.float32, dev, fill=-1.0)
    ws = ps.workspace(ps.OP_NVFP4, B=B, N=N, d=d)
    ps.ps_nvfp4_residual(H, mu, assign, rho, codes.t, scales.t, S.t, ws=ws)
    torch.cuda.synchronize()
    ps.ps_check()
    assert codes.intact() and scales.intact() and S.intact()
    return np_(codes.t), np_(scales.t), np_(S.t)


def run_proxy(Q, chat, Wk, Hkv, A_prev=None):
    B, N, Hq, dh = Q.shape
    C, d = chat.shape[1], chat.shape[2]
    A = Guarded((B, N, C), torch.float32, Q.device, fill=-5.0)
    D = Guarded((B, N), torch.float32, Q.device, fill=-5.0)
    ws = ps.workspace(ps.OP_PROXY_KL, B=B, N=N, d=d, C=C, Hq=Hq, Hkv=Hkv, dh=dh)
    ps.ps_proxy_attn_kl(Q, chat, Wk, A_prev, A.t, D.t, Hkv, ws=ws)
    torch.cuda.synchronize()
    ps.ps_check()
    assert A.intact() and D.intact()
    return A.t.clone(), D.t.clone()


def run_topk(D, assign, counts, k):
    B, N = D.shape
    dev = D.device
    sel = Guarded((B, k), torch.int32, dev, fill=-9)
    sc = Guarded((B, k), torch.float32, dev, fill=-9.0)
    pos = Guarded((B, N), torch.int32, dev, fill=-9)
    npos = Guarded((B,), torch.int32, dev, fill=-9)
    mask = Guarded((B, N), torch.uint8, dev, fill=9)
    ps.ps_topk_drift(D, assign, counts, k, sel.t, sc.t, pos.t, npos.t, mask.t)
    torch.cuda.synchronize()
    ps.ps_check()
    assert all(g.intact() for g in (sel, sc, pos, npos, mask))
    return np_(sel.t), np_(sc.t), np_(pos.t), np_(npos.t), np_(mask.t), pos.t, npos.t


def run_commit(logits, role, undecided, D_blk, d_ld, d_sum, d_cnt, d_prev, suffix_sel,
               params):
    B, P, V = logits.shape
    dev = logits.device
    und = undecided.clone()
    s, n, pv = d_sum.clone(), d_cnt.clone(), d_prev.clone()
    token = Guarded((B, P), torch.int32, dev, fill=-9)
    conf = Guarded((B, P), torch.float32, dev, fill=-9.0)
    com = Guarded((B, P), torch.uint8, dev, fill=9)
    ws = ps.workspace(ps.OP_COMMIT, B=B, P=P, V=V)
    ps.ps_commit(logits, role, und, D_blk, d_ld, s, n, pv, suffix_sel, P, params,
                 token.t, conf.t, com.t, ws=ws)
    torch.cuda.synchronize()
    ps.ps_check()
    assert token.intact() and conf.intact() and com.intact()
    return dict(token=np_(token.t), conf=np_(conf.t), commit=np_(com.t),
                undecided=np_(und), d_sum=np_(s), d_cnt=np_(n), d_prev=np_(pv))
