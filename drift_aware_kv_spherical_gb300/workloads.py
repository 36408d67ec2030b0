"""Seeded synthetic workloads shared by the tests, the smoke run and the bench.

This module only draws random numbers and lays them out; it holds none of the
drift-scoring arithmetic.  The shapes follow the model layers the Polestar
explainer evaluates on (LLaDA-8B: d = 4096, 32 heads x 128; Dream-7B:
d = 3584, 28 query / 4 KV heads x 128), with hidden states built around
planted cluster directions so that spherical k-means has structure to find.
No dataset, checkpoint or trained weight is used.

Seeds: base 20260717 + workload index; per layer + 1000 * layer; per step + t.
"N(0, s)" means standard deviation s.
"""

from dataclasses import dataclass, field
import math

import torch

BASE_SEED = 20260717

ROLE_CURRENT, ROLE_SUFFIX, ROLE_INACTIVE = 0, 1, 2
MODE_DELTA_DROP, MODE_DELTA_RISE, MODE_RATIO = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    N: int
    d: int
    Hq: int
    Hkv: int
    dh: int
    C: int
    iters: int
    k: int
    P: int
    V: int
    dtype: str              # "f32" or "bf16": hidden states, queries, weights, cache
    planted: int            # planted cluster directions
    noise: float            # tiny: additive N(0, noise); others: mixing recipe
    drift_frac: float       # fraction of non-block rows that drift per step
    drift_std: float
    blk_start: int          # first window position of the current block
    logit_std: float
    wq_std: float
    wkv_std: float = 0.02
    layers: int = 1
    mode: int = MODE_DELTA_DROP
    tau_s: float = 0.9
    alpha: float = 1.0
    ratio: float = 0.1
    walk: bool = False      # 32-layer loop: decaying random walk on all rows
    logits: str = "f32"     # dtype the block's logits arrive in: "f32" where the
                            # workload states it, else the model's own ("bf16")
    desc: str = field(default="", compare=False)

    @property
    def G(self):
        return self.Hq // self.Hkv

    @property
    def Ncache(self):
        return self.N

    @property
    def seed(self):
        return BASE_SEED + self.index


WORKLOADS = [
    Workload("tiny_d256_n128", 0, B=1, N=128, d=256, Hq=4, Hkv=4, dh=64, C=8,
             iters=5, k=2, P=16, V=1024, dtype="f32", planted=8, noise=0.1,
             drift_frac=0.10, drift_std=0.5, blk_start=56, logit_std=2.0,
             wq_std=40.0,
             desc="tiny single layer, batch 1, fp32"),
    Workload("llada8b_layer_n1024", 1, B=1, N=1024, d=4096, Hq=32, Hkv=32,
             dh=128, C=64, iters=10, k=8, P=32, V=126464, dtype="bf16",
             planted=64, noise=1.0, drift_frac=0.05, drift_std=0.5,
             blk_start=512, logit_std=2.0, wq_std=0.02, logits="bf16",
             desc="LLaDA-8B-shaped layer, batch 1, window 1024"),
    Workload("dream7b_gqa_b8_n2048", 2, B=8, N=2048, d=3584, Hq=28, Hkv=4,
             dh=128, C=128, iters=10, k=12, P=32, V=152064, dtype="bf16",
             planted=128, noise=1.0, drift_frac=0.05, drift_std=0.5,
             blk_start=1024, logit_std=3.0, wq_std=0.02,
             desc="Dream-7B-shaped GQA layer, batch 8, window 2048"),
    Workload("llada8b_loop32_b4_n768", 3, B=4, N=768, d=4096, Hq=32, Hkv=32,
             dh=128, C=64, iters=10, k=8, P=32, V=126464, dtype="bf16",
             planted=64, noise=1.0, drift_frac=1.0, drift_std=0.3,
             blk_start=512, logit_std=2.0, wq_std=0.02, layers=32,
             mode=MODE_RATIO, ratio=0.1, walk=True, logits="bf16",
             desc="32-layer LLaDA-8B-shaped step loop, batch 4"),
    Workload("stress_b32_n4096_l32", 4, B=32, N=4096, d=4096, Hq=32, Hkv=32,
             dh=128, C=256, iters=15, k=16, P=64, V=126464, dtype="bf16",
             planted=256, noise=1.0, drift_frac=0.05, drift_std=0.5,
             blk_start=2048, logit_std=2.0, wq_std=0.02, layers=32,
             desc="stress: 32 layers, batch 32, window 4096"),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def torch_dtype(w):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, g, device, std=1.0):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def make_layer(w, layer=0, device="cpu", B=None):
    """Hidden states and projection weights of one layer of workload `w`.

    Returns a dict with H [B][N][d], Wq [d][Hq*dh], Wk/Wv [d][Hkv*dh] (all in
    the workload's dtype), the planted directions U [planted][d] fp32 and the
    planted label z [B][N]."""
    B = w.B if B is None else B
    seed = w.seed + 1000 * layer
    g = _gen(seed, device)
    U = _randn((w.planted, w.d), g, device)
    U = U / U.norm(dim=1, keepdim=True)
    z = torch.randint(0, w.planted, (B, w.N), generator=g, device=device)
    if w.dtype == "f32":
        H = U[z] + _randn((B, w.N, w.d), g, device, w.noise)
    else:
        eps = _randn((B, w.N, w.d), g, device)
        H = (eps + math.sqrt(w.d) * U[z]) / math.sqrt(2.0)
    dt = torch_dtype(w)
    Wq = _randn((w.d, w.Hq * w.dh), g, device, w.wq_std).to(dt)
    Wk = _randn((w.d, w.Hkv * w.dh), g, device, w.wkv_std).to(dt)
    Wv = _randn((w.d, w.Hkv * w.dh), g, device, w.wkv_std).to(dt)
    return dict(H=H.to(dt), Wq=Wq, Wk=Wk, Wv=Wv, U=U, z=z)


def drift_rows(w, H, step, layer=0):
    """Hidden states of step `step` >= 1 from those of step - 1.

    Decaying random walk on every row (sigma_t = drift_std * 0.9^t) for the
    32-layer loop; otherwise the current block plus a seeded fraction of the
    other rows move by N(0, drift_std)."""
    device = H.device
    g = _gen(w.seed + 1000 * layer + 7919 * step, device)
    B, N, d = H.shape
    Hf = H.float()
    if w.walk:
        Hf = Hf + _randn((B, N, d), g, device, w.drift_std * 0.9 ** step)
    else:
        mask = torch.rand((B, N), generator=g, device=device) < w.drift_frac
        mask[:, w.blk_start:w.blk_start + w.P] = True
        Hf = Hf + _randn((B, N, d), g, device, w.drift_std) * mask[..., None]
    return Hf.to(H.dtype)


def drift_inplace(w, H, Q, Wq, step, layer=0):
    """Step `step` >= 1 of the drift, applied in place to H [B][N][d] and to
    the rows of Q = H Wq that moved: the same recipe as drift_rows (a seeded
    share of the rows plus the current block move by N(0, drift_std); the
    32-layer loop's random walk moves every row), drawn only for the rows
    that move, so a large window drifts without a second copy of it."""
    device = H.device
    g = _gen(w.seed + 1000 * layer + 7919 * step + 3, device)
    B, N, d = H.shape
    if w.walk:
        H.copy_((H.float() + _randn((B, N, d), g, device, w.drift_std * 0.9 ** step))
                .to(H.dtype))
        Q.copy_(make_queries(w, H, Wq))
        return
    mask = torch.rand((B, N), generator=g, device=device) < w.drift_frac
    mask[:, w.blk_start:w.blk_start + w.P] = True
    rows = mask.reshape(-1).nonzero().squeeze(1)
    Hf = H.view(B * N, d)
    moved = (Hf[rows].float() + _randn((rows.numel(), d), g, device, w.drift_std)).to(H.dtype)
    Hf[rows] = moved
    q = (moved @ Wq) if H.is_cuda else (moved.float() @ Wq.float())
    Q.view(B * N, -1)[rows] = q.to(Q.dtype)


def make_queries(w, H, Wq):
    """Q = H Wq laid out [B][N][Hq][dh] in the workload dtype (input
    synthesis; the drift path takes Q as given)."""
    B, N, d = H.shape
    if H.is_cuda:
        Q = (H.reshape(B * N, d) @ Wq).float()
    else:
        Q = H.reshape(B * N, d).float() @ Wq.float()
    return Q.reshape(B, N, w.Hq, w.dh).to(H.dtype).contiguous()


def logits_dtype(w):
    """The dtype a workload's block logits arrive in."""
    return torch.float32 if w.logits == "f32" else torch.bfloat16


def make_uniforms(w, layer=0, device="cpu", B=None):
    """The k-means++ draws, [B][C] fp64 in [0, 1)."""
    B = w.B if B is None else B
    g = _gen(w.seed + 1000 * layer + 17, device)
    return torch.rand((B, w.C), generator=g, device=device, dtype=torch.float64)


def make_logits(w, step=0, device="cpu", B=None, P=None, V=None):
    """Block logits [B][P][V] fp32 ~ N(0, logit_std), with a planted peak in a
    seeded half of the rows: token t gets max(row) + ln(10 V) + u, u ~ U[0, 1),
    which puts that row's confidence in (0.9, 1)."""
    B = w.B if B is None else B
    P = w.P if P is None else P
    V = w.V if V is None else V
    g = _gen(w.seed + 31 * step + 5, device)
    L = _randn((B, P, V), g, device, w.logit_std)
    peaked = torch.rand((B, P), generator=g, device=device) < 0.5
    tok = torch.randint(0, V, (B, P), generator=g, device=device)
    bump = torch.rand((B, P), generator=g, device=device)
    height = L.max(dim=2).values + math.log(10.0 * V) + bump
    rows = peaked.nonzero(as_tuple=True)
    L[rows[0], rows[1], tok[rows]] = height[rows]
    return L.contiguous()


def make_roles(w):
    """Block roles: every position of the P-token block is current-block."""
    return torch.full((w.P,), ROLE_CURRENT, dtype=torch.uint8)
