"""Offload of the quantised clusters and their reconstruction (oracle).

Test infrastructure: only tests/, __graft_entry__.smoke() and bench.py's CPU
legs use this module; it shares no code with the CUDA path.

[Polestar §2.C, CPU offloading]: the quantised hidden-state clusters are
offloaded to pinned CPU memory while only the centroids stay on the GPU, and
the top-k clusters are fetched back asynchronously.  [Polestar §2.A, local
window & clustering]: the NVFP4 residuals are compact proxies of the hidden
states.  The page gives neither a store layout nor the reconstruction; the
readings taken:

* store: one record per row, grouped by cluster in ascending cluster id and,
  inside a cluster, in ascending position; a record is the row's E2M1 codes
  (d/2 bytes) then its E4M3 block scales (d/16 bytes), each part zero-padded
  to a multiple of 16 bytes; `order[r]` is the position of record r and
  `cl_off[c]` the first record of cluster c (cl_off[C] = N);
* reconstruction of row i of cluster c, element e of block b, in fp32 with
  one rounding per operation (no fused multiply-add), mirroring the
  quantiser's divisor fl(s_b * S):
      g = fl(s_b * S),  deq = fl(v_e * g),  t = fl(rho_i * mu_c[e]),
      h~ = fl(t + deq),
  with v_e the E2M1 value of the element's code and s_b the E4M3 value of
  the block's scale; the refresh takes h~ rounded to bf16 (nearest-even).
"""

import numpy as np

from .nvfp4 import e2m1_decode, e4m3_decode

_F32 = np.float32


def record_bytes(d):
    """Bytes of one store record: codes then scales, each padded to 16."""
    def up16(x):
        return (x + 15) // 16 * 16
    return up16(d // 2) + up16(d // 16)


def pack_clusters(codes, scales, assign, C):
    """Store of one window: (store [N][rec] u8, order [N] i64, cl_off [C+1] i64).

    codes [N][d/2] u8, scales [N][d/16] u8, assign [N] in [0, C)."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    assign = np.asarray(assign, dtype=np.int64)
    N, half = codes.shape
    d = 2 * half
    rec = record_bytes(d)
    off_s = (half + 15) // 16 * 16  # start of the scales part
    order = []
    cl_off = np.zeros(C + 1, dtype=np.int64)
    for c in range(C):
        members = [i for i in range(N) if assign[i] == c]   # ascending position
        cl_off[c + 1] = cl_off[c] + len(members)
        order.extend(members)
    order = np.array(order, dtype=np.int64)
    store = np.zeros((N, rec), dtype=np.uint8)
    for r, i in enumerate(order):
        store[r, :half] = codes[i]
        store[r, off_s:off_s + d // 16] = scales[i]
    return store, order, cl_off


def reconstruct_row(code_row, scale_row, S, mu_c, rho_i):
    """h~ of one row (fp32 [d]) from its codes [d/2], scales [d/16], the
    window's tensor scale S, its centroid mu_c [d] and rho_i."""
    code_row = np.asarray(code_row, dtype=np.int64)
    d = 2 * code_row.shape[0]
    nib = np.empty(d, dtype=np.int64)
    nib[0::2] = code_row & 0xF            # element 2j: low nibble of byte j
    nib[1::2] = code_row >> 4
    v = e2m1_decode(nib).astype(_F32)
    s = e4m3_decode(np.asarray(scale_row, dtype=np.int64)).astype(_F32)
    g = (s * _F32(S)).astype(_F32)                       # fl(s_b * S)
    deq = (v * np.repeat(g, 16)).astype(_F32)            # fl(v * g)
    t = (_F32(rho_i) * np.asarray(mu_c, dtype=_F32)).astype(_F32)   # fl(rho * mu)
    return (t + deq).astype(_F32)                        # fl(t + deq)


def fetch_reconstruct(store, order, cl_off, sel, mu, rho, S, d):
    """{position: h~ fp32 [d]} of every member of the selected clusters
    (entries of sel < 0 ignored), read from the store."""
    store = np.asarray(store, dtype=np.uint8)
    half = d // 2
    off_s = (half + 15) // 16 * 16
    out = {}
    for c in sel:
        c = int(c)
        if c < 0:
            continue
        for r in range(int(cl_off[c]), int(cl_off[c + 1])):
            i = int(order[r])
            out[i] = reconstruct_row(store[r, :half], store[r, off_s:off_s + d // 16], S,
                                     mu[c], rho[i])
    return out
