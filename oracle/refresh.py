"""Sparse K/V refresh of the selected positions (oracle).

[Polestar §2.A, sparse updates]: a sparse forward pass on only the positions
of the top-k clusters produces an update packet that refreshes the matching
KV-cache entries.

Readings taken where the page is silent:
* the refresh recomputes K = h W_k and V = h W_v from the window's current
  hidden states (no bias, no rotary embedding);
* window position p is cache row cache_off + p;
* rows not selected are left untouched;
* a bf16 cache stores the product rounded to bf16 (round-to-nearest-even,
  through fp32); an fp32 cache stores it rounded to fp32.
The part of the update packet that refreshes hidden states of later layers
needs a full transformer layer with trained weights and is not restated.
"""

import numpy as np


def bf16_round(x):
    """Round to bf16 (RNE on the fp32 bit pattern); returned as float32."""
    f = np.array(x, dtype=np.float32, ndmin=1)
    bits = f.view(np.uint32).astype(np.uint64)
    bias = ((bits >> 16) & 1) + 0x7FFF
    out = (((bits + bias) >> 16) << 16).astype(np.uint32)
    return out.view(np.float32).reshape(np.shape(x))


def refresh_kv(H, pos, npos, Wk, Wv, Kcache, Vcache, cache_off, bf16_cache):
    """One window.  H [N][d]; pos [N]; W [d][Hkv*dh];
    Kcache/Vcache [Ncache][Hkv*dh] float32 arrays (bf16 values when
    bf16_cache).  Returns updated copies of both caches."""
    H = np.asarray(H, np.float64)
    Wk = np.asarray(Wk, np.float64)
    Wv = np.asarray(Wv, np.float64)
    Kc = np.array(Kcache, dtype=np.float32, copy=True)
    Vc = np.array(Vcache, dtype=np.float32, copy=True)
    rnd = bf16_round if bf16_cache else (lambda v: np.asarray(v, np.float32))
    for j in range(npos):
        p = int(pos[j])
        Kc[cache_off + p] = rnd(H[p] @ Wk)
        Vc[cache_off + p] = rnd(H[p] @ Wv)
    return Kc, Vc
