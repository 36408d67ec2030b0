"""Proxy attention on cluster centroids and the per-position KL drift (oracle).

[Polestar §2.A, sparse updates]: every step computes a proxy attention of the
window's queries against the cluster centroids instead of all keys.
[Polestar §2.A, drift measurement]: the drift of position i at step t is
D_i = KL(A_i^(t) || A_i^(t-1)), A_i the attention distribution of that token.

Readings taken where the page is silent:
* the centroid keys are the centroid proxies pushed through the key
  projection, K~_c = C_hat_c W_k (one key per cluster and KV head);
* head h attends with KV head floor(h / G), G = Hq / Hkv, scale 1/sqrt(dh);
* a token's distribution over the C clusters is the mean over its Hq heads of
  the per-head softmax;
* no previous distribution (first step of a window) gives D = 0;
* terms with A[c] = 0 contribute 0; A_prev[c] is floored at 1e-30;
* D is floored at 0 (KL >= 0 holds exactly, the floor only removes rounding).
"""

import numpy as np

KL_PREV_FLOOR = 1e-30


def centroid_keys(chat, Wk):
    """K~ = C_hat W_k: [C][d] x [d][Hkv*dh] -> [C][Hkv*dh], fp64."""
    return np.asarray(chat, np.float64) @ np.asarray(Wk, np.float64)


def kl_divergence_rows(A, A_prev):
    """Row-wise KL(A || A_prev) with the conventions above, floored at 0."""
    A = np.asarray(A, np.float64)
    Ap = np.maximum(np.asarray(A_prev, np.float64), KL_PREV_FLOOR)
    terms = np.zeros_like(A)
    pos = A > 0
    terms[pos] = A[pos] * (np.log(A[pos]) - np.log(Ap[pos]))
    return np.maximum(terms.sum(axis=1), 0.0)


def proxy_attn_kl(Q, Kt, Hq, Hkv, dh, A_prev=None):
    """One window's proxy attention and drift.

    Q [N][Hq][dh] queries; Kt [C][Hkv*dh] centroid keys; A_prev [N][C] or None.
    Returns (A [N][C], D [N]) in fp64."""
    Q = np.asarray(Q, np.float64)
    Kt = np.asarray(Kt, np.float64)
    N = Q.shape[0]
    C = Kt.shape[0]
    G = Hq // Hkv
    A = np.zeros((N, C))
    for h in range(Hq):
        g = h // G
        s = Q[:, h, :] @ Kt[:, g * dh:(g + 1) * dh].T / np.sqrt(dh)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        A += p / p.sum(axis=1, keepdims=True)
    A /= Hq
    D = np.zeros(N) if A_prev is None else kl_divergence_rows(A, A_prev)
    return A, D
