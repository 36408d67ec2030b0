"""Spherical k-means over a window's hidden states (oracle, fp64).

[Polestar §2.A, local window & clustering]: the hidden states of the local
window (prefix, current and suffix blocks) are clustered with spherical
k-means.  The page names the algorithm only; the steps below are the textbook
spherical k-means of Dhillon & Modha (2001): points and centroids live on the
unit sphere, a point joins the centroid of largest cosine, a centroid is the
normalised sum of its members.

Readings taken where the page is silent:
* ties in the assignment go to the lowest cluster index;
* an empty cluster (or one whose member sum is the zero vector) keeps its
  centroid;
* after the last update one more assignment pass runs with the final
  centroids, so the returned assignment and centroids agree;
* rho_i = <h_i, mu_{a_i}> is the length of h_i along its centroid, and the
  centroid's hidden-space proxy is C_hat_c = mean(rho over members) * mu_c;
  an empty cluster keeps the caller's C_hat_c;
* a row of zero norm normalises to the zero vector (all its cosines are 0, so
  it joins cluster 0 with rho = 0);
* seeding is k-means++ (Arthur & Vassilvitskii, 2007) on the sphere, with the
  uniforms it draws passed in by the caller (see ``kmeanspp_init``).
"""

import numpy as np


def normalize_rows(H):
    """x_hat_i = h_i / ||h_i|| in fp64; zero rows stay zero."""
    H = np.asarray(H, dtype=np.float64)
    norms = np.sqrt(np.sum(H * H, axis=1))
    out = np.zeros_like(H)
    nz = norms > 0
    out[nz] = H[nz] / norms[nz, None]
    return out


def kmeanspp_init(H, C, u, return_margin=False):
    """k-means++ seeding on the unit sphere.

    H: [N][d] hidden states of one window; u: C uniforms in [0, 1) supplied by
    the caller (the random draws of the seeding are inputs, not generated
    here).  The distance of a point to the chosen set is the chordal one,
    ||x - mu||^2 / 2 = 1 - cos, so the weight of row i is
    w_i = 1 - max_{chosen j} cos(x_hat_i, x_hat_j), floored at 0, and exactly
    0 for rows already chosen.

    * first centre: row floor(u_0 * N) (clamped to N - 1);
    * centre r >= 1: the smallest row i whose inclusive prefix sum of w (fp64,
      in row order) exceeds u_r * sum(w); if sum(w) == 0 the smallest row not
      yet chosen.

    Returns (mu [C][d] fp64 unit rows, chosen row indices [C]).  With
    return_margin=True also the smallest distance, relative to sum(w), of any
    draw u_r * sum(w) from a prefix-sum boundary (a draw that close to a
    boundary may legitimately pick the neighbouring row under a different
    summation order).
    """
    Xh = normalize_rows(H)
    N = Xh.shape[0]
    u = np.asarray(u, dtype=np.float64)
    first = min(int(np.floor(u[0] * N)), N - 1)
    chosen = [first]
    w = np.maximum(0.0, 1.0 - Xh @ Xh[first])
    w[first] = 0.0
    margin = np.inf
    for r in range(1, C):
        prefix = np.cumsum(w)          # sequential, in row order
        total = prefix[-1]
        pick = -1
        if total > 0:
            target = u[r] * total
            above = np.nonzero(prefix > target)[0]
            if above.size:
                pick = int(above[0])
                lo = prefix[pick - 1] if pick > 0 else 0.0
                margin = min(margin, (prefix[pick] - target) / total,
                             (target - lo) / total)
        if pick < 0:
            taken = set(chosen)
            pick = next(i for i in range(N) if i not in taken)
        chosen.append(pick)
        w = np.minimum(w, np.maximum(0.0, 1.0 - Xh @ Xh[pick]))
        for j in chosen:
            w[j] = 0.0
    mu, idx = Xh[chosen].copy(), np.array(chosen, dtype=np.int64)
    return (mu, idx, margin) if return_margin else (mu, idx)


def _assign(Xh, mu):
    """Cosine of every row with every centroid; first-maximum argmax."""
    S = Xh @ mu.T                                   # [N][C]
    a = np.argmax(S, axis=1)                        # numpy: first maximum
    best = S[np.arange(S.shape[0]), a]
    if S.shape[1] > 1:
        masked = S.copy()
        masked[np.arange(S.shape[0]), a] = -np.inf
        margin = best - masked.max(axis=1)
    else:
        margin = np.full(S.shape[0], np.inf)
    return a, best, margin


def kmeans_spherical(H, mu0, iters, chat_in=None):
    """Spherical k-means of one window, warm-started from mu0.

    H: [N][d]; mu0: [C][d] initial centroids (used as given); iters: number of
    centroid updates I >= 0.  Passes t = 0..I each assign every row; passes
    t < I then update the centroids.

    Returns a dict:
      mu      [C][d] final centroids (mu^(I))
      assign  [N]    a^(I), from the final centroids
      rho     [N]    <h_i, mu_{a_i}>
      counts  [C]    cluster sizes n_c
      chat    [C][d] mean(rho over members) * mu_c, or chat_in[c] if n_c = 0
      obj     [I+1]  sum_i cos(x_hat_i, mu^(t)_{a_i^(t)}) for every pass
      margin  [I+1][N] top-2 cosine margin of every row in every pass
      mus     list of the I+1 centroid sets each pass assigned against
    """
    H = np.asarray(H, dtype=np.float64)
    mu = np.array(mu0, dtype=np.float64, copy=True)
    C = mu.shape[0]
    Xh = normalize_rows(H)
    obj, margins, mus = [], [], []
    a = None
    for t in range(iters + 1):
        mus.append(mu.copy())
        a, best, margin = _assign(Xh, mu)
        obj.append(best.sum())
        margins.append(margin)
        if t < iters:
            for c in range(C):
                members = a == c
                if not members.any():
                    continue
                uc = Xh[members].sum(axis=0)
                nu = np.sqrt(np.dot(uc, uc))
                if nu > 0:
                    mu[c] = uc / nu
    rho = np.sum(H * mu[a], axis=1)
    counts = np.bincount(a, minlength=C).astype(np.int64)
    chat = (np.zeros_like(mu) if chat_in is None
            else np.array(chat_in, dtype=np.float64, copy=True))
    for c in range(C):
        if counts[c] > 0:
            chat[c] = (rho[a == c].sum() / counts[c]) * mu[c]
    return dict(mu=mu, assign=a.astype(np.int64), rho=rho, counts=counts,
                chat=chat, obj=np.array(obj), margin=np.array(margins),
                mus=mus)
