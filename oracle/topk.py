"""Top-k most-drifting clusters and the positions they cover (oracle).

[Polestar §2.A, sparse updates]: the top-k clusters with the largest drift are
identified and a sparse forward pass runs on only their positions.

Readings taken where the page is silent:
* a cluster's drift is the mean of D over its members, summed in fp64 one
  member at a time in ascending position order, then divided by n_c;
* empty clusters are never selected;
* ranking is by that mean, descending, ties to the lower cluster index;
  fewer than k non-empty clusters pad `sel` with -1 and `sel_score` with -inf;
* the refreshed positions are every i whose cluster is selected, ascending;
  `pos` is padded with -1 beyond `npos`.
"""

import numpy as np


def topk_drift(D, assign, counts, k):
    """One window.  D [N] fp32, assign [N], counts [C], k <= C.

    Returns (sel [k] int32, sel_score [k] float32, pos [N] int32, npos int,
    posmask [N] uint8, score [C] fp64 with NaN for empty clusters)."""
    D = np.asarray(D, dtype=np.float32)
    assign = np.asarray(assign)
    counts = np.asarray(counts)
    N, C = D.shape[0], counts.shape[0]
    sums = [0.0] * C
    for i in range(N):                       # ascending i, one add at a time
        sums[int(assign[i])] += float(D[i])
    score = np.full(C, np.nan)
    live = []
    for c in range(C):
        if counts[c] > 0:
            score[c] = sums[c] / float(counts[c])
            live.append(c)
    ranked = sorted(live, key=lambda c: (-score[c], c))[:k]
    sel = np.full(k, -1, dtype=np.int32)
    sel_score = np.full(k, -np.inf, dtype=np.float32)
    for r, c in enumerate(ranked):
        sel[r] = c
        sel_score[r] = np.float32(score[c])
    chosen = set(ranked)
    posmask = np.array([1 if int(assign[i]) in chosen else 0 for i in range(N)],
                       dtype=np.uint8)
    hits = np.nonzero(posmask)[0]
    pos = np.full(N, -1, dtype=np.int32)
    pos[:hits.size] = hits
    return sel, sel_score, pos, int(hits.size), posmask, score
