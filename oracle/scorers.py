"""Alternative drift signals of the ablation (oracle).

Test infrastructure: only tests/ and bench.py's CPU legs use this module; it
shares no code with the library.

[Polestar §2.A, drift measurement]: the KL divergence between a token's
attention distributions at consecutive steps tracks contextual shifts more
closely than cosine dissimilarity on subsets.  [Polestar §4, ablation
studies]: KL-based drift beats cosine similarity and uncertainty-based
selection.  The page defines neither alternative; the readings taken, both
on the same proxy attention distributions A_i (rows of [N][C]) that the KL
scorer uses, so that only the signal differs:

* cosine dissimilarity: D_i = 1 - <A_i, A'_i> / (||A_i|| ||A'_i||), A'_i the
  previous step's distribution ("on subsets": the C cluster entries stand for
  the subset of keys); 0 without a previous step;
* uncertainty: D_i = -sum_c A_ic ln A_ic, the entropy of the current
  distribution (terms with A_ic = 0 are 0); it needs no previous step;
* KL, for the same interface: D_i = sum_c A_ic ln(A_ic / A'_ic) over
  A_ic > 0, clamped at 0, as the fused proxy drift computes it.
fp64 throughout.
"""

import numpy as np

SCORER_KL, SCORER_COSINE, SCORER_ENTROPY = 0, 1, 2


def drift_score(A, A_prev, scorer):
    """D [N] of distributions A [N][C] against A_prev [N][C] (or None)."""
    A = np.asarray(A, np.float64)
    N = A.shape[0]
    D = np.zeros(N)
    if scorer == SCORER_ENTROPY:
        for i in range(N):
            a = A[i][A[i] > 0]
            D[i] = -np.sum(a * np.log(a))
        return D
    if A_prev is None:
        return D
    Ap = np.asarray(A_prev, np.float64)
    for i in range(N):
        if scorer == SCORER_COSINE:
            na, npv = np.linalg.norm(A[i]), np.linalg.norm(Ap[i])
            D[i] = 1.0 - np.dot(A[i], Ap[i]) / (na * npv) if na > 0 and npv > 0 else 0.0
        elif scorer == SCORER_KL:
            m = A[i] > 0
            D[i] = max(0.0, np.sum(A[i][m] * np.log(A[i][m] / np.maximum(Ap[i][m], 1e-30))))
        else:
            raise ValueError(f"unknown scorer {scorer}")
    return D
