"""Drift-aware token commitment (oracle).

[Polestar §2.B, current block commitment]: the drift delta Delta_j is the
deviation of the current drift from its historical mean; token j commits when
Delta_j exceeds tau_d,j = alpha (tau_s - c_j)^2, c_j its confidence.
[Polestar §2.B, suffix block commitment]: when the last layer's top-drift
clusters include the suffix window's, a suffix token commits only if its
confidence is at least tau_s.

Readings taken where the page is silent or inconsistent:
* confidence c_j is the largest softmax probability of row j's logits and the
  token is the first arg-max (standard diffusion-LM confidence);
* the confidence rule c_j >= tau_s commits on its own (the static threshold
  the drift rule extends);
* the historical mean is d_sum / d_cnt over earlier steps of the current block
  (the caller zeroes the state at block start); with d_cnt = 0 there is no
  drift rule yet;
* the sign of Delta: the technical summary reads "sharp positive delta"
  while the lay text commits when the drift settles; mode DELTA_DROP
  (Delta = mean - D) is the default, DELTA_RISE (Delta = D - mean) and RATIO
  (D < ratio * previous D) are the alternatives;
* a suffix token is "among the top-drift clusters" when the last layer's
  position mask selects it;
* ensure_progress: if no current-block token commits while some are
  undecided, the undecided current token with the largest c commits (ties to
  the lower j), as semi-autoregressive diffusion decoders do;
* after the decision every undecided current-block token folds its D into the
  state (d_sum = fl32(d_sum + D), d_cnt += 1, d_prev = D), then committed
  tokens become decided.
Roles: 0 current block, 1 suffix block, 2 inactive (no decision, no state).
"""

from dataclasses import dataclass

import numpy as np

ROLE_CURRENT, ROLE_SUFFIX, ROLE_INACTIVE = 0, 1, 2
MODE_DELTA_DROP, MODE_DELTA_RISE, MODE_RATIO = 0, 1, 2


@dataclass
class CommitParams:
    tau_s: float = 0.9
    alpha: float = 1.0
    ratio: float = 0.1
    mode: int = MODE_DELTA_DROP
    ensure_progress: int = 1


def confidence(logits_row):
    """(token, c): first arg-max and 1 / sum_v exp(l_v - max), fp64."""
    l = np.asarray(logits_row, np.float64)
    m = l.max()
    token = int(np.nonzero(l == m)[0][0])
    return token, 1.0 / np.exp(l - m).sum()


def commit_rule(logits, role, undecided, D_blk, d_sum, d_cnt, d_prev,
                suffix_sel, p):
    """One batch element's block of P positions.

    logits [P][V]; role [P]; undecided [P] (0/1); D_blk [P] fp32 drift of the
    last layer; d_sum/d_prev [P] fp32, d_cnt [P] int; suffix_sel [P] or None.
    Returns dict(token, conf, commit, undecided, d_sum, d_cnt, d_prev,
    margin) where margin[j] is the smallest relative distance of any decision
    input of row j from its threshold (for tie-band accounting)."""
    # thresholds cross the C ABI as fp32: decide with the same values
    p = CommitParams(tau_s=float(np.float32(p.tau_s)), alpha=float(np.float32(p.alpha)),
                     ratio=float(np.float32(p.ratio)), mode=p.mode,
                     ensure_progress=p.ensure_progress)
    P = len(role)
    token = np.zeros(P, np.int32)
    conf = np.zeros(P)
    for j in range(P):
        token[j], conf[j] = confidence(logits[j])
    commit = np.zeros(P, np.uint8)
    margin = np.full(P, np.inf)
    und = np.array(undecided, dtype=np.uint8, copy=True)
    s = np.array(d_sum, dtype=np.float32, copy=True)
    n = np.array(d_cnt, dtype=np.int64, copy=True)
    prev = np.array(d_prev, dtype=np.float32, copy=True)
    Dv = np.asarray(D_blk, dtype=np.float32)

    def rel(x, t):
        return abs(x - t) / max(abs(t), 1e-30)

    for j in range(P):
        if not und[j]:
            continue
        c = conf[j]
        if role[j] == ROLE_CURRENT:
            ok = c >= p.tau_s
            margin[j] = rel(c, p.tau_s)
            if n[j] >= 1:
                D = float(Dv[j])
                mean = float(s[j]) / float(n[j])
                if p.mode == MODE_RATIO:
                    thr = p.ratio * float(prev[j])
                    ok = ok or D < thr
                    margin[j] = min(margin[j], rel(D, thr))
                else:
                    delta = mean - D if p.mode == MODE_DELTA_DROP else D - mean
                    thr = p.alpha * (p.tau_s - c) ** 2
                    ok = ok or delta > thr
                    margin[j] = min(margin[j], rel(delta, thr))
            commit[j] = 1 if ok else 0
        elif role[j] == ROLE_SUFFIX:
            sel = suffix_sel is not None and suffix_sel[j] != 0
            commit[j] = 1 if (sel and c >= p.tau_s) else 0
            if sel:
                margin[j] = rel(c, p.tau_s)
    cur = [j for j in range(P) if role[j] == ROLE_CURRENT and und[j]]
    if p.ensure_progress and cur and not any(commit[j] for j in cur):
        best = max(cur, key=lambda j: (conf[j], -j))
        commit[best] = 1
        for j in cur:                         # the pick must be unambiguous
            if j != best:
                margin[best] = min(margin[best], rel(conf[j], conf[best]))
    for j in cur:
        s[j] = np.float32(s[j] + Dv[j])
        n[j] += 1
        prev[j] = Dv[j]
    und[commit == 1] = 0
    return dict(token=token, conf=conf, commit=commit, undecided=und,
                d_sum=s, d_cnt=n.astype(np.int32), d_prev=prev, margin=margin)
