"""Pins of the oracle's confidence and drift-aware commit rule.

Every expected value below is worked by hand from the rule as stated on the
page (technical summary 2.B): commit when c >= tau_s, or when the drift delta
exceeds alpha (tau_s - c)^2; suffix tokens need c >= tau_s and a selected
cluster."""
import math

import numpy as np

from oracle import CommitParams, commit_rule, confidence

CUR, SUF, OFF = 0, 1, 2
DROP, RISE, RATIO = 0, 1, 2


def test_uniform_and_one_hot_confidence():
    tok, c = confidence(np.full(1000, 3.25))
    assert tok == 0 and math.isclose(c, 1 / 1000, rel_tol=1e-14)
    L, V = 7.0, 512
    row = np.zeros(V); row[77] = L
    tok, c = confidence(row)
    assert tok == 77 and math.isclose(c, 1 / (1 + (V - 1) * math.exp(-L)), rel_tol=1e-14)
    row[300] = L                                   # a tie -> first arg-max
    assert confidence(row)[0] == 77


def _logits_with_conf(cs, V=64):
    """Rows whose confidence is exactly c: one peak of height ln(c (V-1)/(1-c))."""
    rows = []
    for c in cs:
        r = np.zeros(V)
        r[5] = math.log(c * (V - 1) / (1 - c))
        rows.append(r)
    return np.array(rows)


def _run(cs, role, D, s, n, prev, p, und=None, sel=None):
    P = len(cs)
    und = np.ones(P, np.uint8) if und is None else np.array(und, np.uint8)
    return commit_rule(_logits_with_conf(cs), np.array(role), und,
                       np.array(D, np.float32), np.array(s, np.float32),
                       np.array(n), np.array(prev, np.float32), sel, p)


def test_confidence_rule_and_no_drift_history():
    p = CommitParams(tau_s=0.9, alpha=1.0, ensure_progress=0)
    r = _run([0.95, 0.5, 0.89], [CUR] * 3, [0, 0, 0], [0, 0, 0], [0, 0, 0], [0, 0, 0], p)
    assert list(r["commit"]) == [1, 0, 0]
    assert np.allclose(r["conf"], [0.95, 0.5, 0.89], rtol=1e-12)
    # state folded in for every undecided current token, then decided
    assert list(r["d_cnt"]) == [1, 1, 1] and list(r["undecided"]) == [0, 1, 1]


def test_delta_drop_threshold():
    # c = 0.5: tau_d = 1.0 * (0.9 - 0.5)^2 = 0.16
    # mean = 0.4 / 2 = 0.2; D = 0.03 -> Delta = 0.17 > 0.16 commits
    #                           D = 0.05 -> Delta = 0.15 does not
    p = CommitParams(tau_s=0.9, alpha=1.0, mode=DROP, ensure_progress=0)
    r = _run([0.5, 0.5], [CUR, CUR], [0.03, 0.05], [0.4, 0.4], [2, 2], [0, 0], p)
    assert list(r["commit"]) == [1, 0]
    assert np.isclose(r["d_sum"][0], np.float32(np.float32(0.4) + np.float32(0.03)))
    assert list(r["d_prev"]) == [np.float32(0.03), np.float32(0.05)]


def test_delta_rise_and_alpha_zero():
    p = CommitParams(tau_s=0.9, alpha=0.0, mode=RISE, ensure_progress=0)
    # alpha = 0: any positive Delta = D - mean commits
    r = _run([0.2, 0.2, 0.2], [CUR] * 3, [0.31, 0.3, 0.29], [0.3, 0.3, 0.3], [1, 1, 1],
             [0, 0, 0], p)
    assert list(r["commit"]) == [1, 0, 0]


def test_tau_above_one_disables_confidence():
    p = CommitParams(tau_s=1.01, alpha=1.0, ensure_progress=0)
    r = _run([0.999, 0.999], [CUR, SUF], [0, 0], [0, 0], [0, 0], [0, 0], p,
             sel=np.array([1, 1]))
    assert list(r["commit"]) == [0, 0]


def test_ratio_edge_is_strict():
    p = CommitParams(tau_s=0.9, ratio=0.5, mode=RATIO, ensure_progress=0)
    # prev 0.5 -> threshold 0.25: D = 0.25 stays, 0.2499 commits, no history: no rule
    r = _run([0.1, 0.1, 0.1], [CUR] * 3, [0.25, 0.2499, 0.0], [1, 1, 0], [1, 1, 0],
             [0.5, 0.5, 0.5], p)
    assert list(r["commit"]) == [0, 1, 0]


def test_suffix_rule_and_inactive():
    p = CommitParams(tau_s=0.9, ensure_progress=0)
    r = _run([0.95, 0.95, 0.5, 0.99], [SUF, SUF, SUF, OFF], [0] * 4, [0] * 4, [0] * 4,
             [0] * 4, p, sel=np.array([1, 0, 1, 1]))
    assert list(r["commit"]) == [1, 0, 0, 0]
    assert list(r["d_cnt"]) == [0, 0, 0, 0]        # only current tokens keep state
    r = _run([0.95], [SUF], [0], [0], [0], [0], p, sel=None)
    assert list(r["commit"]) == [0]


def test_ensure_progress_and_decided_tokens():
    p = CommitParams(tau_s=0.9, ensure_progress=1)
    r = _run([0.3, 0.6, 0.6, 0.8], [CUR] * 4, [0] * 4, [0] * 4, [0] * 4, [0] * 4, p,
             und=[1, 1, 1, 0])
    assert list(r["commit"]) == [0, 1, 0, 0]       # best undecided, lower j on ties
    assert list(r["d_cnt"]) == [1, 1, 1, 0]        # decided tokens keep their state
    assert list(r["undecided"]) == [1, 0, 1, 0]
