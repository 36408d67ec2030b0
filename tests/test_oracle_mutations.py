"""The pins catch plausible mistakes: each test plants one mistake in a copy
of an oracle function (on the CPU), runs the pins of that function against
the copy, and requires at least one of them to fail."""
import numpy as np
import pytest

from oracle import schedule as sched_mod
from oracle import scorers as scorers_mod
from tests import test_oracle_schedule as sched_pins
from tests import test_oracle_scorers as scorer_pins

SCHED_PINS = [sched_pins.test_every_step_when_tau_is_zero,
              sched_pins.test_tau_counts_committed_tokens,
              sched_pins.test_every_second_refresh_is_full,
              sched_pins.test_block_done_slides_and_restarts]
SCORER_PINS = [scorer_pins.test_entropy_closed_forms, scorer_pins.test_entropy_matches_scipy,
               scorer_pins.test_cosine_closed_forms,
               scorer_pins.test_cosine_matches_scipy_and_is_scale_free,
               scorer_pins.test_kl_agrees_with_the_proxy_drift_and_scipy,
               scorer_pins.test_scorers_rank_a_shifted_row_first]


def _some_pin_fails(pins):
    for pin in pins:
        try:
            pin()
        except AssertionError:
            return True
    return False


R, F, S, I = sched_mod.REFRESH, sched_mod.FULL, sched_mod.SLIDE, sched_mod.REINIT


def _sched_strict_threshold(tau, full, blk, st, committed, done):
    st.since += committed
    if done:
        st.block_start += blk
        st.since = st.refreshes = 0
        return R | F | S | I
    if st.since <= tau and tau > 0:          # mistake: needs more than tau tokens
        return 0
    st.since = 0
    st.refreshes += 1
    return R | (F if full > 0 and st.refreshes % full == 0 else 0)


def _sched_full_off_by_one(tau, full, blk, st, committed, done):
    st.since += committed
    if done:
        st.block_start += blk
        st.since = st.refreshes = 0
        return R | F | S | I
    if st.since < tau:
        return 0
    st.since = 0
    st.refreshes += 1
    return R | (F if full > 0 and st.refreshes % full == 1 else 0)   # mistake


def _sched_slide_keeps_count(tau, full, blk, st, committed, done):
    st.since += committed
    if done:
        st.block_start += blk
        st.refreshes = 0                      # mistake: the token count survives the slide
        return R | F | S | I
    if st.since < tau:
        return 0
    st.since = 0
    st.refreshes += 1
    return R | (F if full > 0 and st.refreshes % full == 0 else 0)


@pytest.mark.parametrize("mutant", [_sched_strict_threshold, _sched_full_off_by_one,
                                    _sched_slide_keeps_count])
def test_schedule_pins_catch(monkeypatch, mutant):
    monkeypatch.setattr(sched_pins, "schedule_step", mutant)
    assert _some_pin_fails(SCHED_PINS)


def test_schedule_pins_pass_on_the_oracle():
    assert not _some_pin_fails(SCHED_PINS)


def _score_mutant(kind):
    real = scorers_mod.drift_score

    def f(A, A_prev, scorer):
        A = np.asarray(A, np.float64)
        if kind == "entropy_sign" and scorer == scorers_mod.SCORER_ENTROPY:
            return -real(A, A_prev, scorer)
        if kind == "entropy_log2" and scorer == scorers_mod.SCORER_ENTROPY:
            return real(A, A_prev, scorer) / np.log(2.0)
        if kind == "cosine_unnormalised" and scorer == scorers_mod.SCORER_COSINE:
            if A_prev is None:
                return np.zeros(A.shape[0])
            return 1.0 - np.sum(A * np.asarray(A_prev, np.float64), axis=1)
        if kind == "kl_swapped" and scorer == scorers_mod.SCORER_KL and A_prev is not None:
            return real(A_prev, A, scorer)
        return real(A, A_prev, scorer)
    return f


@pytest.mark.parametrize("kind", ["entropy_sign", "entropy_log2", "cosine_unnormalised",
                                  "kl_swapped"])
def test_scorer_pins_catch(monkeypatch, kind):
    monkeypatch.setattr(scorer_pins, "drift_score", _score_mutant(kind))
    assert _some_pin_fails(SCORER_PINS)


def test_scorer_pins_pass_on_the_oracle():
    assert not _some_pin_fails(SCORER_PINS)


# ---- the hot path's oracle functions
import oracle                                         # noqa: E402
from tests import test_oracle_commit as commit_pins    # noqa: E402
from tests import test_oracle_offload as offload_pins  # noqa: E402
from tests import test_oracle_proxy_kl as proxy_pins   # noqa: E402
from tests import test_oracle_refresh as refresh_pins  # noqa: E402
from tests import test_oracle_topk as topk_pins        # noqa: E402


def _pins(mod):
    return [getattr(mod, n) for n in dir(mod) if n.startswith("test_")]


def _kl_swapped(A, A_prev):
    return oracle.kl_divergence_rows(A_prev, A)


def _proxy_unscaled(Q, Kt, Hq, Hkv, dh, A_prev=None):
    return oracle.proxy_attn_kl(np.asarray(Q, np.float64) * np.sqrt(dh), Kt, Hq, Hkv, dh, A_prev)


def _topk_by_sum(D, assign, counts, k):
    D = np.asarray(D, np.float64)
    n = np.asarray(counts)[np.asarray(assign)]
    return oracle.topk_drift((D * n).astype(np.float32), assign, counts, k)


def _commit_sign_flipped(logits, role, undecided, D_blk, d_sum, d_cnt, d_prev, suffix_sel, p):
    q = oracle.CommitParams(p.tau_s, p.alpha, p.ratio, {0: 1, 1: 0}.get(p.mode, p.mode),
                            p.ensure_progress)
    return oracle.commit_rule(logits, role, undecided, D_blk, d_sum, d_cnt, d_prev, suffix_sel, q)


def _commit_suffix_ignores_mask(logits, role, undecided, D_blk, d_sum, d_cnt, d_prev,
                                suffix_sel, p):
    sel = None if suffix_sel is None else np.ones_like(np.asarray(suffix_sel))
    return oracle.commit_rule(logits, role, undecided, D_blk, d_sum, d_cnt, d_prev, sel, p)


def _refresh_ignores_offset(H, pos, npos, Wk, Wv, Kcache, Vcache, cache_off, bf16_cache):
    return oracle.refresh_kv(H, pos, npos, Wk, Wv, Kcache, Vcache, 0, bf16_cache)


def _reconstruct_nibbles_swapped(code_row, scale_row, S, mu_c, rho_i):
    c = np.asarray(code_row, np.int64)
    return oracle.reconstruct_row(((c & 0xF) << 4) | (c >> 4), scale_row, S, mu_c, rho_i)


@pytest.mark.parametrize("mod,name,mutant", [
    (proxy_pins, "kl_divergence_rows", _kl_swapped),
    (proxy_pins, "proxy_attn_kl", _proxy_unscaled),
    (topk_pins, "topk_drift", _topk_by_sum),
    (commit_pins, "commit_rule", _commit_sign_flipped),
    (commit_pins, "commit_rule", _commit_suffix_ignores_mask),
    (refresh_pins, "refresh_kv", _refresh_ignores_offset),
    (offload_pins, "reconstruct_row", _reconstruct_nibbles_swapped),
])
def test_hot_path_pins_catch(monkeypatch, mod, name, mutant):
    monkeypatch.setattr(mod, name, mutant)
    assert _some_pin_fails(_pins(mod)), (mod.__name__, mutant.__name__)


# ---- k-means and NVFP4
from tests import test_oracle_kmeans as kmeans_pins   # noqa: E402
from tests import test_oracle_nvfp4 as nvfp4_pins     # noqa: E402

_E2M1_ALL = np.arange(16)


def _e2m1_toward_zero(x):
    """E2M1 rounding toward zero instead of to nearest-even."""
    x = np.asarray(x, np.float32)
    vals = oracle.e2m1_decode(_E2M1_ALL[:8]).astype(np.float64)       # 0 .. 6
    mag = np.minimum(np.abs(x.astype(np.float64)), 6.0)
    idx = np.searchsorted(vals, mag, side="right") - 1
    return (idx | np.where(np.signbit(x), 8, 0)).astype(np.int64)


def _residual_one_rounding(H, mu, assign, rho):
    """r = fl(h - rho mu) with the product kept in fp64 (one rounding)."""
    if mu is None:
        return oracle.nvfp4_residual(H, mu, assign, rho)
    H = np.asarray(H, np.float64)
    t = np.asarray(rho, np.float64)[:, None] * np.asarray(mu, np.float64)[np.asarray(assign)]
    R = (H - t).astype(np.float32)
    codes, scales, S = oracle.nvfp4_quantize(R)
    return codes, scales, S, R


def _kmeans_ties_high(H, mu0, iters, chat_in=None):
    """Ties to the higher cluster index: the oracle run on reversed centroids."""
    C = np.asarray(mu0).shape[0]
    rev = np.asarray(mu0)[::-1]
    o = oracle.kmeans_spherical(H, rev, iters, None if chat_in is None else chat_in[::-1])
    o = dict(o)
    o["assign"] = C - 1 - np.asarray(o["assign"])
    for k in ("mu", "chat", "counts"):
        o[k] = np.asarray(o[k])[::-1]
    return o


def _kmeanspp_first_pick_up(H, C, u, return_margin=False):
    """The first centre one row later (ceil instead of floor)."""
    u = np.array(u, np.float64)
    u[0] = min(u[0] + 1.0 / np.asarray(H).shape[0], 1 - 1e-12)
    return oracle.kmeanspp_init(H, C, u, return_margin)


@pytest.mark.parametrize("mod,name,mutant", [
    (nvfp4_pins, "e2m1_encode", _e2m1_toward_zero),
    (nvfp4_pins, "nvfp4_residual", _residual_one_rounding),
    (kmeans_pins, "kmeans_spherical", _kmeans_ties_high),
    (kmeans_pins, "kmeanspp_init", _kmeanspp_first_pick_up),
])
def test_kmeans_and_nvfp4_pins_catch(monkeypatch, mod, name, mutant):
    monkeypatch.setattr(mod, name, mutant)
    assert _some_pin_fails(_pins(mod)), (mod.__name__, mutant.__name__)
