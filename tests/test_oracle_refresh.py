"""Pins of the oracle's sparse K/V refresh."""
import json
import os

import numpy as np
import torch

from oracle import bf16_round, refresh_kv

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                   "nvfp4_formats.json")))


def test_bf16_rounding_cases_and_library():
    for x, want in GOLD["bf16_round"]:
        assert float(bf16_round(np.float32(x))) == want
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(10000) * 10.0 ** rng.integers(-10, 10, 10000)).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(bf16_round(x), lib)


def _setup(seed, N=12, d=16, n=8, ncache=20):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, d))
    Wk = rng.standard_normal((d, n)) * 0.1
    Wv = rng.standard_normal((d, n)) * 0.1
    Kc = rng.standard_normal((ncache, n)).astype(np.float32)
    Vc = rng.standard_normal((ncache, n)).astype(np.float32)
    return H, Wk, Wv, Kc, Vc


def test_selected_rows_equal_dense_recompute_others_untouched():
    H, Wk, Wv, Kc, Vc = _setup(1)
    pos = np.array([1, 4, 5, 11] + [-1] * 8)
    K2, V2 = refresh_kv(H, pos, 4, Wk, Wv, Kc, Vc, cache_off=3, bf16_cache=False)
    dense_k = (H @ Wk).astype(np.float32)
    dense_v = (H @ Wv).astype(np.float32)
    for p in range(12):
        r = 3 + p
        if p in (1, 4, 5, 11):
            assert np.array_equal(K2[r], dense_k[p]) and np.array_equal(V2[r], dense_v[p])
        else:
            assert np.array_equal(K2[r], Kc[r]) and np.array_equal(V2[r], Vc[r])
    for r in (0, 1, 2, 15, 16, 17, 18, 19):
        assert np.array_equal(K2[r], Kc[r])


def test_all_rows_is_the_textbook_gemm_and_empty_is_identity():
    H, Wk, Wv, Kc, Vc = _setup(2, ncache=12)
    K2, V2 = refresh_kv(H, np.arange(12), 12, Wk, Wv, Kc, Vc, 0, bf16_cache=True)
    assert np.array_equal(K2, bf16_round(H @ Wk))
    assert np.array_equal(V2, bf16_round(H @ Wv))
    K3, V3 = refresh_kv(H, np.full(12, -1), 0, Wk, Wv, Kc, Vc, 0, bf16_cache=True)
    assert np.array_equal(K3, Kc) and np.array_equal(V3, Vc)
