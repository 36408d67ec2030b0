"""Pins of the offload oracle (store layout and reconstruction) against
brute force, hand-known values and the NVFP4 error bound."""
import numpy as np

import oracle
from oracle.offload import fetch_reconstruct, pack_clusters, reconstruct_row, record_bytes


def _quantised(N, d, C, seed):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, d)).astype(np.float32)
    mu = oracle.normalize_rows(rng.standard_normal((C, d))).astype(np.float32)
    assign = rng.integers(0, C, N)
    rho = np.sum(H * mu[assign], axis=1).astype(np.float32)
    codes, scales, S, _ = oracle.nvfp4_residual(H, mu, assign, rho)
    return H, mu, assign, rho, codes, scales, S


def test_record_bytes():
    assert record_bytes(64) == 32 + 16          # 32 code bytes, 4 scale bytes -> 16
    assert record_bytes(4096) == 2048 + 256
    assert record_bytes(3584) == 1792 + 224


def test_pack_layout_brute_force():
    N, d, C = 37, 64, 5
    _, _, assign, _, codes, scales, _ = _quantised(N, d, C, 1)
    store, order, cl_off = pack_clusters(codes, scales, assign, C)
    assert sorted(order.tolist()) == list(range(N))          # every row once
    assert cl_off[0] == 0 and cl_off[-1] == N
    assert np.array_equal(np.diff(cl_off), np.bincount(assign, minlength=C))
    for c in range(C):
        rows = order[cl_off[c]:cl_off[c + 1]]
        assert np.all(assign[rows] == c) and np.all(np.diff(rows) > 0)
    for r, i in enumerate(order):
        assert np.array_equal(store[r, :32], codes[i])
        assert np.array_equal(store[r, 32:36], scales[i])
        assert not store[r, 36:].any()                       # zero padding


def test_reconstruct_hand_values():
    # S = 1, block scale E4M3 1.0 (0x38): every code decodes to its E2M1 value
    vals = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    nib = np.array([k for k in range(8)] * 2 + [8 + k for k in range(8)] * 2)   # d = 32
    code_row = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    scale_row = np.array([0x38, 0x38], np.uint8)
    want = np.array(vals * 2 + [-v for v in vals] * 2, np.float32)
    got = reconstruct_row(code_row, scale_row, 1.0, np.zeros(32, np.float32), 0.0)
    assert np.array_equal(got, want)
    # the centroid component is added: rho 2, mu 0.25 -> t = 0.5
    got = reconstruct_row(code_row, scale_row, 1.0, np.full(32, 0.25, np.float32), 2.0)
    assert np.array_equal(got, (want + np.float32(0.5)).astype(np.float32))
    # block scale 2.0 (0x40) and S = 0.5 give g = 1 for block 0, E4M3 0.5 (0x30) for block 1
    got = reconstruct_row(code_row, np.array([0x40, 0x30], np.uint8), 0.5,
                          np.zeros(32, np.float32), 0.0)
    assert np.array_equal(got[:16], want[:16]) and np.array_equal(got[16:], want[16:] * 0.25)


def test_zero_residual_reconstructs_the_centroid_component():
    rng = np.random.default_rng(2)
    d, C = 64, 3
    mu = oracle.normalize_rows(rng.standard_normal((C, d))).astype(np.float32)
    assign = np.array([0, 2, 1, 2])
    rho = np.array([1.5, -0.25, 3.0, 0.75], np.float32)
    H = (rho[:, None] * mu[assign]).astype(np.float32)          # r = 0 exactly
    codes, scales, S, _ = oracle.nvfp4_residual(H, mu, assign, rho)
    for i in range(4):
        got = reconstruct_row(codes[i], scales[i], S, mu[assign[i]], rho[i])
        assert np.array_equal(got, H[i])


def test_round_trip_within_the_nvfp4_bound():
    """|h - h~| <= g + rounding for every element, g = s_b S the block's step
    factor: the E2M1 grid's widest gap is 2 (4 to 6) and the scale's rounding
    can push a block maximum at most 6.4 g before saturation."""
    N, d, C = 24, 128, 4
    H, mu, assign, rho, codes, scales, S = _quantised(N, d, C, 3)
    s = oracle.e4m3_decode(scales.astype(np.int64)).astype(np.float32)
    for i in range(N):
        h_t = reconstruct_row(codes[i], scales[i], S, mu[assign[i]], rho[i])
        g = np.repeat((s[i] * np.float32(S)).astype(np.float32), 16).astype(np.float64)
        err = np.abs(H[i].astype(np.float64) - h_t)
        assert np.all(err <= 1.0001 * g + 1e-6 * np.abs(H[i]) + 1e-30)


def test_fetch_returns_exactly_the_selected_members():
    N, d, C = 40, 64, 6
    _, mu, assign, rho, codes, scales, S = _quantised(N, d, C, 4)
    store, order, cl_off = pack_clusters(codes, scales, assign, C)
    sel = np.array([4, -1, 1])
    got = fetch_reconstruct(store, order, cl_off, sel, mu, rho, S, d)
    assert set(got) == {i for i in range(N) if assign[i] in (4, 1)}
    for i, row in got.items():
        assert np.array_equal(row, reconstruct_row(codes[i], scales[i], S, mu[assign[i]],
                                                   rho[i]))
