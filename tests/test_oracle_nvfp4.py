"""Pins of the oracle's NVFP4 stage against the format definitions."""
import json
import os

import numpy as np

from oracle import (e2m1_decode, e2m1_encode, e4m3_decode, e4m3_encode,
                    nvfp4_quantize, nvfp4_residual)

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                   "nvfp4_formats.json")))


def test_decode_tables_match_format_definitions():
    for code, val in GOLD["e2m1_decode"].items():
        got = float(e2m1_decode(int(code)))
        assert got == val and np.signbit(got) == np.signbit(val), code
    for code, val in GOLD["e4m3_decode"].items():
        got = float(e4m3_decode(int(code)))
        assert got == val and np.signbit(got) == np.signbit(val), code
    assert np.isnan(e4m3_decode(0x7F)) and np.isnan(e4m3_decode(0xFF))


def test_hand_worked_rounding_cases():
    for x, code in GOLD["e2m1_round"]:
        assert int(e2m1_encode(np.float32(x))) == code, (x, code)
    for x, code in GOLD["e4m3_round"]:
        assert int(e4m3_encode(np.float32(x))) == code, (x, code)


def test_decode_then_encode_is_identity():
    c = np.arange(16)
    assert np.array_equal(e2m1_encode(e2m1_decode(c).astype(np.float32)), c)
    c = np.array([i for i in range(256) if (i & 0x7F) != 0x7F])
    assert np.array_equal(e4m3_encode(e4m3_decode(c).astype(np.float32)), c)


def _nearest_brute(x, table):
    """Nearest representable by exhaustive distance scan (ties -> even)."""
    best = None
    for code, v in enumerate(table):
        dist = abs(x - v)
        if best is None or dist < best[0] or (dist == best[0] and code % 2 == 0):
            best = (dist, code)
    return best[1]


def test_encode_matches_exhaustive_scan_on_dense_grid():
    t2 = [float(v) for v in e2m1_decode(np.arange(8))]
    t4 = [float(v) for v in e4m3_decode(np.arange(127))]
    rng = np.random.default_rng(3)
    xs = np.concatenate([np.linspace(0, 6, 2401), rng.uniform(0, 6, 500)])
    for x in xs.astype(np.float32):
        assert int(e2m1_encode(x)) == _nearest_brute(float(x), t2)
    xs4 = np.concatenate([np.ldexp(rng.uniform(1, 2, 400), rng.integers(-12, 9, 400)),
                          np.linspace(0, 448, 1793)])
    for x in xs4.astype(np.float32):
        assert int(e4m3_encode(x)) == _nearest_brute(float(x), t4)


def test_quantize_round_trips_representable_tensor():
    rng = np.random.default_rng(7)
    N, d = 5, 64
    S = np.float32(0.125)
    sb_codes = rng.integers(0x20, 0x7E, size=(N, d // 16))
    sb_codes[0, 0] = 0x7E                      # amax = 6 * 448 * S = 2688 S
    sb = e4m3_decode(sb_codes).astype(np.float32)
    q = rng.integers(0, 16, size=(N, d // 16, 16))
    q[:, :, 3] = 7                             # a +-6 element in every block
    vals = (e2m1_decode(q) * sb[:, :, None] * S).astype(np.float32)
    codes, scales, S_got = nvfp4_quantize(vals.reshape(N, d))
    assert S_got == S
    assert np.array_equal(scales, sb_codes.astype(np.uint8))
    qq = q.reshape(N, d)
    qq = np.where(qq == 8, 0, qq)              # -0 never comes from a value
    want = (qq[:, 0::2] | (qq[:, 1::2] << 4)).astype(np.uint8)
    got = codes.astype(np.int64)
    got_lo = np.where((got & 0xF) == 8, 0, got & 0xF)
    got_hi = np.where((got >> 4) == 8, 0, got >> 4)
    assert np.array_equal(got_lo | (got_hi << 4), want)


def test_zero_tensor():
    codes, scales, S = nvfp4_quantize(np.zeros((3, 32), np.float32))
    assert S == 1.0 and not codes.any() and not scales.any()


def test_error_bound_and_packing():
    rng = np.random.default_rng(11)
    R = rng.standard_normal((8, 128)).astype(np.float32)
    codes, scales, S = nvfp4_quantize(R)
    assert S == np.float32(np.abs(R).max() / np.float32(2688))
    q = np.empty((8, 128), np.int64)
    q[:, 0::2] = codes & 0xF
    q[:, 1::2] = codes >> 4
    deq = e2m1_decode(q) * np.repeat(e4m3_decode(scales), 16, axis=1) * S
    # within half an E2M1 step of the block grid, which is at most 1 (of 6)
    step = np.repeat(e4m3_decode(scales), 16, axis=1) * S
    assert np.all(np.abs(deq - R) <= step * 1.0 + 1e-30)
    assert np.all(np.sign(deq[deq != 0]) == np.sign(R[deq != 0]))


def test_residual_is_two_fp32_roundings():
    H = np.array([[1.0, 2.0, 3.0, 4.0] * 4], np.float32)
    mu = np.array([[0.5] * 16], np.float32)
    rho = np.array([np.float32(1) / np.float32(3)], np.float32)
    _, _, _, R = nvfp4_residual(H, mu, np.array([0]), rho)
    t = np.float32(np.float32(1 / 3) * np.float32(0.5))
    assert np.array_equal(R[0], (H[0] - t).astype(np.float32))
    # a product that fp32 must round: fl(fl(1/3) * fl(1.3)) = 0.43333333730697632, the exact
    # product 0.43333333035310060; IEEE fp32 subtraction of the rounded product gives the
    # values below, which a single rounding of h - rho mu would miss (0.0666666701436042...)
    H2 = np.array([[0.5, 2.0] * 8], np.float32)
    _, _, _, R2 = nvfp4_residual(H2, np.array([[1.3] * 16], np.float32), np.array([0]), rho)
    assert R2[0, 0] == np.float32(0.06666666269302368)
    assert R2[0, 1] == np.float32(1.566666603088379)
    _, _, _, R0 = nvfp4_residual(H, None, None, None)
    assert np.array_equal(R0, H)
