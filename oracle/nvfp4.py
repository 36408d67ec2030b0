"""NVFP4 quantisation of the k-means residuals (oracle).

[Polestar §2.A, local window & clustering]: the residuals of the clustered
hidden states are quantised with NVFP4 to give compact proxy representations.
The page names the format only.  NVFP4 is taken as: E2M1 element codes, one
E4M3 scale per block of 16 consecutive elements, one fp32 scale per tensor,
round-to-nearest-even with saturation to the largest finite value.  The two
element formats follow their bit-level definitions in the OCP Microscaling
Formats (MX) specification v1.0:

* E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit; magnitudes
  {0, 0.5, 1, 1.5, 2, 3, 4, 6}; no inf/NaN.
* E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; subnormals
  m * 2^-9; largest finite 448 (0x7E); 0x7F is NaN.

This stage is defined in fp32 so its integer outputs are exact.  Readings
taken where the page is silent:
* the residual is the part of h orthogonal-ish to its centroid,
  r = h - rho * mu_a, computed as two IEEE fp32 operations
  t = fl(rho * mu_a), r = fl(h - t)  (no fused multiply-add);
* tensor scale S = max(fl(amax / 2688), FLT_MIN) for 0 < amax < inf, else 1,
  with amax the largest |r| of the batch element and 2688 = 6 * 448;
* block scale code = E4M3(fl(amax_blk / fl(6 * S))), its value s_b;
* element code = E2M1(fl(r / fl(s_b * S))), or 0 for the whole block when
  s_b = 0;
* a negative value that rounds to zero keeps its sign (code 0x8 / 0x80);
* packing: byte j of a row holds element 2j in its low nibble and element
  2j + 1 in its high nibble.
"""

import numpy as np

_F32 = np.float32
FLT_MIN = float(np.finfo(np.float32).tiny)


def e2m1_decode(code):
    code = np.asarray(code, dtype=np.int64)
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return np.where(s == 1, -mag, mag)


def e4m3_decode(code):
    code = np.asarray(code, dtype=np.int64)
    s = (code >> 7) & 1
    e = (code >> 3) & 15
    m = code & 7
    mag = np.where(e == 0, np.ldexp(m.astype(np.float64), -9),
                   np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def _rne_encode(x, table, sign_shift):
    """Round |x| to the nearest entry of `table` (the non-negative finite
    values in code order), ties to the even code, saturating above the last
    entry; then put the sign of x (IEEE signbit, so -0 keeps it) on top."""
    x = np.asarray(x, dtype=np.float32)
    mag = np.abs(x.astype(np.float64))
    top = len(table) - 1
    hi = np.clip(np.searchsorted(table, mag, side="left"), 0, top)
    lo = np.clip(hi - 1, 0, top)
    d_lo = mag - table[lo]
    d_hi = table[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(mag >= table[top], top, code)        # saturate (incl. inf)
    code = np.where(mag == 0, 0, code)
    return code.astype(np.int64) | (np.signbit(x).astype(np.int64) << sign_shift)


_E2M1_TABLE = e2m1_decode(np.arange(8))          # 0, .5, 1, 1.5, 2, 3, 4, 6
_E4M3_TABLE = e4m3_decode(np.arange(127))        # 0 .. 448 (0x00..0x7E)


def e2m1_encode(x):
    """fp32 -> E2M1 code (0..15), round-to-nearest-even, saturating."""
    return _rne_encode(x, _E2M1_TABLE, 3)


def e4m3_encode(x):
    """fp32 -> E4M3 code (0..255), round-to-nearest-even, saturating to 448;
    NaN -> 0x7F with its sign."""
    x = np.asarray(x, dtype=np.float32)
    code = _rne_encode(x, _E4M3_TABLE, 7)
    return np.where(np.isnan(x), 0x7F | (np.signbit(x).astype(np.int64) << 7),
                    code)


def nvfp4_quantize(R):
    """Quantise one batch element's fp32 residuals R [N][d] (d % 16 == 0).

    Returns (codes [N][d/2] uint8, scales [N][d/16] uint8, S float32)."""
    R = np.asarray(R, dtype=np.float32)
    N, d = R.shape
    amax = _F32(np.max(np.abs(R))) if R.size else _F32(0)
    if amax > 0 and np.isfinite(amax):
        S = max(_F32(amax / _F32(2688.0)), _F32(FLT_MIN))
    else:
        S = _F32(1.0)
    S = _F32(S)
    blocks = R.reshape(N, d // 16, 16)
    amax_blk = np.max(np.abs(blocks), axis=2)                  # fp32, exact
    six_s = _F32(_F32(6.0) * S)
    sbf = (amax_blk / six_s).astype(np.float32)                # one rounding
    scode = e4m3_encode(sbf)
    sb = e4m3_decode(scode).astype(np.float32)                 # exact
    den = (sb * S).astype(np.float32)                          # one rounding
    q = np.zeros((N, d // 16, 16), dtype=np.int64)
    live = sb != 0
    if live.any():
        ratio = (blocks[live] / den[live][:, None]).astype(np.float32)
        q[live] = e2m1_encode(ratio)
    q = q.reshape(N, d)
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return codes, scode.astype(np.uint8), S


def nvfp4_residual(H, mu, assign, rho):
    """Residual of one window against its centroids, then NVFP4.

    H [N][d] (fp32, or bf16 values widened to fp32), mu [C][d] fp32,
    assign [N], rho [N] fp32.  mu=None quantises H itself.
    Returns (codes, scales, S, R) with R the fp32 residual."""
    H = np.asarray(H, dtype=np.float32)
    if mu is None:
        R = H.copy()
    else:
        mu = np.asarray(mu, dtype=np.float32)
        rho = np.asarray(rho, dtype=np.float32)
        t = (rho[:, None] * mu[np.asarray(assign)]).astype(np.float32)
        R = (H - t).astype(np.float32)
    codes, scales, S = nvfp4_quantize(R)
    return codes, scales, S, R
