"""MXFP4 quantization and its exact three-way error decomposition
(test infrastructure only).

Source: "Decomposing MXFP4 quantization error ..." (arXiv 2605.20402v2),
abstract.  MXFP4 block scales are powers of two; the quantization error is
proved to split exactly into three additive components: scale bias (from
rounding the scale to a power of two), deadzone truncation (small values
zeroed) and grid noise (rounding to the nearest 4-bit grid point).  The
abstract gives names and exactness but no formulas.

Readings:

* Format (OCP MX): 32-element blocks along K, E2M1 elements, one E8M0
  scale 2**e per block with e = floor(log2 a) - 2 (a = max |x|, 2 = the
  exponent of E2M1's largest power of two), clamped to [-127, 127]; a == 0
  gives e = -127.  code_i = E2M1(x_i * 2**-e) (fp32 multiply, RNE,
  satfinite so 6 < |y| < 8 saturates to 6, sign kept).  Scale byte = e + 127.
* Decomposition, telescoping through the ideal real scale s* = a / 6 (the
  scale that puts the block maximum exactly on the grid's top level):
      Q_s(x)  = 2**e * E2M1(x / 2**e)         (what MXFP4 stores)
      Q*(x)   = s*   * E2M1(x / s*)           (same grid, ideal scale)
      E = Q_s - x                              total error
      B = Q_s - Q*                             scale bias
      D = (Q* - x) where E2M1(x / s*) == 0     deadzone truncation
      G = (Q* - x) where E2M1(x / s*) != 0     grid noise
  so E = B + D + G exactly.  s* and x / s* are computed in fp32 (the
  precision of the kernel) so both sides take the same rounding decisions;
  the four components are then formed in fp64, where they are exact.
  A block with a == 0 has every component 0.
* Per-block statistics: [|B|^2, |D|^2, |G|^2, |E|^2] summed over the block,
  and the deadzone count = #{i : E2M1(x_i / s*) == 0 and x_i != 0}.

Corrections.  The abstract names "macro-block scaling" (reduces the scale
bias) and "Outlier Fallback" (recovers deadzone entries and partly reduces
the scale-bias error) without defining either; the readings below are the
plainest that fit those effects and a W4A4 GEMM:

* Macro-block = one row of the operand (all K/32 blocks of a token, or of a
  weight row): the largest group over which a GEMM can apply a
  non-power-of-two factor exactly, outside its sum over K.  Its scale is
  the mantissa of the row's ideal scale: t = RN(A / 6) (A = max |x| over the
  row), m = t / 2^floor(log2 t) in [1, 2) (m = 1 when t == 0 or t < 2^-126).
  The row is multiplied by rho = RN(1 / m) (fp32, RN) and MXFP4-quantized
  as above; its values are m * 2^e * E2M1(code).  The block holding the row
  maximum then sits on the grid's top level (scale bias ~ 0 there).
* Outlier Fallback = a channel set S (the outlier channels, chosen offline
  like the compensation channels) leaves the MXFP4 operand: x[:, S] is set
  to 0 before the row scale, the block scales and the codes, so the blocks
  that held outliers take smaller scales (their small entries leave the
  deadzone, their scale bias shrinks), and the fallback values
  bf16(RN(x[:, S] * rho)) are multiplied in BF16.  Both GEMM operands
  take the same S.
* Corrected GEMM: Y = m_a m_b^T * (deq(q(X'')) . deq(q(W''))^T + F_a . F_b^T),
  F the fallback values; the decomposition statistics of a corrected row are
  those of its scaled operand X'' = RN(X' * rho) (units of m^2).
"""

import numpy as np

from .formats import bf16_round, e2m1_encode, e2m1_value
from .nvfp4 import pack

BLOCK = 32


def block_exponent(a):
    """e = floor(log2 a) - 2 clamped to [-127, 127]; a == 0 -> -127.
    floor(log2 a) is read exactly from frexp (a = m * 2**q, 0.5 <= m < 1)."""
    a = np.asarray(a, dtype=np.float64)
    _, q = np.frexp(a)
    e = np.where(a > 0, q - 1 - 2, -127)
    return np.clip(e, -127, 127).astype(np.int64)


def quantize(x):
    """MXFP4-quantize float32 values of bf16 numbers ``x`` [M, K], K % 32 == 0.

    Returns dict(codes [M,K] uint8, packed [M,K/2], scale [M,K/32] uint8 E8M0,
    e [M,K/32] int64).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    xb = x.reshape(M, K // BLOCK, BLOCK)
    a = np.max(np.abs(xb), axis=2)
    e = block_exponent(a)
    inv = np.power(2.0, -e).astype(np.float32)          # exact power of two
    y = (xb * inv[:, :, None]).astype(np.float32)
    codes = e2m1_encode(y).reshape(M, K)
    return dict(codes=codes, packed=pack(codes), scale=(e + 127).astype(np.uint8), e=e)


def dequantize(codes, scale):
    M, K = codes.shape
    v = e2m1_value(codes).reshape(M, K // BLOCK, BLOCK)
    return (v * np.power(2.0, scale.astype(np.float64) - 127.0)[:, :, None]).reshape(M, K)


def decompose(x):
    """Elementwise decomposition of the MXFP4 error of ``x`` [M, K].

    Returns dict(E, B, D, G) as float64 [M, K], ``dead`` bool [M, K] (the
    deadzone mask) and the quantize() outputs."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    q = quantize(x)
    xb = x.reshape(M, K // BLOCK, BLOCK)
    a = np.max(np.abs(xb), axis=2)
    Qs = dequantize(q["codes"], q["scale"]).reshape(M, K // BLOCK, BLOCK)
    nz = a > 0
    s_star = np.where(nz, a / np.float32(6.0), np.float32(1.0)).astype(np.float32)
    y_star = (xb / s_star[:, :, None]).astype(np.float32)
    c_star = e2m1_encode(y_star)
    Qstar = e2m1_value(c_star) * s_star.astype(np.float64)[:, :, None]
    x64 = xb.astype(np.float64)
    dead = ((c_star & 0x7) == 0)
    E = Qs - x64
    B = Qs - Qstar
    D = np.where(dead, Qstar - x64, 0.0)
    G = np.where(dead, 0.0, Qstar - x64)
    zero_blk = ~nz[:, :, None]
    B = np.where(zero_blk, 0.0, B)
    D = np.where(zero_blk, 0.0, D)
    G = np.where(zero_blk, 0.0, G)
    E = np.where(zero_blk, 0.0, E)
    deadzone = dead & (x64 != 0) & ~zero_blk
    r = lambda t: t.reshape(M, K)
    return dict(E=r(E), B=r(B), D=r(D), G=r(G), dead=r(deadzone), **q)


def block_stats(x):
    """Per-block statistics [M, K/32, 4] = (|B|^2, |D|^2, |G|^2, |E|^2) in
    fp64 and the deadzone count [M, K/32] (uint8)."""
    d = decompose(x)
    M, K = d["E"].shape
    sq = lambda t: np.sum(t.reshape(M, K // BLOCK, BLOCK) ** 2, axis=2)
    stats = np.stack([sq(d["B"]), sq(d["D"]), sq(d["G"]), sq(d["E"])], axis=-1)
    cnt = np.sum(d["dead"].reshape(M, K // BLOCK, BLOCK), axis=2).astype(np.uint8)
    return stats, cnt, d


def macro_scale(x):
    """Row macro-block scales m [M] (float32, in [1, 2)) of ``x`` [M, K]:
    the mantissa of t = RN(max|x_row| / 6); 1 where t == 0 or t < 2^-126."""
    x = np.asarray(x, dtype=np.float32)
    A = np.max(np.abs(x), axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    t = (A / np.float32(6.0)).astype(np.float32)
    mant, q = np.frexp(t.astype(np.float64))      # t = mant * 2^q, mant in [0.5, 1)
    m = (mant * 2.0).astype(np.float32)           # exact: t / 2^(q - 1)
    return np.where(t >= np.float32(2.0 ** -126), m, np.float32(1.0)).astype(np.float32)


def quantize_corrected(x, macro=False, fallback=None):
    """MXFP4 with the corrections of the readings above, ``x`` [M, K] float32
    values of bf16 numbers.  macro: row macro-block scales; fallback: sorted
    channel indices S leaving the FP4 operand.

    Returns quantize() of the scaled operand xs = RN(x' * rho) (x' = x with
    S zeroed) plus m [M], rho [M] (float32), xs, fb [M, k] (float32 values of
    bf16(RN(x[:, S] * rho))), stats [M, K/32, 4], dead [M, K/32]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    x0 = x.copy()
    S = np.zeros(0, np.int64) if fallback is None else np.asarray(fallback, dtype=np.int64)
    x0[:, S] = 0.0
    m = macro_scale(x0) if macro else np.ones(M, np.float32)
    rho = (np.float32(1.0) / m).astype(np.float32)
    xs = (x0 * rho[:, None]).astype(np.float32)
    q = quantize(xs)
    fb = bf16_round((x[:, S] * rho[:, None]).astype(np.float32))
    stats, dead, _ = block_stats(xs)
    return dict(q, m=m, rho=rho, xs=xs, fb=fb, stats=stats, dead=dead)


def gemm_corrected(qa, qb):
    """Y = m_a m_b^T * (deq(qa) . deq(qb)^T + fb_a . fb_b^T) in fp64 for two
    quantize_corrected() results (W^T for qb), the same channel set S."""
    a = dequantize(qa["codes"], qa["scale"])
    b = dequantize(qb["codes"], qb["scale"])
    y = a @ b.T
    if qa["fb"].shape[1]:
        y = y + np.asarray(qa["fb"], np.float64) @ np.asarray(qb["fb"], np.float64).T
    return y * (np.asarray(qa["m"], np.float64)[:, None] * np.asarray(qb["m"], np.float64)[None, :])
