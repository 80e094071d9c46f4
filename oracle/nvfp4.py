"""NVFP4 quantization, dequantization and the compensation residual slice
(test infrastructure only).

Sources.  QUADS abstract (arXiv 2607.15810): NVFP4 is fine-grained block
scaling over E2M1 elements, and rollout activations are quantized online.
gist.science explainer of QUADS, Technisches Resuemee section 2.2 B: the
compensation term is the activation's quantization residual (Delta X_q) on a
set of high-error channels.  FourSight abstract (arXiv 2611.04887): those
channels are kept in BF16.

Readings (the pages name NVFP4 but do not define its arithmetic):

* 16-element blocks along K, one unsigned E4M3 block scale each, under one
  FP32 tensor scale g.
* Dynamic tensor scale: g = amax(|X|) / 2688 in fp32 (2688 = 6 * 448, the
  largest E2M1 magnitude times the largest E4M3 value); g = 1 when X is all
  zero.
* Block scale: sigma = E4M3(( a / 6 ) / g), a = max |x| over the block, two
  fp32 divisions in that order, RNE, saturating at 448.
* Block decode scale d = fp32(sigma) * g (fp32 multiply).  If d == 0 every
  code of the block is +0.  Otherwise r = 1 / d (fp32 division) and
  code_i = E2M1(x_i * r) (fp32 multiply, RNE, satfinite, sign kept).
* Dequantized value used by the residual: deq_i = fp32(E2M1(code_i) * d);
  residual R_i = x_i - deq_i in fp32; the emitted slice is bf16(R_i) on the
  channel set S.  The exact value of the quantized representation (used by
  the reference GEMM) is E2M1(code) * sigma * g in fp64.
* Pre-scaled residual (an operand form for the GEMM, not a different
  method): the fp32 residual R_i times fp32(1 / g) (the correctly rounded
  reciprocal of the tensor scale, fp32 multiply), rounded once to bf16.  The
  GEMM multiplies the compensation product by g again, so R_S . W_S is
  unchanged up to that rounding.
* Quantized residual (the explainer's "second-pass quantization" of the
  high-residual channels, section 2.2 B; the spec's residual stays BF16):
  the pre-scaled fp32 residual R_i * fp32(1 / g) rounded once to FP8 E4M3
  (RNE, satfinite, sign kept).  |R_i / g| is at most about the block's E4M3
  scale, so the value lands in E4M3's range without a scale of its own.  The
  matching weight rows are E4M3(E2M1(code) * sigma * 2^-3): the largest
  product 6 * 448 = 2688 times 2^-3 is 336 <= 448; the GEMM multiplies the
  FP8 product by 2^3 again.
* Trainer-side fake quantization (QDQ, asymmetric W4A16 QAT): the same
  codes and scales, and per element bf16_rn(deq_i), deq_i as above (the
  fp32 product rounded once more to bf16, the trainer's weight dtype).
* Packing: two codes per byte, byte j = code[2j] | code[2j+1] << 4.
* Block-scale storage for the GEMM: 128-row x 4-scale tiles of 512 bytes,
  byte offset inside a tile = (r % 32) * 16 + ((r % 128) // 32) * 4 + (s % 4)
  for row r and scale index s; tiles ordered by (row tile, scale-column tile).
  This is the tile the block-scaled tensor-core MMA reads; the oracle keeps
  row-major scales and maps them through :func:`scale_tile_offsets`.
"""

import numpy as np

from .formats import (bf16_round, e2m1_encode, e2m1_value, e4m3_decode,
                      e4m3_encode, e4m3_encode_signed)

BLOCK = 16
AMAX_TO_G = np.float32(2688.0)  # 6 * 448
_CHUNK_ROWS = 512


def tensor_scale(x):
    """Dynamic FP32 tensor decode scale g = amax|x| / 2688 (1 if all zero)."""
    amax = np.float32(np.max(np.abs(np.asarray(x, dtype=np.float32)))) if np.size(x) else np.float32(0)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax / AMAX_TO_G)


def _quantize_rows(x, g):
    """Quantize float32 rows [R, K] (K % 16 == 0) with tensor scale g.

    Returns (codes [R,K] uint8 unpacked, sigma [R,K/16] uint8, resid_f32 [R,K]).
    """
    R, K = x.shape
    xb = x.reshape(R, K // BLOCK, BLOCK)
    a = np.max(np.abs(xb), axis=2)                             # exact
    t = (a / np.float32(6.0)) / g                              # two fp32 divisions
    sigma = e4m3_encode(t.astype(np.float64))                  # RNE, satfinite
    d = (e4m3_decode(sigma).astype(np.float32) * g).astype(np.float32)
    nz = d != 0
    r = np.where(nz, np.float32(1.0) / np.where(nz, d, np.float32(1.0)), np.float32(0.0)).astype(np.float32)
    y = (xb * r[:, :, None]).astype(np.float32)
    codes = e2m1_encode(y)
    codes = np.where(nz[:, :, None], codes, np.uint8(0)).astype(np.uint8)
    deq = (e2m1_value(codes).astype(np.float32) * d[:, :, None]).astype(np.float32)
    resid = (xb - deq).astype(np.float32)
    return codes.reshape(R, K), sigma, resid.reshape(R, K)


def quantize(x, g=None, chan=None):
    """NVFP4-quantize activations (or W^T) ``x`` [M, K] given as float32
    values of bf16 numbers.

    g: FP32 tensor scale; None -> dynamic (:func:`tensor_scale`).
    chan: sorted int channel indices S (len k) for the residual slice, or None.

    Returns a dict with
      codes   [M, K]    uint8  unpacked E2M1 codes
      packed  [M, K/2]  uint8  two codes per byte, low nibble = even k
      sigma   [M, K/16] uint8  E4M3 block scales (row-major)
      g       float32          tensor scale used
      resid_f32 [M, K]  float32 residual x - deq (before bf16 rounding)
      resid   [M, k]    float32 bf16-rounded residual on S (if chan given)
      resid_scaled [M, k] float32 bf16(resid_f32 * fp32(1/g)) on S (if chan given)
      resid_fp8 [M, k]  uint8  E4M3 bytes of fp32(resid_f32 * fp32(1/g)) on S
                               (the quantized residual; if chan given)
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 16")
    g = tensor_scale(x) if g is None else np.float32(g)
    codes = np.empty((M, K), np.uint8)
    sigma = np.empty((M, K // BLOCK), np.uint8)
    resid_f32 = np.empty((M, K), np.float32)
    for r0 in range(0, M, _CHUNK_ROWS):
        r1 = min(M, r0 + _CHUNK_ROWS)
        c, s, rf = _quantize_rows(x[r0:r1], g)
        codes[r0:r1], sigma[r0:r1], resid_f32[r0:r1] = c, s, rf
    out = dict(codes=codes, packed=pack(codes), sigma=sigma, g=g, resid_f32=resid_f32)
    if chan is not None:
        chan = np.asarray(chan, dtype=np.int64)
        out["resid"] = bf16_round(resid_f32[:, chan])
        pre = (resid_f32[:, chan] * reciprocal(g)).astype(np.float32)
        out["resid_scaled"] = bf16_round(pre)
        out["resid_fp8"] = e4m3_encode_signed(pre)
    return out


def reciprocal(g):
    """fp32(1 / g): numpy's float32 division is the correctly rounded IEEE
    quotient."""
    return np.float32(np.float32(1.0) / np.float32(g))


def quantize_grouped(x, offsets, chan, g=None):
    """Quantize expert-sorted rows; row r of expert e (offsets[e] <= r <
    offsets[e+1]) takes its residual slice on that expert's channels chan[e].
    One tensor scale over all rows (reading: the routed activations are one
    tensor)."""
    out = quantize(x, g=g)
    offsets = np.asarray(offsets, dtype=np.int64)
    chan = np.asarray(chan, dtype=np.int64)
    M = x.shape[0]
    k = chan.shape[1]
    resid = np.zeros((M, k), np.float32)
    resid_scaled = np.zeros((M, k), np.float32)
    rg = reciprocal(out["g"])
    for e in range(len(offsets) - 1):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            rf = out["resid_f32"][lo:hi][:, chan[e]]
            resid[lo:hi] = bf16_round(rf)
            resid_scaled[lo:hi] = bf16_round((rf * rg).astype(np.float32))
    out["resid"] = resid
    out["resid_scaled"] = resid_scaled
    return out


def pack(codes):
    """Pack E2M1 codes [.., K] two per byte: low nibble = even index."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] & 0xF) | ((codes[..., 1::2] & 0xF) << 4)


def unpack(packed):
    """Inverse of :func:`pack`."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def qdq(x, g=None):
    """Trainer-side weight fake quantization (quantize, then dequantize) of
    ``x`` [M, K] (float32 values of bf16 numbers, K the reduction axis).

    Source: gist.science explainer of QUADS, Technisches Resuemee 2.2 A
    (asymmetric W4A16 QAT: the trainer fake-quantizes its weights to NVFP4 so
    its forward pass sees the discretized weights the rollout engine uses;
    activations stay BF16) and section 2.1 (the same quantize-dequantize path
    on both sides removes the weight-induced mismatch).

    Reading: the same quantization as :func:`quantize` (same g, sigma and
    codes), and the element value the residual is measured against,
    deq = fp32(E2M1(code) * d), delivered in the trainer's dtype:
    bf16_rn(deq).  Returns (w_qdq [M, K] float32 holding bf16 values, the
    :func:`quantize` dict).
    """
    q = quantize(x, g=g)
    M, K = q["codes"].shape
    d = (e4m3_decode(q["sigma"]).astype(np.float32) * np.float32(q["g"])).astype(np.float32)
    v = e2m1_value(q["codes"]).astype(np.float32).reshape(M, K // BLOCK, BLOCK)
    deq = (v * d[:, :, None]).astype(np.float32).reshape(M, K)
    return bf16_round(deq), q


def dequantize(codes, sigma, g):
    """Exact value of the quantized tensor in fp64: E2M1(code) * sigma * g."""
    M, K = codes.shape
    v = e2m1_value(codes).reshape(M, K // BLOCK, BLOCK)
    s = e4m3_decode(sigma)[:, :, None] * np.float64(np.float32(g))
    return (v * s).reshape(M, K)


# ------------------------------------------------------ scale-tile layout ----

def scale_rows_padded(M):
    return -(-M // 128) * 128


def scale_cols_padded(K):
    return -(-(K // BLOCK) // 4) * 4


def scale_bytes(M, K):
    """Size in bytes of the tiled block-scale buffer for an [M, K] operand."""
    return scale_rows_padded(M) * scale_cols_padded(K)


def tile_offset(row, s, n_scale_cols_padded):
    """Byte offset of scale index ``s`` of (tile-layout) row ``row``."""
    row = np.asarray(row, dtype=np.int64)
    s = np.asarray(s, dtype=np.int64)
    n_ct = n_scale_cols_padded // 4
    tile = (row // 128) * n_ct + s // 4
    return tile * 512 + (row % 32) * 16 + ((row % 128) // 32) * 4 + (s % 4)


def scale_tile_offsets(M, n_scale):
    """[M, n_scale] byte offsets of row-major scales in the tiled buffer."""
    ncp = -(-n_scale // 4) * 4
    r = np.arange(M)[:, None]
    s = np.arange(n_scale)[None, :]
    return tile_offset(r, s, ncp)


def grouped_row_map(offsets):
    """Tile-layout row of each expert-sorted row: each expert's rows start at
    a 128-aligned tile row (its padded base), so every 128-row M tile of the
    grouped GEMM reads whole scale tiles of one expert."""
    offsets = np.asarray(offsets, dtype=np.int64)
    M = int(offsets[-1])
    prow = np.empty(M, np.int64)
    base = 0
    for e in range(len(offsets) - 1):
        lo, hi = offsets[e], offsets[e + 1]
        prow[lo:hi] = base + np.arange(hi - lo)
        base += -(-(hi - lo) // 128) * 128
    return prow


def grouped_scale_bytes(M_total, K, E):
    """Upper bound of the grouped tiled scale buffer (any routing)."""
    return (-(-M_total // 128) + E) * 128 * scale_cols_padded(K)


def grouped_scale_tile_offsets(offsets, n_scale):
    ncp = -(-n_scale // 4) * 4
    prow = grouped_row_map(offsets)[:, None]
    s = np.arange(n_scale)[None, :]
    return tile_offset(prow, s, ncp)


def comp_weights(codes_w, sigma_w, chan):
    """Compensation weight rows for the default mode, without the tensor
    scale: Wt_S[n, i] = E2M1(code_w[n, S_i]) * sigma_w[n, S_i // 16], shape
    [N, k] (W^T columns on S).  Exact in bf16: a 2-bit by 4-bit significand
    product has at most 6 significant bits."""
    chan = np.asarray(chan, dtype=np.int64)
    v = e2m1_value(codes_w[:, chan])
    s = e4m3_decode(sigma_w[:, chan // BLOCK])
    return v * s


#: power-of-two factor of the FP8 compensation weight rows (2688 * 2^-3 <= 448)
COMP_FP8_SHIFT = 3


def comp_weights_fp8(codes_w, sigma_w, chan):
    """FP8 compensation weight rows: E4M3 bytes (sign in bit 7) of
    :func:`comp_weights` times 2^-3, shape [N, k].  The product with 2^-3 is
    exact in fp64; the one rounding is to E4M3 (RNE, satfinite)."""
    return e4m3_encode_signed(comp_weights(codes_w, sigma_w, chan) * 2.0 ** -COMP_FP8_SHIFT)
