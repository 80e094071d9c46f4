"""Shared test helpers: tolerance of the GEMM parity check and conversions."""

import numpy as np
import torch

from oracle import nvfp4 as onv

# GEMM tolerance (problem statement): |y - y_ref| <= 4e-3 |y_ref| + 1e-3 rms(Y_ref),
# elementwise, against the fp64 product of the same dequantized operands.
REL_TOL = 4e-3
RMS_TOL = 1e-3


def gemm_within_tol(y, y_ref, rms=None):
    """Returns (ok, worst ratio of error to allowance, rms used)."""
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    if rms is None:
        rms = float(np.sqrt(np.mean(y_ref ** 2))) if y_ref.size else 0.0
    allow = REL_TOL * np.abs(y_ref) + RMS_TOL * rms
    err = np.abs(y - y_ref)
    ratio = float(np.max(err / np.maximum(allow, 1e-300))) if y.size else 0.0
    return bool(np.all(err <= allow)), ratio, rms


def f32(t):
    """torch tensor -> float32 numpy (bf16 values are exact)."""
    return t.detach().float().cpu().numpy()


def u8(t):
    return t.detach().cpu().numpy().astype(np.uint8)


def gather_scales(buf, offsets):
    """Pick the row-major [rows, n] scales out of a tiled scale buffer."""
    b = u8(buf).ravel()
    return b[offsets]


def tiled_scales_dense(buf, M, K, block=16):
    return gather_scales(buf, onv.scale_tile_offsets(M, K // block))


def bf16_bits_of(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)
