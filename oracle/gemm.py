"""fp64 reference GEMM with the compensation term (test infrastructure only).

Sources.  QUADS abstract (arXiv 2607.15810): the main product stays a native
W4A4 GEMM and Residual Activation Compensation corrects high-error
activation channels.  gist.science explainer of QUADS, Technisches Resuemee
section 2.2 B: the residual term computed on the selected channels is added
to the quantized output.  FourSight abstract (arXiv 2611.04887): the
selected channels are kept in BF16.

Definition (activations X [M, K], weights W [K, N] stored as W^T [N, K]):

    Y = deq(q(X)) . deq(q(W^T))^T  +  R_S . W_S^T

with R_S [M, k] the bf16 residual slice on channels S and W_S [N, k] the
columns S of W^T: deq(q(W^T))[:, S] by default (so the correction uses the
same quantized weights as the rollout GEMM), or the original bf16 W^T[:, S]
under the BF16-weight flag.  Everything is formed in fp64, where the
dequantized operands are exact.

Quantized-residual variant (the explainer's "second-pass quantization" of
the high-residual channels, section 2.2 B, read as FP8 E4M3 operands for
the compensation product):

    Y = deq(q(X)) . deq(q(W^T))^T  +  2^3 g_a g_w  R8 . W8^T

with R8 [M, k] the E4M3 residual of the residual pre-scaled by 1/g_a
(nvfp4.quantize's resid_fp8) and W8 [N, k] the E4M3 weight rows
E2M1 * sigma * 2^-3 (nvfp4.comp_weights_fp8), both decoded exactly in fp64.
"""

import numpy as np

from . import nvfp4
from .formats import e4m3_value


def reference(a_deq, b_deq, resid=None, w_sel=None):
    """Y = a_deq . b_deq^T (+ resid . w_sel^T), fp64.

    a_deq [M, K], b_deq [N, K], resid [M, k], w_sel [N, k]."""
    y = np.asarray(a_deq, np.float64) @ np.asarray(b_deq, np.float64).T
    if resid is not None and resid.shape[1] > 0:
        y = y + np.asarray(resid, np.float64) @ np.asarray(w_sel, np.float64).T
    return y


def naive(a_deq, b_deq, resid=None, w_sel=None):
    """Pure-Python triple loop of the same definition (tiny shapes only)."""
    M, K = a_deq.shape
    N = b_deq.shape[0]
    k = 0 if resid is None else resid.shape[1]
    y = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = 0.0
            for j in range(K):
                s += float(a_deq[m, j]) * float(b_deq[n, j])
            for i in range(k):
                s += float(resid[m, i]) * float(w_sel[n, i])
            y[m, n] = s
    return y


def comp_weight_rows(qw, chan, wt_bf16=None):
    """W_S [N, k] for the compensation term: dequantized NVFP4 columns S of
    W^T by default, the original bf16 columns when ``wt_bf16`` is given."""
    chan = np.asarray(chan, dtype=np.int64)
    if wt_bf16 is not None:
        return np.asarray(wt_bf16, np.float64)[:, chan]
    return nvfp4.comp_weights(qw["codes"], qw["sigma"], chan) * np.float64(qw["g"])


def linear_comp(x, wt, chan, g_x=None, bf16_weights=False):
    """Whole dense layer: quantize X (dynamic scale unless g_x given) and
    W^T (dynamic scale), then the reference product with compensation.
    Returns (Y fp64, qx, qw)."""
    qx = nvfp4.quantize(x, g=g_x, chan=chan)
    qw = nvfp4.quantize(wt)
    a = nvfp4.dequantize(qx["codes"], qx["sigma"], qx["g"])
    b = nvfp4.dequantize(qw["codes"], qw["sigma"], qw["g"])
    if len(chan):
        ws = comp_weight_rows(qw, chan, wt if bf16_weights else None)
        y = reference(a, b, qx["resid"], ws)
    else:
        y = reference(a, b)
    return y, qx, qw


def comp_term_fp8(resid_fp8, w_fp8, g_a, g_w):
    """The quantized-residual compensation term 2^3 g_a g_w R8 . W8^T in
    fp64, R8 [M, k] and W8 [N, k] E4M3 bytes."""
    r = e4m3_value(resid_fp8)
    w = e4m3_value(w_fp8)
    f = np.float64(2.0 ** nvfp4.COMP_FP8_SHIFT) * np.float64(g_a) * np.float64(g_w)
    return f * (r @ w.T)


def linear_comp_fp8(x, wt, chan, g_x=None):
    """Whole dense layer with the quantized-residual compensation: quantize X
    (dynamic scale unless g_x given) and W^T (dynamic scale), then
    deq . deq^T + comp_term_fp8.  Returns (Y fp64, qx, qw, w_fp8)."""
    qx = nvfp4.quantize(x, g=g_x, chan=chan)
    qw = nvfp4.quantize(wt)
    a = nvfp4.dequantize(qx["codes"], qx["sigma"], qx["g"])
    b = nvfp4.dequantize(qw["codes"], qw["sigma"], qw["g"])
    y = reference(a, b)
    w8 = nvfp4.comp_weights_fp8(qw["codes"], qw["sigma"], chan)
    if len(chan):
        y = y + comp_term_fp8(qx["resid_fp8"], w8, qx["g"], qw["g"])
    return y, qx, qw, w8


def grouped_reference(a_deq, offsets, b_deq, resid=None, w_sel=None):
    """Per-expert reference: rows [offsets[e], offsets[e+1]) of a_deq times
    expert e's b_deq[e] [N, K] (plus resid rows times w_sel[e] [N, k])."""
    offsets = np.asarray(offsets, dtype=np.int64)
    M = int(offsets[-1])
    N = b_deq.shape[1]
    y = np.zeros((M, N))
    for e in range(len(offsets) - 1):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        y[lo:hi] = reference(a_deq[lo:hi], b_deq[e],
                             None if resid is None else resid[lo:hi],
                             None if w_sel is None else w_sel[e])
    return y
