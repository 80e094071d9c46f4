"""Channel selection for the compensation term (test infrastructure only).

Sources.  FourSight abstract (arXiv 2611.04887): quantization error
concentrates in a few high-variance activation channels, and only the
top-variance channels are kept in BF16.  gist.science explainer of QUADS,
Technisches Resuemee section 2.2 B: a binary channel mask picks the channels
with the largest residual.

Reading: on a calibration batch X_cal (same distribution, its own dynamic
tensor scale), form the fp32 residual R = x - deq(q(x)) of NVFP4
quantization, take the population variance of each channel (column) over
the rows in fp64, and keep the k channels with the largest variance; ties go
to the lower channel index; the set is returned sorted ascending.  The
explainer's "top-k% (e.g. 50%)" is not followed: k is a fixed small count.
For MoE, each expert's set comes from the calibration rows routed to it; an
expert with fewer than 2 such rows uses all rows.
"""

import numpy as np

from . import nvfp4


def channel_variance(resid_f32):
    """Population variance of each column of R over rows, fp64 two-pass."""
    r = np.asarray(resid_f32, dtype=np.float64)
    mu = r.mean(axis=0)
    return ((r - mu) ** 2).mean(axis=0)


def top_k(var, k):
    """Indices of the k largest values (ties -> lower index), ascending."""
    var = np.asarray(var, dtype=np.float64)
    idx = np.arange(var.size)
    order = np.lexsort((idx, -var))
    return np.sort(order[:k]).astype(np.int32)


def calibrate(x_cal, k):
    """Channel set S (int32 [k]) of a dense layer from a calibration batch."""
    if k == 0:
        return np.zeros(0, np.int32)
    q = nvfp4.quantize(x_cal)
    return top_k(channel_variance(q["resid_f32"]), k)


def calibrate_grouped(x_cal, offsets_cal, k):
    """Per-expert channel sets int32 [E, k] from expert-sorted calibration rows."""
    q = nvfp4.quantize(x_cal)
    rf = q["resid_f32"]
    offsets_cal = np.asarray(offsets_cal, dtype=np.int64)
    E = len(offsets_cal) - 1
    out = np.zeros((E, k), np.int32)
    var_all = channel_variance(rf)
    for e in range(E):
        lo, hi = offsets_cal[e], offsets_cal[e + 1]
        var = channel_variance(rf[lo:hi]) if hi - lo >= 2 else var_all
        out[e] = top_k(var, k)
    return out
