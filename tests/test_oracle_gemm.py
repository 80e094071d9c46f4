"""Pins of the oracle's reference GEMM, compensation and calibration (CPU only)."""

import numpy as np

from oracle import calib, gemm, nvfp4, formats as F
from nvfp4_w4a4_gemm_gb300 import workloads as W


def _tiny(k=8):
    d = W.dense_inputs("tiny")
    x = d["x"].float().numpy()
    wt = d["wt"].float().numpy()
    xc = W.dense_inputs("tiny", calibration=True, with_weights=False)["x"].float().numpy()
    return x, wt, xc


def test_brute_force_small_shapes():
    rng = np.random.default_rng(0)
    for (M, N, K, k) in [(3, 5, 32, 0), (4, 3, 64, 16), (1, 7, 16, 1)]:
        x = F.bf16_round(rng.standard_normal((M, K)).astype(np.float32) * 3)
        wt = F.bf16_round(rng.standard_normal((N, K)).astype(np.float32) * 0.05)
        chan = np.sort(rng.choice(K, size=k, replace=False))
        y, qx, qw = gemm.linear_comp(x, wt, chan)
        a = nvfp4.dequantize(qx["codes"], qx["sigma"], qx["g"])
        b = nvfp4.dequantize(qw["codes"], qw["sigma"], qw["g"])
        ws = gemm.comp_weight_rows(qw, chan) if k else None
        yn = gemm.naive(a, b, qx.get("resid") if k else None, ws)
        np.testing.assert_allclose(y, yn, rtol=1e-13, atol=1e-13)


def test_full_compensation_reproduces_w4a16_product():
    # k = K with the default weight rows: deq(qX) + R = X up to the bf16
    # rounding of R, so Y = X . deq(qW)^T -- the W4A16 product the QUADS
    # trainer computes (gist.science explainer, Technisches Resuemee 2.2 A).
    x, wt, _ = _tiny()
    K = x.shape[1]
    y, qx, qw = gemm.linear_comp(x, wt, np.arange(K))
    b = nvfp4.dequantize(qw["codes"], qw["sigma"], qw["g"])
    y16 = x.astype(np.float64) @ b.T
    # |R - bf16(R)| <= 2^-9 |R| and |R| <= d (half the coarsest grid step)
    bound = (np.abs(qx["resid_f32"]).astype(np.float64) * 2.0 ** -8) @ np.abs(b).T
    assert np.all(np.abs(y - y16) <= bound + 1e-12)
    # and without compensation the error is far larger
    y0, _, _ = gemm.linear_comp(x, wt, np.zeros(0, np.int64))
    assert np.linalg.norm(y0 - y16) > 50 * np.linalg.norm(y - y16)


def test_compensation_error_shrinks_with_k():
    # gist.science explainer 2.2 B: compensation reduces the distance to the
    # unquantized-activation output; nested channel sets by residual variance.
    x, wt, xc = _tiny()
    K = x.shape[1]
    var = calib.channel_variance(nvfp4.quantize(xc)["resid_f32"])
    order = np.lexsort((np.arange(K), -var))
    qw = nvfp4.quantize(wt)
    b = nvfp4.dequantize(qw["codes"], qw["sigma"], qw["g"])
    y16 = x.astype(np.float64) @ b.T
    errs = []
    for k in (0, 4, 8, 32, 128, 256):
        y, _, _ = gemm.linear_comp(x, wt, np.sort(order[:k]))
        errs.append(np.linalg.norm(y - y16))
    assert all(e1 < e0 for e0, e1 in zip(errs, errs[1:])), errs


def test_bf16_weight_flag_uses_original_weights():
    x, wt, _ = _tiny()
    chan = np.array([3, 100, 200])
    yq, qx, qw = gemm.linear_comp(x, wt, chan)
    yb, _, _ = gemm.linear_comp(x, wt, chan, bf16_weights=True)
    diff = yb - yq
    want = qx["resid"].astype(np.float64) @ (wt[:, chan].astype(np.float64)
                                             - gemm.comp_weight_rows(qw, chan)).T
    np.testing.assert_allclose(diff, want, rtol=1e-9, atol=1e-9)


def test_grouped_reference_is_per_expert_dense():
    rng = np.random.default_rng(4)
    offs = np.array([0, 5, 5, 12])
    a = rng.standard_normal((12, 32))
    b = rng.standard_normal((3, 8, 32))
    y = gemm.grouped_reference(a, offs, b)
    np.testing.assert_allclose(y[:5], a[:5] @ b[0].T)
    np.testing.assert_allclose(y[5:], a[5:] @ b[2].T)


def test_calibration_finds_the_outlier_channels():
    # tiny workload: 4 channels scaled x50 dominate the residual variance,
    # so all 4 are among the k = 8 selected channels.
    _, _, xc = _tiny()
    S = calib.calibrate(xc, 8)
    ids = W.outlier_channels(256, 4, 0).numpy()
    assert set(ids) <= set(S.tolist())
    assert list(S) == sorted(S) and len(set(S)) == 8


def test_top_k_ties_to_lower_index():
    var = np.array([1.0, 3.0, 3.0, 2.0, 3.0])
    assert list(calib.top_k(var, 2)) == [1, 2]
    assert list(calib.top_k(var, 4)) == [1, 2, 3, 4]


def test_grouped_calibration_small_expert_uses_all_rows():
    x = W.activations(20, 64, 2, "x50", 1, 1).float().numpy()
    offs = np.array([0, 1, 20])
    S = calib.calibrate_grouped(x, offs, 4)
    assert np.array_equal(S[0], calib.calibrate(x, 4))
    assert np.array_equal(S[1], calib.top_k(calib.channel_variance(
        nvfp4.quantize(x)["resid_f32"][1:20]), 4))
