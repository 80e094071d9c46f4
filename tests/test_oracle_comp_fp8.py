"""Pins of the oracle's quantized-residual (FP8 E4M3) compensation (CPU
only): the signed E4M3 encoder against torch's float8 conversion, the
hand-derived worked examples, and the whole layer against the exact
compensation within the E4M3 rounding bound."""

import json
import os

import numpy as np
import torch

from oracle import formats as F
from oracle import gemm, nvfp4
from nvfp4_w4a4_gemm_gb300 import workloads as W


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "comp_fp8_worked.json")) as f:
        return json.load(f)


def _all_bf16_values():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    return v[np.isfinite(v)]


def test_signed_e4m3_matches_torch_float8():
    # every finite bf16 value below the overflow midpoint (464 = (448 + 480) / 2)
    v = _all_bf16_values()
    v = v[np.abs(v) < 464.0]
    ours = F.e4m3_encode_signed(v)
    ref = torch.from_numpy(v.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_signed_e4m3_saturates_and_keeps_sign():
    assert list(F.e4m3_encode_signed(np.array([464.0, 1e6, -500.0, -0.0, 0.0]))) == [0x7E, 0x7E, 0xFE, 0x80, 0x00]


def test_e4m3_value_inverts_the_encoder():
    b = np.array([i for i in range(256) if (i & 0x7F) != 0x7F], np.uint8)
    v = F.e4m3_value(b)
    assert np.array_equal(F.e4m3_encode_signed(v), b)
    assert F.e4m3_value(np.uint8(0x7E)) == 448.0 and F.e4m3_value(np.uint8(0x81)) == -(2.0 ** -9)


def test_residual_worked_examples(golden_dir):
    for ex in _golden(golden_dir)["residual_examples"]:
        x = np.array(ex["x"], np.float32)[None, :]
        assert np.array_equal(F.bf16_round(x), x), "fixture values must be bf16-exact"
        q = nvfp4.quantize(x, g=ex["g"], chan=np.array(ex["chan"]))
        assert list(q["resid_fp8"][0]) == ex["resid_fp8"]


def test_weight_rows_worked_example(golden_dir):
    w = _golden(golden_dir)["weight_examples"]
    codes = np.array(w["codes"], np.uint8)[None, :]
    sigma = np.full((1, 1), w["sigma"], np.uint8)
    assert list(nvfp4.comp_weights_fp8(codes, sigma, np.array(w["chan"]))[0]) == w["w_fp8"]


def test_term_worked_example(golden_dir):
    t = _golden(golden_dir)["term_example"]
    y = gemm.comp_term_fp8(np.array(t["resid_fp8"], np.uint8), np.array(t["w_fp8"], np.uint8), t["g_a"], t["g_w"])
    assert np.array_equal(y, np.array(t["y"]))


def _e4m3_err_bound(v):
    """Largest |E4M3(v) - v| for |v| <= 448: half a spacing, 2^-4 |v| for
    normals and 2^-10 in the subnormal range."""
    return np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10)


def test_layer_within_e4m3_bound_of_exact_compensation():
    # the FP8 layer differs from the exact compensation deq.deq + R . W_S
    # (fp32 residual, exact dequantized weight columns) only by the two E4M3
    # roundings of each product's factors
    M, N, K, k = 24, 32, 256, 16
    x = W.activations(M, K, 7, "t3x20", 1, 2).float().numpy()
    wt = W.weights_t(N, K, 8).float().numpy()
    chan = np.sort(np.random.default_rng(3).choice(K, size=k, replace=False))
    y8, qx, qw, w8 = gemm.linear_comp_fp8(x, wt, chan)
    a = nvfp4.dequantize(qx["codes"], qx["sigma"], qx["g"])
    b = nvfp4.dequantize(qw["codes"], qw["sigma"], qw["g"])
    g_a, g_w = np.float64(qx["g"]), np.float64(qw["g"])
    w_units = nvfp4.comp_weights(qw["codes"], qw["sigma"], chan)  # E2M1 * sigma
    r_exact = qx["resid_f32"][:, chan].astype(np.float64)
    y_exact = gemm.reference(a, b, r_exact, w_units * g_w)
    pre = r_exact / g_a                       # the pre-scaled residual, exactly
    w_sc = w_units * 2.0 ** -3
    er = _e4m3_err_bound(pre) + np.abs(pre) * 2.0 ** -22  # + the fp32 product's rounding
    ew = _e4m3_err_bound(w_sc)
    bound = 8.0 * g_a * g_w * ((np.abs(pre) + er) @ ew.T + er @ np.abs(w_sc).T)
    assert np.all(np.abs(y8 - y_exact) <= bound + 1e-12 * np.abs(y_exact))
    # the bound is the E4M3 relative error of the products (not vacuous) ...
    mag = 8.0 * g_a * g_w * (np.abs(pre) @ np.abs(w_sc).T)
    assert np.median(bound / mag) < 0.15
    # ... and tight enough that a dropped 2^3, a residual not divided by g_a
    # or a flipped sign of the term falls outside it
    main = gemm.reference(a, b)
    comp8 = y8 - main
    for bad in (main + comp8 / 8.0, main + comp8 * g_a, main - comp8):
        assert np.any(np.abs(bad - y_exact) > bound + 1e-12 * np.abs(y_exact))
    # the E4M3 operands really are those of the quantizer and weight-row helpers
    assert np.array_equal(w8, nvfp4.comp_weights_fp8(qw["codes"], qw["sigma"], chan))
    assert np.array_equal(qx["resid_fp8"], F.e4m3_encode_signed((qx["resid_f32"][:, chan] * nvfp4.reciprocal(qx["g"])).astype(np.float32)))
