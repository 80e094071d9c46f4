"""Pins of the oracle's corrected MXFP4 (macro-block scaling and Outlier
Fallback; CPU only): the hand-derived worked row, the reductions to plain
MXFP4, the closed forms of the macro scale, the exact product when every
channel falls back, and the effects the corrections are named for (less
scale bias, fewer deadzone entries, a smaller GEMM error)."""

import json
import os

import numpy as np

from oracle import formats as F
from oracle import mxfp4 as mx
from nvfp4_w4a4_gemm_gb300 import workloads as W


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "mxfp4_corrected_worked.json")) as f:
        return json.load(f)


def test_worked_row(golden_dir):
    g = _golden(golden_dir)
    x = np.zeros((1, g["K"]), np.float32)
    for j, v in g["x_nonzero"].items():
        x[0, int(j)] = v
    q = mx.quantize_corrected(x, macro=True, fallback=g["fallback"])
    assert q["m"][0] == np.float32(g["m"]) and q["rho"][0] == np.float32(g["rho"])
    assert list(q["scale"][0]) == g["scale_bytes"]
    for j, c in g["codes_at"].items():
        assert q["codes"][0, int(j)] == c
    assert list(q["fb"][0]) == g["fb"]


def _outlier_rows(M=64, K=512, seed=4):
    return W.activations(M, K, 6, "t3x20", seed, seed + 1).float().numpy()


def test_no_correction_is_plain_mxfp4():
    x = _outlier_rows()
    q = mx.quantize_corrected(x)
    p = mx.quantize(x)
    st, dead, _ = mx.block_stats(x)
    assert np.all(q["m"] == 1) and np.array_equal(q["codes"], p["codes"]) and np.array_equal(q["scale"], p["scale"])
    assert np.array_equal(q["stats"], st) and np.array_equal(q["dead"], dead) and q["fb"].shape == (x.shape[0], 0)


def test_macro_scale_closed_forms():
    rng = np.random.default_rng(7)
    x = F.bf16_round((rng.standard_normal((200, 96)) * np.exp(rng.uniform(-20, 20, (200, 1)))).astype(np.float32))
    m = mx.macro_scale(x)
    t = (np.max(np.abs(x), axis=1) / np.float32(6)).astype(np.float32)
    assert np.all((m >= 1) & (m < 2))
    # m * 2^floor(log2 t) == t exactly
    fl = np.floor(np.log2(t.astype(np.float64)))
    assert np.array_equal(m.astype(np.float64) * np.power(2.0, fl), t.astype(np.float64))
    # rows whose max / 6 is a power of two: m = 1 and the plain quantization
    y = x.copy()
    y[:, 0] = (6.0 * np.power(2.0, rng.integers(-20, 20, 200))).astype(np.float32)
    y[:, 1:] = np.clip(y[:, 1:], -np.abs(y[:, :1]), np.abs(y[:, :1]))
    q = mx.quantize_corrected(y, macro=True)
    assert np.all(q["m"] == 1) and np.array_equal(q["codes"], mx.quantize(y)["codes"])
    # zero rows: m = 1
    assert mx.macro_scale(np.zeros((2, 32), np.float32)).tolist() == [1.0, 1.0]


def test_row_maximum_lands_on_the_top_level():
    x = _outlier_rows(M=128)
    q = mx.quantize_corrected(x, macro=True)
    deq = mx.dequantize(q["codes"], q["scale"]) * q["m"].astype(np.float64)[:, None]
    j = np.argmax(np.abs(x), axis=1)
    r = np.arange(x.shape[0])
    assert np.all(q["codes"][r, j] & 7 == 7)  # the top level, 6
    assert np.all(np.abs(deq[r, j] - x[r, j]) <= 2.0 ** -21 * np.abs(x[r, j]))


def test_full_fallback_is_the_exact_product():
    # every channel falls back and no macro scale: the FP4 operands are zero
    # and the BF16 side product is X . W^T exactly
    x = _outlier_rows(M=16, K=128)
    wt = W.weights_t(24, 128, 3).float().numpy()
    S = np.arange(128)
    qa, qb = mx.quantize_corrected(x, fallback=S), mx.quantize_corrected(wt, fallback=S)
    assert np.all(qa["codes"] & 7 == 0) and np.all(qb["codes"] & 7 == 0)
    assert np.array_equal(mx.gemm_corrected(qa, qb), x.astype(np.float64) @ wt.astype(np.float64).T)


def test_fallback_values_and_zeroed_channels():
    x = _outlier_rows()
    S = W.outlier_channels(x.shape[1], 6, 4)
    q = mx.quantize_corrected(x, macro=True, fallback=S)
    assert np.all(q["codes"][:, S] & 7 == 0)
    assert np.array_equal(q["fb"], F.bf16_round((x[:, S] * q["rho"][:, None]).astype(np.float32)))


def test_corrections_reduce_their_components():
    x = _outlier_rows(M=256, K=1024, seed=9)
    S = W.outlier_channels(1024, 6, 9)
    plain = mx.quantize_corrected(x)
    mac = mx.quantize_corrected(x, macro=True)
    fb = mx.quantize_corrected(x, fallback=S)
    m2 = (mac["m"].astype(np.float64) ** 2)[:, None]
    # macro scaling: less scale-bias energy (in the row's own units)
    assert np.sum(mac["stats"][..., 0] * m2) < 0.9 * np.sum(plain["stats"][..., 0])
    # Outlier Fallback: fewer deadzone entries and less deadzone energy
    assert np.sum(fb["dead"]) < 0.5 * np.sum(plain["dead"])
    assert np.sum(fb["stats"][..., 1]) < 0.5 * np.sum(plain["stats"][..., 1])


def test_corrected_gemm_is_closer_to_the_bf16_product():
    x = _outlier_rows(M=64, K=1024, seed=11)
    wt = W.weights_t(128, 1024, 12).float().numpy()
    S = W.outlier_channels(1024, 6, 11)
    exact = x.astype(np.float64) @ wt.astype(np.float64).T
    err = lambda y: np.linalg.norm(y - exact)
    plain = mx.gemm_corrected(mx.quantize_corrected(x), mx.quantize_corrected(wt))
    both = mx.gemm_corrected(mx.quantize_corrected(x, True, S), mx.quantize_corrected(wt, True, S))
    assert err(both) < 0.7 * err(plain)
