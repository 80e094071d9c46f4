"""Pins of the oracle's MXFP4 quantizer and error decomposition (CPU only)."""

import json
import os

import numpy as np

from oracle import mxfp4, formats as F
from nvfp4_w4a4_gemm_gb300 import workloads as W


def test_worked_example(golden_dir):
    with open(os.path.join(golden_dir, "mxfp4_worked.json")) as f:
        ex = json.load(f)
    x = np.zeros((1, ex["block_len"]), np.float32)
    x[0, :4] = ex["x_head"]
    d = mxfp4.decompose(x)
    assert d["scale"][0, 0] == ex["scale_byte"]
    assert list(d["codes"][0, :4]) == ex["codes_head"]
    assert np.all(d["codes"][0, 4:] == 0)
    for key in "EBDG":
        np.testing.assert_allclose(d[key][0, :4], ex[key + "_head"], rtol=0, atol=1e-12)
        assert np.all(d[key][0, 4:] == 0)
    assert d["dead"].sum() == ex["deadzone_count"]


def test_scales_are_powers_of_two_and_cover_the_block():
    # Decomposing MXFP4 error abstract: scales come from power-of-two rounding.
    x = W.activations(32, 512, 6, "t3x20", 4, 4).float().numpy()
    q = mxfp4.quantize(x)
    s = F.e8m0_value(q["scale"])
    assert np.all(np.log2(s) == np.round(np.log2(s)))
    a = np.abs(x).reshape(32, 16, 32).max(-1)
    ratio = a / s
    assert np.all((ratio >= 4) & (ratio < 8))       # e = floor(log2 a) - 2


def test_roundtrip_of_grid_representable_blocks():
    rng = np.random.default_rng(2)
    M, nb = 6, 8
    e = rng.integers(-20, 20, size=(M, nb))
    c = rng.integers(0, 16, size=(M, nb, 32))
    c[:, :, 0] = np.where(rng.random((M, nb)) < 0.5, 6, 7)   # max |c| in {4, 6}
    # keep the block max at index 0: cap other magnitudes at the chosen max
    top = F.e2m1_value(c[:, :, 0])
    others = np.minimum(np.abs(F.e2m1_value(c[:, :, 1:])), top[:, :, None])
    sign = np.where(c[:, :, 1:] & 8, -1.0, 1.0)
    x = np.concatenate([top[:, :, None], others * sign], axis=2)
    x = (x * np.power(2.0, e)[:, :, None]).reshape(M, nb * 32).astype(np.float32)
    q = mxfp4.quantize(x)
    assert np.array_equal(q["e"], e)
    assert np.array_equal(mxfp4.dequantize(q["codes"], q["scale"]), x.astype(np.float64))


def test_decomposition_is_exact_and_additive():
    x = W.activations(64, 1024, 10, "t3x20", 5, 5).float().numpy()
    d = mxfp4.decompose(x)
    # E = B + D + G holds exactly (every term is exact in fp64)
    assert np.array_equal(d["B"] + d["D"] + d["G"], d["E"])
    assert np.array_equal(d["E"], mxfp4.dequantize(d["codes"], d["scale"]) - x)
    # D and G have disjoint supports
    assert not np.any((d["D"] != 0) & (d["G"] != 0))
    # deadzone entries are exactly those zeroed at the ideal scale: D = -x
    assert np.array_equal(d["D"][d["dead"]], -x[d["dead"]].astype(np.float64))


def test_no_scale_bias_when_block_max_is_six_times_power_of_two():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 64)).astype(np.float32)
    x = F.bf16_round(x)
    x = np.clip(x, -2.9, 2.9)
    x[:, 0] = 6.0 * 0.5     # a = 3 = 6 * 2^-1 -> s* = s = 2^-1
    x[:, 32] = -6.0 * 2.0 ** 3
    d = mxfp4.decompose(x)
    assert np.all(d["B"] == 0)


def test_no_grid_noise_or_deadzone_on_grid_at_ideal_scale():
    s = 2.0 ** -2
    c = np.array([6, -4, 3, 0.5, -1.5, 2, 1, 0] * 4, np.float64)
    x = (c * s).astype(np.float32)[None, :]
    d = mxfp4.decompose(x)
    assert np.all(d["D"] == 0) and np.all(d["G"] == 0)


def test_deadzone_special_case():
    # every |x| <= a/24 except the max -> those entries are all deadzone
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 24.0
    x[0, 1:] = F.bf16_round(np.linspace(-0.99, 0.99, 31).astype(np.float32))
    d = mxfp4.decompose(x)
    nz = x[0, 1:] != 0
    assert np.all(d["dead"][0, 1:][nz])
    assert np.array_equal(d["D"][0, 1:], -x[0, 1:].astype(np.float64))


def test_block_stats_consistent():
    x = W.activations(16, 256, 3, "t3x20", 6, 6).float().numpy()
    st, cnt, d = mxfp4.block_stats(x)
    assert st.shape == (16, 8, 4) and cnt.shape == (16, 8)
    np.testing.assert_allclose(st[..., 3], (d["E"] ** 2).reshape(16, 8, 32).sum(-1))
    assert np.array_equal(cnt, d["dead"].reshape(16, 8, 32).sum(-1))


def test_block_exponent_closed_forms():
    # e = floor(log2 a) - 2: exact powers of two, their bf16 neighbours below,
    # zero, and both clamps
    from oracle.mxfp4 import block_exponent
    ks = np.arange(-120, 121, 7)
    assert np.array_equal(block_exponent(2.0 ** ks), ks - 2)
    below = (2.0 ** ks) * (1 - 2.0 ** -8)     # the next bf16 value down
    assert np.array_equal(block_exponent(below), ks - 3)
    assert block_exponent(np.array([0.0]))[0] == -127
    assert block_exponent(np.array([2.0 ** 200]))[0] == 127
    assert block_exponent(np.array([2.0 ** -140]))[0] == -127


# --- block_stats energy columns (|B|^2, |D|^2, |G|^2), pinned to values that
# do not come from the oracle: the hand-derived components of the worked
# example and two closed-form blocks ("Decomposing MXFP4 quantization
# error", abstract: the error splits exactly into scale bias, deadzone
# truncation and grid noise).

def _stats_pins(stats_fn, golden_dir):
    """Raise AssertionError unless ``stats_fn(x) -> (stats [M, nb, 4], ...)``
    gives the independently derived energies on three blocks."""
    with open(os.path.join(golden_dir, "mxfp4_worked.json")) as f:
        ex = json.load(f)
    # 1) the worked block: its non-zero head holds every non-zero component,
    #    so each energy is the sum of squares of the hand-derived head values
    x = np.zeros((1, ex["block_len"]), np.float32)
    x[0, :4] = ex["x_head"]
    st = stats_fn(x)[0][0, 0]
    want = [sum(v * v for v in ex[k + "_head"]) for k in "BDGE"]
    np.testing.assert_allclose(st, want, rtol=1e-12, atol=1e-15)
    # 2) deadzone block: a = 24 = 6 * 2^2 puts the maximum on the grid at
    #    both scales (s = s* = 4) and every other |x| < 1 < s/2 is zeroed at
    #    both, so B = G = 0 and D = E = -x on the small entries
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 24.0
    x[0, 1:] = F.bf16_round(np.linspace(-0.99, 0.99, 31).astype(np.float32))
    small = float(np.sum(x[0, 1:].astype(np.float64) ** 2))
    np.testing.assert_allclose(stats_fn(x)[0][0, 0], [0.0, small, 0.0, small], rtol=1e-12, atol=0)
    # 3) bias-only block: a = 7 with every entry in {+-7, +-3.5, +-1.75} puts
    #    each x/s* (s* = 7/6, fp32) within fp32 rounding of a grid point
    #    {6, 3, 1.5}, so G is a few fp32 ulps; at s = 1 they round to 6, 4
    #    (tie 3.5 -> even code 4) and 2 (tie 1.75 -> 2): the whole error is
    #    scale bias, B = E up to those ulps, and D = 0
    x = np.array([[7, -3.5, 1.75, -7] * 8], np.float32)
    st = stats_fn(x)[0][0, 0]
    e_energy = 8 * (1.0 + 0.25 + 0.0625 + 1.0)
    assert st[1] == 0.0
    assert st[2] < 1e-9
    np.testing.assert_allclose(st[3], e_energy, rtol=0, atol=0)
    np.testing.assert_allclose(st[0], e_energy, rtol=1e-6)


def test_block_stats_energy_columns_pinned(golden_dir):
    _stats_pins(mxfp4.block_stats, golden_dir)


def test_block_stats_pins_reject_planted_mistakes(golden_dir):
    import pytest

    def swapped_bd(x):
        st, cnt, d = mxfp4.block_stats(x)
        return st[..., [1, 0, 2, 3]], cnt, d

    def swapped_dg(x):
        st, cnt, d = mxfp4.block_stats(x)
        return st[..., [0, 2, 1, 3]], cnt, d

    def no_square(x):
        d = mxfp4.decompose(x)
        M, K = d["E"].shape
        s1 = lambda t: np.sum(np.abs(t.reshape(M, K // 32, 32)), axis=2)
        sq = lambda t: np.sum(t.reshape(M, K // 32, 32) ** 2, axis=2)
        return np.stack([s1(d["B"]), s1(d["D"]), s1(d["G"]), sq(d["E"])], -1), None, d

    def bias_against_x(x):   # B measured as Q_s - x (i.e. the total error)
        st, cnt, d = mxfp4.block_stats(x)
        st = st.copy()
        st[..., 0] = st[..., 3]
        return st, cnt, d

    for bad in (swapped_bd, swapped_dg, no_square, bias_against_x):
        with pytest.raises(AssertionError):
            _stats_pins(bad, golden_dir)
