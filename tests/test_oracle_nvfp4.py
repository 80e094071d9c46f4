"""Pins of the oracle's NVFP4 quantizer (CPU only)."""

import json
import os

import numpy as np
import pytest

from oracle import nvfp4, formats as F
from nvfp4_w4a4_gemm_gb300 import workloads as W


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "nvfp4_worked.json")) as f:
        return json.load(f)["examples"]


@pytest.mark.parametrize("idx", [0, 1])
def test_worked_examples(golden_dir, idx):
    ex = _golden(golden_dir)[idx]
    x = np.array(ex["x"], np.float32)[None, :]
    assert np.array_equal(F.bf16_round(x), x), "fixture values must be bf16-exact"
    q = nvfp4.quantize(x, chan=np.array(ex["chan"]))
    assert q["g"] == np.float32(ex["g"])
    assert list(q["sigma"][0]) == ex["sigma"]
    assert list(q["codes"][0]) == ex["codes"]
    assert np.array_equal(q["resid"][0], np.array(ex["resid"], np.float32))
    if "packed_block1" in ex:
        assert list(q["packed"][0, 8:16]) == ex["packed_block1"]


def test_roundtrip_of_grid_representable_blocks():
    # g = 2^j; block 0 carries sigma = 448 and a +-6 code so that
    # amax = 2688 g exactly; other blocks any E4M3 sigma_b with a +-6 code.
    rng = np.random.default_rng(1)
    for j in (-8, -3, 0, 2):
        g = 2.0 ** j
        M, nb = 8, 12
        sig = rng.integers(0x08, 0x7F, size=(M, nb))  # normal E4M3 scales
        sig[0, 0] = 0x7E
        c = rng.integers(0, 16, size=(M, nb, 16))
        c[:, :, 3] = 7  # +6 in every block so sigma_b is recovered exactly
        x = F.e2m1_value(c) * F.e4m3_decode(sig)[:, :, None] * g
        x = x.reshape(M, nb * 16).astype(np.float32)
        assert np.array_equal(F.bf16_round(x), x)
        q = nvfp4.quantize(x)
        assert q["g"] == np.float32(g)
        assert np.array_equal(q["sigma"], sig.astype(np.uint8))
        deq = nvfp4.dequantize(q["codes"], q["sigma"], q["g"])
        # exact values (negative zero codes compare equal to 0)
        assert np.array_equal(deq, x.astype(np.float64))
        assert np.all(q["resid_f32"] == 0)


def test_zero_tensor_and_zero_blocks():
    x = np.zeros((3, 32), np.float32)
    q = nvfp4.quantize(x, chan=np.array([0, 31]))
    assert q["g"] == 1.0
    assert np.all(q["sigma"] == 0) and np.all(q["codes"] == 0)
    assert np.all(q["resid"] == 0)


def test_scale_is_max_over_block_and_bounded():
    # invariants on heavy-tailed data: sigma*g*6 >= a up to E4M3 rounding
    # (< 2^-4 relative for normals), codes within the grid, |y| <= 6.
    x = W.activations(64, 512, 8, "t3x20", 3, 3).float().numpy()
    q = nvfp4.quantize(x)
    a = np.abs(x).reshape(64, 32, 16).max(-1)
    s = F.e4m3_decode(q["sigma"]) * q["g"]
    nz = q["sigma"] >= 8
    assert np.all(np.abs(s[nz] * 6 - a[nz]) <= a[nz] * 2.0 ** -4 + 1e-30)
    # the block maximum lands on a top code (6 or 4 after rounding)
    deq = nvfp4.dequantize(q["codes"], q["sigma"], q["g"])
    err = np.abs(deq - x).reshape(64, 32, 16).max(-1)
    assert np.all(err <= s * 1.0 + 1e-30)     # at most half the coarsest step (2) times d


def test_tile_layout_positions():
    # byte offset of (row, scale index) in the 128x4 tile layout
    off = nvfp4.scale_tile_offsets(256, 8)  # 2 row tiles x 2 column tiles
    assert off[0, 0] == 0 and off[0, 1] == 1 and off[0, 3] == 3
    assert off[1, 0] == 16 and off[31, 0] == 496
    assert off[32, 0] == 4 and off[64, 0] == 8 and off[96, 3] == 15
    assert off[0, 4] == 512 and off[128, 0] == 1024 and off[128, 4] == 1536
    assert len(np.unique(off)) == off.size == nvfp4.scale_bytes(256, 128)


def test_tile_layout_ragged_padding():
    assert nvfp4.scale_bytes(1, 16) == 128 * 4
    assert nvfp4.scale_bytes(130, 80) == 256 * 8
    off = nvfp4.scale_tile_offsets(130, 5)
    assert off.max() < nvfp4.scale_bytes(130, 80) and len(np.unique(off)) == off.size


def test_grouped_row_map():
    offs = np.array([0, 3, 3, 200, 201])
    prow = nvfp4.grouped_row_map(offs)
    assert list(prow[:3]) == [0, 1, 2]
    assert prow[3] == 128 and prow[199] == 128 + 196 and prow[200] == 384
    assert prow.max() < (2 + 4) * 128  # within the stated upper bound


def test_grouped_residual_uses_each_experts_channels():
    x = W.random_bf16((10, 64), 5).float().numpy()
    offs = np.array([0, 4, 10])
    chan = np.array([[0, 5], [7, 63]])
    q = nvfp4.quantize_grouped(x, offs, chan)
    assert np.array_equal(q["resid"][:4], F.bf16_round(q["resid_f32"][:4][:, [0, 5]]))
    assert np.array_equal(q["resid"][4:], F.bf16_round(q["resid_f32"][4:][:, [7, 63]]))


def test_pack_unpack():
    c = np.random.default_rng(0).integers(0, 16, (3, 32)).astype(np.uint8)
    p = nvfp4.pack(c)
    assert p.shape == (3, 16) and p[0, 0] == (c[0, 0] | (c[0, 1] << 4))
    assert np.array_equal(nvfp4.unpack(p), c)


def test_comp_weights_exact_in_bf16():
    wt = W.weights_t(32, 128, 9).float().numpy()
    q = nvfp4.quantize(wt)
    chan = np.array([1, 17, 64, 127])
    ws = nvfp4.comp_weights(q["codes"], q["sigma"], chan)
    assert np.array_equal(F.bf16_round(ws.astype(np.float32)).astype(np.float64), ws)
    deq = nvfp4.dequantize(q["codes"], q["sigma"], q["g"])
    assert np.array_equal(ws * np.float64(q["g"]), deq[:, chan])


# ------------------------------------------------------------ QDQ pins ----
@pytest.mark.parametrize("idx", [0, 1])
def test_qdq_worked_examples(golden_dir, idx):
    ex = _golden(golden_dir)[idx]
    x = np.array(ex["x"], np.float32)[None, :]
    w, q = nvfp4.qdq(x)
    want = np.array(ex["qdq"], np.float32)
    assert np.array_equal(w[0], want)
    assert np.array_equal(np.signbit(w[0]), np.signbit(want)), "signs of zero"


def _e4m3_values():
    """Every finite non-negative E4M3 value from the format definition
    (4 exponent bits, bias 7, 3 mantissa bits, subnormals at exponent 0)."""
    b = np.arange(0x7F)
    e, m = b >> 3, b & 7
    return np.where(e == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * 2.0 ** (e - 7.0))


def _nearest_even(values, t):
    """Index of the entry of sorted `values` nearest to each t (ties: even
    index), saturating at the ends: a brute-force search."""
    dist = np.abs(values[None, :] - t[:, None])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    idx = np.where(cand, np.arange(len(values))[None, :], 1 << 20)
    even = np.where(cand & (np.arange(len(values))[None, :] % 2 == 0), idx, 1 << 20).min(axis=1)
    return np.where(even < (1 << 20), even, idx.min(axis=1))


def _qdq_brute_force(x, g):
    """QDQ of a [1, 16*nb] row re-derived by enumeration over both grids."""
    import torch
    f = np.float32
    xb = x.reshape(-1, 16).astype(np.float32)
    e4 = _e4m3_values()
    e2 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    out = np.zeros_like(xb)
    for i, blk in enumerate(xb):
        a = np.max(np.abs(blk))
        t = f(f(a / f(6)) / f(g))
        sig = e4[min(_nearest_even(e4, np.array([float(t)]))[0], 0x7E)]
        d = f(f(sig) * f(g))
        if d == 0:
            continue
        y = (blk * f(f(1) / d)).astype(np.float32)
        mag = e2[_nearest_even(e2, np.minimum(np.abs(y).astype(np.float64), 6.0))]
        val = np.where(np.signbit(y), -mag, mag).astype(np.float32)
        deq = (val * d).astype(np.float32)
        out[i] = torch.from_numpy(deq).to(torch.bfloat16).float().numpy()
    return out.reshape(x.shape)


@pytest.mark.parametrize("g", [None, 1.0, 1.0 / 3.0, 0.0123, 2.0 ** -9])
def test_qdq_matches_brute_force_grids(g):
    x = W.activations(6, 256, 4, "t3x20", 5, 6).float().numpy()
    w, q = nvfp4.qdq(x, g=g)
    gg = q["g"]
    for r in range(x.shape[0]):
        want = _qdq_brute_force(x[r], gg)
        assert np.array_equal(w[r], want), f"row {r}"
        assert np.array_equal(np.signbit(w[r]), np.signbit(want))


@pytest.mark.parametrize("j", [-12, -4, 0, 3])
def test_qdq_idempotent_under_power_of_two_scale(j):
    g = np.float32(2.0 ** j)
    x = W.activations(8, 512, 5, "t3x20", 7, 8).float().numpy() * np.float32(2.0 ** (j + 8))
    w1, q1 = nvfp4.qdq(x, g=g)
    w2, q2 = nvfp4.qdq(w1, g=g)
    assert np.array_equal(w1, w2)
    assert np.array_equal(q1["codes"] & 7, q2["codes"] & 7) and np.array_equal(q1["sigma"], q2["sigma"])


def test_qdq_error_within_one_scale_step():
    x = W.activations(16, 1024, 10, "t3x20", 9, 10).float().numpy()
    w, q = nvfp4.qdq(x)
    d = (F.e4m3_decode(q["sigma"]) * np.float64(q["g"])).repeat(16, axis=1)
    err = np.abs(w.astype(np.float64) - x)
    # E2M1 steps are at most 2 d apart (4 -> 6): rounding moves by <= d, the
    # bf16 rounding of the product by <= 2^-9 of it
    assert np.all(err <= d * (1 + 2.0 ** -20) + np.abs(w) * 2.0 ** -9)


# A block where the two readings of "round E2M1(code) * d to bf16" differ.
# g = 1.0130208730697632 is an fp32 value (8498517 * 2^-23); a = 6 gives
# (6 / 6) / g = 0.98715 -> sigma = E4M3(0.98715) = 1, d = g.  x = 3.03125 has
# x / d = 2.9923 -> code 5 (E2M1 3).  3 d = 3.0390626192... is not an fp32
# value: fp32(3 d) = 3.0390625, exactly halfway between the bf16 neighbours
# 3.03125 (even mantissa) and 3.046875, so bf16(fp32(3 d)) = 3.03125 while
# rounding the exact product once would give 3.046875.
DOUBLE_ROUNDING_G = 1.0130208730697632
DOUBLE_ROUNDING_X = [6.0, 3.03125, -3.03125, 0.0] + [0.0] * 12


def test_qdq_rounds_the_fp32_product_to_bf16():
    g = np.float32(DOUBLE_ROUNDING_G)
    assert float(g) == DOUBLE_ROUNDING_G
    x = np.array([DOUBLE_ROUNDING_X], np.float32)
    w, q = nvfp4.qdq(x, g=g)
    assert q["sigma"][0, 0] == 0x38 and list(q["codes"][0, :3]) == [7, 5, 13]
    assert w[0, 1] == np.float32(3.03125) and w[0, 2] == np.float32(-3.03125)
    # the block maximum too: 6 d = 6.0781252384... -> fp32 6.078125, halfway
    # between bf16 6.0625 (even) and 6.09375 -> 6.0625
    assert w[0, 0] == np.float32(6.0625)


def test_grouped_scale_offsets_are_distinct_and_in_bounds():
    # every (row, scale) of an expert-sorted operand gets its own byte inside
    # the grouped buffer, each expert's rows starting on a fresh 128-row tile
    offs = np.array([0, 0, 5, 135, 136, 400, 400, 529])
    E, K = len(offs) - 1, 192
    o = nvfp4.grouped_scale_tile_offsets(offs, K // 16)
    assert o.shape == (offs[-1], K // 16)
    assert len(np.unique(o)) == o.size
    assert o.min() >= 0 and o.max() < nvfp4.grouped_scale_bytes(int(offs[-1]), K, E)
    rows = nvfp4.grouped_row_map(offs)
    for e in range(E):
        if offs[e + 1] > offs[e]:
            assert rows[offs[e]] % 128 == 0


# --- the pre-scaled residual (the GEMM's compensation operand R / g) -----

def test_prescaled_residual_power_of_two_scale_is_exact_rescaling():
    # with g = 2^j, fp32(1/g) = 2^-j exactly and the product is exact, so the
    # pre-scaled residual is the bf16 residual times 2^-j, bit for bit (the
    # values stay far from the subnormal and overflow ranges)
    x = F.bf16_round(np.random.default_rng(5).standard_normal((24, 128)).astype(np.float32) * 3)
    chan = np.arange(0, 128, 5)
    for j in (-9, -3, 0, 4, 11):
        q = nvfp4.quantize(x, g=np.float32(2.0 ** j), chan=chan)
        assert np.array_equal(q["resid_scaled"], (q["resid"] * np.float32(2.0 ** -j)).astype(np.float32))


def test_prescaled_residual_within_one_bf16_rounding_of_the_quotient():
    # any g: |resid_scaled - R/g| <= 2^-8 |R/g| (one bf16 rounding, plus the
    # fp32 reciprocal's and product's 2^-24-level errors); the dynamic scale
    # of a workload, and a planted mistake (R * g) must fail the bound
    x = W.activations(64, 512, 5, "t3x20", 1, 2).float().numpy()
    chan = np.arange(1, 512, 7)
    q = nvfp4.quantize(x, chan=chan)
    exact = q["resid_f32"][:, chan].astype(np.float64) / np.float64(q["g"])
    err = np.abs(q["resid_scaled"] - exact)
    assert np.all(err <= 2.0 ** -8 * np.abs(exact) + 1e-45)
    wrong = q["resid"] * np.float64(q["g"])
    assert not np.all(np.abs(wrong - exact) <= 2.0 ** -8 * np.abs(exact) + 1e-45)


def test_prescaled_residual_grouped_matches_dense_rows():
    # grouped: each expert's rows take that expert's channels, same rule
    x = W.activations(40, 256, 3, "t3x20", 3, 4).float().numpy()
    offs = np.array([0, 10, 10, 31, 40])
    chan = np.array([[0, 16, 100, 255], [1, 2, 3, 4], [5, 50, 150, 250], [7, 8, 9, 200]])
    qg = nvfp4.quantize_grouped(x, offs, chan)
    qd = nvfp4.quantize(x)
    rg = nvfp4.reciprocal(qd["g"])
    for e in range(4):
        lo, hi = offs[e], offs[e + 1]
        want = np.asarray(torch_free_bf16(qd["resid_f32"][lo:hi][:, chan[e]] * rg))
        assert np.array_equal(qg["resid_scaled"][lo:hi], want)


def torch_free_bf16(v):
    """bf16 round-to-nearest-even of float32 values by bit arithmetic (an
    independent restatement of the rounding, not the library routine)."""
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)
