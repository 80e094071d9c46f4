"""Pins of the oracle's element encodings (CPU only)."""

import numpy as np
import torch

from oracle import formats as F


def test_e2m1_grid_is_the_eight_levels():
    # QUADS abstract: "coarse E2M1 grid"; gist.science explainer of QUADS,
    # Technisches Resuemee section 1: 8 non-negative levels per sign.
    grid = F.e2m1_value(np.arange(8))
    assert list(grid) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(F.e2m1_value(np.arange(8, 16))) == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    assert len(set(np.abs(F.e2m1_value(np.arange(16))))) == 8


def test_e2m1_ties_go_to_even_code():
    # half-way points between neighbours -> the even code
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for y, c in ties.items():
        assert F.e2m1_encode(np.float32(y)) == c, y
        assert F.e2m1_encode(np.float32(-y)) == c | 8, -y


def test_e2m1_against_midpoint_thresholds_all_bf16():
    # independent derivation: RNE onto the grid == comparison against the 7
    # midpoints, where a value exactly on a midpoint goes up only if the
    # upper neighbour's code is even.  Checked on every finite bf16 number.
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = F.bf16_from_bits(bits)
    v = v[np.isfinite(v)]
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    up_on_tie = [False, True, False, True, False, True, False]  # upper code 1,2,3,4,5,6,7
    mag = np.abs(v.astype(np.float64))
    want = np.zeros(mag.shape, np.int64)
    for m, up in zip(mids, up_on_tie):
        want += (mag > m) | ((mag == m) & up)
    want = want | (np.signbit(v).astype(np.int64) << 3)
    got = F.e2m1_encode(v)
    assert np.array_equal(got, want)


def test_e2m1_saturates():
    assert F.e2m1_encode(np.float32(7.9)) == 7
    assert F.e2m1_encode(np.float32(1e30)) == 7
    assert F.e2m1_encode(np.float32(-100)) == 15


def test_e4m3_table_endpoints():
    v = F.E4M3_VALUES
    assert v[0] == 0 and v[1] == 2.0 ** -9 and v[8] == 2.0 ** -6
    assert v[0x7E] == 448.0 and len(v) == 127
    assert np.all(np.diff(v) > 0)


def test_e4m3_encode_matches_torch_in_range():
    # library routine pin: torch's float32 -> float8_e4m3fn conversion is
    # round-to-nearest-even; compare on a dense sweep of [0, 448] including
    # every exact half-way point between neighbours.
    vals = F.E4M3_VALUES
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(0)
    sweep = np.concatenate([vals, mids, rng.uniform(0, 448, 200000),
                            np.exp(rng.uniform(np.log(1e-6), np.log(448), 200000))])
    sweep = sweep.astype(np.float32)
    got = F.e4m3_encode(sweep)
    want = torch.from_numpy(sweep).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


def test_e4m3_saturates():
    assert F.e4m3_encode(np.float32(448.0)) == 0x7E
    assert F.e4m3_encode(np.float32(470.0)) == 0x7E
    assert F.e4m3_encode(np.float32(1e9)) == 0x7E
    assert F.e4m3_encode(np.float32(2.0 ** -10)) == 0   # tie 0 / 2^-9 -> even (0)
    assert F.e4m3_encode(np.float32(1.5 * 2.0 ** -10)) == 1


def test_e8m0_powers_of_two():
    assert F.e8m0_value(127) == 1.0
    assert F.e8m0_value(0) == 2.0 ** -127
    assert F.e8m0_value(254) == 2.0 ** 127


def test_bf16_roundtrip():
    x = np.array([0.1, 1.0, 3.14159, -2.5e-3], np.float32)
    b = F.bf16_round(x)
    assert np.array_equal(F.bf16_from_bits(F.bf16_bits(x)), b)
    assert b[1] == 1.0 and abs(b[0] - 0.1) < 0.1 * 2 ** -8
