"""Pins of the oracle's MoE pieces (CPU only): the gated activation, the
routing weights, the weighted combine and the gate/up row interleave."""

import math

import numpy as np

from oracle import moe
from oracle.formats import bf16_round
from nvfp4_w4a4_gemm_gb300 import workloads as W


def test_silu_closed_forms():
    z = np.array([0.0, 1.0, -1.0, 2.0, 40.0, -40.0])
    want = [0.0, 1 / (1 + math.e ** -1), -1 / (1 + math.e), 2 / (1 + math.e ** -2), 40.0, -40 * math.exp(-40)]
    np.testing.assert_allclose(moe.silu(z), want, rtol=1e-15, atol=1e-300)
    # silu(z) - silu(-z) = z for every z (z * (s(z) + s(-z) - 1) ... with s(z) + s(-z) = 1)
    r = np.random.default_rng(0).standard_normal(1000) * 8
    np.testing.assert_allclose(moe.silu(r) - moe.silu(-r), r, rtol=1e-13, atol=1e-13)


def test_swiglu_with_unit_up_is_rounded_silu_and_is_linear_in_up():
    a = bf16_round(np.random.default_rng(1).standard_normal((8, 64)).astype(np.float32) * 3)
    ones = np.ones_like(a)
    assert np.array_equal(moe.swiglu(a, ones), bf16_round(moe.silu(a).astype(np.float32)))
    assert np.array_equal(moe.swiglu(a, 2 * ones), 2 * moe.swiglu(a, ones))     # power-of-two scaling is exact
    assert np.array_equal(moe.swiglu(a, -ones), -moe.swiglu(a, ones))


def test_route_weights_renormalized_top8_and_ties():
    rng = np.random.default_rng(2)
    lg = rng.standard_normal((50, 128))
    ex, w = moe.route_weights(lg, 8)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)
    assert np.all(np.diff(w, axis=1) <= 1e-15)                 # descending
    for t in range(50):                                         # the 8 largest logits
        assert set(ex[t]) == set(np.argsort(-lg[t], kind="stable")[:8])
    ex, w = moe.route_weights(np.zeros((3, 128)), 8)           # all tied -> experts 0..7, uniform
    assert np.array_equal(ex, np.tile(np.arange(8), (3, 1)))
    np.testing.assert_allclose(w, 1 / 8, rtol=0, atol=1e-15)


def test_workload_routing_matches_oracle_experts_and_weights():
    s = W.SPECS["moe"]
    tok, offs, w_rows, logits = W.route(256, s.experts, s.top, 11, with_weights=True)
    ex, w = moe.route_weights(logits.numpy(), s.top)
    want = moe.row_weights(ex, w, tok.numpy(), offs.numpy())
    np.testing.assert_allclose(w_rows.numpy(), want, rtol=2e-6, atol=0)   # fp32 draw vs fp64 oracle


def test_combine_reduces_to_a_permutation_for_one_expert_per_token():
    rng = np.random.default_rng(3)
    T, N = 20, 7
    perm = rng.permutation(T)
    y = rng.standard_normal((T, N))
    out = moe.combine(y, perm, np.ones(T), T)
    assert np.array_equal(out[perm], y)


def test_combine_of_identical_rows_with_normalized_weights_is_the_row():
    rng = np.random.default_rng(4)
    lg = rng.standard_normal((6, 16))
    ex, w = moe.route_weights(lg, 4)
    tok = np.repeat(np.arange(6), 4)
    order = np.lexsort((tok, ex.reshape(-1)))
    tok_sorted = tok[order]
    counts = np.bincount(ex.reshape(-1), minlength=16)
    offs = np.concatenate([[0], np.cumsum(counts)])
    w_rows = moe.row_weights(ex, w, tok_sorted, offs)
    row = rng.standard_normal(5)
    out = moe.combine(np.tile(row, (24, 1)), tok_sorted, w_rows, 6)
    np.testing.assert_allclose(out, np.tile(row, (6, 1)), rtol=1e-14, atol=1e-14)


def test_interleave_gate_up_layout():
    inter, K = 384, 8
    wt = np.arange(2 * inter)[:, None] * np.ones((1, K))
    p, perm = moe.interleave_gate_up(wt)
    assert np.array_equal(np.sort(perm), np.arange(2 * inter))
    for j in range(inter // 128):
        assert np.array_equal(perm[256 * j: 256 * j + 128], np.arange(128 * j, 128 * j + 128))
        assert np.array_equal(perm[256 * j + 128: 256 * j + 256], inter + np.arange(128 * j, 128 * j + 128))
    assert np.array_equal(p[:, 0], perm)
