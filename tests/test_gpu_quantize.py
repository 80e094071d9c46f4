"""GPU parity of the quantizers against the oracle: codes, scale bytes and the
bf16 residual must be bit-exact; MXFP4 decomposition statistics within
fp32-vs-fp64 rounding, deadzone counts exact."""

import json
import os

import numpy as np
import pytest
import torch

from oracle import calib, mxfp4 as omx, nvfp4 as onv, formats as F
from nvfp4_w4a4_gemm_gb300 import workloads as W
from tests.helpers import bf16_bits_of, f32, gather_scales, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from nvfp4_w4a4_gemm_gb300 import binding
    binding.load()
    return binding


def _check_nvfp4(nv, x_cpu, chan=None, g=None, resid_scaled=False):
    x = x_cpu.cuda()
    ch = None if chan is None else torch.as_tensor(chan, dtype=torch.int32).cuda()
    gt = None if g is None else torch.tensor([g], dtype=torch.float32).cuda()
    q = nv.nvfp4_quantize(x, g=gt, chan=ch, resid_scaled=resid_scaled)
    torch.cuda.synchronize()
    ref = onv.quantize(f32(x_cpu), g=g, chan=chan)
    M, K = x_cpu.shape
    assert f32(q["g"])[0] == ref["g"]
    assert np.array_equal(u8(q["codes"]), ref["packed"]), "codes differ"
    sc = gather_scales(q["scales"], onv.scale_tile_offsets(M, K // 16))
    assert np.array_equal(sc, ref["sigma"]), "scale bytes differ"
    if chan is not None and len(chan):
        want = F.bf16_bits(ref["resid_scaled"] if resid_scaled else ref["resid_f32"][:, np.asarray(chan)])
        assert np.array_equal(bf16_bits_of(q["resid"]), want), "residual differs"
    return q, ref


@pytest.mark.parametrize("idx", [0, 1])
def test_worked_examples(nv, golden_dir, idx):
    with open(os.path.join(golden_dir, "nvfp4_worked.json")) as f:
        ex = json.load(f)["examples"][idx]
    x = torch.tensor([ex["x"]], dtype=torch.float32).to(torch.bfloat16)
    q, _ = _check_nvfp4(nv, x, chan=ex["chan"])
    assert list(u8(q["codes"])[0][: len(ex["codes"]) // 2]) == list(onv.pack(np.array(ex["codes"])))
    np.testing.assert_array_equal(f32(q["resid"])[0], np.array(ex["resid"], np.float32))


def test_tiny_workload(nv):
    d = W.dense_inputs("tiny")
    chan = calib.calibrate(W.dense_inputs("tiny", True, False)["x"].float().numpy(), 8)
    _check_nvfp4(nv, d["x"], chan=chan)
    _check_nvfp4(nv, d["wt"])


@pytest.mark.parametrize("M,K,k", [(1, 16, 1), (3, 48, 5), (130, 80, 7), (257, 1040, 33), (64, 4096, 128),
                                   (517, 2064, 64),
                                   # decode-sized inputs (a few CTAs: the grid barrier over few arrivals)
                                   (16, 4096, 64), (31, 2000, 8), (65, 1024, 16), (8, 8192, 32)])
def test_ragged_shapes(nv, M, K, k):
    x = W.activations(M, K, max(1, K // 100), "t3x20", M + K, M * 7 + 1)
    rng = np.random.default_rng(M * 31 + K)
    chan = np.sort(rng.choice(K, size=k, replace=False))
    _check_nvfp4(nv, x, chan=chan)


@pytest.mark.parametrize("M,K,k,g", [(130, 80, 7, None), (257, 1040, 33, None), (517, 2064, 64, None),
                                     (16, 4096, 64, None), (64, 4096, 128, 0.0123), (300, 512, 32, 2.0 ** -7)])
def test_prescaled_residual(nv, M, K, k, g):
    # the residual divided by the tensor scale, bit-exact with the oracle's
    # bf16(fp32(x - deq) * fp32(1/g)); codes and scales unchanged
    x = W.activations(M, K, max(1, K // 100), "t3x20", M + 3 * K, M + 5)
    rng = np.random.default_rng(M * 3 + K)
    chan = np.sort(rng.choice(K, size=k, replace=False))
    _check_nvfp4(nv, x, chan=chan, g=g, resid_scaled=True)


def test_static_scale_and_g_out(nv):
    x = W.random_bf16((40, 96), 3, scale=2.0)
    _check_nvfp4(nv, x, chan=[0, 95], g=0.0123)


def test_edge_blocks(nv):
    # zero blocks, all-equal blocks, +-6 saturation, subnormal-scale and
    # zero-scale blocks, negative values rounding to zero.
    rows = []
    rows.append([0.0] * 64)
    rows.append([1.5] * 64)
    rows.append([2688.0] + [-2688.0] * 15 + [3.0] * 16 + [1e-3] * 16 + [-1e-6, 1e-6] * 8)
    rows.append([1e-5 * (i - 32) for i in range(64)])
    rows.append([-0.01] * 16 + [600.0] + [0.0] * 15 + [7.9] * 16 + [-100.0] + [0.1] * 15)
    x = torch.tensor(rows, dtype=torch.float32).to(torch.bfloat16)
    _check_nvfp4(nv, x, chan=list(range(0, 64, 3)))


def test_exhaustive_e2m1_rounding_of_bf16(nv):
    # With g = 1 and one 6.0 per block, sigma = 1 and d = 1, so code = E2M1(x)
    # exactly: every bf16 value in [-6, 6] goes through the GPU conversion.
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = F.bf16_from_bits(bits)
    v = v[np.isfinite(v) & (np.abs(v) <= 6.0)]
    per = 15
    nb = -(-len(v) // per)
    flat = np.zeros(nb * per, np.float32)
    flat[: len(v)] = v
    body = np.zeros((nb, 16), np.float32)
    body[:, 0] = 6.0
    body[:, 1:] = flat.reshape(nb, per)
    head = np.zeros((1, 16), np.float32)
    head[0, 0] = 2688.0                      # tensor amax -> g = 1
    pad = np.zeros(((-(nb + 1)) % 16, 16), np.float32)
    pad[:, 0] = 6.0
    x = np.concatenate([head, body, pad]).reshape(-1, 256)
    _check_nvfp4(nv, torch.from_numpy(x).to(torch.bfloat16))


def test_exhaustive_e4m3_block_scales_of_bf16(nv):
    # every positive bf16 block maximum up to 2688 with g = 1
    bits = np.arange(1, 0x7F80, dtype=np.uint32).astype(np.uint16)
    a = F.bf16_from_bits(bits)
    a = a[(a > 0) & (a <= 2688.0)]
    n = -(-len(a) // 16) * 16
    col = np.zeros(n, np.float32)
    col[: len(a)] = a
    col[0] = 2688.0
    x = np.zeros((n, 16), np.float32)
    x[:, 0] = col
    x[:, 1] = col * np.float32(0.37)
    _check_nvfp4(nv, torch.from_numpy(F.bf16_round(x.reshape(-1, 64))).to(torch.bfloat16))


def _g_values():
    """Static tensor scales that stress the block-scale step: exact powers of
    two (E4M3 midpoints reached exactly), all-ones significands, thirds, the
    edges of the reciprocal-multiply range [2^-100, 2^100] and just outside
    it, and seeded random scales over 2^-40 .. 2^40."""
    fixed = [1.0, 0.125, 0.75, 2.0 ** -100, 2.0 ** -101, 2.0 ** 100, 2.0 ** 101, 2.0 ** -20, 2.0 ** 17,
             float(np.float32(1.0) / np.float32(3.0)), float(np.float32(1.0) / np.float32(2688.0))]
    ones = [float(np.array([b], np.uint32).view(np.float32)[0]) for b in (0x3F7FFFFF, 0x43FFFFFF, 0x2E7FFFFF)]
    rng = np.random.default_rng(11)
    exps = rng.integers(127 - 40, 127 + 40, 10).astype(np.uint32)
    mants = rng.integers(0, 1 << 23, 10).astype(np.uint32)
    rand = [float(v) for v in ((exps << 23) | mants).view(np.float32)]
    return fixed + ones + rand


@pytest.mark.parametrize("g", _g_values())
def test_block_scales_every_bf16_max_static_g(nv, g):
    # every positive finite bf16 value is the maximum of one block, under a
    # static tensor scale g: scale bytes and codes bit-exact with the oracle
    # (maxima whose quotient (a / 6) / g overflows fp32 are left out: the
    # scale step is defined for finite quotients only)
    bits = np.arange(1, 0x7F80, dtype=np.uint32).astype(np.uint16)
    a = F.bf16_from_bits(bits)
    a = a[np.isfinite(a) & (a > 0) & (a.astype(np.float64) / 6.0 / g < 2.0 ** 127)]
    n = -(-len(a) // 64) * 64
    col = np.zeros(n, np.float32)
    col[: len(a)] = a
    x = np.zeros((n, 16), np.float32)
    x[:, 0] = col
    x[:, 5] = -col * np.float32(0.37)
    x[:, 11] = col * np.float32(0.61)
    _check_nvfp4(nv, torch.from_numpy(F.bf16_round(x.reshape(-1, 1024))).to(torch.bfloat16), g=g)


def test_clustered_channel_set(nv):
    # whole blocks of compensated channels (16 per block, 80 slots in one
    # 1024-column unit: several passes of the warp over the unit's slots)
    # plus scattered ones; ragged row count
    rng = np.random.default_rng(21)
    M, K = 203, 2048
    chan = np.sort(np.concatenate([np.arange(32, 112), np.arange(1040, 1056), rng.choice(np.arange(1200, 2048), 24,
                                                                                         replace=False)]))
    x = W.activations(M, K, 20, "t3x20", 5, 6)
    _check_nvfp4(nv, x, chan=chan.astype(np.int32))


def test_grouped_quantize_channel_lists_without_prefix_tables(nv):
    # 100 experts x K = 4096: the per-expert channel bitmaps would not fit in
    # shared memory, so each unit finds its slots by binary search
    rng = np.random.default_rng(22)
    E, K, k = 100, 4096, 16
    sizes = rng.integers(0, 9, E)
    sizes[3] = 0
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    x = W.activations(int(offs[-1]), K, 10, "t3x20", 7, 8)
    chan = np.stack([np.sort(rng.choice(K, k, replace=False)) for _ in range(E)]).astype(np.int32)
    q = nv.nvfp4_quantize_grouped(x.cuda(), torch.from_numpy(offs).cuda(), torch.from_numpy(chan).cuda())
    torch.cuda.synchronize()
    ref = onv.quantize_grouped(f32(x), offs, chan)
    assert f32(q["g"])[0] == ref["g"]
    assert np.array_equal(u8(q["codes"]), ref["packed"])
    sc = gather_scales(q["scales"], onv.grouped_scale_tile_offsets(offs, K // 16))
    assert np.array_equal(sc, ref["sigma"])
    assert np.array_equal(bf16_bits_of(q["resid"]), F.bf16_bits(ref["resid"]))


def test_grouped_quantize_prescaled_residual(nv):
    rng = np.random.default_rng(23)
    E, K, k = 9, 1024, 24
    sizes = rng.integers(0, 150, E)
    sizes[2] = 0
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    x = W.activations(int(offs[-1]), K, 10, "t3x20", 17, 18)
    chan = np.stack([np.sort(rng.choice(K, k, replace=False)) for _ in range(E)]).astype(np.int32)
    q = nv.nvfp4_quantize_grouped(x.cuda(), torch.from_numpy(offs).cuda(), torch.from_numpy(chan).cuda(),
                                  resid_scaled=True)
    torch.cuda.synchronize()
    ref = onv.quantize_grouped(f32(x), offs, chan)
    assert f32(q["g"])[0] == ref["g"]
    assert np.array_equal(u8(q["codes"]), ref["packed"])
    assert np.array_equal(bf16_bits_of(q["resid"]), F.bf16_bits(ref["resid_scaled"]))


def test_grouped_quantize(nv):
    d = W.moe_inputs(with_weights=False, which=("gate_up",))
    offs = d["offsets"].numpy()
    E = int(np.searchsorted(offs, 3000, side="right")) - 1   # experts fully below row 3000
    offs_c = offs[: E + 1].astype(np.int32)
    x = d["x_gate_up"][: int(offs_c[-1])]
    rng = np.random.default_rng(0)
    chan = np.stack([np.sort(rng.choice(2048, 32, replace=False)) for _ in range(E)]).astype(np.int32)
    q = nv.nvfp4_quantize_grouped(x.cuda(), torch.from_numpy(offs_c).cuda(), torch.from_numpy(chan).cuda())
    torch.cuda.synchronize()
    ref = onv.quantize_grouped(f32(x), offs_c, chan)
    assert f32(q["g"])[0] == ref["g"]
    assert np.array_equal(u8(q["codes"]), ref["packed"])
    sc = gather_scales(q["scales"], onv.grouped_scale_tile_offsets(offs_c, 2048 // 16))
    assert np.array_equal(sc, ref["sigma"])
    assert np.array_equal(bf16_bits_of(q["resid"]), F.bf16_bits(ref["resid"]))


def _check_gather(nv, xt, tok, offs, chan, g=None, resid_scaled=False):
    """The routed quantize read through the row table against the oracle on
    the gathered rows (the test gathers them on the CPU)."""
    K = xt.shape[1]
    gt = None if g is None else torch.tensor([g], dtype=torch.float32).cuda()
    q = nv.nvfp4_quantize_grouped_gather(xt.cuda(), torch.from_numpy(tok).cuda(), torch.from_numpy(offs).cuda(),
                                         torch.from_numpy(chan).cuda(), g=gt, resid_scaled=resid_scaled)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    ref = onv.quantize_grouped(f32(xt)[tok], offs, chan, g=g)
    assert f32(q["g"])[0] == ref["g"]
    assert np.array_equal(u8(q["codes"]), ref["packed"]), "codes differ"
    sc = gather_scales(q["scales"], onv.grouped_scale_tile_offsets(offs, K // 16))
    assert np.array_equal(sc, ref["sigma"]), "scale bytes differ"
    want = ref["resid_scaled"] if resid_scaled else ref["resid"]
    assert np.array_equal(bf16_bits_of(q["resid"]), F.bf16_bits(want)), "residual differs"
    return q


@pytest.mark.parametrize("resid_scaled", [False, True])
def test_grouped_gather_quantize(nv, resid_scaled):
    # the MoE workload's routing on its first experts, read from all 4096 token rows
    d = W.moe_inputs(with_weights=False, which=("gate_up",))
    offs = d["offsets"].numpy()
    E = int(np.searchsorted(offs, 2500, side="right")) - 1
    offs_c = offs[: E + 1].astype(np.int32)
    tok = d["token_of_row"].numpy()[: int(offs_c[-1])].astype(np.int32)
    rng = np.random.default_rng(5)
    chan = np.stack([np.sort(rng.choice(2048, 32, replace=False)) for _ in range(E)]).astype(np.int32)
    q = _check_gather(nv, d["x_tokens"], tok, offs_c, chan, resid_scaled=resid_scaled)
    # bit-identical to the grouped quantizer on the materialized rows
    qm = nv.nvfp4_quantize_grouped(d["x_tokens"][tok].cuda(), torch.from_numpy(offs_c).cuda(),
                                   torch.from_numpy(chan).cuda(), resid_scaled=resid_scaled)
    for key in ("g", "codes", "resid"):
        assert torch.equal(q[key], qm[key]), key
    # the scale bytes of the rows (the padding rows between experts are not written)
    tiles = onv.grouped_scale_tile_offsets(offs_c, 2048 // 16)
    assert np.array_equal(gather_scales(q["scales"], tiles), gather_scales(qm["scales"], tiles))


@pytest.mark.parametrize("K,static", [(160, False), (1056, True), (3072, False)])
def test_grouped_gather_ragged(nv, K, static):
    # rows past the last full 1024-column group, repeated and unused tokens,
    # empty experts, experts of one row, a static tensor scale
    rng = np.random.default_rng(K)
    T, E, k = 37, 7, 8
    sizes = np.array([5, 0, 1, 130, 0, 19, 3])
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    tok = rng.integers(0, T - 3, int(offs[-1])).astype(np.int32)  # the last three tokens never routed
    tok[:4] = 0
    xt = W.activations(T, K, 3, "t3x20", K + 1, K + 2)
    xt[T - 1, 5] = 1000.0  # an unrouted outlier must not enter the dynamic scale
    chan = np.stack([np.sort(rng.choice(K, k, replace=False)) for _ in range(E)]).astype(np.int32)
    g = 0.75 * onv.tensor_scale(f32(xt)[tok]) if static else None
    _check_gather(nv, xt, tok, offs, chan, g=g, resid_scaled=static)


@pytest.mark.parametrize("M,K", [(64, 256), (33, 160), (256, 5120)])
def test_mxfp4_quantize_and_decomposition(nv, M, K):
    x = W.activations(M, K, max(1, K // 100), "t3x20", K, M + 3)
    q = nv.mxfp4_quantize(x.cuda(), stats=True)
    torch.cuda.synchronize()
    st, cnt, d = omx.block_stats(f32(x))
    assert np.array_equal(u8(q["codes"]), d["packed"])
    sc = gather_scales(q["scales"], onv.scale_tile_offsets(M, K // 32))
    assert np.array_equal(sc, d["scale"])
    assert np.array_equal(u8(q["dead"]).reshape(M, K // 32), cnt)
    g = f32(q["stats"]).reshape(M, K // 32, 4).astype(np.float64)
    # fp32 kernel vs fp64 oracle: per-block relative 1e-5 of the block's
    # total error energy (the components' products of s* round in fp32)
    tol = 1e-5 * (st[..., 3:4] + st.sum(-1, keepdims=True)) + 1e-30
    assert np.all(np.abs(g - st) <= tol)


def _mx_midpoint_blocks():
    """32-element blocks whose elements sit on (or next to) the E2M1 rounding
    midpoints at the ideal scale s* = a/6: exact s* (a = 6 * 2^k, 6 * 1.5 * 2^k)
    puts x/s* exactly on 0.25, 0.75, ... 5 (ties to even), inexact s*
    (a = 7 * 2^k) puts it within rounding noise of them, and bf16 neighbours of
    the midpoint elements land just off them."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    rows = []
    for amax in (6.0, 9.0, 7.0, 6.0 * 2.0 ** -9, 9.0 * 2.0 ** 11, 7.0 * 2.0 ** -20):
        s_star = amax / 6.0
        for sign in (1.0, -1.0):
            v = np.zeros(32)
            v[0] = amax
            v[1:8] = sign * mids * s_star
            v[8:15] = sign * mids * s_star
            rows.append(v)
    x = F.bf16_round(np.stack(rows).astype(np.float32))
    # bf16 neighbours of elements 8..14 (one step up / down in the bit pattern)
    up, dn = x.copy(), x.copy()
    b = F.bf16_bits(x[:, 8:15]).astype(np.int32)
    up[:, 8:15] = F.bf16_from_bits((b + 1).astype(np.uint16))
    dn[:, 8:15] = F.bf16_from_bits((b - 1).astype(np.uint16))
    return np.concatenate([x, up, dn]).reshape(-1, 128)


def _check_elementwise(nv, x):
    """Per-element (B, D, G) of the GPU against the oracle's fp64 components:
    each within fp32 rounding of the block's scale, D and G on the same
    elements, and B + D + G equal to the oracle's E."""
    M, K = x.shape
    bdg = f32(nv.mxfp4_decompose_elements(x.cuda())).astype(np.float64)
    torch.cuda.synchronize()
    d = omx.decompose(f32(x))
    blk = np.abs(f32(x)).reshape(M, K // 32, 32).max(axis=2).repeat(32, axis=1).astype(np.float64)
    tol = blk * 2.0 ** -20 + 1e-38
    for i, name in enumerate(("B", "D", "G")):
        assert np.all(np.abs(bdg[..., i] - d[name]) <= tol), name
    dead_at_star = (d["D"] != 0) | d["dead"]
    assert not np.any((bdg[..., 2] != 0) & dead_at_star), "grid noise on a deadzone element"
    assert not np.any((bdg[..., 1] != 0) & ~dead_at_star), "deadzone error on a non-deadzone element"
    assert np.all(np.abs(bdg.sum(-1) - d["E"]) <= 3 * tol)


@pytest.mark.parametrize("M,K", [(64, 256), (33, 160), (8, 1024)])
def test_mxfp4_decomposition_per_element(nv, M, K):
    x = W.activations(M, K, max(1, K // 100), "t3x20", K + 11, M + 13).clone()
    x[0, :32] = 0                                   # zero block: all components 0
    x[1, :32] = torch.tensor([3.0] + [0.01] * 31)   # mostly deadzone at s* = 0.5
    x[2, :32] = torch.tensor([6.0 * 2.0 ** 3] * 32)  # a = 6 * 2^k: no scale bias
    _check_elementwise(nv, x)


def test_mxfp4_decomposition_per_element_at_midpoints(nv):
    x = torch.from_numpy(_mx_midpoint_blocks().astype(np.float32)).to(torch.bfloat16)
    _check_elementwise(nv, x)


def test_mxfp4_ideal_scale_codes_at_midpoints(nv):
    x = torch.from_numpy(_mx_midpoint_blocks()).to(torch.bfloat16)
    M, K = x.shape
    q = nv.mxfp4_quantize(x.cuda(), stats=True)
    torch.cuda.synchronize()
    st, cnt, d = omx.block_stats(f32(x))
    assert np.array_equal(u8(q["codes"]), d["packed"])
    assert np.array_equal(gather_scales(q["scales"], onv.scale_tile_offsets(M, K // 32)), d["scale"])
    assert np.array_equal(u8(q["dead"]).reshape(M, K // 32), cnt)
    assert cnt.sum() > 0  # the 0.25 midpoints tie to code 0
    g = f32(q["stats"]).reshape(M, K // 32, 4).astype(np.float64)
    tol = 1e-5 * (st[..., 3:4] + st.sum(-1, keepdims=True)) + 1e-30
    assert np.all(np.abs(g - st) <= tol)


def test_comp_weights_both_modes(nv):
    wt = W.weights_t(256, 512, 11)
    qw = nv.nvfp4_quantize(wt.cuda())
    chan = torch.tensor([0, 15, 16, 100, 511], dtype=torch.int32).cuda()
    ws = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], chan)
    wb = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], chan, flags=nv.COMP_W_BF16, wt=wt.cuda())
    torch.cuda.synchronize()
    ref = onv.quantize(f32(wt))
    want = onv.comp_weights(ref["codes"], ref["sigma"], chan.cpu().numpy())
    assert np.array_equal(f32(ws).astype(np.float64), want)
    assert np.array_equal(f32(wb), f32(wt)[:, chan.cpu().numpy()])


def test_calibration_selects_like_oracle(nv):
    for name in ("tiny", "decode"):
        xc = W.dense_inputs(name, calibration=True, with_weights=False)["x"]
        k = W.SPECS[name].k
        got = nv.nvfp4_calibrate_channels(xc.cuda(), k).cpu().numpy()
        want = calib.calibrate(f32(xc), k)
        if not np.array_equal(np.sort(got), want):
            # only near-ties at the boundary may differ (fp64 summation order)
            var = calib.channel_variance(onv.quantize(f32(xc))["resid_f32"])
            diff = set(got.tolist()) ^ set(want.tolist())
            kth = np.sort(var)[::-1][k - 1]
            assert all(abs(var[j] - kth) <= 1e-9 * kth for j in diff)


def _same_up_to_near_ties(got, want, var, k):
    """The selected sets agree except for channels whose variance ties the
    k-th largest within fp64 summation-order noise."""
    if np.array_equal(np.sort(got), want):
        return True
    diff = set(np.asarray(got).tolist()) ^ set(np.asarray(want).tolist())
    kth = np.sort(var)[::-1][k - 1]
    return all(abs(var[j] - kth) <= 1e-9 * kth for j in diff)


@pytest.mark.parametrize("which", ["gate_up", "down"])
def test_grouped_calibration_selects_like_oracle(nv, which):
    # per-expert channel sets of the MoE calibration batch: residual variance
    # over each expert's routed rows (experts with < 2 rows use all rows)
    s = W.SPECS["moe"]
    d = W.moe_inputs(calibration=True, with_weights=False, which=(which,))
    x = d["x_gate_up"] if which == "gate_up" else d["x_down"]
    offs = d["offsets"].numpy().astype(np.int64)
    got = nv.nvfp4_calibrate_channels(x.cuda(), s.k, offsets=d["offsets"].cuda()).cpu().numpy()
    want = calib.calibrate_grouped(f32(x), offs, s.k)
    rf = onv.quantize(f32(x))["resid_f32"]
    var_all = calib.channel_variance(rf)
    for e in range(s.experts):
        lo, hi = offs[e], offs[e + 1]
        var = calib.channel_variance(rf[lo:hi]) if hi - lo >= 2 else var_all
        assert np.all(np.diff(got[e]) > 0), f"expert {e}: set not sorted / unique"
        assert _same_up_to_near_ties(got[e], want[e], var, s.k), f"expert {e}"


def test_grouped_calibration_small_experts_use_all_rows(nv):
    # experts with 0 and 1 calibration rows take the all-row statistics
    x = W.activations(40, 256, 3, "t3x20", 51, 52)
    offs = np.array([0, 0, 1, 20, 40], np.int32)
    k = 16
    got = nv.nvfp4_calibrate_channels(x.cuda(), k, offsets=torch.from_numpy(offs).cuda()).cpu().numpy()
    want = calib.calibrate_grouped(f32(x), offs, k)
    rf = onv.quantize(f32(x))["resid_f32"]
    var_all = calib.channel_variance(rf)
    assert _same_up_to_near_ties(got[0], want[0], var_all, k)
    assert _same_up_to_near_ties(got[1], want[1], var_all, k)
    assert np.array_equal(np.sort(got[0]), np.sort(got[1]))

