"""GPU parity of the W4A4 GEMM with compensation against the fp64 oracle.
Tolerance (problem statement): |y - y_ref| <= 4e-3 |y_ref| + 1e-3 rms(Y_ref)
elementwise, y_ref the fp64 product of the same dequantized operands."""

import numpy as np
import pytest
import torch

from oracle import gemm as og, mxfp4 as omx, nvfp4 as onv
from nvfp4_w4a4_gemm_gb300 import workloads as W
from tests.helpers import f32, gemm_within_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from nvfp4_w4a4_gemm_gb300 import binding
    binding.load()
    return binding


def _dense_case(nv, x, wt, chan, flags=0, resid_scaled=False):
    """Run quantize(X) + quantize(W^T) + comp weights + GEMM on the GPU and
    the oracle on the same inputs; returns (y_gpu fp64, y_ref fp64).
    resid_scaled: the quantizer emits the residual divided by g_x and the GEMM
    consumes it as such (the reference keeps the plain bf16 residual: the two
    differ by one bf16 rounding of the compensation operand)."""
    N = wt.shape[0]
    ch = torch.as_tensor(np.asarray(chan), dtype=torch.int32).cuda() if len(chan) else None
    qx = nv.nvfp4_quantize(x.cuda(), chan=ch, resid_scaled=resid_scaled)
    qw = nv.nvfp4_quantize(wt.cuda())
    ws = None
    if len(chan):
        ws = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], ch, flags=flags,
                                           wt=wt.cuda() if flags else None)
    y = nv.w4a4_gemm_comp(qx, qw, N, resid=qx["resid"] if len(chan) else None, w_sel=ws, flags=flags)
    torch.cuda.synchronize()
    st, _ = nv.check_status()
    assert st == 0, f"device status {st}"
    y_ref, _, _ = og.linear_comp(f32(x), f32(wt), np.asarray(chan, np.int64), bf16_weights=bool(flags))
    return f32(y).astype(np.float64), y_ref


def _assert_close(y, y_ref):
    ok, ratio, rms = gemm_within_tol(y, y_ref)
    assert ok, f"max err/allowance = {ratio:.3f} (rms {rms:.4g})"


def test_tiny_workload(nv):
    from oracle import calib
    d = W.dense_inputs("tiny")
    chan = calib.calibrate(W.dense_inputs("tiny", True, False)["x"].float().numpy(), 8)
    y, y_ref = _dense_case(nv, d["x"], d["wt"], chan)
    _assert_close(y, y_ref)


@pytest.mark.parametrize("M,N,K,k", [(128, 128, 256, 0), (300, 384, 1024, 64), (77, 256, 320, 72),
                                     (1, 128, 64, 8), (513, 128, 2048, 128), (16, 640, 4096, 64),
                                     # up to 64 tokens the operands are swapped (MMA N = M rounded up to 16)
                                     (40, 256, 1024, 16), (5, 384, 512, 24), (64, 128, 768, 0), (17, 1024, 2048, 64)])
@pytest.mark.parametrize("resid_scaled", [False, True])
def test_shapes(nv, M, N, K, k, resid_scaled):
    x = W.activations(M, K, max(1, K // 100), "t3x20", K + 1, M + 2)
    wt = W.weights_t(N, K, N + K)
    rng = np.random.default_rng(M + N + K)
    chan = np.sort(rng.choice(K, size=k, replace=False))
    y, y_ref = _dense_case(nv, x, wt, chan, resid_scaled=resid_scaled)
    _assert_close(y, y_ref)


@pytest.mark.parametrize("M", [200, 700])
@pytest.mark.parametrize("resid_scaled", [False, True])
def test_bf16_weight_flag(nv, M, resid_scaled):
    # 700 rows: the 256 x 256 pair-tile kernel; 200: the 128-row kernel
    x = W.activations(M, 512, 5, "t3x20", 9, 9)
    wt = W.weights_t(256, 512, 10)
    chan = np.arange(0, 512, 8)
    y, y_ref = _dense_case(nv, x, wt, chan, flags=1, resid_scaled=resid_scaled)
    _assert_close(y, y_ref)


def test_bf16_weight_flag_swapped_operands(nv):
    x = W.activations(48, 512, 5, "t3x20", 11, 11)
    wt = W.weights_t(384, 512, 12)
    chan = np.arange(3, 512, 16)
    y, y_ref = _dense_case(nv, x, wt, chan, flags=1)
    _assert_close(y, y_ref)


def test_full_compensation_k_equals_K(nv):
    x = W.activations(64, 256, 4, "x50", 1, 1)
    wt = W.weights_t(128, 256, 2)
    y, y_ref = _dense_case(nv, x, wt, np.arange(256))
    _assert_close(y, y_ref)


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (200, 384, 640), (8192 // 16, 5120 // 10, 5120),
                                   (16, 256, 512), (33, 384, 1024)])
def test_mxfp4_gemm(nv, M, N, K):
    N = (N + 127) // 128 * 128
    x = W.activations(M, K, max(1, K // 100), "t3x20", 5, M)
    wt = W.weights_t(N, K, 6)
    qx = nv.mxfp4_quantize(x.cuda())
    qw = nv.mxfp4_quantize(wt.cuda())
    y = nv.w4a4_gemm_comp(dict(codes=qx["codes"], scales=qx["scales"]), dict(codes=qw["codes"], scales=qw["scales"]),
                          N, fmt=nv.FMT_MXFP4)
    torch.cuda.synchronize()
    ax = omx.quantize(f32(x))
    aw = omx.quantize(f32(wt))
    y_ref = og.reference(omx.dequantize(ax["codes"], ax["scale"]), omx.dequantize(aw["codes"], aw["scale"]))
    _assert_close(f32(y), y_ref)


@pytest.mark.parametrize("resid_scaled", [False, True])
def test_grouped_gemm_small(nv, resid_scaled):
    # 6 experts with ragged (and one empty) row counts
    counts = [0, 5, 130, 1, 256, 77]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M, K, N, k = int(offs[-1]), 512, 256, 32
    E = len(counts)
    x = W.activations(M, K, 5, "t3x20", 3, 4)
    wt = W.weights_t(N, K, 7, experts=E)
    rng = np.random.default_rng(1)
    chan = np.stack([np.sort(rng.choice(K, k, replace=False)) for _ in range(E)]).astype(np.int32)
    offs_t = torch.from_numpy(offs).cuda()
    chan_t = torch.from_numpy(chan).cuda()
    qx = nv.nvfp4_quantize_grouped(x.cuda(), offs_t, chan_t, resid_scaled=resid_scaled)
    # per-expert weight quantization (each expert its own tensor scale)
    codes, scales, gs = [], [], []
    for e in range(E):
        q = nv.nvfp4_quantize(wt[e].cuda())
        codes.append(q["codes"]); scales.append(q["scales"]); gs.append(q["g"])
    b_codes = torch.stack(codes)
    b_scales = torch.cat(scales)
    g_b = torch.cat(gs)
    w_sel = nv.nvfp4_prepare_comp_weights(b_codes, b_scales, chan_t, E=E)
    y = nv.w4a4_grouped_gemm_comp(qx, offs_t, b_codes, b_scales, g_b, N, resid=qx["resid"], w_sel=w_sel)
    torch.cuda.synchronize()
    st, _ = nv.check_status()
    assert st == 0
    rq = onv.quantize_grouped(f32(x), offs, chan)
    a = onv.dequantize(rq["codes"], rq["sigma"], rq["g"])
    bq = [onv.quantize(f32(wt[e])) for e in range(E)]
    b = np.stack([onv.dequantize(q["codes"], q["sigma"], q["g"]) for q in bq])
    ws = np.stack([og.comp_weight_rows(bq[e], chan[e]) for e in range(E)])
    y_ref = og.grouped_reference(a, offs, b, rq["resid"], ws)
    _assert_close(f32(y), y_ref)


@pytest.mark.parametrize("bf16_w,resid_scaled", [(False, False), (False, True), (True, False), (True, True)])
def test_grouped_gemm_pair_tiles(nv, bf16_w, resid_scaled):
    # experts averaging >= 192 rows take 256-row tiles on CTA pairs: empty,
    # one-row, exactly-one-tile and one-past-a-tile experts, a ragged last
    # 256-column tile (N % 256 = 128), a partial last k-tile (K % 256 = 64),
    # a partial compensation tile (k = 72), per-expert weight scales
    counts = [300, 0, 128, 257, 1, 513, 255, 129]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M, K, N, k = int(offs[-1]), 576, 384, 72
    E = len(counts)
    assert M >= 192 * E
    x = W.activations(M, K, 5, "t3x20", 13, 14)
    wt = W.weights_t(N, K, 15, experts=E)
    rng = np.random.default_rng(11)
    chan = np.stack([np.sort(rng.choice(K, k, replace=False)) for _ in range(E)]).astype(np.int32)
    offs_t = torch.from_numpy(offs).cuda()
    chan_t = torch.from_numpy(chan).cuda()
    qs = [nv.nvfp4_quantize(wt[e].cuda()) for e in range(E)]
    b_codes = torch.stack([q["codes"] for q in qs])
    b_scales = torch.cat([q["scales"] for q in qs])
    g_b = torch.cat([q["g"] for q in qs])
    if bf16_w:
        w_sel = nv.nvfp4_prepare_comp_weights(b_codes, b_scales, chan_t, flags=nv.COMP_W_BF16, wt=wt.cuda(), E=E)
        flags = nv.COMP_W_BF16
    else:
        w_sel = nv.nvfp4_prepare_comp_weights(b_codes, b_scales, chan_t, E=E)
        flags = nv.COMP_W_DEQ
    xd = x.cuda()
    torch.cuda.synchronize()
    ys = []
    for ready in (False, True):
        qx = nv.nvfp4_quantize_grouped(xd, offs_t, chan_t, resid_scaled=resid_scaled)
        ys.append(nv.w4a4_grouped_gemm_comp(qx, offs_t, b_codes, b_scales, g_b, N, resid=qx["resid"], w_sel=w_sel,
                                            flags=flags, weights_ready=ready))
    torch.cuda.synchronize()
    st, _ = nv.check_status()
    assert st == 0
    assert torch.equal(ys[0], ys[1])
    rq = onv.quantize_grouped(f32(x), offs, chan)
    a = onv.dequantize(rq["codes"], rq["sigma"], rq["g"])
    bq = [onv.quantize(f32(wt[e])) for e in range(E)]
    b = np.stack([onv.dequantize(q["codes"], q["sigma"], q["g"]) for q in bq])
    ws = np.stack([og.comp_weight_rows(bq[e], chan[e], f32(wt[e]) if bf16_w else None) for e in range(E)])
    y_ref = og.grouped_reference(a, offs, b, rq["resid"], ws)
    _assert_close(f32(ys[0]), y_ref)


@pytest.mark.parametrize("M,N,K,k", [(16, 1024, 4096, 64), (200, 384, 1024, 32), (600, 512, 2048, 128)])
def test_weights_ready_overlap_is_bit_identical(nv, M, N, K, k):
    """The GEMM starts while the activation quantizer before it still runs
    (programmatic dependent launch).  With the weights-ready flag it also
    streams weight tiles before waiting for that quantizer: the output must be
    bit-identical to the default order, and within tolerance of the oracle."""
    x = W.activations(M, K, max(1, K // 100), "t3x20", 21, 22)
    wt = W.weights_t(N, K, 23)
    ch = torch.arange(0, K, K // k, dtype=torch.int32)[:k].cuda().contiguous()
    qw = nv.nvfp4_quantize(wt.cuda())
    ws = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], ch)
    xd = x.cuda()
    torch.cuda.synchronize()
    ys = []
    for ready in (False, True, True):
        qx = nv.nvfp4_quantize(xd, chan=ch)  # the kernel just before the GEMM
        ys.append(nv.w4a4_gemm_comp(qx, qw, N, resid=qx["resid"], w_sel=ws, weights_ready=ready))
    torch.cuda.synchronize()
    st, _ = nv.check_status()
    assert st == 0
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])
    y_ref, _, _ = og.linear_comp(f32(x), f32(wt), ch.cpu().numpy().astype(np.int64))
    _assert_close(f32(ys[1]).astype(np.float64), y_ref)


def test_weights_ready_grouped_and_mxfp4(nv):
    counts = [3, 0, 200, 57]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M, K, N, k, E = int(offs[-1]), 1024, 256, 16, len(counts)
    x = W.activations(M, K, 5, "t3x20", 31, 32).cuda()
    wt = W.weights_t(N, K, 33, experts=E)
    rng = np.random.default_rng(3)
    chan_t = torch.from_numpy(np.stack([np.sort(rng.choice(K, k, replace=False)) for _ in range(E)])
                              .astype(np.int32)).cuda()
    offs_t = torch.from_numpy(offs).cuda()
    qs = [nv.nvfp4_quantize(wt[e].cuda()) for e in range(E)]
    b_codes = torch.stack([q["codes"] for q in qs])
    b_scales = torch.cat([q["scales"] for q in qs])
    g_b = torch.cat([q["g"] for q in qs])
    w_sel = nv.nvfp4_prepare_comp_weights(b_codes, b_scales, chan_t, E=E)
    torch.cuda.synchronize()
    ys = []
    for ready in (False, True):
        qx = nv.nvfp4_quantize_grouped(x, offs_t, chan_t)
        ys.append(nv.w4a4_grouped_gemm_comp(qx, offs_t, b_codes, b_scales, g_b, N, resid=qx["resid"], w_sel=w_sel,
                                            weights_ready=ready))
    xm = W.activations(48, 512, 5, "t3x20", 34, 35).cuda()
    qwm = nv.mxfp4_quantize(W.weights_t(256, 512, 36).cuda())
    torch.cuda.synchronize()
    ym = []
    for ready in (False, True):
        qxm = nv.mxfp4_quantize(xm)
        ym.append(nv.w4a4_gemm_comp(dict(codes=qxm["codes"], scales=qxm["scales"]),
                                    dict(codes=qwm["codes"], scales=qwm["scales"]), 256, fmt=nv.FMT_MXFP4,
                                    weights_ready=ready))
    torch.cuda.synchronize()
    st, _ = nv.check_status()
    assert st == 0
    assert torch.equal(ys[0], ys[1])
    assert torch.equal(ym[0], ym[1])
