"""GPU parity of the quantized-residual (FP8 E4M3) compensation against the
oracle: the E4M3 residual bytes and weight rows bit-exact, the GEMM with the
FP8 term within the GEMM tolerance |y - y_ref| <= 4e-3 |y_ref| + 1e-3
rms(y_ref) of the fp64 product of the same operands, on the 128-row kernel
(swapped operands up to 64 rows), the 256-row pair kernel, and the prefill
workload at full size on sampled outputs."""

import numpy as np
import pytest
import torch

from oracle import gemm as og, nvfp4 as onv
from nvfp4_w4a4_gemm_gb300 import workloads as W
from tests.helpers import f32, gather_scales, gemm_within_tol, tiled_scales_dense, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from nvfp4_w4a4_gemm_gb300 import binding
    binding.load()
    assert binding.check_status()[0] == 0
    return binding


def _chan(K, k, seed, must=()):
    """k sorted distinct channels of K: those in `must` first, the rest drawn."""
    rng = np.random.default_rng(seed)
    c = list(dict.fromkeys(int(v) for v in must))[:k]
    taken = set(c)
    rest = [int(v) for v in rng.permutation(K) if int(v) not in taken]
    return np.sort(np.array(c + rest[:k - len(c)], np.int32))


@pytest.mark.parametrize("M,K,k,static", [(37, 4096, 128, False), (300, 1552, 48, True), (129, 2048, 16, False),
                                          (5, 64, 16, True), (1000, 1024, 1024, False)])
def test_quantize_resid_fp8_bit_exact(nv, M, K, k, static):
    x = W.activations(M, K, max(1, K // 100), "t3x20", K + 3, M + 5)
    xf = f32(x)
    chan = _chan(K, k, M + K)
    g = onv.tensor_scale(xf) * np.float32(1.25) if static else None
    gd = torch.tensor([g], dtype=torch.float32, device="cuda") if static else None
    q = nv.nvfp4_quantize(x.cuda(), g=gd, chan=torch.from_numpy(chan).cuda(), resid_fp8=True)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    ref = onv.quantize(xf, g=g, chan=chan)
    assert f32(q["g"])[0] == ref["g"]
    assert np.array_equal(u8(q["codes"]), ref["packed"])
    assert np.array_equal(tiled_scales_dense(q["scales"], M, K), ref["sigma"])
    r8 = u8(q["resid"])
    bad = np.argwhere(r8 != ref["resid_fp8"])
    assert bad.size == 0, (f"{len(bad)} residual bytes differ, first {bad[:4].tolist()}: "
                           f"{r8[tuple(bad[0])]:#x} vs {ref['resid_fp8'][tuple(bad[0])]:#x}")
    # the cases cover negative and positive residuals and both zeros
    assert (ref["resid_fp8"] & 0x80).any() and ((ref["resid_fp8"] & 0x80) == 0).any()


def test_comp_weights_fp8_bit_exact(nv):
    N, K, k = 384, 1024, 64
    wt = W.weights_t(N, K, 21)
    wf = f32(wt)
    # the column of the largest |w| (scale 448, code +-6: 2688 * 2^-3 = 336,
    # a tie that rounds to 320) is among the channels
    j_max = int(np.unravel_index(np.argmax(np.abs(wf)), wf.shape)[1])
    chan = _chan(K, k, 5, must=[j_max])
    qw = nv.nvfp4_quantize(wt.cuda())
    w8 = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], torch.from_numpy(chan).cuda(),
                                       flags=nv.COMP_W_DEQ_FP8)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    rq = onv.quantize(wf)
    ref = onv.comp_weights_fp8(rq["codes"], rq["sigma"], chan)
    assert w8.dtype == torch.uint8 and np.array_equal(u8(w8), ref)
    assert (ref & 0x7F).max() == 0x7A


def _fp8_case(nv, x, wt, chan):
    N = wt.shape[0]
    ch = torch.from_numpy(chan).cuda()
    qx = nv.nvfp4_quantize(x.cuda(), chan=ch, resid_fp8=True)
    qw = nv.nvfp4_quantize(wt.cuda())
    w8 = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], ch, flags=nv.COMP_W_DEQ_FP8)
    y = nv.w4a4_gemm_comp(qx, qw, N, resid=qx["resid"], w_sel=w8)
    y0 = nv.w4a4_gemm_comp(qx, qw, N)  # the same product without the term
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    y_ref, rq, rw, w8_ref = og.linear_comp_fp8(f32(x), f32(wt), chan)
    assert np.array_equal(u8(qx["resid"]), rq["resid_fp8"]) and np.array_equal(u8(w8), w8_ref)
    term = og.comp_term_fp8(rq["resid_fp8"], w8_ref, rq["g"], rw["g"])
    return f32(y).astype(np.float64), f32(y0).astype(np.float64), y_ref, term


@pytest.mark.parametrize("M,N,K,k", [(1, 128, 256, 16), (40, 256, 1024, 48), (64, 128, 512, 128),
                                     (100, 384, 1024, 144), (256, 256, 2048, 128), (300, 384, 1024, 64),
                                     (777, 256, 1024, 272), (513, 128, 2048, 128)])
def test_gemm_fp8_compensation(nv, M, N, K, k):
    n_out = max(2, K // 64)  # outlier channels, all compensated: the term is 13-21x the bf16 output rounding
    x = W.activations(M, K, n_out, "t3x20", K + 7, M + 11)
    wt = W.weights_t(N, K, N + K + 1)
    chan = _chan(K, k, M + N + K, must=W.outlier_channels(K, n_out, K + 7))
    y, y0, y_ref, term = _fp8_case(nv, x, wt, chan)
    ok, ratio, rms = gemm_within_tol(y, y_ref)
    assert ok, f"max err/allowance {ratio:.3f} (rms {rms:.4g})"
    # the term is there, once, at its scale: the product without it misses
    # the reference by the term, the product with it only by the bf16 rounding
    d_ok, d_none = np.linalg.norm(y - y_ref), np.linalg.norm(y0 - y_ref)
    assert np.linalg.norm(term) > 8 * 2.0 ** -9 * np.linalg.norm(y_ref)
    assert d_ok < 0.25 * d_none, (d_ok, d_none)


def test_prefill_full_size_fp8(nv):
    s = W.SPECS["prefill"]
    d = W.dense_inputs("prefill")
    x, wt = d["x"], d["wt"]
    rng = np.random.default_rng(12)
    chan = np.sort(rng.choice(s.K, size=s.k, replace=False)).astype(np.int32)
    ch = torch.from_numpy(chan).cuda()
    qx = nv.nvfp4_quantize(x.cuda(), chan=ch, resid_fp8=True)
    qw = nv.nvfp4_quantize(wt.cuda())
    w8 = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], ch, flags=nv.COMP_W_DEQ_FP8)
    y = nv.w4a4_gemm_comp(qx, qw, s.N, resid=qx["resid"], w_sel=w8)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    xf, wf = f32(x), f32(wt)
    g_x, g_w = onv.tensor_scale(xf), onv.tensor_scale(wf)
    rows = np.unique(np.concatenate([rng.choice(s.M, 254, replace=False), [0, s.M - 1]]))
    cols = np.sort(rng.choice(s.N, 384, replace=False))
    rq = onv.quantize(xf[rows], g=g_x, chan=chan)
    cq = onv.quantize(wf[cols], g=g_w)
    assert np.array_equal(u8(qx["resid"])[rows], rq["resid_fp8"])
    off = onv.scale_tile_offsets(s.M, s.K // 16)[rows]
    assert np.array_equal(gather_scales(qx["scales"], off), rq["sigma"])
    w8_ref = onv.comp_weights_fp8(cq["codes"], cq["sigma"], chan)
    assert np.array_equal(u8(w8)[cols], w8_ref)
    a = onv.dequantize(rq["codes"], rq["sigma"], g_x)
    b = onv.dequantize(cq["codes"], cq["sigma"], g_w)
    y_ref = og.reference(a, b) + og.comp_term_fp8(rq["resid_fp8"], w8_ref, g_x, g_w)
    ok, ratio, rms = gemm_within_tol(f32(y)[np.ix_(rows, cols)], y_ref)
    assert ok, f"max err/allowance {ratio:.3f} (rms {rms:.4g})"


def test_fp8_flag_combinations_rejected(nv):
    M, N, K, k = 300, 256, 512, 32
    x = W.activations(M, K, 5, "t3x20", 1, 2).cuda()
    wt = W.weights_t(N, K, 3).cuda()
    ch = torch.arange(0, K, K // k, dtype=torch.int32, device="cuda")
    qx = nv.nvfp4_quantize(x, chan=ch, resid_fp8=True)
    qw = nv.nvfp4_quantize(wt)
    w8 = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], ch, flags=nv.COMP_W_DEQ_FP8)
    # FP8 operands with the BF16-weight mode: an argument error, nothing launched
    with pytest.raises(RuntimeError):
        nv.w4a4_gemm_comp(qx, qw, N, resid=qx["resid"], w_sel=w8, flags=nv.COMP_W_BF16)
    # k not a multiple of 16: unsupported, nothing launched
    with pytest.raises(RuntimeError):
        nv.w4a4_gemm_comp(qx, qw, N, resid=qx["resid"][:, :24].contiguous(), w_sel=w8[:, :24].contiguous())
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0


@pytest.mark.parametrize("M", [40, 200, 700])
def test_fp8_weights_ready_overlap_is_bit_identical(nv, M):
    # the GEMM with the FP8 term started as a programmatic dependent of the
    # quantizer before it, with and without streaming weights before its wait
    N, K, k = 384, 1024, 64
    x = W.activations(M, K, 8, "t3x20", 41, 42).cuda()
    wt = W.weights_t(N, K, 43).cuda()
    ch = torch.arange(0, K, K // k, dtype=torch.int32, device="cuda")
    qw = nv.nvfp4_quantize(wt)
    w8 = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], ch, flags=nv.COMP_W_DEQ_FP8)
    torch.cuda.synchronize()
    ys = []
    for ready in (False, True, True):
        qx = nv.nvfp4_quantize(x, chan=ch, resid_fp8=True)
        ys.append(nv.w4a4_gemm_comp(qx, qw, N, resid=qx["resid"], w_sel=w8, weights_ready=ready))
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])
