"""GPU parity of the one-launch decode layer (w4a4_decode_linear): every CTA
quantizes the 1..16 token rows itself and runs the swapped-operand GEMM with
the compensation term.

* Against the oracle: y within |y - y_ref| <= 4e-3 |y_ref| + 1e-3 rms(y_ref)
  of the fp64 product of the oracle's dequantized operands, and the tensor
  scale bit-exact (dynamic: amax / 2688; static: the one given).
* Against the two-launch path (nvfp4_quantize_ex with the pre-scaled residual,
  then w4a4_gemm_comp): bit-identical output wherever that GEMM does not split
  K across CTAs (at least 76 output tiles of 128 columns; with fewer tiles it
  sums fp32 partials in a different order).
"""

import ctypes

import numpy as np
import pytest
import torch

from oracle import gemm as og, nvfp4 as onv
from nvfp4_w4a4_gemm_gb300 import workloads as W
from tests.helpers import f32, gemm_within_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from nvfp4_w4a4_gemm_gb300 import binding
    binding.load()
    return binding


def _case(nv, M, N, K, k, seed, static=False, flags=0):
    x = W.activations(M, K, max(1, K // 100), "t3x20", seed, seed + 1)
    wt = W.weights_t(N, K, seed + 2)
    rng = np.random.default_rng(seed)
    chan = np.sort(rng.choice(K, size=k, replace=False)).astype(np.int32)
    ch = torch.from_numpy(chan).cuda() if k else None
    qw = nv.nvfp4_quantize(wt.cuda())
    ws = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], ch, flags=flags,
                                       wt=wt.cuda() if flags else None) if k else None
    g_x = None
    if static:
        g_x = np.float32(onv.tensor_scale(f32(x)) * np.float32(1.5))  # a calibrated scale with headroom
    g_t = torch.tensor([g_x], dtype=torch.float32).cuda() if static else None
    return dict(x=x, wt=wt, chan=chan, ch=ch, qw=qw, ws=ws, g_x=g_x, g_t=g_t, flags=flags)


def _fused(nv, c, N, **kw):
    g_out = torch.zeros(1, dtype=torch.float32, device="cuda")
    y = nv.w4a4_decode_linear(c["x"].cuda(), c["qw"], N, chan=c["ch"], w_sel=c["ws"], g=c["g_t"],
                              flags=c["flags"], g_out=g_out, **kw)
    torch.cuda.synchronize()
    st, det = nv.check_status()
    assert st == 0, (st, det)
    return y, f32(g_out)[0]


def _two_launch(nv, c, N):
    qx = nv.nvfp4_quantize(c["x"].cuda(), g=c["g_t"], chan=c["ch"], resid_scaled=True)
    y = nv.w4a4_gemm_comp(qx, c["qw"], N, resid=qx["resid"] if c["ch"] is not None else None, w_sel=c["ws"],
                          flags=c["flags"])
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("M,N,K,k", [(16, 384, 1024, 64), (1, 128, 64, 8), (5, 256, 320, 24), (16, 128, 4096, 256),
                                     (9, 640, 8192, 72), (16, 256, 4160, 0), (12, 1152, 2048, 128)])
@pytest.mark.parametrize("static", [False, True])
def test_decode_layer_vs_oracle(nv, M, N, K, k, static):
    c = _case(nv, M, N, K, k, 11 + M + K, static)
    y, g = _fused(nv, c, N)
    xf = f32(c["x"])
    g_ref = c["g_x"] if static else onv.tensor_scale(xf)
    assert g == np.float32(g_ref)
    y_ref, _, _ = og.linear_comp(xf, f32(c["wt"]), c["chan"].astype(np.int64), g_x=c["g_x"])
    ok, ratio, rms = gemm_within_tol(f32(y).astype(np.float64), y_ref)
    assert ok, f"max err/allowance {ratio:.3f} (rms {rms:.4g})"


def test_decode_layer_bf16_weight_columns(nv):
    c = _case(nv, 7, 256, 1024, 32, 5, flags=1)
    y, _ = _fused(nv, c, 256)
    y_ref, _, _ = og.linear_comp(f32(c["x"]), f32(c["wt"]), c["chan"].astype(np.int64), bf16_weights=True)
    ok, ratio, _ = gemm_within_tol(f32(y).astype(np.float64), y_ref)
    assert ok, ratio


@pytest.mark.parametrize("M,K,k,static,flags", [(16, 1024, 64, False, 0), (3, 2048, 16, True, 0),
                                                (16, 512, 40, False, 1), (11, 4160, 0, False, 0)])
def test_decode_layer_bit_identical_to_two_launches(nv, M, K, k, static, flags):
    N = 76 * 128  # enough output tiles that the two-launch GEMM keeps K whole
    c = _case(nv, M, N, K, k, 40 + M, static, flags)
    y2 = _two_launch(nv, c, N)
    y1, _ = _fused(nv, c, N)
    y1r, _ = _fused(nv, c, N, weights_ready=True)
    assert torch.equal(y1, y2)
    assert torch.equal(y1r, y2)


def test_decode_layer_full_size(nv):
    """The decode workload (16 x 4096 tokens, W^T 14336 x 4096, k = 64 channels
    calibrated on the calibration batch): bit-identical to the two-launch
    path, sampled columns within tolerance of the oracle."""
    s = W.SPECS["decode"]
    d = W.dense_inputs("decode")
    x, wt = d["x"].cuda(), d["wt"].cuda()
    ch = nv.nvfp4_calibrate_channels(W.dense_inputs("decode", True, False)["x"].cuda(), s.k)
    qw = nv.nvfp4_quantize(wt)
    ws = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], ch)
    c = dict(x=d["x"], ch=ch, qw=qw, ws=ws, g_t=None, flags=0)
    y2 = _two_launch(nv, c, s.N)
    y1, g = _fused(nv, c, s.N, weights_ready=True)
    assert torch.equal(y1, y2)
    xf = f32(d["x"])
    assert g == np.float32(onv.tensor_scale(xf))
    # sampled output columns: the oracle quantizes those weight rows with the
    # tensor scale of the whole weight
    rng = np.random.default_rng(3)
    cols = np.sort(rng.choice(s.N, 768, replace=False))
    chan = ch.cpu().numpy().astype(np.int64)
    wf = f32(d["wt"])
    g_w = onv.tensor_scale(wf)
    rq = onv.quantize(xf, chan=chan)
    cq = onv.quantize(wf[cols], g=g_w)
    a = onv.dequantize(rq["codes"], rq["sigma"], rq["g"])
    b = onv.dequantize(cq["codes"], cq["sigma"], g_w)
    y_ref = og.reference(a, b, rq["resid"], og.comp_weight_rows(cq, chan))
    ok, ratio, _ = gemm_within_tol(f32(y1)[:, cols].astype(np.float64), y_ref)
    assert ok, ratio


def test_decode_layer_rejects_unsupported_shapes(nv):
    lib = nv.load()
    x = torch.zeros((17, 256), dtype=torch.bfloat16, device="cuda")
    q = nv.nvfp4_quantize(torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda"))
    y = torch.empty((17, 128), dtype=torch.bfloat16, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    args = lambda M, N, K, k: (M, N, K, p(x), 256, None, None, None, k, p(q["codes"]), p(q["scales"]), None, None,
                               0, p(y), None)
    assert lib.w4a4_decode_linear(*args(17, 128, 256, 0)) == nv.ERR_UNSUPPORTED   # more than 16 tokens
    assert lib.w4a4_decode_linear(*args(0, 128, 256, 0)) == nv.ERR_INVALID_ARG    # no tokens
    assert lib.w4a4_decode_linear(*args(4, 100, 256, 0)) == nv.ERR_UNSUPPORTED    # N % 128
