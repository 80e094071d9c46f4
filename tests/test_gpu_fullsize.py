"""Full-size parity on the five workloads' shapes, in the launch configuration
bench.py times.  The GPU runs the whole problem; the oracle recomputes the
rows it needs (with the tensor scale of the full tensor) and checks codes and
scale bytes bit-exactly on those rows and the GEMM on sampled outputs, with
the tolerance |y - y_ref| <= 4e-3 |y_ref| + 1e-3 rms(y_ref), rms taken over
the sample."""

import numpy as np
import pytest
import torch

from oracle import formats as F, gemm as og, mxfp4 as omx, nvfp4 as onv
from nvfp4_w4a4_gemm_gb300 import workloads as W
from tests.helpers import bf16_bits_of, f32, gather_scales, gemm_within_tol, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from nvfp4_w4a4_gemm_gb300 import binding
    binding.load()
    return binding


def _rows_quantized(x_rows, g):
    """Oracle quantization of selected rows with a given tensor scale."""
    return onv.quantize(x_rows, g=np.float32(g))


def _assert_close(y, y_ref, what):
    ok, ratio, rms = gemm_within_tol(y, y_ref)
    assert ok, f"{what}: max err/allowance {ratio:.3f} (rms {rms:.4g})"


def _dense(nv, name, rows, cols, seed):
    s = W.SPECS[name]
    d = W.dense_inputs(name)
    x, wt = d["x"], d["wt"]
    rng = np.random.default_rng(seed)
    chan = np.sort(rng.choice(s.K, size=s.k, replace=False)).astype(np.int32)
    ch = torch.from_numpy(chan).cuda()
    qx = nv.nvfp4_quantize(x.cuda(), chan=ch)
    qw = nv.nvfp4_quantize(wt.cuda())
    ws = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], ch)
    y = nv.w4a4_gemm_comp(qx, qw, s.N, resid=qx["resid"], w_sel=ws)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    xf, wf = f32(x), f32(wt)
    g_x, g_w = onv.tensor_scale(xf), onv.tensor_scale(wf)
    assert f32(qx["g"])[0] == g_x and f32(qw["g"])[0] == g_w
    rq = _rows_quantized(xf[rows], g_x)
    rq_res = onv.quantize(xf[rows], g=g_x, chan=chan)
    cq = _rows_quantized(wf[cols], g_w)
    # codes / scales / residual of the sampled rows, bit-exact
    assert np.array_equal(u8(qx["codes"])[rows], rq["packed"])
    off = onv.scale_tile_offsets(s.M, s.K // 16)[rows]
    assert np.array_equal(gather_scales(qx["scales"], off), rq["sigma"])
    assert np.array_equal(f32(qx["resid"])[rows], rq_res["resid"])
    assert np.array_equal(u8(qw["codes"])[cols], cq["packed"])
    # GEMM on the (rows x cols) block
    a = onv.dequantize(rq["codes"], rq["sigma"], g_x)
    b = onv.dequantize(cq["codes"], cq["sigma"], g_w)
    w_sel = onv.comp_weights(cq["codes"], cq["sigma"], chan) * np.float64(g_w)
    y_ref = og.reference(a, b, rq_res["resid"], w_sel)
    _assert_close(f32(y)[np.ix_(rows, cols)], y_ref, name)


def test_decode_full_size(nv):
    s = W.SPECS["decode"]
    rng = np.random.default_rng(1)
    _dense(nv, "decode", np.arange(s.M), np.sort(rng.choice(s.N, 1024, replace=False)), 1)


def test_prefill_full_size(nv):
    s = W.SPECS["prefill"]
    rng = np.random.default_rng(2)
    rows = np.sort(np.concatenate([rng.choice(s.M, 254, replace=False), [0, s.M - 1]]))
    _dense(nv, "prefill", np.unique(rows), np.sort(rng.choice(s.N, 384, replace=False)), 2)


@pytest.mark.parametrize("which", ["gate_up", "down"])
def test_moe_full_size(nv, which):
    s = W.SPECS["moe"]
    d = W.moe_inputs(which=(which,))
    x = d["x_gate_up"] if which == "gate_up" else d["x_down"]
    wt = d["wt_gate_up"] if which == "gate_up" else d["wt_down"]
    E, N, K = wt.shape
    offs = d["offsets"].numpy().astype(np.int32)
    # per-expert channel sets calibrated on the calibration batch (residual
    # variance over the rows routed to each expert), as the bench uses them
    dc = W.moe_inputs(calibration=True, with_weights=False, which=(which,))
    xc = dc["x_gate_up"] if which == "gate_up" else dc["x_down"]
    chan_t = nv.nvfp4_calibrate_channels(xc.cuda(), s.k, offsets=dc["offsets"].cuda())
    chan = chan_t.cpu().numpy().astype(np.int32)
    offs_t = torch.from_numpy(offs).cuda()
    qx = nv.nvfp4_quantize_grouped(x.cuda(), offs_t, chan_t, resid_scaled=True)
    if which == "gate_up":
        # the bench's form: read through the routing table from the token rows
        qg = nv.nvfp4_quantize_grouped_gather(d["x_tokens"].cuda(), d["token_of_row"].to(torch.int32).cuda(),
                                              offs_t, chan_t, resid_scaled=True)
        for key in ("g", "codes", "resid"):
            assert torch.equal(qg[key], qx[key]), key
        tiles = onv.grouped_scale_tile_offsets(offs, K // 16)
        assert np.array_equal(gather_scales(qg["scales"], tiles), gather_scales(qx["scales"], tiles))
        del qg
    codes, scales, gs = [], [], []
    for e in range(E):
        q = nv.nvfp4_quantize(wt[e].cuda())
        codes.append(q["codes"]); scales.append(q["scales"]); gs.append(q["g"])
    b_codes, b_scales, g_b = torch.stack(codes), torch.cat(scales), torch.cat(gs)
    w_sel = nv.nvfp4_prepare_comp_weights(b_codes, b_scales, chan_t, E=E)
    y = nv.w4a4_grouped_gemm_comp(qx, offs_t, b_codes, b_scales, g_b, N, resid=qx["resid"], w_sel=w_sel)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    xf = f32(x)
    g_x = onv.tensor_scale(xf)
    assert f32(qx["g"])[0] == g_x
    yg = f32(y)
    prow = onv.grouped_row_map(offs)
    for e in (0, 37, 77, E - 1):
        lo, hi = offs[e], offs[e + 1]
        if hi == lo:
            continue
        rows = np.arange(lo, hi)
        rq = onv.quantize(xf[rows], g=g_x, chan=chan[e])
        assert np.array_equal(u8(qx["codes"])[rows], rq["packed"])
        off = onv.tile_offset(prow[rows][:, None], np.arange(K // 16)[None, :], -(-(K // 16) // 4) * 4)
        assert np.array_equal(gather_scales(qx["scales"], off), rq["sigma"])
        wq = onv.quantize(f32(wt[e]))
        assert f32(g_b)[e] == wq["g"]
        a = onv.dequantize(rq["codes"], rq["sigma"], g_x)
        b = onv.dequantize(wq["codes"], wq["sigma"], wq["g"])
        ws = og.comp_weight_rows(wq, chan[e])
        # the GEMM consumed the pre-scaled residual: bit-exact against the
        # oracle's, and the output within tolerance of the plain-residual product
        assert np.array_equal(bf16_bits_of(qx["resid"][lo:hi]), F.bf16_bits(rq["resid_scaled"]))
        _assert_close(yg[rows], og.reference(a, b, rq["resid"], ws), f"moe {which} expert {e}")


def test_mxfp4_full_size(nv):
    s = W.SPECS["mxfp4"]
    d = W.dense_inputs("mxfp4")
    x, wt = d["x"], d["wt"]
    qx = nv.mxfp4_quantize(x.cuda(), stats=True)
    qw = nv.mxfp4_quantize(wt.cuda())
    y = nv.w4a4_gemm_comp(dict(codes=qx["codes"], scales=qx["scales"]),
                          dict(codes=qw["codes"], scales=qw["scales"]), s.N, fmt=nv.FMT_MXFP4)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(s.M, 256, replace=False))
    cols = np.sort(rng.choice(s.N, 384, replace=False))
    st, cnt, dx = omx.block_stats(f32(x)[rows])
    assert np.array_equal(u8(qx["codes"])[rows], dx["packed"])
    off = onv.scale_tile_offsets(s.M, s.K // 32)[rows]
    assert np.array_equal(gather_scales(qx["scales"], off), dx["scale"])
    nb = s.K // 32
    assert np.array_equal(u8(qx["dead"]).reshape(s.M, nb)[rows], cnt)
    g = f32(qx["stats"]).reshape(s.M, nb, 4)[rows].astype(np.float64)
    assert np.all(np.abs(g - st) <= 1e-5 * (st[..., 3:4] + st.sum(-1, keepdims=True)) + 1e-30)
    wq = omx.quantize(f32(wt)[cols])
    assert np.array_equal(u8(qw["codes"])[cols], wq["packed"])
    y_ref = og.reference(omx.dequantize(dx["codes"], dx["scale"]), omx.dequantize(wq["codes"], wq["scale"]))
    _assert_close(f32(y)[np.ix_(rows, cols)], y_ref, "mxfp4")
