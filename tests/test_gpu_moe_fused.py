"""GPU parity of the fused MoE epilogues against the oracle.

* Gate/up projection with SwiGLU and the down input's NVFP4 quantize in its
  epilogue (w4a4_grouped_gemm_swiglu_quant): the activation h it computes is
  within one bf16 rounding of the oracle's SwiGLU of the projection's bf16
  output (fp32 with expf against fp64), and its codes, scale bytes and
  residual slice are bit-exact with the oracle's static-scale quantization of
  that same h.
* Down projection with the routing-weighted combine in its epilogue
  (w4a4_grouped_gemm_combine): every token's fp32 output within the GEMM
  tolerance of the fp64 oracle chain (dequantized operands, compensation,
  renormalized top-k weights).
"""

import numpy as np
import pytest
import torch

from oracle import formats as F, gemm as og, moe as omoe, nvfp4 as onv
from nvfp4_w4a4_gemm_gb300 import workloads as W
from tests.helpers import bf16_bits_of, f32, gather_scales, gemm_within_tol, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from nvfp4_w4a4_gemm_gb300 import binding
    binding.load()
    return binding


def _quant_experts(nv, wt):
    """Per-expert NVFP4 weights: (codes [E,N,K/2], scales, g [E], per-expert oracle dicts)."""
    qs = [nv.nvfp4_quantize(wt[e].cuda()) for e in range(wt.shape[0])]
    return (torch.stack([q["codes"] for q in qs]), torch.cat([q["scales"] for q in qs]),
            torch.cat([q["g"] for q in qs]))


def _gate_up_case(nv, counts, K, inter, k, h_k, seed, resid_scaled, h_resid_scaled):
    E = len(counts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(offs[-1])
    x = W.activations(M, K, max(1, K // 100), "t3x20", seed, seed + 1)
    wt = W.weights_t(2 * inter, K, seed + 2, experts=E)
    wt_int = torch.from_numpy(omoe.interleave_gate_up(wt.view(torch.int16).numpy())[0]).view(torch.bfloat16)
    rng = np.random.default_rng(seed)
    chan = np.stack([np.sort(rng.choice(K, k, replace=False)) for _ in range(E)]).astype(np.int32)
    h_chan = np.stack([np.sort(rng.choice(inter, h_k, replace=False)) for _ in range(E)]).astype(np.int32)
    offs_t, chan_t, h_chan_t = (torch.from_numpy(a).cuda() for a in (offs, chan, h_chan))
    b_codes, b_scales, g_b = _quant_experts(nv, wt_int)
    w_sel = nv.nvfp4_prepare_comp_weights(b_codes, b_scales, chan_t, E=E)
    qx = nv.nvfp4_quantize_grouped(x.cuda(), offs_t, chan_t, resid_scaled=resid_scaled)
    # the unfused projection (bf16 output, interleaved columns) gives the
    # gate / up values the fused epilogue starts from
    y = nv.w4a4_grouped_gemm_comp(qx, offs_t, b_codes, b_scales, g_b, 2 * inter, resid=qx["resid"], w_sel=w_sel)
    y = f32(y).reshape(M, inter // 128, 2, 128)
    gate = y[:, :, 0, :].reshape(M, inter)
    up = y[:, :, 1, :].reshape(M, inter)
    h_ref = omoe.swiglu(gate, up)
    g_h = np.float32(onv.tensor_scale(h_ref) * np.float32(1.25))   # a static scale with some headroom
    g_h_t = torch.tensor([g_h], dtype=torch.float32).cuda()
    fused = nv.w4a4_grouped_gemm_swiglu_quant(qx, offs_t, b_codes, b_scales, g_b, 2 * inter, g_h_t, h_chan_t,
                                              resid=qx["resid"], w_sel=w_sel, h_resid_scaled=h_resid_scaled,
                                              with_h=True)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    return dict(offs=offs, h_chan=h_chan, g_h=g_h, h_ref=h_ref, fused=fused, M=M, E=E)


@pytest.mark.parametrize("counts,K,inter,k,h_k", [([40, 0, 130, 7, 1, 82], 512, 256, 32, 16),
                                                  ([256, 129, 300], 1024, 384, 64, 32)])
@pytest.mark.parametrize("scaled", [False, True])
def test_swiglu_quant_epilogue(nv, counts, K, inter, k, h_k, scaled):
    c = _gate_up_case(nv, counts, K, inter, k, h_k, 7 + K, scaled, scaled)
    fz = c["fused"]
    h = f32(fz["h"])
    h_ref = c["h_ref"]
    # fp32 SwiGLU with expf against fp64: at most one bf16 rounding apart
    assert np.all(np.abs(h - h_ref) <= 2.0 ** -7 * np.abs(h_ref) + 1e-30), np.max(np.abs(h - h_ref))
    ref = onv.quantize_grouped(h, c["offs"], c["h_chan"], g=c["g_h"])
    assert np.array_equal(u8(fz["codes"]), ref["packed"]), "codes"
    sc = gather_scales(fz["scales"], onv.grouped_scale_tile_offsets(c["offs"], inter // 16))
    assert np.array_equal(sc, ref["sigma"]), "scale bytes"
    want = ref["resid_scaled"] if scaled else ref["resid"]
    assert np.array_equal(bf16_bits_of(fz["resid"]), F.bf16_bits(want)), "residual"


@pytest.mark.parametrize("T,E,top", [(96, 12, 4), (512, 4, 2)])  # small experts: 128-row tiles; large: pair tiles
def test_combine_epilogue(nv, T, E, top):
    K, N, k = 512, 384, 32
    tok, offs, w_rows, logits = W.route(T, E, top, 31, with_weights=True)
    ex, w = omoe.route_weights(logits.numpy(), top)
    w_oracle = omoe.row_weights(ex, w, tok.numpy(), offs.numpy())
    np.testing.assert_allclose(w_rows.numpy(), w_oracle, rtol=2e-6)
    M = int(offs[-1])
    x = W.activations(M, K, 5, "t3x20", 32, 33)
    wt = W.weights_t(N, K, 34, experts=E)
    rng = np.random.default_rng(35)
    chan = np.stack([np.sort(rng.choice(K, k, replace=False)) for _ in range(E)]).astype(np.int32)
    offs_t, chan_t = offs.cuda(), torch.from_numpy(chan).cuda()
    b_codes, b_scales, g_b = _quant_experts(nv, wt)
    w_sel = nv.nvfp4_prepare_comp_weights(b_codes, b_scales, chan_t, E=E)
    qx = nv.nvfp4_quantize_grouped(x.cuda(), offs_t, chan_t, resid_scaled=True)
    out = nv.w4a4_grouped_gemm_combine(qx, offs_t, b_codes, b_scales, g_b, N, tok.to(torch.int32).cuda(),
                                       w_rows.cuda(), T, resid=qx["resid"], w_sel=w_sel)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    rq = onv.quantize_grouped(f32(x), offs.numpy(), chan)
    a = onv.dequantize(rq["codes"], rq["sigma"], rq["g"])
    bq = [onv.quantize(f32(wt[e])) for e in range(E)]
    b = np.stack([onv.dequantize(q["codes"], q["sigma"], q["g"]) for q in bq])
    ws = np.stack([og.comp_weight_rows(bq[e], chan[e]) for e in range(E)])
    y_rows = og.grouped_reference(a, offs.numpy(), b, rq["resid"], ws)
    ref = omoe.combine(y_rows, tok.numpy(), w_oracle, T)
    ok, ratio, _ = gemm_within_tol(f32(out), ref)
    assert ok, f"max err/allowance {ratio:.3f}"


def test_fused_moe_layer_full_size(nv):
    """The MoE workload (4096 tokens, top-8 of 128 experts, hidden 2048,
    intermediate 768) through both fused GEMMs; h of sampled experts checked
    as above, the output of sampled tokens against the oracle chain started
    from the GPU's quantized h."""
    s = W.SPECS["moe"]
    d = W.moe_inputs(which=("gate_up", "down"))
    dc = W.moe_inputs(calibration=True, with_weights=False)
    E, inter, hidden = s.experts, s.inter, s.hidden
    offs = d["offsets"]
    offs_t = offs.cuda()
    x = d["x_gate_up"].cuda()
    wt_int = torch.from_numpy(omoe.interleave_gate_up(d["wt_gate_up"].view(torch.int16).numpy())[0]).view(torch.bfloat16)
    chan = nv.nvfp4_calibrate_channels(dc["x_gate_up"].cuda(), s.k, offsets=dc["offsets"].cuda())
    h_chan = nv.nvfp4_calibrate_channels(dc["x_down"].cuda(), s.k, offsets=dc["offsets"].cuda())
    b_codes, b_scales, g_b = _quant_experts(nv, wt_int)
    w_sel = nv.nvfp4_prepare_comp_weights(b_codes, b_scales, chan, E=E)
    d_codes, d_scales, g_d = _quant_experts(nv, d["wt_down"])
    wd_sel = nv.nvfp4_prepare_comp_weights(d_codes, d_scales, h_chan, E=E)
    qx = nv.nvfp4_quantize_grouped(x, offs_t, chan, resid_scaled=True)
    g_h = torch.tensor([0.05], dtype=torch.float32).cuda()
    qh = nv.w4a4_grouped_gemm_swiglu_quant(qx, offs_t, b_codes, b_scales, g_b, 2 * inter, g_h, h_chan,
                                           resid=qx["resid"], w_sel=w_sel, h_resid_scaled=True, with_h=True)
    tok = d["token_of_row"].to(torch.int32)
    out = nv.w4a4_grouped_gemm_combine(qh, offs_t, d_codes, d_scales, g_d, hidden, tok.cuda(),
                                       d["route_weight"].cuda(), s.tokens, resid=qh["resid"], w_sel=wd_sel)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    offs_np = offs.numpy()
    h = f32(qh["h"])
    hc = h_chan.cpu().numpy()
    for e in (0, 41, E - 1):
        lo, hi = offs_np[e], offs_np[e + 1]
        rq = onv.quantize(h[lo:hi], g=0.05, chan=hc[e])
        assert np.array_equal(u8(qh["codes"])[lo:hi], rq["packed"])
        assert np.array_equal(bf16_bits_of(qh["resid"][lo:hi]), F.bf16_bits(rq["resid_scaled"]))
    # sampled tokens: the oracle chain from the GPU's h through the down projection
    rng = np.random.default_rng(9)
    toks = np.sort(rng.choice(s.tokens, 12, replace=False))
    tok_np = tok.numpy()
    w_np = d["route_weight"].numpy().astype(np.float64)
    wdq = {}
    ref = np.zeros((toks.size, hidden))
    for i, t in enumerate(toks):
        for r in np.nonzero(tok_np == t)[0]:
            e = int(np.searchsorted(offs_np, r, side="right")) - 1
            if e not in wdq:
                q = onv.quantize(f32(d["wt_down"][e]))
                wdq[e] = (onv.dequantize(q["codes"], q["sigma"], q["g"]), og.comp_weight_rows(q, hc[e]))
            rq = onv.quantize(h[r:r + 1], g=0.05, chan=hc[e])
            a = onv.dequantize(rq["codes"], rq["sigma"], rq["g"])
            ref[i] += w_np[r] * og.reference(a, wdq[e][0], rq["resid"], wdq[e][1])[0]
    ok, ratio, _ = gemm_within_tol(f32(out)[toks], ref)
    assert ok, f"max err/allowance {ratio:.3f}"
