"""Empty inputs through every entry point: no rows (M = 0, or experts that
all route zero rows) must return NVFP4_OK and write nothing but the tensor
scale, which is the oracle's scale of an empty tensor (1) when it is dynamic
and the given one when it is static."""

import numpy as np
import pytest
import torch

from oracle import nvfp4 as onv
from nvfp4_w4a4_gemm_gb300 import workloads as W
from tests.helpers import f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from nvfp4_w4a4_gemm_gb300 import binding
    binding.load()
    assert binding.check_status()[0] == 0
    return binding


def test_oracle_scale_of_empty_tensor():
    assert onv.tensor_scale(np.zeros((0, 64), np.float32)) == np.float32(1.0)


@pytest.mark.parametrize("static", [False, True])
def test_quantize_no_rows(nv, static):
    K, k = 256, 8
    x = torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    chan = torch.arange(0, K, K // k, dtype=torch.int32, device="cuda")
    g = torch.tensor([0.125], device="cuda") if static else None
    q = nv.nvfp4_quantize(x, g=g, chan=chan)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    assert q["codes"].shape == (0, K // 2) and q["resid"].shape == (0, k)
    assert f32(q["g"])[0] == (np.float32(0.125) if static else onv.tensor_scale(np.zeros((0, K), np.float32)))


def test_static_scale_reported_without_rows(nv):
    # the grouped quantizer and the trainer-side QDQ also hand back the given scale
    E, K = 2, 128
    g = torch.tensor([0.375], device="cuda")
    offs = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    chan = torch.stack([torch.arange(0, K, 16, dtype=torch.int32)] * E).cuda()
    qg = nv.nvfp4_quantize_grouped(torch.empty((0, K), dtype=torch.bfloat16, device="cuda"), offs, chan, g=g)
    r = nv.nvfp4_qdq(torch.empty((0, K), dtype=torch.bfloat16, device="cuda"), g=g)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    assert f32(qg["g"])[0] == np.float32(0.375) and float(r["g"].item()) == 0.375


def test_grouped_quantize_all_experts_empty(nv):
    E, K, k = 3, 256, 8
    x = torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    offs = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    chan = torch.stack([torch.arange(0, K, K // k, dtype=torch.int32)] * E).cuda()
    q = nv.nvfp4_quantize_grouped(x, offs, chan)
    xt = W.activations(5, K, 2, "t3x20", 1, 2).cuda()  # token rows that no row routes to
    qg = nv.nvfp4_quantize_grouped_gather(xt, torch.empty(0, dtype=torch.int32, device="cuda"), offs, chan)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    assert f32(q["g"])[0] == np.float32(1.0) and f32(qg["g"])[0] == np.float32(1.0)
    assert q["codes"].shape == (0, K // 2) and qg["codes"].shape == (0, K // 2)


def test_gemms_no_rows(nv):
    N, K, k, E = 256, 256, 8, 3
    wt = W.weights_t(N, K, 3).cuda()
    qw = nv.nvfp4_quantize(wt)
    chan = torch.arange(0, K, K // k, dtype=torch.int32, device="cuda")
    ws = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], chan)
    qx = nv.nvfp4_quantize(torch.empty((0, K), dtype=torch.bfloat16, device="cuda"), chan=chan)
    y = nv.w4a4_gemm_comp(qx, qw, N, resid=qx["resid"], w_sel=ws)
    # grouped: every expert routes zero rows
    wte = torch.stack([W.weights_t(N, K, 10 + e) for e in range(E)]).cuda()
    qs = [nv.nvfp4_quantize(wte[e]) for e in range(E)]
    b_codes = torch.stack([s["codes"] for s in qs])
    b_scales = torch.cat([s["scales"] for s in qs])
    g_b = torch.cat([s["g"] for s in qs])
    chan_e = torch.stack([chan] * E)
    w_sel = nv.nvfp4_prepare_comp_weights(b_codes, b_scales, chan_e, E=E)
    offs = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    qa = nv.nvfp4_quantize_grouped(torch.empty((0, K), dtype=torch.bfloat16, device="cuda"), offs, chan_e)
    yg = nv.w4a4_grouped_gemm_comp(qa, offs, b_codes, b_scales, g_b, N, resid=qa["resid"], w_sel=w_sel)
    # MXFP4 quantize of no rows
    qm = nv.mxfp4_quantize(torch.empty((0, 512), dtype=torch.bfloat16, device="cuda"), stats=True)
    torch.cuda.synchronize()
    assert nv.check_status()[0] == 0
    assert y.shape == (0, N) and yg.shape == (0, N)
    assert qm["codes"].shape == (0, 256) and qm["stats"].shape == (0, 4)
