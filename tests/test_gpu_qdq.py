"""GPU parity of the trainer-side weight fake quantization (QDQ) against the
oracle: bit-exact bf16 values (signs of zero included), and the codes and
scales it can emit bit-identical to the quantizer's."""

import numpy as np
import pytest
import torch

from oracle import nvfp4 as onv
from oracle.formats import bf16_bits
from nvfp4_w4a4_gemm_gb300 import workloads as W
from tests.helpers import f32, gather_scales, u8
from tests.test_oracle_nvfp4 import DOUBLE_ROUNDING_G, DOUBLE_ROUNDING_X

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from nvfp4_w4a4_gemm_gb300 import binding
    binding.load()
    return binding


def _bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _check(nv, w, g=None, with_codes=True):
    gd = None if g is None else torch.tensor([g], dtype=torch.float32).cuda()
    r = nv.nvfp4_qdq(w, g=gd, with_codes=with_codes)
    torch.cuda.synchronize()
    want, q = onv.qdq(f32(w), g=g)
    assert float(r["g"].item()) == float(q["g"])
    assert np.array_equal(_bits(r["w_qdq"]), bf16_bits(want))
    if with_codes:
        M, K = w.shape
        ref = nv.nvfp4_quantize(w, g=gd)
        assert torch.equal(r["codes"], ref["codes"])
        assert np.array_equal(u8(r["codes"]), q["packed"])
        offs = onv.scale_tile_offsets(M, K // 16)
        assert np.array_equal(gather_scales(r["scales"], offs), q["sigma"])
        assert np.array_equal(gather_scales(r["scales"], offs), gather_scales(ref["scales"], offs))


@pytest.mark.parametrize("M,K,g", [(64, 256, None), (300, 1040, None), (128, 4096, 2.0 ** -7),
                                   (77, 2048, 0.0123), (1, 16, None), (33, 3072, 1.0 / 3.0)])
def test_qdq_matches_oracle(nv, M, K, g):
    w = W.weights_t(M, K, M + K).cuda()
    w[0, :16] = 0  # an all-zero block
    _check(nv, w, g)


def test_qdq_outlier_rows_without_codes(nv):
    x = W.activations(96, 2048, 20, "t3x20", 4, 5).cuda()
    _check(nv, x, None, with_codes=False)


def test_qdq_double_rounding_block(nv):
    x = torch.tensor([DOUBLE_ROUNDING_X * 4] * 3, dtype=torch.bfloat16).cuda()
    r = nv.nvfp4_qdq(x, g=torch.tensor([DOUBLE_ROUNDING_G], dtype=torch.float32).cuda())
    torch.cuda.synchronize()
    got = f32(r["w_qdq"])
    assert got[0, 1] == np.float32(3.03125) and got[0, 2] == np.float32(-3.03125) and got[0, 0] == np.float32(6.0625)
    _check(nv, x, DOUBLE_ROUNDING_G)


def test_qdq_strided_input_and_output(nv):
    big = W.weights_t(40, 1536, 8).cuda()
    w = big[:, 256:1280]  # row stride 1536
    out = torch.full((40, 1104), 7.0, dtype=torch.bfloat16).cuda()
    r = nv.nvfp4_qdq(w, out=out[:, :1024])
    torch.cuda.synchronize()
    want, _ = onv.qdq(f32(w))
    assert np.array_equal(_bits(r["w_qdq"]), bf16_bits(want))
    assert torch.all(out[:, 1024:] == 7.0)  # nothing written past the row


def test_qdq_empty(nv):
    r = nv.nvfp4_qdq(torch.empty((0, 64), dtype=torch.bfloat16).cuda())
    torch.cuda.synchronize()
    assert r["w_qdq"].numel() == 0 and float(r["g"].item()) == 1.0


def test_qdq_full_size_prefill_weight_sampled_rows(nv):
    s = W.SPECS["prefill"]
    wt = W.weights_t(s.N, s.K, 3).cuda()
    r = nv.nvfp4_qdq(wt, with_codes=True)
    torch.cuda.synchronize()
    g = np.float32(r["g"].item())
    # tensor scale from the whole matrix, the rows checked one by one under it
    assert g == onv.tensor_scale(f32(wt))
    rows = np.sort(np.random.default_rng(5).choice(s.N, 48, replace=False))
    want, q = onv.qdq(f32(wt[rows]), g=g)
    assert np.array_equal(_bits(r["w_qdq"][rows]), bf16_bits(want))
    assert np.array_equal(u8(r["codes"][rows]), q["packed"])
