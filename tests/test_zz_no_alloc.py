"""The allocation-free quantizer entry point (nvfp4_quantize_noalloc).

Some callers cannot allocate device memory (an engine that owns all of it
through its own allocator, or a hot path that must never call cudaMalloc),
so they cannot hand nvfp4_quantize the workspace its dynamic tensor scale
needs.  nvfp4_quantize_noalloc keeps that scratch in a device array owned by
the library.  This test calls it through the C ABI and checks that its codes,
scale bytes, tensor scale and residuals are identical to those of the
allocating entry point, on three calls in a row with different inputs (the
shared scratch keeps the previous call's contents).  This file is collected
last on purpose.
"""

import numpy as np
import pytest
import torch

from nvfp4_w4a4_gemm_gb300 import workloads as W
from tests.helpers import bf16_bits_of, u8

pytestmark = pytest.mark.gpu


def test_noalloc_matches_allocating_quantizer_on_successive_calls():
    from nvfp4_w4a4_gemm_gb300 import binding as nv
    nv.load()
    # the third call follows the large second one with a much smaller shape
    # and a 1000x smaller amax: the scratch then still holds the second
    # call's larger partial maxima past the third call's own partials, so a
    # read past them would change the tensor scale
    shapes = [(300, 1040, 33, 21, 1.0), (517, 4096, 128, 22, 1.0), (40, 512, 16, 23, 1e-3)]
    for call, (M, K, k, seed, amp) in enumerate(shapes):
        x = (W.activations(M, K, max(1, K // 100), "t3x20", seed, seed).float() * amp).bfloat16().cuda()
        rng = np.random.default_rng(seed)
        chan = torch.from_numpy(np.sort(rng.choice(K, size=k, replace=False)).astype(np.int32)).cuda()
        ref = nv.nvfp4_quantize(x, chan=chan)            # existing entry point, caller workspace
        got = nv.nvfp4_quantize_noalloc(x, chan=chan)    # library-owned scratch
        torch.cuda.synchronize()
        assert nv.check_status()[0] == 0
        assert float(got["g"].item()) == float(ref["g"].item()), f"call {call}: tensor scale"
        assert np.array_equal(u8(got["codes"]), u8(ref["codes"])), f"call {call}: codes"
        n = nv.scale_bytes(M, K)
        assert np.array_equal(u8(got["scales"])[:n], u8(ref["scales"])[:n]) or _same_scales(got, ref, M, K), \
            f"call {call}: scale bytes"
        assert np.array_equal(bf16_bits_of(got["resid"]), bf16_bits_of(ref["resid"])), f"call {call}: residual"


def _same_scales(a, b, M, K):
    # padding bytes of the tiled layout are unspecified: compare the real ones
    from oracle import nvfp4 as onv
    off = onv.scale_tile_offsets(M, K // 16).ravel()
    return np.array_equal(u8(a["scales"])[off], u8(b["scales"])[off])
