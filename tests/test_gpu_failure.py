"""Failure detection on the GPU without a fault: a bounded device-side wait
that runs out, and routing offsets that do not partition the rows.

* The dynamic-scale quantizer's grid barrier is started one arrival short
  (nvfp4_inject_barrier_timeout), so no CTA is ever released.  With a 1 ms
  wait limit every CTA gives up, latches NVFP4_ERR_TIMEOUT at the grid
  barrier's wait site and returns before its quantize phase: none of the
  outputs may change.  The next call in the same process must be bit-exact
  with the oracle again (the context stays usable).
* Grouped launches given offsets that are not a partition of the rows
  latch NVFP4_ERR_INVALID_ARG and write nothing instead of indexing past
  the buffers.
* The routed quantizer given a token index outside [0, T) latches
  NVFP4_ERR_INVALID_ARG and reads token row 0 for that row instead.

Nothing here faults, traps or hangs a GPU: every wait is bounded and every
rejected launch returns before touching its outputs.
"""

import numpy as np
import pytest
import torch

from oracle import formats as F, nvfp4 as onv
from nvfp4_w4a4_gemm_gb300 import workloads as W
from tests.helpers import bf16_bits_of, f32, gather_scales, u8

pytestmark = pytest.mark.gpu

GRID_BARRIER_SITE = 20


@pytest.fixture(scope="module")
def nv():
    from nvfp4_w4a4_gemm_gb300 import binding
    binding.load()
    assert binding.check_status()[0] == 0
    yield binding
    binding.set_wait_limit_ns(2_000_000_000)


def _sentinel_outputs(M, K, k, nv):
    dev = torch.device("cuda")
    return dict(codes=torch.full((M, K // 2), 0xA5, dtype=torch.uint8, device=dev),
                scales=torch.full((nv.scale_bytes(M, K),), 0x5A, dtype=torch.uint8, device=dev),
                resid=torch.full((M, k), -3.0, dtype=torch.bfloat16, device=dev),
                ws=torch.zeros(nv.load().nvfp4_quantize_workspace_bytes(), dtype=torch.uint8, device=dev))


@pytest.mark.parametrize("M,K,k", [(512, 4096, 128), (16, 4096, 64)])
def test_grid_barrier_timeout_reported_then_recovers(nv, M, K, k):
    x_cpu = W.activations(M, K, 41, "t3x20", 90 + M, 91 + M)
    x = x_cpu.cuda()
    rng = np.random.default_rng(M)
    chan_np = np.sort(rng.choice(K, size=k, replace=False))
    chan = torch.from_numpy(chan_np.astype(np.int32)).cuda()
    out = _sentinel_outputs(M, K, k, nv)
    g_out = torch.full((1,), -7.0, dtype=torch.float32, device="cuda")

    nv.set_wait_limit_ns(1_000_000)
    nv.inject_barrier_timeout()
    nv.nvfp4_quantize(x, chan=chan, out=out, g_out=g_out)
    st, where = nv.check_status()          # synchronizes, then clears the latch
    assert st == nv.ERR_TIMEOUT and where == GRID_BARRIER_SITE, (st, where)
    # no CTA passed the barrier: every output keeps its sentinel
    assert bool((out["codes"] == 0xA5).all())
    assert bool((out["scales"] == 0x5A).all())
    assert bool((out["resid"] == -3.0).all())
    assert float(g_out.item()) == -7.0

    # the same process, the same buffers: the next call is exact again
    nv.set_wait_limit_ns(2_000_000_000)
    q = nv.nvfp4_quantize(x, chan=chan, out=out, g_out=g_out)
    assert nv.check_status()[0] == 0
    ref = onv.quantize(f32(x_cpu), chan=chan_np)
    assert f32(q["g"])[0] == ref["g"]
    assert np.array_equal(u8(q["codes"]), ref["packed"])
    assert np.array_equal(gather_scales(q["scales"], onv.scale_tile_offsets(M, K // 16)), ref["sigma"])
    assert np.array_equal(bf16_bits_of(q["resid"]), F.bf16_bits(ref["resid_f32"][:, chan_np]))


def test_qdq_grid_barrier_timeout(nv):
    w = W.weights_t(256, 1024, 5).cuda()
    y = torch.full_like(w, 9.0)
    nv.set_wait_limit_ns(1_000_000)
    nv.inject_barrier_timeout()
    nv.nvfp4_qdq(w, out=y)
    st, where = nv.check_status()
    assert st == nv.ERR_TIMEOUT and where == GRID_BARRIER_SITE
    assert bool((y == 9.0).all())
    nv.set_wait_limit_ns(2_000_000_000)
    r = nv.nvfp4_qdq(w, out=y)
    assert nv.check_status()[0] == 0
    want, _ = onv.qdq(f32(w.cpu()))
    assert np.array_equal(bf16_bits_of(r["w_qdq"]), F.bf16_bits(want))


@pytest.mark.parametrize("bad", ["decreasing", "first_nonzero", "last_short", "last_long"])
def test_grouped_offsets_not_a_partition_are_rejected(nv, bad):
    E, K, N, k = 6, 256, 256, 16
    counts = [40, 0, 130, 7, 1, 82]
    M = sum(counts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    if bad == "decreasing":
        offs[3] = offs[2] - 5
    elif bad == "first_nonzero":
        offs[0] = 3
    elif bad == "last_short":
        offs[-1] = M - 1
    else:
        offs[-1] = M + 64
    x = W.activations(M, K, 3, "t3x20", 31, 32).cuda()
    offsets = torch.from_numpy(offs).cuda()
    chan = torch.stack([torch.arange(0, 256, 16, dtype=torch.int32)] * E).cuda()
    with torch.no_grad():
        q = nv.nvfp4_quantize_grouped(x, offsets, chan, g=torch.ones(1, device="cuda"))
    st, where = nv.check_status()
    assert st == nv.ERR_INVALID_ARG and where == 0x200, (st, where)

    # the grouped GEMM with the same bad table: no tile runs, Y keeps its sentinel
    good = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).cuda()
    qa = nv.nvfp4_quantize_grouped(x, good, chan)
    wt = torch.stack([W.weights_t(N, K, 40 + e) for e in range(E)]).cuda()
    qs = [nv.nvfp4_quantize(wt[e]) for e in range(E)]
    b_codes = torch.stack([s["codes"] for s in qs])
    b_scales = torch.cat([s["scales"] for s in qs])
    g_b = torch.cat([s["g"] for s in qs])
    w_sel = nv.nvfp4_prepare_comp_weights(b_codes, b_scales, chan, E=E)
    assert nv.check_status()[0] == 0
    y = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
    nv.w4a4_grouped_gemm_comp(qa, offsets, b_codes, b_scales, g_b, N, resid=qa["resid"], w_sel=w_sel, y=y)
    st, where = nv.check_status()
    assert st == nv.ERR_INVALID_ARG and where == 0x300, (st, where)
    assert bool((y == 5.0).all())
    # and with the good table the same call runs and leaves no error behind
    nv.w4a4_grouped_gemm_comp(qa, good, b_codes, b_scales, g_b, N, resid=qa["resid"], w_sel=w_sel, y=y)
    assert nv.check_status()[0] == 0
    assert not bool((y == 5.0).all())


@pytest.mark.parametrize("bad", ["decreasing", "last_long"])
def test_grouped_pair_tiles_reject_bad_offsets(nv, bad):
    # experts large enough for the 256-row pair tiles: the pair kernel checks
    # the table before any copy, and both CTAs of every pair return
    E, K, N = 3, 256, 256
    counts = [300, 260, 250]
    M = sum(counts)
    good = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    offs = good.copy()
    if bad == "decreasing":
        offs[2] = offs[1] - 7
    else:
        offs[-1] = M + 256
    x = W.activations(M, K, 3, "t3x20", 51, 52).cuda()
    chan = torch.stack([torch.arange(0, 256, 16, dtype=torch.int32)] * E).cuda()
    qa = nv.nvfp4_quantize_grouped(x, torch.from_numpy(good).cuda(), chan)
    wt = torch.stack([W.weights_t(N, K, 60 + e) for e in range(E)]).cuda()
    qs = [nv.nvfp4_quantize(wt[e]) for e in range(E)]
    b_codes = torch.stack([s["codes"] for s in qs])
    b_scales = torch.cat([s["scales"] for s in qs])
    g_b = torch.cat([s["g"] for s in qs])
    w_sel = nv.nvfp4_prepare_comp_weights(b_codes, b_scales, chan, E=E)
    assert nv.check_status()[0] == 0
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    nv.w4a4_grouped_gemm_comp(qa, torch.from_numpy(offs).cuda(), b_codes, b_scales, g_b, N, resid=qa["resid"],
                              w_sel=w_sel, y=y)
    st, where = nv.check_status()
    assert st == nv.ERR_INVALID_ARG and where == 0x300, (st, where)
    assert bool(torch.isnan(y).all())
    # the good table writes every row
    nv.w4a4_grouped_gemm_comp(qa, torch.from_numpy(good).cuda(), b_codes, b_scales, g_b, N, resid=qa["resid"],
                              w_sel=w_sel, y=y)
    assert nv.check_status()[0] == 0
    assert not bool(torch.isnan(y).any())


@pytest.mark.parametrize("bad", [-1, 37, 1 << 30])
def test_gather_index_out_of_range_reported(nv, bad):
    T, K, E, k = 37, 256, 3, 8
    offs = torch.tensor([0, 10, 10, 25], dtype=torch.int32).cuda()
    tok = torch.arange(25, dtype=torch.int32) % T
    tok[7] = bad
    xt = W.activations(T, K, 3, "t3x20", 41, 42)
    chan = torch.stack([torch.arange(0, K, K // k, dtype=torch.int32)] * E).cuda()
    g = torch.ones(1, device="cuda")
    q = nv.nvfp4_quantize_grouped_gather(xt.cuda(), tok.cuda(), offs, chan, g=g)
    st, where = nv.check_status()
    assert st == nv.ERR_INVALID_ARG and where == 0x210, (st, where)
    # the bad row was read as token row 0; every other row is its token's
    good = tok.clone()
    good[7] = 0
    ref = nv.nvfp4_quantize_grouped(xt[good.long()].cuda(), offs, chan, g=g)
    assert nv.check_status()[0] == 0
    for key in ("codes", "resid"):
        assert torch.equal(q[key], ref[key]), key
    tiles = onv.grouped_scale_tile_offsets(offs.cpu().numpy(), K // 16)
    assert np.array_equal(gather_scales(q["scales"], tiles), gather_scales(ref["scales"], tiles))
