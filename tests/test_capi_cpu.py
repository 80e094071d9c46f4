"""C-ABI surface checks that need no GPU: the library loads, exports every
symbol include/nvfp4w4a4.h declares, the size helpers agree with the oracle's
layout, and argument errors are reported before anything touches a device."""

import ctypes
import os
import re

import pytest

from oracle import nvfp4 as onv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4w4a4.h")


@pytest.fixture(scope="module")
def lib():
    from nvfp4_w4a4_gemm_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from nvfp4_w4a4_gemm_gb300 import build
        build.build()
    return binding.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return")))


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for n in ("nvfp4_quantize", "mxfp4_quantize", "w4a4_gemm_comp", "w4a4_grouped_gemm_comp"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from nvfp4_w4a4_gemm_gb300 import binding
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(binding.EXPORTED)


def test_version_and_status_strings(lib):
    assert lib.nvfp4_version() >= 10000
    assert lib.nvfp4_status_string(0) == b"ok"
    assert b"argument" in lib.nvfp4_status_string(1)


@pytest.mark.parametrize("M,K", [(1, 16), (64, 256), (130, 80), (8192, 4096), (16, 4096)])
def test_scale_bytes_match_oracle_layout(lib, M, K):
    assert lib.nvfp4_scale_bytes(M, K) == onv.scale_bytes(M, K)
    off = onv.scale_tile_offsets(M, K // 16)
    assert off.max() < lib.nvfp4_scale_bytes(M, K)


def test_grouped_scale_bytes_bound(lib):
    assert lib.nvfp4_grouped_scale_bytes(32768, 2048, 128) == onv.grouped_scale_bytes(32768, 2048, 128)


def test_invalid_arguments_rejected_on_host(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: validation fails first
    # K not a multiple of 16
    assert lib.nvfp4_quantize(fake, 4, 24, 24, None, None, fake, fake, None, 0, None, None, 0, None) == 1
    # misaligned x
    assert lib.nvfp4_quantize(P((1 << 20) + 2), 4, 32, 32, fake, None, fake, fake, None, 0, None, None, 0,
                              None) == 1
    # ldx < K
    assert lib.nvfp4_quantize(fake, 4, 32, 16, fake, None, fake, fake, None, 0, None, None, 0, None) == 1
    # k > 0 without channel list
    assert lib.nvfp4_quantize(fake, 4, 32, 32, fake, None, fake, fake, None, 4, fake, None, 0, None) == 1
    # MXFP4 needs K % 32
    assert lib.mxfp4_quantize(fake, 4, 48, 48, fake, fake, None, None, None) == 1
    # code buffers only 8-byte aligned (the kernels store 8 and 16 bytes at a time)
    odd8 = P((1 << 20) + 8)
    assert lib.nvfp4_quantize(fake, 4, 32, 32, fake, None, odd8, fake, None, 0, None, None, 0, None) == 1
    assert lib.mxfp4_quantize(fake, 4, 64, 64, odd8, fake, None, None, None) == 1
    # GEMM: bad format / flag / N not a multiple of 128
    assert lib.w4a4_gemm_comp(7, 4, 128, 64, fake, fake, None, fake, fake, None, None, None, 0, 0, fake,
                              None, 0, None) == 1
    assert lib.w4a4_gemm_comp(0, 4, 128, 64, fake, fake, None, fake, fake, None, None, None, 0, 9, fake,
                              None, 0, None) == 1
    assert lib.w4a4_gemm_comp(0, 4, 100, 64, fake, fake, None, fake, fake, None, None, None, 0, 0, fake,
                              None, 0, None) == 2
    # MXFP4: the fallback term takes the plain mode only, dense GEMMs only;
    # row scales are MXFP4's
    assert lib.w4a4_gemm_comp(1, 4, 128, 128, fake, fake, None, fake, fake, None, fake, fake, 16, 0x200, fake,
                              None, 0, None) == 1
    assert lib.w4a4_gemm_comp(1, 4, 128, 128, fake, fake, None, fake, fake, None, fake, fake, 16, 1, fake,
                              None, 0, None) == 1
    assert lib.w4a4_gemm_comp(0, 4, 128, 128, fake, fake, None, fake, fake, None, None, None, 0, 0x800, fake,
                              None, 0, None) == 1
    assert lib.w4a4_grouped_gemm_comp(1, 4, fake, 8, 128, 128, fake, fake, None, fake, fake, None, fake, fake,
                                      16, 0, fake, None, 0, None) == 2
    # corrected MXFP4 quantize: flag bits, row scales with the macro flag, the fallback list
    mxq = lambda flags, rs=fake, chan=None, k=0, fb=None: lib.mxfp4_quantize_ex(
        fake, 4, 64, 64, chan, k, flags, rs, fb, fake, fake, None, None, None)
    assert mxq(2) == 1
    assert mxq(1, rs=None) == 1
    assert mxq(0, k=8) == 1
    # grouped: missing offsets
    assert lib.w4a4_grouped_gemm_comp(0, 4, None, 8, 128, 64, fake, fake, None, fake, fake, None, None, None,
                                      0, 0, fake, None, 0, None) == 1
    # dynamic tensor scale without workspace
    assert lib.nvfp4_quantize(fake, 4, 32, 32, None, None, fake, fake, None, 0, None, None, 0, None) == 5
    # GEMM flag bits: the compensation mode, the weights-ready, the
    # pre-scaled-residual and the FP8-compensation bits; FP8 needs the
    # pre-scaled residual and the dequantized-weight mode
    for bad in (2, 0x400, 0x101 | 0x400, 0x800 | 0x200, 0x601):
        assert lib.w4a4_gemm_comp(0, 4, 128, 64, fake, fake, None, fake, fake, None, None, None, 0, bad, fake,
                                  None, 0, None) == 1
    assert lib.w4a4_grouped_gemm_comp(0, 4, fake, 8, 128, 64, fake, fake, None, fake, fake, None, None, None,
                                      0, 0x500, fake, None, 0, None) == 1
    # fused MoE GEMMs: the SwiGLU tile needs N % 256, h flags, h_k within N/2, the combine its row tables
    assert lib.w4a4_grouped_gemm_swiglu_quant(4, fake, 8, 384, 64, fake, fake, None, fake, fake, None, None, None,
                                              0, 0, fake, fake, 4, 0, fake, fake, fake, None, None) == 2
    assert lib.w4a4_grouped_gemm_swiglu_quant(4, fake, 8, 512, 64, fake, fake, None, fake, fake, None, None, None,
                                              0, 0, fake, fake, 4, 2, fake, fake, fake, None, None) == 1
    assert lib.w4a4_grouped_gemm_swiglu_quant(4, fake, 8, 512, 64, fake, fake, None, fake, fake, None, None, None,
                                              0, 0, fake, fake, 257, 0, fake, fake, fake, None, None) == 1
    assert lib.w4a4_grouped_gemm_combine(4, fake, 8, 512, 64, fake, fake, None, fake, fake, None, None, None, 0, 0,
                                         None, fake, 2, fake, None) == 1
    # one-launch decode layer: 1..16 tokens, N % 128, K % 64 and <= 8192, k <= 256 and % 8, known flags
    dec = lambda M, N, K, ldx, k, flags, chan=fake, ws=fake: lib.w4a4_decode_linear(
        M, N, K, fake, ldx, None, None, chan, k, fake, fake, None, ws, flags, fake, None)
    assert dec(17, 128, 256, 256, 0, 0) == 2
    assert dec(0, 128, 256, 256, 0, 0) == 1
    assert dec(4, 100, 256, 256, 0, 0) == 2
    assert dec(4, 128, 96, 96, 0, 0) == 2
    assert dec(4, 128, 8448, 8448, 0, 0) == 2
    assert dec(4, 128, 256, 256, 264, 0) == 2
    assert dec(4, 128, 256, 256, 12, 0) == 2
    assert dec(4, 128, 256, 200, 0, 0) == 1
    assert dec(4, 128, 256, 256, 0, 0x200) == 1
    assert dec(4, 128, 256, 256, 8, 0, chan=None) == 1
    # FP8 compensation: NVFP4 only, k % 16, dense GEMMs only
    gf8 = 0x400 | 0x200
    assert lib.w4a4_gemm_comp(1, 4, 128, 128, fake, fake, None, fake, fake, None, None, None, 0, gf8, fake,
                              None, 0, None) == 1
    assert lib.w4a4_gemm_comp(0, 4, 128, 64, fake, fake, None, fake, fake, None, fake, fake, 24, gf8, fake,
                              None, 0, None) == 2
    assert lib.w4a4_grouped_gemm_comp(0, 4, fake, 8, 128, 64, fake, fake, None, fake, fake, None, fake, fake,
                                      16, gf8, fake, None, 0, None) == 2
    assert lib.w4a4_grouped_gemm_combine(4, fake, 8, 512, 64, fake, fake, None, fake, fake, None, fake, fake, 16,
                                         gf8, fake, fake, 2, fake, None) == 2
    # quantizer flags: the pre-scaled-residual bit, and the E4M3-residual bit
    # with it (dense only)
    assert lib.nvfp4_quantize_ex(fake, 4, 32, 32, fake, None, fake, fake, None, 0, None, 2, None, 0, None) == 1
    assert lib.nvfp4_quantize_ex(fake, 4, 32, 32, fake, None, fake, fake, None, 0, None, 4, None, 0, None) == 1
    assert lib.nvfp4_quantize_grouped_ex(fake, 4, 32, 32, 1, fake, fake, None, fake, fake, None, 0, None, 4, None,
                                         0, None) == 1
    assert lib.nvfp4_quantize_grouped_ex(fake, 4, 32, 32, 1, fake, fake, None, fake, fake, None, 0, None, 3, None,
                                         0, None) == 1
    # compensation weight modes 0, 1, 2 (FP8 rows come from the codes)
    assert lib.nvfp4_prepare_comp_weights(1, 128, 64, fake, fake, None, fake, 8, 3, fake, None) == 1
    assert lib.nvfp4_prepare_comp_weights(1, 128, 64, None, None, fake, fake, 8, 2, fake, None) == 1
    # routed gather: token rows and a row table are required; flags and workspace as the grouped quantizer
    gat = lambda T, tok, flags=0, g=fake, ws=fake, wsb=1 << 16: lib.nvfp4_quantize_grouped_gather(
        fake, T, tok, 8, 32, 32, 1, fake, g, None, fake, fake, None, 0, None, flags, ws, wsb, None)
    assert gat(0, fake) == 1
    assert gat(-1, fake) == 1
    assert gat(4, None) == 1
    assert gat(4, P((1 << 20) + 2)) == 1
    assert gat(1 << 31, fake) == 1
    assert gat(4, fake, flags=2) == 1
    assert gat(4, fake, g=None, ws=None, wsb=0) == 5
    # QDQ: K % 16, strides, misaligned buffers, codes without scales, dynamic scale without workspace
    g = fake
    assert lib.nvfp4_qdq(fake, 4, 24, 24, g, None, fake, 24, None, None, None, 0, None) == 1
    assert lib.nvfp4_qdq(fake, 4, 32, 16, g, None, fake, 32, None, None, None, 0, None) == 1
    assert lib.nvfp4_qdq(fake, 4, 32, 32, g, None, fake, 20, None, None, None, 0, None) == 1
    assert lib.nvfp4_qdq(P((1 << 20) + 8), 4, 32, 32, g, None, fake, 32, None, None, None, 0, None) == 1
    assert lib.nvfp4_qdq(fake, 4, 32, 32, g, None, P((1 << 20) + 8), 32, None, None, None, 0, None) == 1
    assert lib.nvfp4_qdq(fake, 4, 32, 32, g, None, fake, 32, fake, None, None, 0, None) == 1
    assert lib.nvfp4_qdq(fake, 4, 32, 32, g, None, fake, 32, odd8, fake, None, 0, None) == 1
    assert lib.nvfp4_qdq(fake, 4, 32, 32, None, None, fake, 32, None, None, None, 0, None) == 5
    # per-element MXFP4 decomposition: K % 32, stride, alignment
    assert lib.mxfp4_decompose_elements(fake, 4, 48, 48, fake, None) == 1
    assert lib.mxfp4_decompose_elements(fake, 4, 64, 32, fake, None) == 1
    assert lib.mxfp4_decompose_elements(P((1 << 20) + 2), 4, 64, 64, fake, None) == 1
    assert lib.mxfp4_decompose_elements(fake, 4, 64, 64, P((1 << 20) + 2), None) == 1
    assert lib.mxfp4_decompose_elements(None, 0, 64, 64, None, None) == 0


def test_empty_problem_is_a_no_op(lib):
    fake = ctypes.c_void_p(1 << 20)
    # M == 0 with a static scale launches nothing and needs no device
    assert lib.w4a4_gemm_comp(0, 0, 128, 64, None, None, None, None, None, None, None, None, 0, 0, None,
                              None, 0, None) == 0
    assert lib.nvfp4_prepare_comp_weights(1, 128, 64, fake, fake, None, fake, 0, 0, fake, None) == 0


def test_binding_fails_loudly_without_the_library(tmp_path):
    # the product path has no fallback: a missing library is an error, not a
    # silent switch to other code
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, %r)\n"
            "from nvfp4_w4a4_gemm_gb300 import binding\n"
            "binding.LIB_PATH = %r\n"
            "try:\n    binding.load()\nexcept RuntimeError as e:\n    print('raised', e)\n") % (ROOT, str(tmp_path / "absent.so"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.startswith("raised"), r.stdout + r.stderr
