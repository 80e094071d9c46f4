"""Thin ctypes binding of ``libnvfp4w4a4.so`` (the C ABI in include/nvfp4w4a4.h).

Argument marshalling only: every function takes torch CUDA tensors, checks
dtype/device/contiguity, allocates the outputs with torch (device memory is
the caller's plumbing), and calls the C entry point of the same name on the
current torch stream.  Every step of the computation runs in the library's
CUDA kernels; there is no fallback path: if the library is missing or the
device is not sm_103, calls raise.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvfp4w4a4.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = range(6)
FMT_NVFP4, FMT_MXFP4 = 0, 1
COMP_W_DEQ, COMP_W_BF16, COMP_W_DEQ_FP8 = 0, 1, 2
GEMM_WEIGHTS_READY = 0x100  # flag bit: the weights are not written by work still pending on the stream
GEMM_RESID_SCALED = 0x200   # flag bit: resid is the pre-scaled residual of nvfp4_quantize(..., resid_scaled=True)
GEMM_COMP_FP8 = 0x400       # flag bit: resid / w_sel are E4M3 bytes (nvfp4_quantize(..., resid_fp8=True),
                            # nvfp4_prepare_comp_weights(..., flags=COMP_W_DEQ_FP8))
QUANT_RESID_SCALED, QUANT_RESID_FP8 = 1, 2
MXFP4_QUANT_MACRO = 1
GEMM_MX_ROW_SCALES = 0x800  # flag bit: MXFP4 operands carry row macro-block scales (g_a [M], g_b [N])

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t

_SIGS = {
    "nvfp4_version": ([], ctypes.c_int),
    "nvfp4_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "nvfp4_device_supported": ([ctypes.c_int], ctypes.c_int),
    "nvfp4_scale_bytes": ([_I64, _I64], _SZ),
    "mxfp4_scale_bytes": ([_I64, _I64], _SZ),
    "nvfp4_grouped_scale_bytes": ([_I64, _I64, _I32], _SZ),
    "nvfp4_quantize_workspace_bytes": ([], _SZ),
    "nvfp4_quantize": ([_P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _I32, _P, _P, _SZ, _P], ctypes.c_int),
    "nvfp4_quantize_grouped": ([_P, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, _P, _I32, _P, _P, _SZ, _P],
                               ctypes.c_int),
    "nvfp4_quantize_ex": ([_P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _I32, _P, ctypes.c_int, _P, _SZ, _P],
                          ctypes.c_int),
    "nvfp4_quantize_grouped_ex": ([_P, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, _P, _I32, _P, ctypes.c_int, _P,
                                   _SZ, _P], ctypes.c_int),
    "nvfp4_quantize_grouped_gather": ([_P, _I64, _P, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, _P, _I32, _P,
                                       ctypes.c_int, _P, _SZ, _P], ctypes.c_int),
    "nvfp4_quantize_noalloc": ([_P, _I64, _I64, _I64, _P, _P, _P, _P, _I32, _P, _P], ctypes.c_int),
    "mxfp4_quantize": ([_P, _I64, _I64, _I64, _P, _P, _P, _P, _P], ctypes.c_int),
    "mxfp4_quantize_ex": ([_P, _I64, _I64, _I64, _P, _I32, ctypes.c_int, _P, _P, _P, _P, _P, _P, _P],
                          ctypes.c_int),
    "mxfp4_decompose_elements": ([_P, _I64, _I64, _I64, _P, _P], ctypes.c_int),
    "nvfp4_qdq": ([_P, _I64, _I64, _I64, _P, _P, _P, _I64, _P, _P, _P, _SZ, _P], ctypes.c_int),
    "nvfp4_prepare_comp_weights": ([_I32, _I64, _I64, _P, _P, _P, _P, _I32, ctypes.c_int, _P, _P], ctypes.c_int),
    "nvfp4_calibrate_workspace_bytes": ([_I64, _I32], _SZ),
    "nvfp4_calibrate_channels": ([_P, _I64, _I64, _I64, _I32, _P, _I32, _P, _P, _SZ, _P], ctypes.c_int),
    "w4a4_gemm_workspace_bytes": ([_I64, _I64, _I64], _SZ),
    "w4a4_gemm_comp": ([ctypes.c_int, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _I32, ctypes.c_int, _P,
                        _P, _SZ, _P], ctypes.c_int),
    "w4a4_grouped_gemm_workspace_bytes": ([_I32, _I64, _I64, _I64], _SZ),
    "w4a4_grouped_gemm_comp": ([ctypes.c_int, _I32, _P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _I32,
                                ctypes.c_int, _P, _P, _SZ, _P], ctypes.c_int),
    "w4a4_grouped_gemm_swiglu_quant": ([_I32, _P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _I32,
                                        ctypes.c_int, _P, _P, _I32, ctypes.c_int, _P, _P, _P, _P, _P],
                                       ctypes.c_int),
    "w4a4_grouped_gemm_combine": ([_I32, _P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _I32, ctypes.c_int,
                                   _P, _P, _I64, _P, _P], ctypes.c_int),
    "w4a4_decode_linear": ([_I64, _I64, _I64, _P, _I64, _P, _P, _P, _I32, _P, _P, _P, _P, ctypes.c_int, _P, _P],
                           ctypes.c_int),
    "nvfp4_check_status": ([ctypes.c_int, ctypes.POINTER(ctypes.c_uint32)], ctypes.c_int),
    "nvfp4_set_wait_limit_ns": ([ctypes.c_uint64], ctypes.c_int),
    "nvfp4_inject_barrier_timeout": ([], None),
}

EXPORTED = tuple(_SIGS)


class NvfpError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({status_string(status)})")


def load(path=None):
    """Load (once) and return the ctypes library; raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} (run `python -m nvfp4_w4a4_gemm_gb300.build`)")
    lib = ctypes.CDLL(p)
    for name, (args, res) in _SIGS.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    if path is None:
        _lib = lib
    return lib


def status_string(status):
    return load().nvfp4_status_string(status).decode()


def _check(fn, status):
    if status != OK:
        raise NvfpError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t, dtype, name):
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor, got {t.dtype} on {t.device}")


def scale_bytes(rows, K):
    return load().nvfp4_scale_bytes(rows, K)


def mx_scale_bytes(rows, K):
    return load().mxfp4_scale_bytes(rows, K)


def grouped_scale_bytes(M_total, K, E):
    return load().nvfp4_grouped_scale_bytes(M_total, K, E)


def nvfp4_quantize(x, g=None, chan=None, out=None, g_out=None, resid_scaled=False, resid_fp8=False):
    """x bf16 [M, K] -> dict(codes u8 [M, K/2], scales u8 tiled, g f32 [1],
    resid bf16 [M, k]).  g: None (dynamic) or device float32 [1].
    resid_scaled: the residual comes divided by g (the GEMM's pre-scaled
    compensation operand; pass resid_scaled=True to the GEMM too).
    resid_fp8: the pre-scaled residual as E4M3 bytes (u8 [M, k]; implies
    resid_scaled), the operand of the FP8 compensation."""
    resid_scaled = resid_scaled or resid_fp8
    lib = load()
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    dev = x.device
    k = 0 if chan is None else int(chan.numel())
    if chan is not None:
        _need(chan, torch.int32, "chan")
    if g is not None:
        _need(g, torch.float32, "g")
    o = out or {}
    codes = o.get("codes") if o.get("codes") is not None else torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    scales = o.get("scales") if o.get("scales") is not None else torch.empty(
        lib.nvfp4_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    rdt = torch.uint8 if resid_fp8 else torch.bfloat16
    resid = o.get("resid") if o.get("resid") is not None else torch.empty((M, k), dtype=rdt, device=dev)
    if k:
        _need(resid, rdt, "resid")
    if g_out is None:
        g_out = torch.empty(1, dtype=torch.float32, device=dev)
    ws = o.get("ws")
    if ws is None and g is None:
        ws = torch.empty(lib.nvfp4_quantize_workspace_bytes(), dtype=torch.uint8, device=dev)
    flags = (QUANT_RESID_SCALED if resid_scaled else 0) | (QUANT_RESID_FP8 if resid_fp8 else 0)
    st = lib.nvfp4_quantize_ex(_ptr(x), M, K, x.stride(0), _ptr(g), _ptr(g_out), _ptr(codes), _ptr(scales),
                               _ptr(chan) if k else None, k, _ptr(resid) if k else None, flags, _ptr(ws),
                               0 if ws is None else ws.numel(), _stream())
    _check("nvfp4_quantize_ex", st)
    return dict(codes=codes, scales=scales, g=g_out, resid=resid, resid_scaled=bool(resid_scaled),
                resid_fp8=bool(resid_fp8))


def _need_rows(t, dtype, name):
    """A CUDA tensor of `dtype` whose rows are contiguous (any row stride)."""
    if not (t.is_cuda and t.dtype == dtype and t.dim() == 2 and t.stride(1) == 1):
        raise ValueError(f"{name}: expected a row-contiguous 2-D CUDA {dtype} tensor")


def nvfp4_qdq(w, g=None, with_codes=False, out=None):
    """Trainer-side fake quantization: w bf16 [M, K] -> dict(w_qdq bf16 [M, K],
    g f32 [1]) and, with with_codes, the packed codes and tiled scales of the
    same quantization (what nvfp4_quantize returns for w)."""
    lib = load()
    _need_rows(w, torch.bfloat16, "w")
    M, K = w.shape
    dev = w.device
    if g is not None:
        _need(g, torch.float32, "g")
    w_qdq = out if out is not None else torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    _need_rows(w_qdq, torch.bfloat16, "out")
    g_out = torch.empty(1, dtype=torch.float32, device=dev)
    codes = scales = None
    if with_codes:
        codes = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
        scales = torch.empty(lib.nvfp4_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    ws = None if g is not None else torch.empty(lib.nvfp4_quantize_workspace_bytes(), dtype=torch.uint8, device=dev)
    st = lib.nvfp4_qdq(_ptr(w), M, K, w.stride(0), _ptr(g), _ptr(g_out), _ptr(w_qdq), w_qdq.stride(0), _ptr(codes),
                       _ptr(scales), _ptr(ws), 0 if ws is None else ws.numel(), _stream())
    _check("nvfp4_qdq", st)
    r = dict(w_qdq=w_qdq, g=g_out)
    if with_codes:
        r.update(codes=codes, scales=scales)
    return r


def mxfp4_decompose_elements(x):
    """x bf16 [M, K] -> float32 [M, K, 3]: per-element (B, D, G) of the MXFP4
    error decomposition (small shapes; a checking aid)."""
    lib = load()
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    out = torch.empty((M, K, 3), dtype=torch.float32, device=x.device)
    st = lib.mxfp4_decompose_elements(_ptr(x), M, K, x.stride(0), _ptr(out), _stream())
    _check("mxfp4_decompose_elements", st)
    return out


def nvfp4_quantize_noalloc(x, chan=None, out=None, g_out=None):
    """nvfp4_quantize with a dynamic tensor scale and no workspace: for
    callers that cannot allocate device memory (the library keeps the
    scratch).  Outputs are allocated here unless given in ``out``."""
    lib = load()
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    dev = x.device
    k = 0 if chan is None else int(chan.numel())
    if chan is not None:
        _need(chan, torch.int32, "chan")
    o = out or {}
    codes = o.get("codes") if o.get("codes") is not None else torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    scales = o.get("scales") if o.get("scales") is not None else torch.empty(
        lib.nvfp4_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    resid = o.get("resid") if o.get("resid") is not None else torch.empty((M, k), dtype=torch.bfloat16, device=dev)
    if g_out is None:
        g_out = torch.empty(1, dtype=torch.float32, device=dev)
    st = lib.nvfp4_quantize_noalloc(_ptr(x), M, K, x.stride(0), _ptr(g_out), _ptr(codes), _ptr(scales),
                                    _ptr(chan) if k else None, k, _ptr(resid) if k else None, _stream())
    _check("nvfp4_quantize_noalloc", st)
    return dict(codes=codes, scales=scales, g=g_out, resid=resid)


def nvfp4_quantize_grouped(x, offsets, chan, g=None, g_out=None, resid_scaled=False):
    """Expert-sorted rows x [M_total, K], offsets int32 [E+1], chan int32 [E, k]."""
    lib = load()
    _need(x, torch.bfloat16, "x")
    _need(offsets, torch.int32, "offsets")
    _need(chan, torch.int32, "chan")
    M, K = x.shape
    E = offsets.numel() - 1
    k = chan.shape[1] if chan.dim() == 2 else 0
    dev = x.device
    codes = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty(lib.nvfp4_grouped_scale_bytes(M, K, E), dtype=torch.uint8, device=dev)
    resid = torch.empty((M, k), dtype=torch.bfloat16, device=dev)
    if g_out is None:
        g_out = torch.empty(1, dtype=torch.float32, device=dev)
    ws = torch.empty(lib.nvfp4_quantize_workspace_bytes(), dtype=torch.uint8, device=dev)
    st = lib.nvfp4_quantize_grouped_ex(_ptr(x), M, K, x.stride(0), E, _ptr(offsets), _ptr(g), _ptr(g_out),
                                       _ptr(codes), _ptr(scales), _ptr(chan) if k else None, k,
                                       _ptr(resid) if k else None, QUANT_RESID_SCALED if resid_scaled else 0,
                                       _ptr(ws), ws.numel(), _stream())
    _check("nvfp4_quantize_grouped_ex", st)
    return dict(codes=codes, scales=scales, g=g_out, resid=resid, resid_scaled=bool(resid_scaled))


def nvfp4_quantize_grouped_gather(x_tokens, token_of_row, offsets, chan, g=None, g_out=None, resid_scaled=False):
    """The routed operand x_tokens[token_of_row] (expert-sorted rows, offsets
    int32 [E+1], chan int32 [E, k]) quantized straight from the token rows
    x_tokens [T, K]; same result as nvfp4_quantize_grouped on the gathered rows."""
    lib = load()
    _need(x_tokens, torch.bfloat16, "x_tokens")
    _need(token_of_row, torch.int32, "token_of_row")
    _need(offsets, torch.int32, "offsets")
    _need(chan, torch.int32, "chan")
    T, K = x_tokens.shape
    M = token_of_row.numel()
    E = offsets.numel() - 1
    k = chan.shape[1] if chan.dim() == 2 else 0
    dev = x_tokens.device
    codes = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty(lib.nvfp4_grouped_scale_bytes(M, K, E), dtype=torch.uint8, device=dev)
    resid = torch.empty((M, k), dtype=torch.bfloat16, device=dev)
    if g_out is None:
        g_out = torch.empty(1, dtype=torch.float32, device=dev)
    ws = torch.empty(lib.nvfp4_quantize_workspace_bytes(), dtype=torch.uint8, device=dev)
    st = lib.nvfp4_quantize_grouped_gather(_ptr(x_tokens), T, _ptr(token_of_row), M, K, x_tokens.stride(0), E,
                                           _ptr(offsets), _ptr(g), _ptr(g_out), _ptr(codes), _ptr(scales),
                                           _ptr(chan) if k else None, k, _ptr(resid) if k else None,
                                           QUANT_RESID_SCALED if resid_scaled else 0, _ptr(ws), ws.numel(),
                                           _stream())
    _check("nvfp4_quantize_grouped_gather", st)
    return dict(codes=codes, scales=scales, g=g_out, resid=resid, resid_scaled=bool(resid_scaled))


def mxfp4_quantize(x, stats=False, chan=None, macro=False):
    """x bf16 [M, K] (K % 32 == 0) -> dict(codes, scales, stats f32 [M*K/32, 4], dead u8 [M*K/32]).
    chan (int32 [k], sorted) / macro: the corrected quantizer (Outlier
    Fallback on those channels, row macro-block scales); the dict then also
    holds fb bf16 [M, k] and m f32 [M] (None without macro)."""
    lib = load()
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    dev = x.device
    codes = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty(lib.mxfp4_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    st_t = torch.empty((M * K // 32, 4), dtype=torch.float32, device=dev) if stats else None
    dead = torch.empty(M * K // 32, dtype=torch.uint8, device=dev) if stats else None
    if chan is None and not macro:
        st = lib.mxfp4_quantize(_ptr(x), M, K, x.stride(0), _ptr(codes), _ptr(scales), _ptr(st_t), _ptr(dead),
                                _stream())
        _check("mxfp4_quantize", st)
        return dict(codes=codes, scales=scales, stats=st_t, dead=dead)
    k = 0 if chan is None else int(chan.numel())
    if k:
        _need(chan, torch.int32, "chan")
    fb = torch.empty((M, k), dtype=torch.bfloat16, device=dev)
    m = torch.empty(M, dtype=torch.float32, device=dev) if macro else None
    st = lib.mxfp4_quantize_ex(_ptr(x), M, K, x.stride(0), _ptr(chan) if k else None, k,
                               MXFP4_QUANT_MACRO if macro else 0, _ptr(m), _ptr(fb) if k else None, _ptr(codes),
                               _ptr(scales), _ptr(st_t), _ptr(dead), _stream())
    _check("mxfp4_quantize_ex", st)
    return dict(codes=codes, scales=scales, stats=st_t, dead=dead, fb=fb, m=m)


def nvfp4_prepare_comp_weights(b_codes, b_scales, chan, flags=COMP_W_DEQ, wt=None, E=1):
    """Compensation weight columns w_sel [E, N, k] (or [N, k] when E == 1):
    bf16, or E4M3 bytes for flags=COMP_W_DEQ_FP8."""
    lib = load()
    _need(chan, torch.int32, "chan")
    k = chan.shape[-1]
    if b_codes.dim() == 2:
        N, Kh = b_codes.shape
    else:
        E, N, Kh = b_codes.shape
    K = Kh * 2
    dev = b_codes.device
    w_sel = torch.empty((E, N, k), dtype=torch.uint8 if flags == COMP_W_DEQ_FP8 else torch.bfloat16, device=dev)
    st = lib.nvfp4_prepare_comp_weights(E, N, K, _ptr(b_codes), _ptr(b_scales), _ptr(wt), _ptr(chan), k, flags,
                                        _ptr(w_sel), _stream())
    _check("nvfp4_prepare_comp_weights", st)
    return w_sel[0] if E == 1 and b_codes.dim() == 2 else w_sel


def nvfp4_calibrate_channels(x_cal, k, offsets=None):
    """Channel sets int32 [k] (dense) or [E, k] (grouped by offsets)."""
    lib = load()
    _need(x_cal, torch.bfloat16, "x_cal")
    M, K = x_cal.shape
    E = 1 if offsets is None else offsets.numel() - 1
    ws = torch.empty(lib.nvfp4_calibrate_workspace_bytes(K, E), dtype=torch.uint8, device=x_cal.device)
    out = torch.empty((E, k), dtype=torch.int32, device=x_cal.device)
    st = lib.nvfp4_calibrate_channels(_ptr(x_cal), M, K, x_cal.stride(0), E, _ptr(offsets), k, _ptr(out),
                                      _ptr(ws), ws.numel(), _stream())
    _check("nvfp4_calibrate_channels", st)
    return out[0] if offsets is None else out


def w4a4_gemm_comp(qa, qb, N, resid=None, w_sel=None, flags=COMP_W_DEQ, fmt=FMT_NVFP4, y=None, ws=None,
                   weights_ready=False):
    """y [M, N] bf16 = block-scaled W4A4 product (+ compensation).  qa / qb
    are the dicts returned by the quantizers (qb for W^T [N, K]).
    weights_ready: qb and w_sel are not being written by work still pending on
    the stream, so the kernel may stream them while the preceding kernel runs."""
    if weights_ready:
        flags |= GEMM_WEIGHTS_READY
    if resid is not None and qa.get("resid_scaled"):
        flags |= GEMM_RESID_SCALED
    if resid is not None and qa.get("resid_fp8"):
        flags |= GEMM_COMP_FP8  # w_sel must then come from COMP_W_DEQ_FP8
    g_a, g_b = qa.get("g"), qb.get("g")
    if fmt == FMT_MXFP4 and (qa.get("m") is not None or qb.get("m") is not None):
        # corrected MXFP4 operands: both sides carry row macro-block scales
        flags |= GEMM_MX_ROW_SCALES
        g_a, g_b = qa["m"], qb["m"]
    lib = load()
    a_codes, b_codes = qa["codes"], qb["codes"]
    M, Kh = a_codes.shape
    K = Kh * 2
    k = 0 if resid is None else resid.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=a_codes.device)
    need = lib.w4a4_gemm_workspace_bytes(M, N, K)
    if need and ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=a_codes.device)
    st = lib.w4a4_gemm_comp(fmt, M, N, K, _ptr(a_codes), _ptr(qa["scales"]), _ptr(g_a),
                            _ptr(b_codes), _ptr(qb["scales"]), _ptr(g_b),
                            _ptr(resid) if k else None, _ptr(w_sel) if k else None, k, flags, _ptr(y),
                            _ptr(ws), 0 if ws is None else ws.numel(), _stream())
    _check("w4a4_gemm_comp", st)
    return y


def w4a4_decode_linear(x, qw, N, chan=None, w_sel=None, g=None, flags=COMP_W_DEQ, y=None, g_out=None,
                       weights_ready=False):
    """The whole layer for 1..16 tokens in one launch: y [M, N] bf16 from the
    bf16 activations x [M, K] (quantized inside the kernel: dynamic tensor
    scale, or g, a device float32 [1]), the quantized weights qw (the dict of
    nvfp4_quantize for W^T [N, K]) and the compensation columns w_sel [N, k]
    of the sorted channel list chan [k].  g_out: optional float32 [1]
    receiving the tensor scale used."""
    if weights_ready:
        flags |= GEMM_WEIGHTS_READY
    lib = load()
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    k = 0 if chan is None else int(chan.numel())
    if chan is not None:
        _need(chan, torch.int32, "chan")
    if g is not None:
        _need(g, torch.float32, "g")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    st = lib.w4a4_decode_linear(M, N, K, _ptr(x), x.stride(0), _ptr(g), _ptr(g_out), _ptr(chan) if k else None, k,
                                _ptr(qw["codes"]), _ptr(qw["scales"]), _ptr(qw.get("g")),
                                _ptr(w_sel) if k else None, flags, _ptr(y), _stream())
    _check("w4a4_decode_linear", st)
    return y


def w4a4_grouped_gemm_comp(qa, offsets, b_codes, b_scales, g_b, N, resid=None, w_sel=None, flags=COMP_W_DEQ,
                           y=None, weights_ready=False):
    """MoE: y [M_total, N] bf16; b_codes [E, N, K/2], b_scales E tiles, g_b [E].
    weights_ready: the weights, g_b, w_sel and offsets are not being written by
    work still pending on the stream."""
    if weights_ready:
        flags |= GEMM_WEIGHTS_READY
    if resid is not None and qa.get("resid_scaled"):
        flags |= GEMM_RESID_SCALED
    if resid is not None and qa.get("resid_fp8"):
        flags |= GEMM_COMP_FP8  # not built for grouped GEMMs: the library refuses it
    lib = load()
    a_codes = qa["codes"]
    M, Kh = a_codes.shape
    K = Kh * 2
    E = offsets.numel() - 1
    k = 0 if resid is None else resid.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=a_codes.device)
    st = lib.w4a4_grouped_gemm_comp(FMT_NVFP4, E, _ptr(offsets), M, N, K, _ptr(a_codes), _ptr(qa["scales"]),
                                    _ptr(qa.get("g")), _ptr(b_codes), _ptr(b_scales), _ptr(g_b),
                                    _ptr(resid) if k else None, _ptr(w_sel) if k else None, k, flags, _ptr(y),
                                    None, 0, _stream())
    _check("w4a4_grouped_gemm_comp", st)
    return y


def w4a4_grouped_gemm_swiglu_quant(qa, offsets, b_codes, b_scales, g_b, N, g_h, h_chan, resid=None, w_sel=None,
                                   flags=COMP_W_DEQ, h_resid_scaled=False, with_h=False, weights_ready=False):
    """MoE gate/up projection with SwiGLU and the down input's NVFP4 quantize
    (static scale g_h) in its epilogue.  b_codes/b_scales/w_sel hold the
    gate/up rows interleaved in blocks of 128 (N = 2 I).  Returns the down
    projection's quantized input dict(codes, scales, g, resid, resid_scaled)
    and, with with_h, h itself (bf16 [M, I])."""
    if weights_ready:
        flags |= GEMM_WEIGHTS_READY
    if resid is not None and qa.get("resid_scaled"):
        flags |= GEMM_RESID_SCALED
    if resid is not None and qa.get("resid_fp8"):
        flags |= GEMM_COMP_FP8  # not built for grouped GEMMs: the library refuses it
    lib = load()
    a_codes = qa["codes"]
    M, Kh = a_codes.shape
    K = Kh * 2
    E = offsets.numel() - 1
    k = 0 if resid is None else resid.shape[1]
    I = N // 2
    _need(h_chan, torch.int32, "h_chan")
    h_k = h_chan.shape[-1]
    dev = a_codes.device
    h_codes = torch.empty((M, I // 2), dtype=torch.uint8, device=dev)
    h_scales = torch.zeros(lib.nvfp4_grouped_scale_bytes(M, I, E), dtype=torch.uint8, device=dev)
    h_resid = torch.empty((M, h_k), dtype=torch.bfloat16, device=dev)
    h_out = torch.empty((M, I), dtype=torch.bfloat16, device=dev) if with_h else None
    st = lib.w4a4_grouped_gemm_swiglu_quant(E, _ptr(offsets), M, N, K, _ptr(a_codes), _ptr(qa["scales"]),
                                            _ptr(qa.get("g")), _ptr(b_codes), _ptr(b_scales), _ptr(g_b),
                                            _ptr(resid) if k else None, _ptr(w_sel) if k else None, k, flags,
                                            _ptr(g_h), _ptr(h_chan), h_k, QUANT_RESID_SCALED if h_resid_scaled else 0,
                                            _ptr(h_codes), _ptr(h_scales), _ptr(h_resid), _ptr(h_out), _stream())
    _check("w4a4_grouped_gemm_swiglu_quant", st)
    out = dict(codes=h_codes, scales=h_scales, g=g_h, resid=h_resid, resid_scaled=bool(h_resid_scaled))
    if with_h:
        out["h"] = h_out
    return out


def w4a4_grouped_gemm_combine(qa, offsets, b_codes, b_scales, g_b, N, token_of_row, w_row, n_tokens, resid=None,
                              w_sel=None, flags=COMP_W_DEQ, out=None, weights_ready=False):
    """MoE down projection with the routing-weighted combine in its epilogue:
    returns out fp32 [n_tokens, N] (zeroed here unless given; the kernel adds)."""
    if weights_ready:
        flags |= GEMM_WEIGHTS_READY
    if resid is not None and qa.get("resid_scaled"):
        flags |= GEMM_RESID_SCALED
    if resid is not None and qa.get("resid_fp8"):
        flags |= GEMM_COMP_FP8  # not built for grouped GEMMs: the library refuses it
    lib = load()
    a_codes = qa["codes"]
    M, Kh = a_codes.shape
    K = Kh * 2
    E = offsets.numel() - 1
    k = 0 if resid is None else resid.shape[1]
    _need(token_of_row, torch.int32, "token_of_row")
    _need(w_row, torch.float32, "w_row")
    if out is None:
        out = torch.zeros((n_tokens, N), dtype=torch.float32, device=a_codes.device)
    st = lib.w4a4_grouped_gemm_combine(E, _ptr(offsets), M, N, K, _ptr(a_codes), _ptr(qa["scales"]),
                                       _ptr(qa.get("g")), _ptr(b_codes), _ptr(b_scales), _ptr(g_b),
                                       _ptr(resid) if k else None, _ptr(w_sel) if k else None, k, flags,
                                       _ptr(token_of_row), _ptr(w_row), n_tokens, _ptr(out), _stream())
    _check("w4a4_grouped_gemm_combine", st)
    return out


def interleave_gate_up_rows(wt):
    """Weight-row layout of w4a4_grouped_gemm_swiglu_quant: W^T [..., 2I, K]
    with gate rows [0, I) and up rows [I, 2I) reordered so rows [256 j, 256 j
    + 128) are gate rows [128 j, 128 j + 128) and the next 128 the matching up
    rows (a one-time, offline reordering of the weights)."""
    two_i = wt.shape[-2]
    inter = two_i // 2
    if inter % 128:
        raise ValueError("the gate width must be a multiple of 128")
    idx = torch.arange(two_i).view(2, inter // 128, 128).transpose(0, 1).reshape(-1)
    return wt.index_select(wt.dim() - 2, idx.to(wt.device))


def check_status(clear=True):
    """Synchronizes and returns (status, detail) of the device error latch."""
    d = ctypes.c_uint32(0)
    st = load().nvfp4_check_status(1 if clear else 0, ctypes.byref(d))
    return st, d.value


def set_wait_limit_ns(ns):
    _check("nvfp4_set_wait_limit_ns", load().nvfp4_set_wait_limit_ns(int(ns)))


def inject_barrier_timeout():
    """Testing aid: the next dynamic-scale quantize launch's grid barrier is
    started one arrival short, so its bounded waits run out (one-shot)."""
    load().nvfp4_inject_barrier_timeout()
