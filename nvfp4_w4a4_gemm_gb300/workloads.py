"""Seeded synthetic inputs for the five NVFP4 / MXFP4 linear-layer workloads.

This module only draws random numbers and arranges them (outlier channels,
MoE routing and the expert sort); it holds none of the quantization or GEMM
arithmetic.  Every draw uses a CPU ``torch.Generator`` so the same seed gives
the same tensors on any machine.

Workloads (shapes from the problem statement; distributions as stated):

tiny     X [64, 256] ~ N(0,1) with 4 fixed channels scaled x50;
         W [256, 128] ~ N(0, 0.02^2); k = 8.
decode   X [16, 4096]: 1 % of channels (41) Student-t(nu=3) x 20, the rest
         N(0,1); W [4096, 14336] ~ N(0, 0.02^2); k = 64.
prefill  X [8192, 4096] with the same outlier mix; W [4096, 4096]; k = 128.
moe      4096 tokens, hidden 2048 (20 outlier channels), 128 experts,
         top-8 of softmax(N(0,1) logits) (ties to the lower expert id);
         routed rows sorted by (expert, token) -> offsets [129];
         gate/up W_e [2048, 1536], down W_e [768, 2048] per expert; the down
         input is its own draw [32768, 768] with 8 outlier channels; k = 32
         per expert.
mxfp4    X [8192, 5120], 51 channels Student-t(3) x 20; W [5120, 5120];
         32-element blocks, no compensation (k = 0).

Weights are returned transposed, W^T [N, K] row-major, which is the layout
the GEMM consumes (both operands block along K); W^T's entries are iid so
drawing W^T directly has the same distribution as drawing W.

Seeds: workload i uses seed i for its data draw; the calibration batch uses
seed + 1000 with the same outlier channel identities (which come from
randperm(K) under the workload seed); weights use seed + 500.
"""

import math
from dataclasses import dataclass

import torch

WORKLOADS = ("tiny", "decode", "prefill", "moe", "mxfp4")


@dataclass(frozen=True)
class Dense:
    name: str
    M: int
    K: int
    N: int
    k: int
    n_out: int
    outlier: str  # "x50" or "t3x20"
    seed: int
    fmt: str = "nvfp4"


@dataclass(frozen=True)
class MoE:
    name: str
    tokens: int
    hidden: int
    inter: int     # down-proj input width (gate/up width is 2 * inter)
    experts: int
    top: int
    k: int
    seed: int


def _n_outliers(K):
    return int(round(0.01 * K))


SPECS = {
    "tiny": Dense("tiny", 64, 256, 128, 8, 4, "x50", 0),
    "decode": Dense("decode", 16, 4096, 14336, 64, _n_outliers(4096), "t3x20", 1),
    "prefill": Dense("prefill", 8192, 4096, 4096, 128, _n_outliers(4096), "t3x20", 2),
    "moe": MoE("moe", 4096, 2048, 768, 128, 8, 32, 3),
    "mxfp4": Dense("mxfp4", 8192, 5120, 5120, 0, _n_outliers(5120), "t3x20", 4, "mxfp4"),
}


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def outlier_channels(K, n, seed):
    """Sorted ids of the n outlier channels: the first n of randperm(K)."""
    perm = torch.randperm(K, generator=_gen(seed))
    return torch.sort(perm[:n]).values


def student_t3(shape, g):
    """Student-t with 3 degrees of freedom: z / sqrt(chi2_3 / 3)."""
    z = torch.randn(shape, generator=g)
    c = torch.randn((3,) + tuple(shape), generator=g).pow(2).sum(0)
    return z / torch.sqrt(c / 3.0)


def activations(M, K, n_out, outlier, channel_seed, value_seed):
    """bf16 [M, K]: N(0,1) with n_out outlier channels."""
    g = _gen(value_seed)
    x = torch.randn(M, K, generator=g)
    ids = outlier_channels(K, n_out, channel_seed)
    if outlier == "x50":
        x[:, ids] *= 50.0
    elif outlier == "t3x20":
        x[:, ids] = student_t3((M, len(ids)), g) * 20.0
    else:
        raise ValueError(outlier)
    return x.to(torch.bfloat16)


def weights_t(N, K, seed, experts=None):
    """bf16 W^T [N, K] (or [E, N, K]) ~ N(0, 0.02^2)."""
    g = _gen(seed)
    shape = (N, K) if experts is None else (experts, N, K)
    w = torch.empty(shape, dtype=torch.bfloat16)
    flat = w.view(-1, K)
    step = 1 << 14
    for r0 in range(0, flat.shape[0], step):   # chunked to bound fp32 temp memory
        r1 = min(flat.shape[0], r0 + step)
        flat[r0:r1] = (torch.randn(r1 - r0, K, generator=g) * 0.02).to(torch.bfloat16)
    return w


def route(tokens, experts, top, seed, with_weights=False):
    """Top-``top`` routing of softmax(N(0,1) logits); routed (token, expert)
    pairs sorted by (expert, token).  Returns (token_of_row int64 [T*top],
    offsets int32 [E+1]); with_weights also returns the routing weight of every
    sorted row (the token's top-``top`` softmax probabilities renormalized to
    sum to 1, fp32; the router's output, an input of the combine) and the
    logits."""
    g = _gen(seed)
    logits = torch.randn(tokens, experts, generator=g)
    p = torch.softmax(logits, dim=1)
    srt = torch.sort(p, dim=1, descending=True, stable=True)
    order = srt.indices[:, :top]
    tok = torch.arange(tokens).repeat_interleave(top)
    exp = order.reshape(-1)
    key = exp * tokens + tok
    perm = torch.sort(key, stable=True).indices
    tok_sorted = tok[perm]
    counts = torch.bincount(exp, minlength=experts)
    offsets = torch.zeros(experts + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(counts, 0).to(torch.int32)
    if not with_weights:
        return tok_sorted, offsets
    w = srt.values[:, :top]
    w = (w / w.sum(dim=1, keepdim=True)).reshape(-1)[perm].to(torch.float32)
    return tok_sorted, offsets, w, logits


def dense_inputs(name, calibration=False, with_weights=True):
    """Inputs of a dense workload as CPU tensors: dict(x, wt, spec)."""
    s = SPECS[name]
    vs = s.seed + (1000 if calibration else 0)
    out = dict(spec=s, x=activations(s.M, s.K, s.n_out, s.outlier, s.seed, vs))
    if with_weights:
        out["wt"] = weights_t(s.N, s.K, s.seed + 500)
    return out


def moe_inputs(calibration=False, with_weights=True, which=("gate_up", "down")):
    """MoE workload inputs (CPU).  Keys: x_tokens [T, hidden] (the token
    rows), x_gate_up [T*top, hidden] (x_tokens[token_of_row]: the sorted
    rows), x_down [T*top, inter], offsets, token_of_row, route_weight (per
    sorted row), and the weights
    wt_gate_up [E, 2*inter, hidden], wt_down [E, hidden, inter]."""
    s = SPECS["moe"]
    vs = s.seed + (1000 if calibration else 0)
    tok, offsets, w_rows, _ = route(s.tokens, s.experts, s.top, vs + 7, with_weights=True)
    out = dict(spec=s, offsets=offsets, token_of_row=tok, route_weight=w_rows)
    if "gate_up" in which:
        xt = activations(s.tokens, s.hidden, _n_outliers(s.hidden), "t3x20", s.seed, vs)
        out["x_tokens"] = xt
        out["x_gate_up"] = xt[tok].contiguous()
    if "down" in which:
        rows = s.tokens * s.top
        out["x_down"] = activations(rows, s.inter, _n_outliers(s.inter), "t3x20", s.seed + 100, vs + 100)
    if with_weights:
        if "gate_up" in which:
            out["wt_gate_up"] = weights_t(2 * s.inter, s.hidden, s.seed + 500, s.experts)
        if "down" in which:
            out["wt_down"] = weights_t(s.hidden, s.inter, s.seed + 600, s.experts)
    return out


def random_bf16(shape, seed, scale=1.0):
    """Plain N(0, scale^2) bf16 tensor for edge-case tests."""
    return (torch.randn(shape, generator=_gen(seed)) * scale).to(torch.bfloat16)


def flops_dense(M, N, K):
    return 2.0 * M * N * K


def ceil_div(a, b):
    return -(-a // b)


__all__ = ["SPECS", "WORKLOADS", "dense_inputs", "moe_inputs", "route", "activations",
           "weights_t", "random_bf16", "outlier_channels", "student_t3", "math"]
