"""MoE pieces around the grouped W4A4 GEMMs (test infrastructure only): the
gated activation between the two projections, the routing weights and the
weighted combine of the experts' outputs.

Source.  QUADS abstract (arXiv 2607.15810): the rollout model is an MoE whose
linear layers run as native W4A4 GEMMs; gist.science explainer of QUADS,
Technisches Resuemee section 4: a 25B-parameter MoE.  The pages name the MoE
but define neither its gated activation nor how the experts' outputs are
combined, so the readings below are this library's.

Readings:

* Gated activation (SwiGLU): the gate/up projection's 2*I outputs of a row
  are I gate values a_j and I up values b_j; h_j = silu(a_j) * b_j with
  silu(z) = z / (1 + exp(-z)).  a_j and b_j are the projection's bf16
  outputs (what the unfused GEMM writes); h is rounded to bf16, the dtype the
  down projection's quantizer reads.
* Down-projection input quantization in the fused path: the static-scale
  NVFP4 quantizer (a tensor scale given, e.g. from a calibration batch), since
  a dynamic scale needs the amax of all of h before any block can be coded.
* Routing weights: softmax over the experts of a token's router logits, the
  top-8 kept (ties to the lower expert id) and renormalized to sum to 1.
* Combine: out[t] = sum over the token's routed rows r of w_r * y_down[r],
  accumulated in fp32 (fp64 here).
"""

import numpy as np

from .formats import bf16_round


def silu(z):
    """z * sigmoid(z) in fp64 (stable for large |z|)."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = z[pos] / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = z[~pos] * ez / (1.0 + ez)
    return out


def swiglu(gate_bf16, up_bf16):
    """h = bf16(silu(a) * b) for bf16-valued a (gate) and b (up), [R, I]."""
    a = np.asarray(gate_bf16, dtype=np.float64)
    b = np.asarray(up_bf16, dtype=np.float64)
    return bf16_round((silu(a) * b).astype(np.float32))


def route_weights(logits, top):
    """Renormalized top-`top` softmax weights.  Returns (experts [T, top]
    int64, weights [T, top] fp64); ties go to the lower expert id."""
    lg = np.asarray(logits, dtype=np.float64)
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    T, E = p.shape
    idx = np.arange(E)
    experts = np.stack([np.lexsort((idx, -p[t]))[:top] for t in range(T)])
    w = np.take_along_axis(p, experts, axis=1)
    return experts.astype(np.int64), w / w.sum(axis=1, keepdims=True)


def row_weights(experts, weights, token_of_row, offsets):
    """Weight of every expert-sorted routed row: row r is token token_of_row[r]
    routed to the expert e with offsets[e] <= r < offsets[e+1]."""
    token_of_row = np.asarray(token_of_row, dtype=np.int64)
    offsets = np.asarray(offsets, dtype=np.int64)
    w = np.zeros(token_of_row.size, np.float64)
    for e in range(offsets.size - 1):
        for r in range(offsets[e], offsets[e + 1]):
            t = token_of_row[r]
            hit = np.nonzero(experts[t] == e)[0]
            if hit.size != 1:
                raise ValueError(f"row {r}: token {t} is not routed to expert {e}")
            w[r] = weights[t, hit[0]]
    return w


def combine(y_rows, token_of_row, w_rows, n_tokens):
    """out[t] = sum_r w_r y_rows[r] over the rows of token t (fp64)."""
    y = np.asarray(y_rows, dtype=np.float64)
    out = np.zeros((n_tokens, y.shape[1]), np.float64)
    np.add.at(out, np.asarray(token_of_row, dtype=np.int64), y * np.asarray(w_rows, np.float64)[:, None])
    return out


def interleave_gate_up(wt_gate_up, tile_cols=256):
    """Row order of a gate/up weight W^T [2I, K] (gate rows 0..I-1, up rows
    I..2I-1) for the fused kernel: each 256-row tile holds 128 gate rows and
    the 128 matching up rows, so one output tile carries both halves of its
    128 activations.  Returns (permuted W^T, perm) with perm[i] = source row of
    permuted row i."""
    w = np.asarray(wt_gate_up)
    two_i = w.shape[-2]
    inter = two_i // 2
    half = tile_cols // 2
    if inter % half:
        raise ValueError("the gate width must be a multiple of 128")
    perm = np.empty(two_i, np.int64)
    for j in range(inter // half):
        perm[j * tile_cols: j * tile_cols + half] = np.arange(j * half, (j + 1) * half)
        perm[j * tile_cols + half: (j + 1) * tile_cols] = inter + np.arange(j * half, (j + 1) * half)
    return np.take(w, perm, axis=-2), perm
