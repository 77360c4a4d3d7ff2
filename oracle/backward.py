"""Training backward of the routed-MoE layer, in plain fp64 numpy.

TEST INFRASTRUCTURE ONLY: part of the CPU oracle (see oracle/moe.py).

What the pages fix: the backward GroupGemm epilogue reads the GEMM output,
computes dSwiGLU, quantises, and writes back (NVIDIA blog "Boosting MoE
training throughput with advanced fusion kernels", kernel families list and
section on GLU epilogue fusion); MXFP8 training keeps a row-quantised copy
and a transposed (column-quantised) copy of each GEMM operand for the
backward (same blog, section on fusing MXFP8/NVFP4 quantisation).

Readings taken (listed in the design notes):
  * every quantiser is straight-through: gradients pass it unchanged;
  * the backward reads the pre-activation h rounded to bf16 (the saved copy);
  * operands contracted over the token axis (wgrad) are MXFP8-quantised in
    blocks of 32 rows within each expert, the expert's rows padded with zero
    rows to a multiple of 32; the activation operand is quantised this way
    from x itself (not from its row-quantised copy), the W2 input from the
    unquantised SwiGLU output y;
  * dgrad GEMMs use weight copies quantised along the other axis;
  * the router Jacobian is the one of softmax over the k selected logits,
    times routed_scale; unselected logits get zero gradient.
Parity pins: tests/test_oracle_backward.py (central finite differences of
the unquantised layer).
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import formats as F
from .moe import Forward, act_bwd, act_fwd, act_plain, act_plain_bwd, gated, values


def _q_rows(v, quant):
    """MXFP8 round trip along the last axis (identity when quant is False)."""
    if not quant:
        return np.asarray(v, np.float64)
    q, s = F.mx_quantize(v)
    return F.mx_dequantize(q, s)


def _q_cols(v, quant):
    """MXFP8 round trip along axis 0 in blocks of 32 rows; rows padded with
    zeros to a multiple of 32 first (identity when quant is False)."""
    v = np.asarray(v, np.float64)
    if not quant:
        return v
    n = v.shape[0]
    npad = (n + 31) // 32 * 32
    p = np.zeros((npad,) + v.shape[1:])
    p[:n] = v
    q, s = F.mx_quantize(p.T)                 # blocks along the padded row axis
    return F.mx_dequantize(q, s).T[:n]


@dataclasses.dataclass
class Backward:
    dx: np.ndarray       # fp64 [T, H]
    dW1: np.ndarray      # fp64 [G, H, 2I]   (logical W1 layout: H x (gate|up); sReLU: [G, H, I])
    dW2: np.ndarray      # fp64 [G, I, H]
    dlogits: np.ndarray  # fp64 [T, E]
    dw_row: np.ndarray   # fp64 [R]
    dh: np.ndarray       # fp64 [R, 2I] (sReLU: [R, I])
    dY1: np.ndarray      # fp64 [R, I]
    db1: np.ndarray      # fp64 [G, 2I]: gradient of W1's bias (gate b then up c)


def layer_backward(fwd: Forward, x_bits, dout_bits, wts: dict, *, E: int, k: int,
                   routed_scale: float = 1.0, act: str = "swiglu", alpha: float = 1.0,
                   limit: float = 0.0, quant: bool = True, experts=None,
                   w1t=None, w2t=None) -> Backward:
    """Gradients of L = sum(dOut * out) for the layer computed by ``fwd``.

    Weights for the dgrad GEMMs come from ``w1t(e)`` -> [H, 2I] ([H, I] for
    the non-gated sReLU) and ``w2t(e)`` -> [I, H] (decoded fp64).
    ``experts`` restricts the work to a subset of expert groups (others
    leave zeros / NaN rows). With a W1 bias (h = xW + b | xV + c) the
    backward is unchanged but for the bias gradient db1[e] = the sum of dh
    over the group's rows. The backward kernel family of the NVIDIA fusion
    blog (GroupGemm + dActivation + Quantize/Transpose) covers SwiGLU, GeGLU
    and sReLU; for sReLU dh = w_row * dY1 * 2 max(h, 0) over W1's I outputs.
    """
    x = values(x_bits)
    dout = values(dout_bits)
    T, H = x.shape
    d = fwd.disp
    G = len(d.counts)
    kp = len(d.inv) // max(T, 1) if T else k
    R = len(d.perm_src)
    I = fwd.y.shape[1]
    N1 = 2 * I if gated(act) else I                    # W1 outputs
    want = np.zeros(G, bool)
    want[list(range(G)) if experts is None else list(experts)] = True
    dY1 = np.full((R, I), np.nan)
    dh = np.full((R, N1), np.nan)
    dXp = np.full((R, H), np.nan)
    dw_row = np.full(R, np.nan)
    dW1 = np.zeros((G, H, N1))
    db1 = np.zeros((G, N1))
    dW2 = np.zeros((G, I, H))
    for e in range(G):
        lo, hi = d.offsets[e], d.offsets[e + 1]
        if not want[e] or hi == lo:
            continue                                   # empty expert: zero grads
        rs = np.arange(lo, hi)
        toks = d.perm_src[rs] // kp
        dz = dout[toks]                                # [n, H]
        # dY1 = dz . W2^T  (contraction over H; W2 copy quantised along H)
        dy = _q_rows(dz, quant) @ w2t(e).T             # [n, I]
        hb = fwd.h[rs]
        if quant:                                      # saved h is bf16
            hb = F.bf16_to_f64(F.f64_to_bf16(hb))
        if gated(act):
            g, u = hb[:, :I], hb[:, I:]
            a_val = act_fwd(g, u, act, alpha, limit)
            dw_row[rs] = (dy * a_val).sum(axis=1)
            dg, du = act_bwd(g, u, d.w_row[rs, None] * dy, act, alpha, limit)
            dhe = np.concatenate([dg, du], axis=1)     # [n, 2I]
        else:
            a_val = act_plain(hb, act)
            dw_row[rs] = (dy * a_val).sum(axis=1)
            dhe = act_plain_bwd(hb, d.w_row[rs, None] * dy, act)   # [n, I]
        # dXp = dh . W1^T (contraction over N1; W1 copy quantised along N1)
        dXp[rs] = _q_rows(dhe, quant) @ w1t(e).T       # [n, H]
        # wgrads: contraction over the expert's rows
        a_cols = _q_cols(x[toks], quant)               # [n, H]
        dW1[e] = a_cols.T @ _q_cols(dhe, quant)        # [H, N1]
        dW2[e] = _q_cols(fwd.y[rs], quant).T @ _q_cols(dz, quant)   # [I, H]
        dY1[rs], dh[rs] = dy, dhe
        db1[e] = dhe.sum(axis=0)
    dx = np.full((T, H), np.nan)
    dlogits = np.zeros((T, E))
    for t in range(T):
        rr = d.inv[t * kp:(t + 1) * kp]
        if np.isnan(dXp[rr, 0]).any():
            dlogits[t] = np.nan
            continue
        acc = np.zeros(H)
        for r in rr:                                   # slot order
            acc = acc + dXp[r]
        dx[t] = acc
        # router: w_j = rs * p_j, p = softmax over the selected logits
        p = fwd.w[t] / routed_scale
        dp = routed_scale * dw_row[rr[:k]]
        dsel = p * (dp - (p * dp).sum())
        dlogits[t, fwd.ids[t]] = dsel
    return Backward(dx, dW1, dW2, dlogits, dw_row, dh, dY1, db1)


# ---------------------------------------------------------------------------
# NVFP4 training recipe: per-tensor amax of the activation output and of its
# transposed Hadamard rotation (NVIDIA blog "Boosting MoE training
# throughput with advanced fusion kernels", section on fusing MXFP8/NVFP4
# quantisation: for NVFP4 the kernel emits the output's per-tensor amax for
# the forward and, for the backward, the amax of the Hadamard rotation of
# the transposed output).
# Reading taken: the rotation is the normalised Sylvester Hadamard matrix of
# order 16, H16 / 4, applied along the token axis in blocks of 16
# consecutive rows of one expert, the expert's rows zero-padded to a
# multiple of 16 (no random sign flips: the page names a Hadamard rotation).
# ---------------------------------------------------------------------------
def sylvester_hadamard(n: int) -> np.ndarray:
    """Sylvester's construction: H1 = [1], H2m = [[Hm, Hm], [Hm, -Hm]]."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def nvfp4_amax(y: np.ndarray, offsets: np.ndarray):
    """(max |y|, max over experts e, 16-row blocks and features of
    |(H16 / 4) @ block|) for y [R, I] in expert order, offsets [G + 1]."""
    y = np.asarray(y, np.float64)
    amax = float(np.abs(y).max(initial=0.0))
    h = sylvester_hadamard(16) / 4.0
    amax_t = 0.0
    for e in range(len(offsets) - 1):
        blk = y[offsets[e]:offsets[e + 1]]
        n = blk.shape[0]
        if n == 0:
            continue
        pad = np.zeros(((n + 15) // 16 * 16, y.shape[1]))
        pad[:n] = blk
        rot = np.einsum("ij,bjf->bif", h, pad.reshape(-1, 16, y.shape[1]))
        amax_t = max(amax_t, float(np.abs(rot).max()))
    return amax, amax_t
