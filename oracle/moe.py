"""Routed-MoE layer, step by step, in plain fp64 numpy.

TEST INFRASTRUCTURE ONLY: the CPU oracle. Only the tests, the smoke check and
the benchmark's CPU-baseline leg may import it; the product path never does.

Steps follow the layer the pages describe:
  GC-MoE summary (arxiv-wiki page "GC-MoE: Overlapping Expert-Parallel Token
  Dispatch with FP8/FP4 Grouped GEMM via CUDA Green Contexts"), Approach:
  role1 aggregates routing counts and moves tokens into expert blocks; role2
  runs W1 with SwiGLU, routing weight and requantisation fused in the
  epilogue, then W2 emitting BF16 fragments; role3 combines.
  NVIDIA blog "Boosting MoE training throughput with advanced fusion kernels":
  SwiGLU(x, W, V, b, c, beta) = Swish_beta(xW + b) * (xV + c) (section on GLU
  epilogue fusion); per-group token counts kept on the device (section on
  removing host-device sync); GroupGemm + dActivation + Quantize/Transpose
  for the backward (kernel families list).

Readings taken where the pages are silent (each listed in the design notes):
  * routing weights: softmax over all logits, keep the top-k, renormalise
    (equal to a softmax over the k selected logits), then x routed_scale;
    ties in the logit order go to the lower expert id;
  * shared experts: every token, weight 1.0, slot k (after the routed slots);
  * rows of an expert are ordered by flat assignment index t*k' + j;
  * W1 holds gate columns [0, I) then up columns [I, 2I); beta = 1; the
    blog's b and c are an optional per-expert fp32 bias vector of W1's 2I
    outputs (b for gate, c for up; the blog's fused epilogues add a "bias
    vector", kernel families section), zero when the weights carry none;
  * sReLU (the blog's non-gated activation) is max(h, 0)^2 of a W1 with I
    outputs, then the routing weight;
  * the clamped variant is g' = clamp(g, -L, L), u' = clamp(u, -L, L),
    act = g' * sigmoid(alpha * g') * u';
  * the routing weight multiplies the SwiGLU output before requantisation;
  * combine sums the k' expert outputs of a token in slot order.

Parity pins: tests/test_oracle_moe.py and tests/test_oracle_backward.py.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import formats as F


# ---------------------------------------------------------------------------
# S1 router logits / S2 top-k routing
# ---------------------------------------------------------------------------
def router_logits(x: np.ndarray, W_r: np.ndarray) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] * W_r[h, e], exactly in fp64."""
    return np.asarray(x, np.float64) @ np.asarray(W_r, np.float64)


def topk_route(logits: np.ndarray, k: int, routed_scale: float = 1.0):
    """Per token: the k experts with the largest logits (ties -> lower id), in
    that order, and their weights softmax(selected logits) * routed_scale.
    Returns (ids int32 [T, k], w fp64 [T, k])."""
    logits = np.asarray(logits, np.float64)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    eid = np.arange(E)
    for t in range(T):
        order = np.lexsort((eid, -logits[t]))[:k]     # primary -logit, then id
        sel = logits[t, order]
        p = np.exp(sel - sel.max())
        ids[t] = order
        w[t] = p / p.sum() * routed_scale
    return ids, w


# ---------------------------------------------------------------------------
# S3 counts + offsets, S4 permutation
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class Dispatch:
    counts: np.ndarray     # int32 [G]   rows per expert group
    offsets: np.ndarray    # int32 [G+1] exclusive prefix sum of counts
    perm_src: np.ndarray   # int32 [R]   row r <- flat assignment t*k' + j
    inv: np.ndarray        # int32 [T*k'] flat assignment -> row
    w_row: np.ndarray      # fp64  [R]   routing weight of row r
    expert: np.ndarray     # int32 [T*k'] expert group of each assignment


def dispatch(ids: np.ndarray, w: np.ndarray, E: int, n_shared: int = 0) -> Dispatch:
    """Group the T*k' assignments by expert. Assignment (t, j) has flat index
    a = t*k' + j; slots j >= k are the shared experts E + (j - k) with weight 1.
    Within an expert, rows keep increasing a (a stable counting sort)."""
    T, k = ids.shape
    kp = k + n_shared
    G = E + n_shared
    expert = np.zeros(T * kp, np.int32)
    weight = np.zeros(T * kp, np.float64)
    for t in range(T):
        for j in range(kp):
            a = t * kp + j
            if j < k:
                expert[a] = ids[t, j]
                weight[a] = w[t, j]
            else:
                expert[a] = E + (j - k)
                weight[a] = 1.0
    counts = np.bincount(expert, minlength=G).astype(np.int32)
    offsets = np.zeros(G + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    perm_src = np.zeros(T * kp, np.int32)
    inv = np.zeros(T * kp, np.int32)
    fill = offsets[:-1].copy()
    for a in range(T * kp):              # ascending a: stable within an expert
        e = expert[a]
        r = fill[e]
        fill[e] += 1
        perm_src[r] = a
        inv[a] = r
    return Dispatch(counts, offsets, perm_src, inv, weight[perm_src], expert)


# ---------------------------------------------------------------------------
# S5 activation function and its derivative
# ---------------------------------------------------------------------------
def sigmoid(v):
    return 1.0 / (1.0 + np.exp(-v))


def gelu_cdf(v):
    """Phi(v), the standard normal CDF, = (1 + erf(v / sqrt 2)) / 2."""
    v = np.asarray(v, np.float64)
    return 0.5 * (1.0 + np.vectorize(math.erf, otypes=[np.float64])(v / math.sqrt(2.0)))


def gelu_pdf(v):
    """phi(v) = exp(-v^2 / 2) / sqrt(2 pi)."""
    v = np.asarray(v, np.float64)
    return np.exp(-0.5 * v * v) / math.sqrt(2.0 * math.pi)


def gated(act: str) -> bool:
    """Whether W1 has gate and up halves (2I outputs) or I outputs."""
    return act != "srelu"


def act_plain(h, act="srelu"):
    """The non-gated activation the blog's fused kernels list (kernel
    families: sReLU): the squared ReLU, max(h, 0)^2, of W1's I outputs."""
    h = np.asarray(h, np.float64)
    assert act == "srelu", act
    return np.square(np.maximum(h, 0.0))


def act_plain_bwd(h, d, act="srelu"):
    """Gradient of sum(d * act_plain(h)) with respect to h: the derivative
    of max(h, 0)^2 is 2 max(h, 0) (the dActivation kernel family of the same
    blog lists sReLU among its activations)."""
    h = np.asarray(h, np.float64)
    assert act == "srelu", act
    return d * 2.0 * np.maximum(h, 0.0)


def act_fwd(g, u, act="swiglu", alpha=1.0, limit=0.0):
    """The gated activations the blog's fused kernels support (NVIDIA blog,
    kernel families: SwiGLU, GeGLU), with b = c = 0:
    'swiglu'        Swish_1(g) * u = g * sigmoid(g) * u;
    'swiglu_clamp'  g and u clamped to [-limit, limit] first, Swish_alpha;
    'geglu'         GELU(g) * u with the exact GELU(v) = v * Phi(v)."""
    g = np.asarray(g, np.float64)
    u = np.asarray(u, np.float64)
    if act == "swiglu":
        return g * sigmoid(g) * u
    if act == "geglu":
        return g * gelu_cdf(g) * u
    gc = np.clip(g, -limit, limit)
    uc = np.clip(u, -limit, limit)
    return gc * sigmoid(alpha * gc) * uc


def act_bwd(g, u, d, act="swiglu", alpha=1.0, limit=0.0):
    """Gradients (dg, du) of sum(d * act(g, u)). The clamp passes gradient
    where -limit <= v <= limit and blocks it outside."""
    g = np.asarray(g, np.float64)
    u = np.asarray(u, np.float64)
    if act == "swiglu":
        s = sigmoid(g)
        return d * (s + g * s * (1.0 - s)) * u, d * g * s
    if act == "geglu":
        c = gelu_cdf(g)
        return d * (c + g * gelu_pdf(g)) * u, d * g * c
    gc = np.clip(g, -limit, limit)
    uc = np.clip(u, -limit, limit)
    s = sigmoid(alpha * gc)
    dg = d * (s + alpha * gc * s * (1.0 - s)) * uc * ((g >= -limit) & (g <= limit))
    du = d * gc * s * ((u >= -limit) & (u <= limit))
    return dg, du


# ---------------------------------------------------------------------------
# weights
# ---------------------------------------------------------------------------
def values(a) -> np.ndarray:
    """bf16 bit patterns (int16/uint16) -> fp64 values; fp64 passes through."""
    a = np.asarray(a)
    if a.dtype == np.float64:
        return a
    return F.bf16_to_f64(a)


def expert_w1(wts: dict, e: int, wfmt: str) -> np.ndarray:
    """Decoded W1 of group e as stored: [2I, H] (row n = output feature n)."""
    if "w1_f64" in wts:
        return np.asarray(wts["w1_f64"][e], np.float64)
    if wfmt == "nvfp4":
        return F.nvfp4_dequantize(wts["w1_q"][e], wts["w1_s"][e], wts["w1_gs"][e])
    if wfmt == "mxfp4":
        return F.mxfp4_dequantize(wts["w1_q"][e], wts["w1_s"][e])
    return F.mx_dequantize(wts["w1_q"][e], wts["w1_s"][e])


def expert_b1(wts: dict, e: int, n: int) -> np.ndarray:
    """W1's bias of group e, [2I] (gate b then up c), zeros if none."""
    if "b1" not in wts:
        return np.zeros(n)
    return np.asarray(wts["b1"][e], np.float64).reshape(n)


def expert_w2(wts: dict, e: int, wfmt: str) -> np.ndarray:
    """Decoded W2 of group e as stored: [H, I]."""
    if "w2_f64" in wts:
        return np.asarray(wts["w2_f64"][e], np.float64)
    if wfmt == "nvfp4":
        return F.nvfp4_dequantize(wts["w2_q"][e], wts["w2_s"][e], wts["w2_gs"][e])
    if wfmt == "mxfp4":
        return F.mxfp4_dequantize(wts["w2_q"][e], wts["w2_s"][e])
    return F.mx_dequantize(wts["w2_q"][e], wts["w2_s"][e])


# ---------------------------------------------------------------------------
# the forward layer
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class Forward:
    ids: np.ndarray
    w: np.ndarray
    disp: Dispatch
    xq: np.ndarray        # uint8 [T, H]   E4M3 codes of x
    xs: np.ndarray        # uint8 [T, H/32] E8M0 scales of x
    h: np.ndarray         # fp64 [R, 2I]  W1 output (gate | up); sReLU: [R, I]
    y: np.ndarray         # fp64 [R, I]   routing weight * act(g, u)
    y1q: np.ndarray       # uint8 [R, I]
    y1s: np.ndarray       # uint8 [R, I/32]
    z: np.ndarray         # fp64 [R, H]   W2 output
    out: np.ndarray       # fp64 [T, H]   combined, unrounded


def layer_forward(x_bits, logits, wts: dict, *, E: int, k: int, n_shared: int = 0,
                  routed_scale: float = 1.0, act: str = "swiglu", alpha: float = 1.0,
                  limit: float = 0.0, wfmt: str = "nvfp4", rows=None,
                  quant: bool = True) -> Forward:
    """The whole forward hot path from bf16 x and fp32/fp64 router logits.

    ``rows`` (optional iterable of row indices) restricts the W1/W2 work to
    those rows; other rows of h/y/z stay NaN and ``out`` only covers tokens
    whose rows were all computed. ``quant=False`` skips both activation
    quantisers (used to pin the gradient formulas by finite differences).
    """
    x = values(x_bits)
    T, H = x.shape
    ids, w = topk_route(logits, k, routed_scale)
    d = dispatch(ids, w, E, n_shared)
    if quant:
        xq, xs = F.mx_quantize(x)
        a_tok = F.mx_dequantize(xq, xs)              # dequantised activations [T, H]
    else:
        xq, xs, a_tok = None, None, x
    kp = k + n_shared
    R = T * kp
    G = E + n_shared
    want = np.zeros(R, bool)
    if rows is None:
        want[:] = True
    else:
        want[np.asarray(list(rows), np.int64)] = True
    I = expert_w2(wts, 0, wfmt).shape[1]
    N1 = 2 * I if gated(act) else I
    h = np.full((R, N1), np.nan)
    y = np.full((R, I), np.nan)
    y1q = np.zeros((R, I), np.uint8)
    y1s = np.zeros((R, max(I // 32, 1)), np.uint8)
    z = np.full((R, H), np.nan)
    for e in range(G):
        lo, hi = d.offsets[e], d.offsets[e + 1]
        rs = [r for r in range(lo, hi) if want[r]]
        if not rs:
            continue                                 # empty expert: nothing to do
        rs = np.asarray(rs)
        toks = d.perm_src[rs] // kp
        A = a_tok[toks]                              # gathered rows [n, H]
        W1 = expert_w1(wts, e, wfmt)                 # [2I, H] (sReLU: [I, H])
        he = A @ W1.T + expert_b1(wts, e, N1)        # [n, 2I]: xW + b | xV + c
        if gated(act):
            ye = d.w_row[rs, None] * act_fwd(he[:, :I], he[:, I:], act, alpha, limit)
        else:
            ye = d.w_row[rs, None] * act_plain(he, act)
        if quant:
            q, s = F.mx_quantize(ye)
            y_in = F.mx_dequantize(q, s)
        else:
            q, s, y_in = 0, 0, ye
        W2 = expert_w2(wts, e, wfmt)                 # [H, I]
        ze = y_in @ W2.T                             # [n, H]
        h[rs], y[rs], y1q[rs], y1s[rs], z[rs] = he, ye, q, s, ze
    out = combine(z, d.inv, T, kp, rows_ok=want)
    return Forward(ids, w, d, xq, xs, h, y, y1q, y1s, z, out)


def combine(z: np.ndarray, inv: np.ndarray, T: int, kp: int, weights=None,
            rows_ok=None) -> np.ndarray:
    """S8: out[t] = sum over slots j = 0..k'-1 (in that order) of
    z[inv[t*k' + j]], optionally times weights[t, j]. Tokens with a row
    outside ``rows_ok`` stay NaN."""
    H = z.shape[1]
    out = np.full((T, H), np.nan)
    for t in range(T):
        rr = inv[t * kp:(t + 1) * kp]
        if rows_ok is not None and not rows_ok[rr].all():
            continue
        acc = np.zeros(H)
        for j, r in enumerate(rr):
            acc = acc + (z[r] if weights is None else weights[t, j] * z[r])
        out[t] = acc
    return out


def dense_forward(x_bits, logits, wts: dict, *, E: int, k: int, n_shared: int = 0,
                  routed_scale: float = 1.0, act: str = "swiglu", alpha: float = 1.0,
                  limit: float = 0.0, wfmt: str = "nvfp4") -> np.ndarray:
    """The same layer written densely: every expert on every token, masked by
    the routing: out[t] = sum_e gate[t, e] * FFN_e(x_t). No permutation, no
    offsets. Used to pin layer_forward's gather/scatter."""
    x = values(x_bits)
    T, H = x.shape
    ids, w = topk_route(logits, k, routed_scale)
    xq, xs = F.mx_quantize(x)
    a = F.mx_dequantize(xq, xs)
    G = E + n_shared
    gate = np.zeros((T, G))
    for t in range(T):
        for j in range(k):
            gate[t, ids[t, j]] += w[t, j]
        for j in range(n_shared):
            gate[t, E + j] = 1.0
    I = expert_w2(wts, 0, wfmt).shape[1]
    out = np.zeros((T, H))
    for e in range(G):
        W1 = expert_w1(wts, e, wfmt)
        W2 = expert_w2(wts, e, wfmt)
        N1 = 2 * I if gated(act) else I
        hh = a @ W1.T + expert_b1(wts, e, N1)
        if gated(act):
            yy = gate[:, e:e + 1] * act_fwd(hh[:, :I], hh[:, I:], act, alpha, limit)
        else:
            yy = gate[:, e:e + 1] * act_plain(hh, act)
        q, s = F.mx_quantize(yy)
        zz = F.mx_dequantize(q, s) @ W2.T
        out += np.where(gate[:, e:e + 1] != 0, zz, 0.0)
    return out
