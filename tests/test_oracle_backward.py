"""Pin the oracle's backward formulas by central finite differences (no GPU).

The quantised backward is the same code with straight-through quantisers, so
pinning the unquantised variant against finite differences of the
unquantised forward fixes the gradient algebra (SwiGLU and clamp derivatives,
routing-weight gradient, router softmax Jacobian, dgrad/wgrad contractions,
the slot-ordered combine backward).
"""
import numpy as np
import pytest

from oracle import backward as B
from oracle import moe as M


def _setup(act, S=0, rs=1.0):
    rng = np.random.default_rng(11)
    T, H, I, E, k = 5, 12, 8, 4, 2
    G = E + S
    x = rng.normal(0, 1, (T, H))
    logits = rng.normal(0, 1, (T, E))
    w1 = rng.normal(0, 0.6, (G, 2 * I, H))
    w2 = rng.normal(0, 0.6, (G, H, I))
    dout = rng.normal(0, 1, (T, H))
    kw = dict(E=E, k=k, n_shared=S, routed_scale=rs, act=act,
              alpha=1.702 if act != "swiglu" else 1.0, limit=1.5 if act != "swiglu" else 0.0)
    return x, logits, w1, w2, dout, kw


def _loss(x, logits, w1, w2, dout, kw):
    f = M.layer_forward(x, logits, {"w1_f64": w1, "w2_f64": w2}, quant=False, **kw)
    return float((f.out * dout).sum())


@pytest.mark.parametrize("act,S,rs", [("swiglu", 0, 1.0), ("swiglu_clamp", 0, 1.0), ("swiglu", 1, 2.5)])
def test_backward_matches_finite_differences(act, S, rs):
    x, logits, w1, w2, dout, kw = _setup(act, S, rs)
    f = M.layer_forward(x, logits, {"w1_f64": w1, "w2_f64": w2}, quant=False, **kw)
    bw = B.layer_backward(f, x, dout, {}, E=kw["E"], k=kw["k"], routed_scale=rs, act=act,
                          alpha=kw["alpha"], limit=kw["limit"], quant=False,
                          w1t=lambda e: w1[e].T, w2t=lambda e: w2[e].T)
    eps = 1e-6

    def fd(arr, idx):
        old = arr[idx]
        arr[idx] = old + eps
        lp = _loss(x, logits, w1, w2, dout, kw)
        arr[idx] = old - eps
        lm = _loss(x, logits, w1, w2, dout, kw)
        arr[idx] = old
        return (lp - lm) / (2 * eps)

    # keep clear of clamp kinks: skip probes whose h lands within 1e-3 of +-limit
    for t in range(x.shape[0]):
        for h in range(0, x.shape[1], 3):
            assert bw.dx[t, h] == pytest.approx(fd(x, (t, h)), rel=1e-5, abs=1e-6)
    for t in range(x.shape[0]):
        for e in range(kw["E"]):
            assert bw.dlogits[t, e] == pytest.approx(fd(logits, (t, e)), rel=1e-5, abs=1e-6)
    G, I2, H = w1.shape
    for e in range(G):
        for n in range(0, I2, 3):
            for h in range(0, H, 5):
                assert bw.dW1[e, h, n] == pytest.approx(fd(w1, (e, n, h)), rel=1e-5, abs=1e-6)
        for h in range(0, H, 4):
            for i in range(0, I2 // 2, 3):
                assert bw.dW2[e, i, h] == pytest.approx(fd(w2, (e, h, i)), rel=1e-5, abs=1e-6)


def test_quantised_backward_close_to_unquantised():
    """With quantisers on, gradients stay within MXFP8 error of the exact ones
    (sanity: the quantised path is the same algebra)."""
    x, logits, w1, w2, dout, kw = _setup("swiglu")
    H = x.shape[1]
    # widen to multiples of 32 for MX blocks
    rng = np.random.default_rng(3)
    T, E, k, I = 6, 4, 2, 32
    H = 64
    x = rng.normal(0, 1, (T, H)); logits = rng.normal(0, 1, (T, E))
    w1 = rng.normal(0, 0.2, (E, 2 * I, H)); w2 = rng.normal(0, 0.2, (E, H, I))
    dout = rng.normal(0, 1, (T, H))
    kw = dict(E=E, k=k, act="swiglu")
    wts = {"w1_f64": w1, "w2_f64": w2}
    outs = []
    for quant in (False, True):
        f = M.layer_forward(x, logits, wts, quant=quant, **kw)
        bw = B.layer_backward(f, x, dout, wts, E=E, k=k, quant=quant,
                              w1t=lambda e: w1[e].T, w2t=lambda e: w2[e].T)
        outs.append(bw)
    for name in ("dx", "dW1", "dW2", "dlogits"):
        a, b = getattr(outs[0], name), getattr(outs[1], name)
        rel = np.linalg.norm(a - b) / np.linalg.norm(a)
        assert rel < 0.15, (name, rel)
