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
from oracle import formats as F
from oracle import moe as M


def _setup(act, S=0, rs=1.0):
    rng = np.random.default_rng(11)
    T, H, I, E, k = 5, 12, 8, 4, 2
    G = E + S
    x = rng.normal(0, 1, (T, H))
    logits = rng.normal(0, 1, (T, E))
    w1 = rng.normal(0, 0.6, (G, I if act == "srelu" else 2 * I, H))
    w2 = rng.normal(0, 0.6, (G, H, I))
    dout = rng.normal(0, 1, (T, H))
    clamp = act == "swiglu_clamp"
    kw = dict(E=E, k=k, n_shared=S, routed_scale=rs, act=act,
              alpha=1.702 if clamp else 1.0, limit=1.5 if clamp else 0.0)
    return x, logits, w1, w2, dout, kw


def _loss(x, logits, w1, w2, dout, kw):
    f = M.layer_forward(x, logits, {"w1_f64": w1, "w2_f64": w2}, quant=False, **kw)
    return float((f.out * dout).sum())


@pytest.mark.parametrize("act,S,rs", [("swiglu", 0, 1.0), ("swiglu_clamp", 0, 1.0), ("swiglu", 1, 2.5),
                                      ("geglu", 0, 1.0), ("srelu", 0, 1.0)])
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
    G, N1, H = w1.shape
    I = w2.shape[2]
    for e in range(G):
        for n in range(0, N1, 3):
            for h in range(0, H, 5):
                assert bw.dW1[e, h, n] == pytest.approx(fd(w1, (e, n, h)), rel=1e-5, abs=1e-6)
        for h in range(0, H, 4):
            for i in range(0, I, 3):
                assert bw.dW2[e, i, h] == pytest.approx(fd(w2, (e, h, i)), rel=1e-5, abs=1e-6)


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_bias_gradient_matches_finite_differences(act):
    """With a W1 bias (gate b, up c) the oracle's db1 is the finite-difference
    gradient of the loss in the bias, and the other gradients still are."""
    x, logits, w1, w2, dout, kw = _setup(act)
    rng = np.random.default_rng(5)
    b1 = rng.normal(0, 0.5, (w1.shape[0], w1.shape[1]))
    wts = {"w1_f64": w1, "w2_f64": w2, "b1": b1}

    def loss():
        f = M.layer_forward(x, logits, wts, quant=False, **kw)
        return float((f.out * dout).sum())

    f = M.layer_forward(x, logits, wts, quant=False, **kw)
    bw = B.layer_backward(f, x, dout, wts, E=kw["E"], k=kw["k"], act=act, quant=False,
                          w1t=lambda e: w1[e].T, w2t=lambda e: w2[e].T)
    eps = 1e-6

    def fd(arr, idx):
        old = arr[idx]
        arr[idx] = old + eps
        lp = loss()
        arr[idx] = old - eps
        lm = loss()
        arr[idx] = old
        return (lp - lm) / (2 * eps)

    for e in range(b1.shape[0]):
        for n in range(b1.shape[1]):
            assert bw.db1[e, n] == pytest.approx(fd(b1, (e, n)), rel=1e-5, abs=1e-6)
    for t in range(0, x.shape[0], 2):
        for h in range(0, x.shape[1], 4):
            assert bw.dx[t, h] == pytest.approx(fd(x, (t, h)), rel=1e-5, abs=1e-6)
    for h in range(0, x.shape[1], 5):
        assert bw.dW1[0, h, 1] == pytest.approx(fd(w1, (0, 1, h)), rel=1e-5, abs=1e-6)


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


def test_q_cols_blocks_of_32_rows_with_trailing_zero_pad():
    """The wgrad operands' quantiser: MXFP8 along the row axis in blocks of 32
    rows, rows padded with zeros AFTER the data to a multiple of 32. A 33-row
    input therefore puts row 32 alone in a second block (its 31 pad rows are
    zero). Expected values worked out by hand from the scale rule (smallest e
    with amax <= 448 * 2^e) and E4M3 round-to-nearest-even:

      column 0, rows 0..31: 1.0 everywhere except row 5 = 448 * 2^10 and
        row 7 = 1.1. amax = 448 * 2^10, so e = 10 and the step near zero is
        the E4M3 subnormal 2^-9 * 2^10 = 2:
          row 5 -> 448 * 2^10 exactly, row 7 -> 1.1 / 1024 = 0.55 steps -> 2.0,
          1.0 -> exactly half a step -> ties to the even code 0 -> 0.0.
      column 0, row 32 (alone): 3.3 -> e = -7 (448 * 2^-7 = 3.5), 3.3 * 128 =
        422.4 -> nearest E4M3 416 -> 3.25.
      column 1: zero except row 32 = -0.2 -> e = -11, -0.2 * 2048 = -409.6 ->
        -416 -> -0.203125.
    Quantising along the other axis (each row's 32 columns), or padding in
    front of the data, gives different values (checked below)."""
    v = np.zeros((33, 32))
    v[:32, 0] = 1.0
    v[5, 0] = 448.0 * 2 ** 10
    v[7, 0] = 1.1
    v[32, 0] = 3.3
    v[32, 1] = -0.2
    got = B._q_cols(v, True)
    assert got.shape == (33, 32)
    assert got[5, 0] == 448.0 * 2 ** 10
    assert got[7, 0] == 2.0
    for r in set(range(32)) - {5, 7}:
        assert got[r, 0] == 0.0
    assert got[32, 0] == 3.25
    assert got[32, 1] == -0.203125
    assert (got[:32, 1] == 0.0).all() and (got[:, 2:] == 0.0).all()
    # the other axis: row 7 alone in its block would give 1.1 -> 1.125, and a
    # row of 1.0 would stay 1.0
    along_rows = B._q_rows(v, True)
    assert along_rows[7, 0] == 1.125 and along_rows[0, 0] == 1.0
    assert not np.array_equal(along_rows, got)
    # padding in front of the data would put row 32 in row 5's block
    front = np.zeros((64, 32))
    front[31:] = v
    q, s = F.mx_quantize(front.T)
    assert F.mx_dequantize(q, s).T[63, 0] == 4.0 != got[32, 0]
    assert np.array_equal(B._q_cols(v, False), v)


def test_backward_reads_bf16_rounded_h():
    """The backward evaluates SwiGLU and its derivative at the saved h rounded
    to bf16, not at the exact h. With g = 1 + 2^-10 (rounds to 1.0 in bf16),
    u = 1, a one-hot upstream gradient and a one-hot W2 copy, the routing-weight
    gradient is act(1, 1) = sigmoid(1) and the gate gradient is the closed form
    d/dg[g sigmoid(g)] at g = 1, sigmoid(1) * (2 - sigmoid(1)); the exact h
    would give values about 1e-3 away."""
    I = H = 32
    ids = np.array([[0]], np.int32)
    w = np.array([[1.0]])
    disp = M.dispatch(ids, w, 1)
    h = np.zeros((1, 2 * I))
    h[0, 0] = 1.0 + 2.0 ** -10          # gate feature 0
    h[0, I] = 1.0                       # up feature 0
    fwd = M.Forward(ids, w, disp, None, None, h, np.zeros((1, I)), None, None, np.zeros((1, H)),
                    np.zeros((1, H)))
    dout = np.zeros((1, H))
    dout[0, 0] = 1.0                    # exact in MXFP8
    w2t = np.zeros((I, H))
    w2t[0, 0] = 1.0                     # dY1 = e_0
    bw = B.layer_backward(fwd, np.zeros((1, H)), dout, {}, E=1, k=1, quant=True,
                          w1t=lambda e: np.zeros((H, 2 * I)), w2t=lambda e: w2t)
    s1 = 0.7310585786300049             # sigmoid(1)
    assert bw.dY1[0, 0] == 1.0
    assert bw.dw_row[0] == pytest.approx(s1, abs=1e-15)
    assert bw.dh[0, 0] == pytest.approx(s1 * (2.0 - s1), abs=1e-15)
    assert bw.dh[0, I] == pytest.approx(s1, abs=1e-15)     # du = g * sigmoid(g) at g = 1
    exact = (1.0 + 2.0 ** -10) / (1.0 + np.exp(-(1.0 + 2.0 ** -10)))
    assert abs(bw.dw_row[0] - exact) > 5e-4


def test_sylvester_hadamard_matches_the_bit_parity_formula():
    """Two constructions of H16 agree: Sylvester's recursion and the closed
    form H[i, j] = (-1)^popcount(i & j); H H^T = 16 I."""
    h = B.sylvester_hadamard(16)
    ref = np.array([[(-1) ** bin(i & j).count("1") for j in range(16)] for i in range(16)], np.float64)
    assert np.array_equal(h, ref)
    assert np.array_equal(h @ h.T, 16 * np.eye(16))


def test_nvfp4_amax_closed_forms():
    """One expert, one feature: a constant block c rotates to (4c, 0, ..., 0)
    (amax 4|c|); a single nonzero v rotates to sixteen values of magnitude
    |v|/4; rows of different experts never share a block (the second expert's
    single row is zero-padded to its own block)."""
    c = 0.75
    y = np.full((16, 1), c)
    assert B.nvfp4_amax(y, np.array([0, 16])) == (c, 4 * c)
    y = np.zeros((16, 2)); y[5, 1] = -3.0
    assert B.nvfp4_amax(y, np.array([0, 16])) == (3.0, 0.75)
    # 15 rows of 1.0 in expert 0 and one row of 1.0 in expert 1: expert 0's
    # padded block rotates to a first entry of 15/4, expert 1's to 1/4 each
    y = np.ones((16, 1))
    amax, amax_t = B.nvfp4_amax(y, np.array([0, 15, 16]))
    assert amax == 1.0 and amax_t == 15 / 4
    # merged into one expert the block would be constant: 16/4
    assert B.nvfp4_amax(y, np.array([0, 16]))[1] == 4.0
