"""Pins for the oracle's routing, dispatch, forward layer and combine (no GPU).

Checks against closed forms, brute force over subsets, invariants and an
independent dense formulation of the layer.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import inputs
from oracle import formats as F
from oracle import moe as M


def _sig(v):
    return 1.0 / (1.0 + math.exp(-v))


# ---- SwiGLU closed forms --------------------------------------------------
def test_swiglu_closed_forms():
    assert M.act_fwd(0.0, 3.0) == 0.0
    assert M.act_fwd(2.0, 0.0) == 0.0
    assert M.act_fwd(1.0, 1.0) == pytest.approx(0.7310585786300049, abs=1e-15)   # sigmoid(1)
    assert M.act_fwd(-1.0, 1.0) == pytest.approx(-0.2689414213699951, abs=1e-15)
    assert M.act_fwd(2.0, 3.0) == pytest.approx(6.0 * _sig(2.0), rel=1e-15)
    assert M.act_fwd(40.0, 0.5) == pytest.approx(20.0, rel=1e-15)                 # -> g*u
    assert M.act_fwd(-40.0, 0.5) == pytest.approx(0.0, abs=1e-15)


def test_swiglu_clamp_closed_forms():
    kw = dict(act="swiglu_clamp", alpha=1.702, limit=7.0)
    assert M.act_fwd(10.0, 10.0, **kw) == pytest.approx(49.0 * _sig(1.702 * 7.0), rel=1e-15)
    assert M.act_fwd(-10.0, -10.0, **kw) == pytest.approx(-7.0 * _sig(-1.702 * 7.0) * -7.0, rel=1e-15)
    assert M.act_fwd(1.0, 2.0, **kw) == pytest.approx(2.0 * _sig(1.702), rel=1e-15)
    # gradient is zero beyond the clamp, nonzero inside
    dg, du = M.act_bwd(np.array([8.0, 1.0]), np.array([1.0, -9.0]), 1.0, **kw)
    assert dg[0] == 0.0 and du[1] == 0.0 and dg[1] != 0.0 and du[0] != 0.0


def test_geglu_closed_forms():
    """GELU(v) = v * Phi(v): Phi(0) = 1/2, Phi(1) = 0.8413447460685429 (the
    normal table), Phi(-1) = 1 - Phi(1); GELU(g) * u -> g * u as g -> +inf
    and -> 0 as g -> -inf."""
    kw = dict(act="geglu")
    assert M.act_fwd(0.0, 3.0, **kw) == 0.0
    assert M.act_fwd(2.0, 0.0, **kw) == 0.0
    assert M.act_fwd(1.0, 1.0, **kw) == pytest.approx(0.8413447460685429, abs=1e-15)
    assert M.act_fwd(-1.0, 2.0, **kw) == pytest.approx(-2.0 * (1.0 - 0.8413447460685429), abs=1e-15)
    assert M.act_fwd(2.0, 1.5, **kw) == pytest.approx(3.0 * 0.9772498680518208, rel=1e-15)   # Phi(2)
    assert M.act_fwd(12.0, 0.5, **kw) == pytest.approx(6.0, rel=1e-15)
    assert M.act_fwd(-12.0, 0.5, **kw) == pytest.approx(0.0, abs=1e-15)


def test_geglu_derivative_closed_form():
    """d/dg [g Phi(g) u] = u (Phi(g) + g phi(g)), d/du = g Phi(g); at g = 1:
    Phi(1) + phi(1) = 0.8413447460685429 + 0.24197072451914337 (the normal
    density at 1); at g = 0 the gate derivative is 1/2."""
    dg, du = M.act_bwd(1.0, 2.0, 1.0, "geglu")
    assert dg == pytest.approx(2.0 * (0.8413447460685429 + 0.24197072451914337), rel=1e-14)
    assert du == pytest.approx(0.8413447460685429, rel=1e-14)
    dg0, du0 = M.act_bwd(0.0, -3.0, 2.0, "geglu")
    assert dg0 == pytest.approx(2.0 * 0.5 * -3.0, rel=1e-15) and du0 == 0.0


def test_swiglu_derivative_closed_form():
    # d/dg [g s(g) u] = u (s + g s (1 - s)); d/du = g s(g)
    g, u = 0.7, -1.3
    s = _sig(g)
    dg, du = M.act_bwd(g, u, 1.0)
    assert dg == pytest.approx(u * (s + g * s * (1 - s)), rel=1e-14)
    assert du == pytest.approx(g * s, rel=1e-14)


# ---- routing ---------------------------------------------------------------
def test_topk_k1_is_argmax():
    rng = np.random.default_rng(0)
    lg = rng.normal(0, 1, (50, 16))
    ids, w = M.topk_route(lg, 1, 2.5)
    assert (ids[:, 0] == lg.argmax(1)).all()
    assert (w == 2.5).all()


def test_topk_kE_is_full_softmax():
    rng = np.random.default_rng(1)
    lg = rng.normal(0, 3, (20, 6))
    ids, w = M.topk_route(lg, 6)
    for t in range(20):
        ex = [math.exp(v) for v in lg[t]]
        tot = sum(ex)
        for j in range(6):
            assert w[t, j] == pytest.approx(ex[ids[t, j]] / tot, rel=1e-13)
        assert list(ids[t]) == sorted(range(6), key=lambda e: -lg[t, e])


def test_topk_brute_force_subsets_and_ties():
    rng = np.random.default_rng(2)
    for trial in range(200):
        E, k = rng.integers(2, 7), None
        k = int(rng.integers(1, E + 1))
        lg = rng.integers(-3, 3, size=(1, E)).astype(np.float64)   # many ties
        ids, _ = M.topk_route(lg, k)
        best = None
        for sub in itertools.combinations(range(E), k):
            key = sorted(((-lg[0, e], e) for e in sub))
            if best is None or key < best:
                best = key
        # the chosen set is the lexicographically best (value desc, id asc) subset, in order
        assert [e for _, e in best] == list(ids[0])


def test_topk_special_values_brute_force():
    """Signed zeros, infinities and subnormals: -0 and +0 compare equal (the
    lower id wins the tie), -inf ranks below every finite number, and the
    selection is the brute-force best (value desc, id asc) subset; a token
    whose selected logits are all -inf has undefined (NaN) weights, every
    other token's weights sum to the routed scale."""
    rng = np.random.default_rng(5)
    pool = np.array([0.0, -0.0, -np.inf, 3.4e38, -3.4e38, 1e-310, -1e-310, 1.0, -1.0])
    for trial in range(300):
        E = int(rng.integers(2, 7))
        k = int(rng.integers(1, E + 1))
        lg = pool[rng.integers(0, len(pool), size=(1, E))]
        with np.errstate(invalid="ignore"):
            ids, w = M.topk_route(lg, k, 2.0)
        best = None
        for sub in itertools.combinations(range(E), k):
            key = sorted(((-lg[0, e], e) for e in sub))
            if best is None or key < best:
                best = key
        assert [e for _, e in best] == list(ids[0])
        if np.isfinite(lg[0, ids[0]]).any():
            assert abs(w[0].sum() - 2.0) < 1e-12
    # all zeros of either sign: ids in order
    ids, _ = M.topk_route(np.array([[-0.0, 0.0, -0.0, 0.0]]), 3)
    assert list(ids[0]) == [0, 1, 2]


# ---- dispatch --------------------------------------------------------------
@pytest.mark.parametrize("T,E,k,S", [(0, 4, 2, 0), (1, 8, 2, 0), (37, 8, 3, 0), (64, 33, 8, 1), (200, 5, 5, 0)])
def test_dispatch_invariants(T, E, k, S):
    rng = np.random.default_rng(T + E)
    lg = rng.normal(0, 1, (T, E))
    ids, w = M.topk_route(lg, k)
    d = M.dispatch(ids, w, E, S)
    kp, G = k + S, E + S
    assert d.counts.sum() == T * kp
    assert (np.diff(d.offsets) == d.counts).all() and d.offsets[0] == 0
    assert sorted(d.perm_src.tolist()) == list(range(T * kp))          # bijection
    assert (d.inv[d.perm_src] == np.arange(T * kp)).all()               # inv o perm = id
    for e in range(G):
        seg = d.perm_src[d.offsets[e]:d.offsets[e + 1]]
        assert (np.diff(seg) > 0).all()                                 # token-major order
        assert (d.expert[seg] == e).all()
    if S:
        assert d.counts[E] == T
    for r in range(T * kp):
        a = d.perm_src[r]
        t, j = divmod(a, kp)
        assert d.w_row[r] == (w[t, j] if j < k else 1.0)


def test_combine_identity_experts():
    """Identity experts: dispatch rows are the weighted token copies; combine
    returns x * sum_j w_j exactly."""
    rng = np.random.default_rng(7)
    T, E, k, H = 40, 6, 3, 16
    x = rng.normal(0, 1, (T, H))
    ids, w = M.topk_route(rng.normal(0, 1, (T, E)), k)
    d = M.dispatch(ids, w, E, 1)
    kp = k + 1
    z = np.stack([x[d.perm_src[r] // kp] * d.w_row[r] for r in range(T * kp)])
    out = M.combine(z, d.inv, T, kp)
    expect = x * (w.sum(1) + 1.0)[:, None]
    assert np.allclose(out, expect, rtol=1e-15, atol=1e-15)


# ---- forward layer ---------------------------------------------------------
def _tiny_case(act="swiglu", wfmt="nvfp4", S=0, rs=1.0, T=16):
    s = inputs.workload("tiny", T=T, n_shared=S, routed_scale=rs, act=act,
                        alpha=1.702 if act != "swiglu" else 1.0,
                        limit=7.0 if act != "swiglu" else 0.0, wfmt=wfmt)
    x = inputs.gen_x(s, 0)
    Wr = inputs.gen_router(s, 0)
    wts = {k: v.numpy() for k, v in inputs.gen_expert_weights(s, 0).items()}
    logits = (x.float() @ Wr).numpy()          # fp32 logits as the routing input
    return s, inputs.bf16_bits(x).numpy(), logits, wts


@pytest.mark.parametrize("act,wfmt,S,rs", [("swiglu", "nvfp4", 0, 1.0), ("swiglu", "nvfp4", 1, 2.5),
                                          ("swiglu_clamp", "mxfp8", 0, 1.0), ("geglu", "nvfp4", 0, 1.0),
                                          ("swiglu", "mxfp4", 0, 1.0), ("srelu", "nvfp4", 0, 1.0),
                                          ("srelu", "mxfp8", 1, 2.5)])
def test_routed_equals_dense_formulation(act, wfmt, S, rs):
    s, xb, lg, wts = _tiny_case(act, wfmt, S, rs)
    kw = dict(E=s.E, k=s.k, n_shared=S, routed_scale=rs, act=s.act, alpha=s.alpha, limit=s.limit, wfmt=wfmt)
    f = M.layer_forward(xb, lg, wts, **kw)
    dense = M.dense_forward(xb, lg, wts, **kw)
    assert np.allclose(f.out, dense, rtol=1e-12, atol=1e-12)
    assert np.isfinite(f.out).all()


def test_w1_bias_is_added_to_gate_and_up_before_the_activation():
    """With W1 = 0 every row's W1 output is exactly its expert's bias (gate
    part b first, up part c second); with W1 as drawn, adding the bias
    shifts each row's W1 output by exactly that vector (up to fp64
    rounding), and the layer equals its dense formulation."""
    s, xb, lg, wts = _tiny_case(T=8)
    G, I, H = s.groups, s.I, s.H
    rng = np.random.default_rng(11)
    b1 = rng.normal(0, 0.5, (G, 2 * I))
    f0 = M.layer_forward(xb, lg, dict(wts, w1_f64=np.zeros((G, 2 * I, H)), b1=b1), E=s.E, k=s.k)
    e_row = f0.disp.expert[f0.disp.perm_src]
    assert (f0.h == b1[e_row]).all()
    # gate from b, up from c: a swapped pair would change y
    g, u = b1[e_row, :I], b1[e_row, I:]
    expect = f0.disp.w_row[:, None] * (g / (1.0 + np.exp(-g))) * u
    assert np.allclose(f0.y, expect, rtol=1e-14, atol=0)
    fa = M.layer_forward(xb, lg, wts, E=s.E, k=s.k)
    fb = M.layer_forward(xb, lg, dict(wts, b1=b1), E=s.E, k=s.k)
    assert np.allclose(fb.h - fa.h, b1[e_row], rtol=0, atol=1e-15)
    dense = M.dense_forward(xb, lg, dict(wts, b1=b1), E=s.E, k=s.k)
    assert np.allclose(fb.out, dense, rtol=1e-12, atol=1e-12)


def test_srelu_is_the_squared_relu_of_a_non_gated_w1():
    """sReLU: W1 has I outputs (no up half); with one-hot W1 rows each output
    is an exact scaled activation, and y = w_row * max(h, 0)^2 exactly:
    negative outputs give 0 (not |h|^2), positive ones their square (not h)."""
    s, xb, lg, wts = _tiny_case(act="srelu", T=8)
    G, I, H = s.groups, s.I, s.H
    assert wts["w1_q"].shape[1] == I
    w1 = np.zeros((G, I, H))
    for n in range(I):
        w1[:, n, (5 * n) % H] = 2.0 ** ((n % 3) - 1)
    f = M.layer_forward(xb, lg, dict(wts, w1_f64=w1), E=s.E, k=s.k, act="srelu")
    a = F.mx_dequantize(f.xq, f.xs)
    t = f.disp.perm_src // s.kp
    assert f.h.shape == (s.T * s.kp, I)
    neg = pos = 0
    for r in range(s.T * s.kp):
        for n in range(0, I, 7):
            v = a[t[r], (5 * n) % H] * 2.0 ** ((n % 3) - 1)
            assert f.h[r, n] == v
            want = f.disp.w_row[r] * (v * v if v > 0 else 0.0)
            assert f.y[r, n] == want
            neg += v < 0
            pos += v > 0
    assert neg > 10 and pos > 10


def test_gemm_brute_force_triple_loop():
    s, xb, lg, wts = _tiny_case(T=3)
    f = M.layer_forward(xb, lg, wts, E=s.E, k=s.k, wfmt="nvfp4")
    a = F.mx_dequantize(f.xq, f.xs)
    kp = s.kp
    for r in range(0, s.T * kp, 2):
        e = f.disp.expert[f.disp.perm_src[r]]
        t = f.disp.perm_src[r] // kp
        W1 = M.expert_w1(wts, e, "nvfp4")
        for n in (0, 5, s.I, 2 * s.I - 1):
            acc = 0.0
            for h in range(s.H):
                acc += a[t, h] * W1[n, h]
            assert f.h[r, n] == pytest.approx(acc, rel=1e-12, abs=1e-14)


def test_one_hot_weights_are_exact():
    """W1 rows that pick single inputs with power-of-two values reproduce the
    dequantised activations exactly."""
    s, xb, lg, wts = _tiny_case(T=8)
    G, I, H = s.groups, s.I, s.H
    w1 = np.zeros((G, 2 * I, H))
    for n in range(2 * I):
        w1[:, n, (3 * n) % H] = 2.0 ** ((n % 5) - 2)
    wts2 = dict(wts, w1_f64=w1)
    f = M.layer_forward(xb, lg, wts2, E=s.E, k=s.k)
    a = F.mx_dequantize(f.xq, f.xs)
    t = f.disp.perm_src // s.kp
    for n in range(2 * I):
        assert (f.h[:, n] == a[t, (3 * n) % H] * 2.0 ** ((n % 5) - 2)).all()


def test_unrouted_expert_has_no_effect():
    s, xb, lg, wts = _tiny_case(T=4)
    f = M.layer_forward(xb, lg, wts, E=s.E, k=s.k)
    empty = [e for e in range(s.E) if f.disp.counts[e] == 0]
    assert empty, "tiny case should leave some expert empty at T=4"
    wts2 = {k: v.copy() for k, v in wts.items()}
    for e in empty:
        wts2["w1_q"][e] ^= 0x77
        wts2["w2_q"][e] ^= 0x11
    f2 = M.layer_forward(xb, lg, wts2, E=s.E, k=s.k)
    assert (f2.out == f.out).all()


def test_row_subset_matches_full():
    s, xb, lg, wts = _tiny_case()
    kw = dict(E=s.E, k=s.k, wfmt="nvfp4")
    full = M.layer_forward(xb, lg, wts, **kw)
    rows = full.disp.inv[3 * s.kp:5 * s.kp]
    part = M.layer_forward(xb, lg, wts, rows=rows, **kw)
    assert (part.out[3:5] == full.out[3:5]).all()
    assert np.isnan(part.out[0]).all()


# ---------------------------------------------------------------------------
# Readings pinned one by one (each on the oracle alone).
# ---------------------------------------------------------------------------
def test_routed_scale_multiplies_renormalised_weights():
    """Routing weights are the softmax over the k selected logits times
    routed_scale: they sum to routed_scale, and scale linearly with it."""
    rng = np.random.default_rng(11)
    logits = rng.normal(size=(5, 16))
    ids1, w1 = M.topk_route(logits, 4, 1.0)
    ids2, w2 = M.topk_route(logits, 4, 2.5)
    assert (ids1 == ids2).all()
    np.testing.assert_allclose(w1.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(w2, 2.5 * w1, rtol=1e-15, atol=0)


def test_shared_expert_slot_and_weight():
    """A shared expert takes slot k (after the routed slots) of every token,
    group E, weight 1.0 regardless of routed_scale, rows in token order."""
    rng = np.random.default_rng(12)
    T, E, k = 6, 8, 2
    ids, w = M.topk_route(rng.normal(size=(T, E)), k, 2.5)
    d = M.dispatch(ids, w, E, n_shared=1)
    kp = k + 1
    assert d.counts[E] == T
    rows = range(d.offsets[E], d.offsets[E + 1])
    assert [d.perm_src[r] for r in rows] == [t * kp + k for t in range(T)]
    assert all(d.w_row[r] == 1.0 for r in rows)
    assert all(d.expert[t * kp + k] == E for t in range(T))


def test_nan_logit_ranks_below_finite():
    """A NaN logit is never chosen while k finite logits remain; the weights
    of the chosen experts stay finite."""
    logits = np.array([[0.5, np.nan, 2.0, -1.0, 1.0]])
    ids, w = M.topk_route(logits, 3)
    assert 1 not in ids[0]
    assert list(ids[0]) == [2, 4, 0]
    assert np.isfinite(w).all()


def test_dispatch_empty_batch():
    """T = 0 is legal: zero counts, zero offsets, no rows."""
    ids = np.zeros((0, 2), np.int32)
    w = np.zeros((0, 2))
    d = M.dispatch(ids, w, 8)
    assert d.counts.shape == (8,) and (d.counts == 0).all()
    assert (d.offsets == 0).all()
    assert d.perm_src.size == 0 and d.inv.size == 0


def test_clamp_gradient_is_inclusive_at_the_limit():
    """The clamped SwiGLU passes gradient at |v| == limit and blocks it just
    outside; inside, both partials match the unclamped form at alpha."""
    lim, a = 7.0, 1.702
    d = np.ones(4)
    g = np.array([lim, -lim, lim * (1 + 1e-12), 0.3])
    u = np.array([0.5, 0.5, 0.5, -lim])
    dg, du = M.act_bwd(g, u, d, "swiglu_clamp", a, lim)
    assert dg[0] != 0 and dg[1] != 0 and dg[2] == 0
    assert du[3] != 0
    s = 1.0 / (1.0 + np.exp(-a * 0.3))
    np.testing.assert_allclose(dg[3], (s + a * 0.3 * s * (1 - s)) * (-lim), rtol=1e-13)
    np.testing.assert_allclose(du[3], 0.3 * s, rtol=1e-13)


# ---- S1 router logits ---------------------------------------------------------
def test_router_logits_one_hot_rows_pick_rows_of_w():
    """x = e_h (a one-hot row) gives logits = W_r[h, :]: the contraction runs
    over H and the result keeps W_r's expert axis. W_r is non-symmetric, so a
    transposed operand or a reduction over the wrong axis changes the rows."""
    W_r = np.array([[0.5, -1.0, 2.0, 0.0],
                    [3.0, 0.25, -4.0, 1.5],
                    [-0.75, 6.0, 1.0, -2.0]])          # H = 3, E = 4
    x = np.zeros((5, 3))
    hs = [2, 0, 1, 2, 0]
    for t, h in enumerate(hs):
        x[t, h] = 1.0
    got = M.router_logits(x, W_r)
    assert got.shape == (5, 4)
    for t, h in enumerate(hs):
        assert list(got[t]) == list(W_r[h])


def test_router_logits_hand_computed_case():
    """Two tokens, H = 4, E = 3, power-of-two entries (every product and sum
    exact); expected values worked out by hand:
      row 0: 1*(1, 0, 2) + 2*(0, 1/4, 1) + 0*(..) - 1*(1, 1, 1) = (0, -1/2, 3)
      row 1: (1/2)*(1, 0, 2) + 4*(-2, 1, 0)                     = (-15/2, 4, 1)"""
    x = np.array([[1.0, 2.0, 0.0, -1.0],
                  [0.5, 0.0, 4.0, 0.0]])
    W_r = np.array([[1.0, 0.0, 2.0],
                    [0.0, 0.25, 1.0],
                    [-2.0, 1.0, 0.0],
                    [1.0, 1.0, 1.0]])
    got = M.router_logits(x, W_r)
    assert got.tolist() == [[0.0, -0.5, 3.0], [-7.5, 4.0, 1.0]]


def test_mxfp4_encoding_scale_rule():
    """The MXFP4 weights the workloads hand the layer: every block's scale is
    the smallest power of two with amax <= 6 * 2^e (so no element saturates,
    and the block maximum lands in the top binade [3, 6]), and decoding
    returns each element within half an E2M1 step of its value."""
    g = torch.Generator().manual_seed(5)
    w = torch.randn(8, 128, generator=g) * 0.02
    packed, sc = inputs.encode_mxfp4(w)
    dec = F.mxfp4_dequantize(packed.numpy(), sc.numpy())
    e = sc.numpy().astype(np.int64) - 127
    blk = w.numpy().astype(np.float64).reshape(8, 4, 32)
    amax = np.abs(blk).max(-1)
    assert (amax <= 6.0 * np.exp2(e)).all() and (amax > 3.0 * np.exp2(e)).all()
    err = np.abs(dec.reshape(8, 4, 32) - blk) / np.exp2(e)[..., None]
    assert err.max() <= 1.0 + 1e-12          # steps of E2M1 are at most 2 (between 4 and 6)
