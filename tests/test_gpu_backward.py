"""Training forward + backward parity (MXFP8 weights, clamped SwiGLU).

A reduced case is checked in full (every gradient entry); the full-size
training workload is checked on the experts of three sampled tokens (the
first, middle and last: their experts' complete weight gradients) and on
those tokens' outputs, dx and router gradients.
"""
import numpy as np
import pytest
import torch

import inputs
import quantized_grouped_gemm_topk_gb300 as m
from oracle import backward as B
from oracle import formats as F
from oracle import moe as M

from gpu_harness import LazyExperts, oracle_forward, oracle_weights, run_forward
from util import assert_close_layer, assert_mx_close, cuda_device, np_

pytestmark = pytest.mark.gpu


def _run_backward(s, r, T, seed=0, db1=None):
    dev = r["x"].device
    cfg = r["cfg"]
    dout = inputs.gen_dout(s, seed, device=dev, T=T)
    packed_d = m.moe_prepack_weights(cfg, r["wts"], m.MOE_PACK_DGRAD)
    dx = torch.empty(T, s.H, dtype=torch.bfloat16, device=dev)
    dW1 = torch.empty(s.E, s.H, s.I if s.act == "srelu" else 2 * s.I, dtype=torch.bfloat16, device=dev)
    dW2 = torch.empty(s.E, s.I, s.H, dtype=torch.bfloat16, device=dev)
    dlog = torch.empty(T, s.E, dtype=torch.float32, device=dev)
    m.moe_layer_backward(cfg, dout, r["x"], T, r["save"], packed_d, dx, dW1, dW2, dlog, r["ws"], db1=db1)
    torch.cuda.synchronize()
    assert m.moe_read_status(cfg, r["ws"]) == 0
    return dout, dx, dW1, dW2, dlog


def _oracle_backward(s, r, f, dout, experts=None):
    wts = oracle_weights(r["wts"])

    def w1t(e):
        from oracle import formats as F
        return F.mx_dequantize(wts["w1t_q"][e], wts["w1t_s"][e])

    def w2t(e):
        from oracle import formats as F
        return F.mx_dequantize(wts["w2t_q"][e], wts["w2t_s"][e])

    return B.layer_backward(f, inputs.bf16_bits(r["x"]).cpu().numpy(), inputs.bf16_bits(dout).cpu().numpy(), wts,
                            E=s.E, k=s.k, routed_scale=s.routed_scale, act=s.act, alpha=s.alpha, limit=s.limit,
                            quant=True, experts=experts, w1t=w1t, w2t=w2t)


@pytest.mark.parametrize("act", ["swiglu_clamp", "geglu", "srelu"])
def test_train_reduced_full_check(act):
    dev = cuda_device()
    s = inputs.workload("train", T=48, E=8, act=act)
    r = run_forward(s, s.T, dev=dev, save=True)
    f = oracle_forward(s, r)
    assert (np_(r["views"]["topk_ids"]) == f.ids).all()
    assert_mx_close(np_(r["views"]["y1_q"]), np_(r["views"]["y1_s"]), f.y1q, f.y1s, "y1")
    assert_close_layer(np_(r["out"].float()), f.out, "out")
    # saved pre-activation h (bf16) against the oracle's h
    h = np_(r["save_bufs"]["h"].view(torch.bfloat16).float())[: s.T * s.kp]
    assert_close_layer(h, f.h, "h")
    dout, dx, dW1, dW2, dlog = _run_backward(s, r, s.T)
    b = _oracle_backward(s, r, f, dout)
    assert_close_layer(np_(dx.float()), b.dx, "dx")
    assert_close_layer(np_(dW1.float()), b.dW1, "dW1")
    assert_close_layer(np_(dW2.float()), b.dW2, "dW2")
    assert_close_layer(np_(dlog), b.dlogits, "dlogits")


def test_nvfp4_recipe_amax():
    """The W1 epilogue's NVFP4-recipe amaxes: max |y| and the amax of the
    16-row Hadamard rotation of y's transpose within each expert, against the
    oracle's on the same routing."""
    dev = cuda_device()
    s = inputs.workload("train", T=56, E=8)
    T = s.T
    r = run_forward(s, T, dev=dev, save=False)
    cfg = r["cfg"]
    st, bufs = m.alloc_train_save(cfg, T, dev, amax=True)
    bufs["amax"].fill_(-1.0)
    out = torch.empty_like(r["out"])
    m.moe_layer_forward(cfg, r["x"], r["Wr"], None, T, r["packed"], out, st, r["ws"])
    torch.cuda.synchronize()
    assert m.moe_read_status(cfg, r["ws"]) == 0
    f = oracle_forward(s, r)
    amax, amax_t = B.nvfp4_amax(f.y, f.disp.offsets)
    got = np_(bufs["amax"])[:2]
    np.testing.assert_allclose(got, [amax, amax_t], rtol=1e-4)
    assert amax_t > 0 and amax > 0


def test_train_empty_expert_grads_are_zero():
    dev = cuda_device()
    s = inputs.workload("train", T=4, E=16)
    r = run_forward(s, s.T, dev=dev, save=True)
    counts = np_(r["views"]["counts"])
    assert (counts == 0).any()
    _, _, dW1, dW2, _ = _run_backward(s, r, s.T)
    for e in np.nonzero(counts == 0)[0]:
        assert (dW1[e] == 0).all() and (dW2[e] == 0).all()


@pytest.mark.slow
def test_train_full_size_sampled():
    dev = cuda_device()
    s = inputs.workload("train")
    T = s.T
    r = run_forward(s, T, dev=dev, save=True)
    ids = np_(r["views"]["topk_ids"])
    toks = [0, T // 2, T - 1]           # first, middle and last token (different row tiles of their experts)
    experts = sorted(set(int(e) for t in toks for e in ids[t]))
    offs = np_(r["views"]["offsets"])
    rows = [rr for e in experts for rr in range(offs[e], offs[e + 1])]
    f = oracle_forward(s, r, rows=rows)
    assert (ids == f.ids).all()
    assert_close_layer(np_(r["out"].float())[toks], f.out[toks], "out[toks]")
    dout, dx, dW1, dW2, dlog = _run_backward(s, r, T)
    b = _oracle_backward(s, r, f, dout, experts=experts)
    assert_close_layer(np_(dx.float())[toks], b.dx[toks], "dx[toks]")
    assert_close_layer(np_(dlog)[toks], b.dlogits[toks], "dlogits[toks]")
    for e in experts:
        assert_close_layer(np_(dW1[e].float()), b.dW1[e], f"dW1[{e}]")
        assert_close_layer(np_(dW2[e].float()), b.dW2[e], f"dW2[{e}]")


@pytest.mark.parametrize("T,E", [(300, 8), (4, 16)])
def test_train_saved_transposed_x_bit_exact(T, E):
    """The transposed MXFP8 copy of the gathered x rows that the training
    forward saves (at_q, at_s) against the oracle's MXFP8 quantisation of
    each expert's rows, zero-padded to a multiple of 128 rows, along the row
    axis: codes and scales byte for byte. H = 2880 spans eleven full
    256-column tiles and a 64-column tail; T = 300 gives experts of several
    32-row blocks with ragged ends, T = 4 empty experts."""
    dev = cuda_device()
    s = inputs.workload("train", T=T, E=E)
    r = run_forward(s, T, dev=dev, save=True)
    assert r["status"] == 0
    f = oracle_forward(s, r)
    offs = f.disp.offsets
    cnt = np.diff(offs)
    poff = np.concatenate([[0], np.cumsum((cnt + 127) // 128 * 128)])
    bufs = r["save_bufs"]
    assert np.array_equal(np_(bufs["poff"])[: len(poff)], poff)
    xv = F.bf16_to_f64(inputs.bf16_bits(r["x"]).cpu().numpy())
    at_q = np_(bufs["at_q"])
    rp = bufs["r_pad"]
    at_s = np_(bufs["at_s"]).reshape(rp // 128, s.H, 4).transpose(1, 0, 2).reshape(s.H, rp // 32)
    for e in range(len(cnt)):
        n = poff[e + 1] - poff[e]
        if n == 0:
            continue
        rows = np.zeros((n, s.H))
        rows[: cnt[e]] = xv[f.disp.perm_src[offs[e]: offs[e + 1]] // s.kp]
        q, sc = F.mx_quantize(rows.T)
        assert np.array_equal(at_q[:, poff[e]: poff[e + 1]], q), f"at_q of expert {e}"
        assert np.array_equal(at_s[:, poff[e] // 32: poff[e + 1] // 32], sc), f"at_s of expert {e}"


@pytest.mark.parametrize("act,T", [("swiglu_clamp", 48), ("geglu", 300)])
def test_train_w1_bias(act, T):
    """Training with a W1 bias (gate b, up c): the forward adds it before the
    activation (saved h includes it), the backward's gradients match the
    oracle's, and db1 (the sum of dh over each group's rows, from the
    dActivation epilogue's per-32-row column sums) matches the oracle's db1.
    T = 300 over 8 experts spans several 128-row tiles per group."""
    dev = cuda_device()
    s = inputs.workload("train", T=T, E=8, act=act, bias=True)
    r = run_forward(s, s.T, dev=dev, save=True)
    assert r["status"] == 0
    f = oracle_forward(s, r)
    assert_close_layer(np_(r["out"].float()), f.out, "out")
    db1 = torch.full((s.E, 2 * s.I), float("nan"), dtype=torch.float32, device=dev)
    dout, dx, dW1, dW2, dlog = _run_backward(s, r, s.T, db1=db1)
    b = _oracle_backward(s, r, f, dout)
    assert_close_layer(np_(dx.float()), b.dx, "dx")
    assert_close_layer(np_(dW1.float()), b.dW1, "dW1")
    assert_close_layer(np_(dW2.float()), b.dW2, "dW2")
    assert_close_layer(np_(dlog), b.dlogits, "dlogits")
    assert_close_layer(np_(db1), b.db1, "db1")
