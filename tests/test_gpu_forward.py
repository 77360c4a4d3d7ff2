"""Forward parity: the CUDA path through the C ABI against the fp64 oracle.

Bit-exact: top-k ids, counts, offsets, permutation, inverse, row weights'
sources, the MXFP8 copy of x. Within tolerance: logits (vs fp64), routing
weights (1e-6 relative), y1 (<= 1 E4M3 step on <= 0.1%), z and out
(rel-L2 <= 5e-3, cosine >= 0.9999).
"""
import numpy as np
import pytest
import torch

import inputs
from oracle import moe as M

from gpu_harness import oracle_forward, run_forward
from util import assert_close_layer, assert_mx_close, cuda_device, np_

pytestmark = pytest.mark.gpu


def _check_dispatch(s, r, f):
    v = r["views"]
    assert (np_(v["topk_ids"]) == f.ids).all()
    np.testing.assert_allclose(np_(v["topk_w"]), f.w, rtol=1e-6, atol=0)
    assert (np_(v["counts"]) == f.disp.counts).all()
    assert (np_(v["offsets"]) == f.disp.offsets).all()
    assert (np_(v["perm_src"]) == f.disp.perm_src).all()
    assert (np_(v["inv"]) == f.disp.inv).all()
    np.testing.assert_allclose(np_(v["w_row"]), f.disp.w_row, rtol=1e-6, atol=0)
    assert (np_(v["xq"]) == f.xq).all()
    assert (np_(v["xs"]) == f.xs).all()


def test_tiny_full_forward():
    dev = cuda_device()
    s = inputs.workload("tiny")
    r = run_forward(s, s.T, dev=dev)
    assert r["status"] == 0
    f = oracle_forward(s, r)
    # logits vs the fp64 product of the same bf16 x and fp32 W_r
    ref_logits = M.router_logits(np_(r["x"].float()), np_(r["Wr"]))
    np.testing.assert_allclose(np_(r["views"]["logits"]), ref_logits, rtol=1e-4, atol=1e-5)
    _check_dispatch(s, r, f)
    v = r["views"]
    assert_mx_close(np_(v["y1_q"]), np_(v["y1_s"]), f.y1q, f.y1s, "y1")
    z = np_(v["z"].view(torch.bfloat16).float())
    assert_close_layer(z, f.z, "z")
    assert_close_layer(np_(r["out"].float()), f.out, "out")


@pytest.mark.parametrize("T", [0, 1, 5, 33])
def test_tiny_ragged_T(T):
    dev = cuda_device()
    s = inputs.workload("tiny")
    r = run_forward(s, T, dev=dev, seed=3)
    if T == 0:
        assert (np_(r["views"]["counts"]) == 0).all() and (np_(r["views"]["offsets"]) == 0).all()
        return
    f = oracle_forward(s, r)
    _check_dispatch(s, r, f)
    assert_close_layer(np_(r["out"].float()), f.out, "out")


@pytest.mark.parametrize("T,E,k,S", [(300, 8, 2, 0), (1000, 64, 6, 1), (70, 33, 8, 0)])
def test_dispatch_multiblock_and_shared(T, E, k, S):
    """Large T takes the multi-block histogram / scan / scatter path."""
    dev = cuda_device()
    s = inputs.workload("tiny", E=E, k=k, n_shared=S, routed_scale=2.5 if S else 1.0)
    r = run_forward(s, T, dev=dev, seed=5)
    f = oracle_forward(s, r)
    _check_dispatch(s, r, f)
    assert_close_layer(np_(r["out"].float()), f.out, "out")


def test_empty_experts_and_skew():
    """Skewed logits: many experts empty; grouped GEMM skips them."""
    dev = cuda_device()
    s = inputs.workload("tiny", E=32, k=4, logits="zipf")
    r = run_forward(s, 64, dev=dev, seed=2)
    f = oracle_forward(s, r)
    assert (f.disp.counts == 0).sum() >= 9
    _check_dispatch(s, r, f)
    assert_mx_close(np_(r["views"]["y1_q"]), np_(r["views"]["y1_s"]), f.y1q, f.y1s, "y1")
    assert_close_layer(np_(r["out"].float()), f.out, "out")


def _sample_tokens(r, s, T, n=16):
    """n tokens spread over the batch, plus the tokens whose rows sit at
    positions 16, 64, 128 and last inside the most loaded expert group (so
    the sample reaches interior and trailing token tiles of the grouped
    GEMMs, whatever tile height they run with)."""
    if T <= n:
        return list(range(T))
    toks = set(int(t) for t in np.linspace(0, T - 1, n - 4).round())
    counts = np_(r["views"]["counts"])
    offs = np_(r["views"]["offsets"])
    perm = np_(r["views"]["perm_src"])
    e = int(np.argmax(counts))
    for pos in (16, 64, 128, int(counts[e]) - 1):
        if 0 <= pos < counts[e]:
            toks.add(int(perm[offs[e] + pos]) // s.kp)
    return sorted(toks)


def _full_size_sampled(s, T, seed, toks=None):
    """Dispatch checked in full; the expert path (y1, out) on the rows of the
    sampled tokens (default: _sample_tokens)."""
    dev = cuda_device()
    r = run_forward(s, T, dev=dev, seed=seed)
    assert r["status"] == 0
    if toks is None:
        toks = _sample_tokens(r, s, T)
    kp = s.kp
    inv = np_(r["views"]["inv"])
    rows = [int(inv[t * kp + j]) for t in toks for j in range(kp)]
    f = oracle_forward(s, r, rows=rows)
    _check_dispatch(s, r, f)
    v = r["views"]
    assert_mx_close(np_(v["y1_q"])[rows], np_(v["y1_s"])[rows], f.y1q[rows], f.y1s[rows], "y1")
    assert_close_layer(np_(r["out"].float())[toks], f.out[toks], "out")
    return r


@pytest.mark.parametrize("T", [1, 8, 32, 128])
def test_dsv3_decode(T):
    """DeepSeek-V3-shaped decode at full size; dispatch checked in full, the
    expert path on up to 16 sampled tokens (all of them for T <= 16)."""
    s = inputs.workload("dsv3", T=T)
    _full_size_sampled(s, T, 0)


@pytest.mark.parametrize("T", [1, 16, 64])
def test_shared_expert_decode(T):
    """Decode with one always-on shared expert at full size (H=6144, I=1536,
    E=160 + 1 shared, top-8, routed weights x2.5)."""
    s = inputs.workload("shared", T=T)
    _full_size_sampled(s, T, 0)


def test_skewed_routing_full_size():
    """Zipf-skewed routing at full size (T=4096, H=4096, I=1536, E=128,
    top-8): 30% of the experts receive no rows, the rest are load-imbalanced;
    multi-block dispatch and 64-token GEMM tiles. The sample includes rows in
    the second and third 64-row tiles of the hottest expert."""
    s = inputs.workload("skewed")
    r = _full_size_sampled(s, s.T, 3)
    counts = np_(r["views"]["counts"])
    assert (counts == 0).sum() >= int(0.3 * s.E)
    assert counts.sum() == s.T * s.k
    assert counts.max() > 192


@pytest.mark.parametrize("T,E,k", [(64, 33, 8), (40, 8, 2)])
def test_route_topk_exact_ties(T, E, k):
    """Integer-valued logits force many exact ties; moe_route_topk must pick
    the same ids as the oracle's rule (larger logit first, the lower expert id
    on a tie) and the same weights."""
    dev = cuda_device()
    import quantized_grouped_gemm_topk_gb300 as m
    s = inputs.workload("tiny", E=E, k=k)
    cfg = m.config_from_shape(s, T_max=T)
    ws = torch.zeros(m.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    g = torch.Generator(device="cpu")
    g.manual_seed(17)
    logits = torch.randint(-3, 4, (T, E), generator=g).to(torch.float32)
    logits[0] = 1.0                      # a token whose logits all tie
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    m.moe_route_topk(cfg, logits.to(dev), T, ids, w, ws)
    torch.cuda.synchronize()
    ref_ids, ref_w = M.topk_route(logits.numpy().astype(np.float64), k, 1.0)
    assert (np_(ids) == ref_ids).all()
    assert list(np_(ids)[0]) == list(range(k))
    np.testing.assert_allclose(np_(w), ref_w, rtol=1e-6, atol=0)
    assert m.moe_read_status(cfg, ws) == 0


@pytest.mark.parametrize("E", [40, 300])
def test_route_topk_special_values(E):
    """Logits with signed zeros, infinities, the largest finite values and
    subnormals (E = 300 keeps 10 logits a lane): -0 and +0 tie (the lower id
    first), -inf ranks below every number, and ids and weights match the
    oracle's rule."""
    dev = cuda_device()
    import quantized_grouped_gemm_topk_gb300 as m
    T, k = 24, 8
    s = inputs.workload("tiny", E=E, k=k)
    cfg = m.config_from_shape(s, T_max=T)
    ws = torch.zeros(m.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    g = torch.Generator(device="cpu")
    g.manual_seed(23)
    pool = torch.tensor([0.0, -0.0, float("-inf"), 3.4e38, -3.4e38, 1e-40, -1e-40, 1.0, -1.0, 2.5],
                        dtype=torch.float32)
    logits = pool[torch.randint(0, len(pool), (T, E), generator=g)]
    logits[0] = -0.0                     # all tie: ids 0..k-1
    logits[0, 5] = 0.0
    logits[1] = float("-inf")            # all -inf: ids 0..k-1 as well
    logits[2] = -0.0
    logits[2, E - 1] = 1e-40             # one subnormal above the zeros
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    m.moe_route_topk(cfg, logits.to(dev), T, ids, w, ws)
    torch.cuda.synchronize()
    with np.errstate(invalid="ignore"):          # the all--inf token's weights are 0/0
        ref_ids, ref_w = M.topk_route(logits.numpy().astype(np.float64), k, 1.0)
    got = np_(ids)
    assert (got == ref_ids).all()
    assert list(got[0]) == list(range(k))
    assert list(got[1]) == list(range(k))
    assert got[2][0] == E - 1 and list(got[2][1:]) == list(range(k - 1))
    fin = np.isfinite(ref_w)
    np.testing.assert_allclose(np_(w)[fin], ref_w[fin], rtol=1e-6, atol=0)
    assert m.moe_read_status(cfg, ws) == 0


@pytest.mark.parametrize("name", ["tiny", "train"])
def test_geglu_forward(name):
    """GeGLU (GELU(gate) * up) through both GEMM paths: the NVFP4 decode GEMM
    with its epilogue kernel, and the block-scaled MXFP8 GEMM with the fused
    epilogue."""
    dev = cuda_device()
    if name == "tiny":
        s = inputs.workload("tiny", act="geglu")
    else:
        s = inputs.workload("train", T=40, E=8, act="geglu")
    r = run_forward(s, s.T, dev=dev, seed=4)
    assert r["status"] == 0
    f = oracle_forward(s, r)
    _check_dispatch(s, r, f)
    assert_mx_close(np_(r["views"]["y1_q"]), np_(r["views"]["y1_s"]), f.y1q, f.y1s, "y1")
    assert_close_layer(np_(r["out"].float()), f.out, "out")


@pytest.mark.parametrize("T,logits", [(16, "router"), (1, "router"), (33, "router"), (64, "zipf"),
                                      (400, "router")])
def test_mxfp4_tiny_forward(T, logits):
    """MXFP4 weights (E2M1 elements, E8M0 scale per 32 along K) through the
    block-scaled GEMM with E2M1 as the weight operand: every output against
    the oracle, ragged token counts included; the Zipf-skewed T = 64 gives
    uneven groups, T = 400 groups of about 100 rows."""
    dev = cuda_device()
    s = inputs.workload("tiny", T=T, wfmt="mxfp4", logits=logits)
    r = run_forward(s, T, dev=dev, seed=5)
    assert r["status"] == 0
    f = oracle_forward(s, r)
    _check_dispatch(s, r, f)
    assert_mx_close(np_(r["views"]["y1_q"]), np_(r["views"]["y1_s"]), f.y1q, f.y1s, "y1")
    assert_close_layer(np_(r["views"]["z"].view(torch.bfloat16).float()), f.z, "z")
    assert_close_layer(np_(r["out"].float()), f.out, "out")


def test_mxfp4_shared_expert():
    """MXFP4 with one always-on shared expert and routed weights x2.5 (a
    multi-tile expert axis: H=512, I=256, E=16)."""
    dev = cuda_device()
    s = inputs.workload("tiny", T=48, H=512, I=256, E=16, k=4, n_shared=1, routed_scale=2.5, wfmt="mxfp4")
    r = run_forward(s, s.T, dev=dev, seed=6)
    assert r["status"] == 0
    f = oracle_forward(s, r)
    _check_dispatch(s, r, f)
    assert_close_layer(np_(r["out"].float()), f.out, "out")


@pytest.mark.parametrize("T", [1, 32, 128])
def test_mxfp4_dsv3_decode(T):
    """DeepSeek-V3-shaped decode (H=7168, I=2048, E=256, top-8) with MXFP4
    weights at full size; dispatch in full, the expert path on up to 16
    sampled tokens."""
    s = inputs.workload("dsv3", T=T, wfmt="mxfp4")
    _full_size_sampled(s, T, 1)


@pytest.mark.parametrize("case", ["nvfp4_fused", "nvfp4_separate", "mxfp8", "mxfp4"])
def test_w1_bias_forward(case):
    """A per-expert W1 bias (gate b, up c, added before the activation) on
    every W1 epilogue: the fused layer's tile epilogue (tiny, T = 4), the
    separate NVFP4 epilogue kernel (tiny, T = 16), and the block-scaled
    GEMM's epilogue with MXFP8 (training shape, reduced) and MXFP4 weights."""
    dev = cuda_device()
    if case == "nvfp4_fused":
        s = inputs.workload("tiny", T=4, bias=True)
    elif case == "nvfp4_separate":
        s = inputs.workload("tiny", T=16, bias=True)
    elif case == "mxfp8":
        s = inputs.workload("train", T=40, E=8, bias=True)
    else:
        s = inputs.workload("tiny", T=16, wfmt="mxfp4", bias=True)
    r = run_forward(s, s.T, dev=dev, seed=7)
    assert r["status"] == 0
    import quantized_grouped_gemm_topk_gb300 as m
    assert m.moe_layer_fused(r["cfg"], s.T) == (case == "nvfp4_fused")
    f = oracle_forward(s, r)
    _check_dispatch(s, r, f)
    assert_mx_close(np_(r["views"]["y1_q"]), np_(r["views"]["y1_s"]), f.y1q, f.y1s, "y1")
    assert_close_layer(np_(r["out"].float()), f.out, "out")


@pytest.mark.parametrize("case", ["nvfp4", "nvfp4_decode", "mxfp8", "mxfp4"])
def test_srelu_forward(case):
    """sReLU (max(h, 0)^2 of a non-gated W1 with I outputs): the NVFP4
    decoding GEMM with its epilogue kernel (tiny T = 16; a decode size,
    where the fused layer declines it) and the block-scaled GEMM's epilogue
    with MXFP8 (training shape, reduced) and MXFP4 weights."""
    dev = cuda_device()
    import quantized_grouped_gemm_topk_gb300 as m
    if case == "nvfp4":
        s = inputs.workload("tiny", T=16, act="srelu")
    elif case == "nvfp4_decode":
        s = inputs.workload("dsv3", T=8, E=32, act="srelu")
    elif case == "mxfp8":
        s = inputs.workload("train", T=40, E=8, act="srelu")
    else:
        s = inputs.workload("tiny", T=16, wfmt="mxfp4", act="srelu")
    r = run_forward(s, s.T, dev=dev, seed=8)
    assert r["status"] == 0
    assert not m.moe_layer_fused(r["cfg"], s.T)
    f = oracle_forward(s, r)
    _check_dispatch(s, r, f)
    assert_mx_close(np_(r["views"]["y1_q"]), np_(r["views"]["y1_s"]), f.y1q, f.y1s, "y1")
    assert_close_layer(np_(r["out"].float()), f.out, "out")


@pytest.mark.parametrize("name,T,E,nd", [("dsv3", 8, 32, 1), ("dsv3", 8, 32, 12), ("dsv3", 1, 256, 8),
                                          ("dsv3", 32, 256, 20), ("shared", 16, 160, 8)])
def test_partitioned_fused_layer(name, T, E, nd):
    """The partitioned fused layer: nd CTAs of the W1 -> W2 kernel gather the
    W1 operand rows group by group and raise ring flags that the other CTAs
    acquire. Its output has the bits of the unpartitioned fused layer (the
    gather as a launch of its own), on two calls in a row through one
    workspace (the routing kernel clears the flags and counters each call),
    and the reduced case matches the oracle."""
    import quantized_grouped_gemm_topk_gb300 as m
    dev = cuda_device()
    s = inputs.workload(name, T=T, E=E)
    r = run_forward(s, T, dev=dev)
    assert r["status"] == 0
    assert m.moe_layer_fused(r["cfg"], T)
    cfg = m.config_from_shape(s, T_max=T, dispatch_sms=nd)
    ws = torch.zeros(m.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    out = torch.empty_like(r["out"])
    for _ in range(2):
        out.fill_(float("nan"))
        m.moe_layer_forward(cfg, r["x"], r["Wr"], r["logits_in"], T, r["packed"], out, None, ws)
        torch.cuda.synchronize()
        assert m.moe_read_status(cfg, ws) == 0
        assert torch.equal(out, r["out"])
    if E <= 32:
        f = oracle_forward(s, r)
        assert_close_layer(np_(out.float()), f.out, "out")
