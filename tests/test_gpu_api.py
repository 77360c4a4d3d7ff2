"""The step-wise C-ABI entry points, CUDA-graph replay, the identity-expert
combine invariant, and the device status word."""
import numpy as np
import pytest
import torch

import inputs
import quantized_grouped_gemm_topk_gb300 as m
from oracle import moe as M

from gpu_harness import oracle_forward, run_forward, weights_for
from util import assert_close_layer, cuda_device, np_

pytestmark = pytest.mark.gpu


GUARD = 64   # guard elements on each side of a guarded buffer (>= 64 bytes)


def _guarded(n, dtype, dev, fill):
    """A buffer of n elements with GUARD canary elements on both sides;
    returns (whole, inner view). The inner view stays 64-byte aligned."""
    whole = torch.full((n + 2 * GUARD,), fill, dtype=dtype, device=dev)
    return whole, whole[GUARD:GUARD + n]


def _guards_intact(whole, n, fill):
    return bool((whole[:GUARD] == fill).all()) and bool((whole[GUARD + n:] == fill).all())


def _alloc_dispatch(s, T, dev, guard=False):
    """Caller-owned dispatch buffers; with guard=True each one sits between
    canary bands (t["_guards"] lists (whole, n, fill) to check afterwards)."""
    R = T * s.kp
    G = s.groups
    spec = {
        "topk_ids": ((T, s.k), torch.int32, 0x5a5a5a5a),
        "topk_w": ((T, s.k), torch.float32, -123.25),
        "counts": ((G,), torch.int32, 0x3c3c3c3c),
        "offsets": ((G + 1 + 3,), torch.int32, 0x3c3c3c3c),
        "perm_src": ((R,), torch.int32, 0x7e7e7e7e),
        "inv": ((R,), torch.int32, 0x7e7e7e7e),
        "w_row": ((R,), torch.float32, -77.5),
        "xq": ((T, s.H), torch.uint8, 0xA5),
        "xs": ((T, s.H // 32), torch.uint8, 0xA5),
    }
    t, guards = {}, []
    for name, (shape, dtype, fill) in spec.items():
        n = int(np.prod(shape))
        if guard:
            whole, inner = _guarded(n, dtype, dev, fill)
            t[name] = inner.view(shape)
            guards.append((name, whole, n, fill))
        else:
            t[name] = torch.empty(shape, dtype=dtype, device=dev)
    t["_guards"] = guards
    return t, m.dispatch_struct(t)


def _check_guards(t):
    for name, whole, n, fill in t["_guards"]:
        assert _guards_intact(whole, n, fill), f"write outside {name}"


@pytest.mark.parametrize("name,S", [("tiny", 0), ("tiny", 1), ("dsv3", 0), ("tiny_small", 0)])
def test_stepwise_equals_layer_forward(name, S):
    """The step-wise calls (router, top-k, dispatch, W1 + epilogue, W2,
    combine: one kernel chain each) give bit for bit what moe_layer_forward
    gives. With at most 2 rows per expert on average the layer runs W1, its
    epilogue and W2 as one persistent launch (DeepSeek-V3 shapes with E=32,
    T=8: 64 token rows over 32 experts; tiny with T=4); tiny at T=16
    (4 rows per expert, with and without a shared expert) takes the
    separate kernels."""
    dev = cuda_device()
    if name == "dsv3":
        s = inputs.workload("dsv3", T=8, E=32)
    elif name == "tiny_small":
        s = inputs.workload("tiny", T=4)
    else:
        s = inputs.workload(name, n_shared=S, routed_scale=2.5 if S else 1.0)
    T = s.T
    r = run_forward(s, T, dev=dev)
    cfg, ws = r["cfg"], r["ws"]
    logits = torch.empty(T, s.E, dtype=torch.float32, device=dev)
    m.moe_router_logits(cfg, r["x"], r["Wr"], T, logits, ws)
    np.testing.assert_allclose(np_(logits), np_(r["views"]["logits"]), rtol=1e-5, atol=1e-6)
    t, d = _alloc_dispatch(s, T, dev)
    m.moe_route_dispatch(cfg, r["views"]["logits"], r["x"], T, d, ws)
    for k in ("topk_ids", "counts", "perm_src", "inv", "xq", "xs"):
        ref = r["views"][k]
        assert torch.equal(t[k][: ref.numel()].view(ref.shape) if k != "counts" else t[k], ref), k
    ids2 = torch.empty_like(t["topk_ids"])
    w2 = torch.empty_like(t["topk_w"])
    m.moe_route_topk(cfg, r["views"]["logits"], T, ids2, w2, ws)
    assert torch.equal(ids2, t["topk_ids"]) and torch.equal(w2, t["topk_w"])
    # dispatch from given ids
    t2, d2 = _alloc_dispatch(s, T, dev)
    t2["topk_ids"].copy_(t["topk_ids"])
    t2["topk_w"].copy_(t["topk_w"])
    m.moe_dispatch(cfg, r["x"], T, d2, ws)
    assert torch.equal(t2["perm_src"], t["perm_src"]) and torch.equal(t2["inv"], t["inv"])
    R = T * s.kp
    y1q = torch.empty(R, s.I, dtype=torch.uint8, device=dev)
    y1s = torch.empty(R, s.I // 32, dtype=torch.uint8, device=dev)
    m.moe_grouped_gemm_w1_swiglu_quant(cfg, d, T, r["packed"], y1q, y1s, None, ws)
    assert torch.equal(y1q, r["views"]["y1_q"]) and torch.equal(y1s, r["views"]["y1_s"])
    z = torch.empty(R, s.H, dtype=torch.bfloat16, device=dev)
    m.moe_grouped_gemm_w2(cfg, d, T, y1q, y1s, r["packed"], z, ws)
    assert torch.equal(z.view(torch.int16), r["views"]["z"])
    out = torch.empty(T, s.H, dtype=torch.bfloat16, device=dev)
    m.moe_combine(cfg, z, t["inv"], None, T, out)
    assert torch.equal(out, r["out"])


def test_identity_experts_combine():
    """Rows copied straight from their tokens and combined with the routing
    weights give x * sum_j w_j."""
    dev = cuda_device()
    s = inputs.workload("tiny", n_shared=1, routed_scale=2.5)
    T = 40
    r = run_forward(s, T, dev=dev)
    v = r["views"]
    tok = (v["perm_src"].long() // s.kp)
    z = r["x"][tok].contiguous()
    out = torch.empty(T, s.H, dtype=torch.bfloat16, device=dev)
    m.moe_combine(r["cfg"], z, v["inv"], v["topk_w"], T, out)
    wsum = v["topk_w"].double().sum(1) + 1.0
    ref = r["x"].double() * wsum[:, None]
    assert_close_layer(np_(out.double()), np_(ref), "identity combine")
    assert (out.double() - ref).abs().max() <= ref.abs().max() * 2 ** -7


@pytest.mark.parametrize("nd", [0, 8])
def test_cuda_graph_replay_matches_eager(nd):
    """One captured layer replayed on new inputs gives the eager bits; with
    nd ring CTAs (the partitioned fused layer) the routing kernel inside the
    graph clears the ring flags and hand-off counters on every replay."""
    dev = cuda_device()
    s = inputs.workload("dsv3", T=8, E=32)
    T = s.T
    r = run_forward(s, T, dev=dev)
    ws, packed, Wr = r["ws"], r["packed"], r["Wr"]
    cfg = m.config_from_shape(s, T_max=T, dispatch_sms=nd)
    x_static = torch.empty_like(r["x"])
    out_static = torch.empty_like(r["out"])
    xs = [inputs.gen_x(s, 100 + i, device=dev, T=T) for i in range(3)]
    eager = []
    for x in xs:
        o = torch.empty_like(out_static)
        m.moe_layer_forward(cfg, x, Wr, None, T, packed, o, None, ws)
        eager.append(o)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    x_static.copy_(xs[0])
    with torch.cuda.graph(g):
        m.moe_layer_forward(cfg, x_static, Wr, None, T, packed, out_static, None, ws)
    for x, ref in zip(xs, eager):
        x_static.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_static, ref)


@pytest.mark.parametrize("T", [8, 40])
def test_bad_expert_ids_flag_status(T):
    """Out-of-range expert ids set MOE_DEV_BAD_EXPERT_ID, their slots are
    skipped (inv = -1), nothing is written past the valid rows, and every
    output buffer's canary bands are untouched. T = 8 (16 assignments) takes
    the routing kernel's direct path for at most 32 assignments, T = 40 its
    histogram and scan path."""
    dev = cuda_device()
    s = inputs.workload("tiny")
    cfg = m.config_from_shape(s, T_max=T)
    ws = torch.zeros(m.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    x = inputs.gen_x(s, 0, device=dev, T=T)
    t, d = _alloc_dispatch(s, T, dev, guard=True)
    t["topk_ids"].copy_(torch.tensor([[0, 1]] * T, dtype=torch.int32))
    t["topk_ids"][3, 1] = s.E + 5            # out of range
    t["topk_ids"][5, 0] = -1
    t["topk_w"].fill_(0.5)
    t["perm_src"].fill_(-7)
    t["w_row"].fill_(-9.0)
    m.moe_dispatch(cfg, x, T, d, ws)
    st = m.moe_read_status(cfg, ws)
    assert st & m.MOE_DEV_BAD_EXPERT_ID
    counts = np_(t["counts"])
    n = T * s.k - 2
    assert counts.sum() == n                               # the bad slots are skipped
    inv = np_(t["inv"])
    assert inv[3 * s.k + 1] == -1 and inv[5 * s.k + 0] == -1
    perm = np_(t["perm_src"])
    assert (perm[:n] >= 0).all() and (perm[n:] == -7).all()  # rows past the valid ones untouched
    assert (np_(t["w_row"])[n:] == -9.0).all()
    _check_guards(t)
    assert m.moe_read_status(cfg, ws) == 0                 # reading clears it


def test_empty_experts_write_nothing_outside_their_rows():
    """Zipf-skewed routing with many empty experts, run step by step into
    caller buffers between canary bands: the dispatch, W1 (y1), W2 (z) and
    combine outputs touch no byte outside their valid rows, and equal the
    layer forward's."""
    dev = cuda_device()
    s = inputs.workload("tiny", E=32, k=4, logits="zipf")
    T = 48
    r = run_forward(s, T, dev=dev, seed=2)
    cfg, ws = r["cfg"], r["ws"]
    counts_ref = np_(r["views"]["counts"])
    assert (counts_ref == 0).sum() >= 9
    t, d = _alloc_dispatch(s, T, dev, guard=True)
    m.moe_route_dispatch(cfg, r["logits_in"], r["x"], T, d, ws)
    R = T * s.kp
    y1q_w, y1q = _guarded(R * s.I, torch.uint8, dev, 0xC3)
    y1s_w, y1s = _guarded(R * s.I // 32, torch.uint8, dev, 0xC3)
    z_w, z = _guarded(R * s.H, torch.int16, dev, 0x1357)
    out_w, out = _guarded(T * s.H, torch.int16, dev, 0x2468)
    y1q, y1s = y1q.view(R, s.I), y1s.view(R, s.I // 32)
    m.moe_grouped_gemm_w1_swiglu_quant(cfg, d, T, r["packed"], y1q, y1s, None, ws)
    m.moe_grouped_gemm_w2(cfg, d, T, y1q, y1s, r["packed"], z.view(R, s.H), ws)
    m.moe_combine(cfg, z.view(R, s.H), t["inv"], None, T, out.view(T, s.H))
    torch.cuda.synchronize()
    assert m.moe_read_status(cfg, ws) == 0
    _check_guards(t)
    assert _guards_intact(y1q_w, R * s.I, 0xC3) and _guards_intact(y1s_w, R * s.I // 32, 0xC3)
    assert _guards_intact(z_w, R * s.H, 0x1357) and _guards_intact(out_w, T * s.H, 0x2468)
    assert torch.equal(t["counts"], r["views"]["counts"])
    assert torch.equal(y1q, r["views"]["y1_q"]) and torch.equal(y1s, r["views"]["y1_s"])
    assert torch.equal(z.view(R, s.H), r["views"]["z"])
    assert torch.equal(out.view(T, s.H), r["out"].view(torch.int16))


def test_nan_logit_flags_status():
    dev = cuda_device()
    s = inputs.workload("tiny")
    T = 4
    cfg = m.config_from_shape(s, T_max=T)
    ws = torch.zeros(m.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    logits = torch.randn(T, s.E, device=dev)
    logits[2, 3] = float("nan")
    ids = torch.empty(T, s.k, dtype=torch.int32, device=dev)
    w = torch.empty(T, s.k, dtype=torch.float32, device=dev)
    m.moe_route_topk(cfg, logits, T, ids, w, ws)
    assert m.moe_read_status(cfg, ws) & m.MOE_DEV_NAN_LOGIT
    assert ((ids >= 0) & (ids < s.E)).all()
    assert 3 not in ids[2].tolist()                         # NaN ranks last


def test_launch_accounting_and_phases():
    dev = cuda_device()
    s = inputs.workload("tiny")
    r = run_forward(s, s.T, dev=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(m.MOE_N_PHASE_EVENTS)]
    for e in ev:
        e.record()
    m.moe_set_phase_events(ev)
    m.moe_layer_forward(r["cfg"], r["x"], r["Wr"], None, s.T, r["packed"], r["out"], None, r["ws"])
    m.moe_set_phase_events(None)
    torch.cuda.synchronize()
    n = m.moe_last_launch_count()
    assert 5 <= n <= 12
    ts = [ev[0].elapsed_time(e) for e in ev]
    assert all(b >= a for a, b in zip(ts, ts[1:]))


@pytest.mark.parametrize("name,which", [("tiny", 0), ("mxfp4", 0), ("srelu", 0), ("srelu_mx", 0), ("train_small", 0),
                                        ("train_small", 1)])
def test_packed_layout_round_trip(name, which):
    """moe_prepack_weights followed by moe_debug_unpack_weights gives back the
    source bytes of both matrices exactly (NVFP4 tiles with gate/up
    interleave; MXFP8 and MXFP4 rows with the 96 + 96 gate/up tiles, and the
    MXFP8 dgrad copies)."""
    dev = cuda_device()
    if name == "tiny":
        s = inputs.workload("tiny", n_shared=1)
    elif name == "mxfp4":
        s = inputs.workload("tiny", H=384, I=384, E=5, k=2, n_shared=1, wfmt="mxfp4")
    elif name == "srelu":
        s = inputs.workload("tiny", I=192, act="srelu")                   # NVFP4 tiles of a non-gated W1
    elif name == "srelu_mx":
        s = inputs.workload("train", T=8, E=5, H=320, I=256, act="srelu")  # MXFP8 rows, no gate / up interleave
    else:
        s = inputs.workload("train", T=8, E=5, H=320, I=128)
    cfg = m.config_from_shape(s, T_max=8)
    wts = inputs.gen_expert_weights(s, 0, device=dev)
    packed = m.moe_prepack_weights(cfg, wts, which)
    suffix = "" if which == m.MOE_PACK_FORWARD else "t"
    for mat in (1, 2):
        src_q, src_s = wts[f"w{mat}{suffix}_q"], wts[f"w{mat}{suffix}_s"]
        q = torch.full_like(src_q, 0x5A)
        sc = torch.full_like(src_s, 0x5A)
        m.moe_debug_unpack_weights(cfg, packed, which, mat, q, sc)
        torch.cuda.synchronize()
        assert torch.equal(q, src_q), f"codes of matrix {mat}"
        assert torch.equal(sc, src_s), f"scales of matrix {mat}"


def test_wrong_pack_sets_status_and_writes_nothing():
    """A blob packed for the dgrad copies handed to the forward sets
    MOE_DEV_BAD_PACK; the GEMMs write nothing."""
    dev = cuda_device()
    s = inputs.workload("train", T=16, E=4, H=320, I=128)
    r = run_forward(s, s.T, dev=dev)
    cfg, ws = r["cfg"], r["ws"]
    wrong = m.moe_prepack_weights(cfg, r["wts"], m.MOE_PACK_DGRAD)
    out = torch.full_like(r["out"], 7.0)
    v = r["views"]
    v["y1_q"].fill_(0x33)
    m.moe_layer_forward(cfg, r["x"], r["Wr"], None, s.T, wrong, out, None, ws)
    torch.cuda.synchronize()
    st = m.moe_read_status(cfg, ws)
    assert st & m.MOE_DEV_BAD_PACK
    assert (v["y1_q"] == 0x33).all()


def test_flag_wait_times_out_and_context_survives():
    """The fused layer's cross-CTA wait is bounded: waiting on a flag that
    nothing sets gives up after the limit and sets MOE_DEV_TIMEOUT; a set
    flag passes; the context stays usable (a layer forward afterwards matches
    one before)."""
    dev = cuda_device()
    s = inputs.workload("tiny", T=4)
    r = run_forward(s, s.T, dev=dev)
    cfg, ws = r["cfg"], r["ws"]
    flag = torch.zeros(4, dtype=torch.int32, device=dev)
    m.moe_debug_flag_wait(cfg, flag, 20_000_000, ws)          # ~10 ms at the top clock
    assert m.moe_read_status(cfg, ws) == m.MOE_DEV_TIMEOUT
    flag.fill_(1)
    m.moe_debug_flag_wait(cfg, flag, 20_000_000, ws)
    assert m.moe_read_status(cfg, ws) == 0
    out2 = torch.empty_like(r["out"])
    m.moe_layer_forward(cfg, r["x"], r["Wr"], None, s.T, r["packed"], out2, None, ws)
    torch.cuda.synchronize()
    assert m.moe_read_status(cfg, ws) == 0
    assert torch.equal(out2, r["out"])


@pytest.mark.parametrize("E", [200, 202])
@pytest.mark.parametrize("T", [1, 5, 16, 17, 32, 33, 100])
def test_router_logits_every_kernel(T, E):
    """Router logits through each kernel the split-K router picks by batch
    size: the register-resident kernel for one token, for T <= 8, <= 16 and
    <= 32, and the staged 64-token x 128-expert tile kernel above that.
    E = 200 leaves the last 64- and 128-expert tiles ragged; E = 202 (rows
    not a multiple of 16 bytes) takes the scalar-load kernel. Against the
    fp64 product of the same bf16 x and fp32 W_r, and the allocation-free
    entry point bit for bit."""
    dev = cuda_device()
    s = inputs.workload("tiny", T=T, H=1024, E=E)
    cfg = m.make_config(s.H, s.I, s.E, s.k, T_max=128)
    x = inputs.gen_x(s, 40 + T, device=dev)
    Wr = inputs.gen_router(s, 40 + T, device=dev)
    ws = torch.zeros(m.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    logits = torch.full((T, s.E), float("nan"), dtype=torch.float32, device=dev)
    m.moe_router_logits(cfg, x, Wr, T, logits, ws)
    got = torch.full((T, s.E), float("nan"), dtype=torch.float32, device=dev)
    m.moe_router_logits_noalloc(cfg, x, Wr, T, got)
    torch.cuda.synchronize()
    ref = M.router_logits(np_(x.float()), np_(Wr))
    np.testing.assert_allclose(np_(logits), ref, rtol=1e-4, atol=1e-5)
    assert torch.equal(got, logits)


def test_router_logits_large_batch():
    """Router logits at a batch whose 64-token x 128-expert tiles fill the
    SMs (the large-batch logits kernel, no split of H), ragged in tokens
    (T % 64 = 36) and in experts (E = 200: the second expert tile is partly
    empty), against the fp64 product of the same bf16 x and fp32 W_r."""
    dev = cuda_device()
    s = inputs.workload("tiny", T=4900, H=512, E=200)
    T = s.T
    cfg = m.make_config(s.H, s.I, s.E, s.k, T_max=T)
    x = inputs.gen_x(s, 5, device=dev)
    Wr = inputs.gen_router(s, 5, device=dev)
    ws = torch.zeros(m.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    logits = torch.full((T, s.E), float("nan"), dtype=torch.float32, device=dev)
    m.moe_router_logits(cfg, x, Wr, T, logits, ws)
    torch.cuda.synchronize()
    ref = M.router_logits(np_(x.float()), np_(Wr))
    np.testing.assert_allclose(np_(logits), ref, rtol=1e-4, atol=1e-5)
