"""The C-ABI library builds, loads, exports every symbol include/moe.h declares,
and rejects bad arguments on the host (no GPU needed: every checked call
returns before touching the device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from quantized_grouped_gemm_topk_gb300 import build as b
    b.build()
    from quantized_grouped_gemm_topk_gb300 import binding
    return binding.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    from quantized_grouped_gemm_topk_gb300 import binding
    names = _declared()
    assert len(names) >= 19
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(binding.EXPORTS) == names


def _cfg(**kw):
    from quantized_grouped_gemm_topk_gb300 import binding as m
    base = dict(H=256, I=128, E=8, k=2, T_max=16)
    base.update(kw)
    return m.make_config(**base)


def test_config_validation(lib):
    from quantized_grouped_gemm_topk_gb300 import binding as m
    assert m.moe_config_validate(_cfg()) == 0
    bad = [dict(H=200), dict(I=96), dict(k=0), dict(k=9), dict(n_shared=2), dict(E=2048, n_shared=1),
           dict(k=32, E=64, n_shared=1), dict(T_max=-1), dict(act="swiglu_clamp", limit=0.0),
           dict(routed_scale=0.0), dict(max_sms=-1)]
    for b in bad:
        assert m.moe_config_validate(_cfg(**b)) == 1, b
    assert m.moe_config_validate(_cfg(act="swiglu_clamp", limit=7.0, alpha=1.702)) == 0
    # MXFP4 rows move in 128-element runs: H and I multiples of 128
    assert m.moe_config_validate(_cfg(wfmt="mxfp4")) == 0
    assert m.moe_config_validate(_cfg(wfmt="mxfp4", H=320)) == 1
    assert m.moe_config_validate(_cfg(wfmt="mxfp4", I=192)) == 1
    assert m.moe_config_validate(_cfg(wfmt="mxfp8", H=320, I=192)) == 0


def test_sizes(lib):
    from quantized_grouped_gemm_topk_gb300 import binding as m
    c = _cfg()
    assert m.moe_workspace_size(c) > 0
    nv = m.moe_packed_weights_size(c)
    # 2 matrices x 8 groups x tiles x chunks x 4608 B, plus header/scales
    assert nv >= 8 * (2 * (256 // 64) + 2 * (128 // 64)) * 4608
    with pytest.raises(m.MoEError):
        m.moe_packed_weights_size(c, m.MOE_PACK_DGRAD)       # NVFP4 has no dgrad copy
    c8 = _cfg(wfmt="mxfp8")
    assert m.moe_packed_weights_size(c8, m.MOE_PACK_DGRAD) > 0
    assert m.moe_train_sizes(c8, 16) % 32 == 0
    with pytest.raises(m.MoEError):
        m.moe_train_sizes(c8, 17)                            # T > T_max
    c4 = _cfg(wfmt="mxfp4")
    # codes K/2 bytes a row (as NVFP4) but E8M0 scales per 32: smaller than MXFP8
    assert 0 < m.moe_packed_weights_size(c4) < m.moe_packed_weights_size(c8)
    with pytest.raises(m.MoEError):
        m.moe_packed_weights_size(c4, m.MOE_PACK_DGRAD)      # forward only


def test_host_errors_enqueue_nothing(lib):
    from quantized_grouped_gemm_topk_gb300 import binding as m
    c = _cfg()
    P = ctypes.c_void_p
    # NULL / misaligned pointers and bad T are rejected before any device work
    assert lib.moe_layer_forward(ctypes.byref(c), None, None, None, 4, None, None, None, None, None) == 1
    assert lib.moe_layer_forward(ctypes.byref(c), 0x1000, 0x1000, 0x2000, 4, 0x3000, 0x4000, None, 0x5000,
                                 None) == 1               # both W_r and logits given
    assert lib.moe_layer_forward(ctypes.byref(c), 0x1001, 0x1000, None, 4, 0x3000, 0x4000, None, 0x5000,
                                 None) == 1               # misaligned x
    assert lib.moe_layer_forward(ctypes.byref(c), 0x1000, 0x1000, None, 17, 0x3000, 0x4000, None, 0x5000,
                                 None) == 1               # T > T_max
    assert lib.moe_combine(ctypes.byref(c), None, P(0x1000), None, 4, P(0x2000), None) == 1
    assert lib.moe_layer_backward(ctypes.byref(c), 0x10, 0x10, 4, None, 0x10, 0x10, 0x10, 0x10, 0x10, None,
                                  0x10, None) == 2        # NVFP4 config: backward unsupported
    assert m.moe_status_string(0) == "ok"


def test_more_host_errors(lib):
    """Further argument checks that return before any device work (on this
    machine without a GPU, a call that reached the CUDA runtime would return
    MOE_ERR_CUDA instead)."""
    from quantized_grouped_gemm_topk_gb300 import binding as m
    c = _cfg()
    P = ctypes.c_void_p
    by = ctypes.byref
    # prepack: destination smaller than moe_packed_weights_size
    src = m.moe_weights_view_t(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000)
    assert lib.moe_prepack_weights(by(c), by(src), m.MOE_PACK_FORWARD, P(0x2000), 16, None) == 3
    # prepack: NVFP4 needs the per-group fp32 scales; `which` out of range
    src_nogs = m.moe_weights_view_t(0x1000, 0x1000, None, 0x1000, 0x1000, None)
    assert lib.moe_prepack_weights(by(c), by(src_nogs), m.MOE_PACK_FORWARD, P(0x2000), 1 << 30, None) == 1
    assert lib.moe_prepack_weights(by(c), by(src), 7, P(0x2000), 1 << 30, None) == 1
    # top-k alone: T > T_max, misaligned output; T = 0 accepts NULL row buffers
    assert lib.moe_route_topk(by(c), P(0x1000), 17, P(0x2000), P(0x3000), P(0x4000), None) == 1
    assert lib.moe_route_topk(by(c), P(0x1000), 4, P(0x2004), P(0x3000), P(0x4000), None) == 1
    assert lib.moe_route_topk(by(c), None, 0, None, None, P(0x4000), None) == 0
    # workspace-free router: NULL W_r, T > T_max; T = 0 is a no-op
    assert lib.moe_router_logits_noalloc(by(c), P(0x1000), None, 4, P(0x2000), None) == 1
    assert lib.moe_router_logits_noalloc(by(c), P(0x1000), P(0x1000), 17, P(0x2000), None) == 1
    assert lib.moe_router_logits_noalloc(by(c), None, P(0x1000), 0, None, None) == 0
    # an invalid config is reported by every entry point
    bad = _cfg(k=0)
    assert lib.moe_layer_forward(by(bad), 0x1000, 0x1000, None, 4, 0x3000, 0x4000, None, 0x5000, None) == 1
    assert lib.moe_route_topk(by(bad), P(0x1000), 4, P(0x2000), P(0x3000), P(0x4000), None) == 1
    # status strings exist for every code
    for code in range(6):
        assert m.moe_status_string(code) not in ("", "unknown status")


def test_layer_fused_rule(lib):
    """The fused W1 -> W2 layer runs for NVFP4 weights, I <= 2048 and at most
    2 token rows per group on average; otherwise the separate kernels."""
    from quantized_grouped_gemm_topk_gb300 import binding as m
    c = m.make_config(H=7168, I=2048, E=256, k=8, T_max=128)
    assert [m.moe_layer_fused(c, T) for T in (0, 1, 8, 32, 64, 65, 128)] == [False, True, True, True, True, False,
                                                                              False]
    assert not m.moe_layer_fused(m.make_config(H=7168, I=2048, E=256, k=8, T_max=128, wfmt="mxfp8"), 8)
    assert not m.moe_layer_fused(m.make_config(H=7168, I=2560, E=256, k=8, T_max=128), 8)
    s = m.make_config(H=6144, I=1536, E=160, k=8, n_shared=1, T_max=64)   # 9 rows a token over 161 groups
    assert m.moe_layer_fused(s, 35) and not m.moe_layer_fused(s, 36)
    with pytest.raises(m.MoEError):
        m.moe_layer_fused(c, 129)                                          # T > T_max


def test_flag_wait_host_errors(lib):
    """moe_debug_flag_wait checks its arguments on the host and enqueues
    nothing on an error."""
    import ctypes
    from quantized_grouped_gemm_topk_gb300 import binding as m
    c = _cfg()
    L = m.load()
    fake = ctypes.c_void_p(4096)
    assert L.moe_debug_flag_wait(ctypes.byref(c), None, 100, fake, None) == 1
    assert L.moe_debug_flag_wait(ctypes.byref(c), fake, 0, fake, None) == 1
    assert L.moe_debug_flag_wait(ctypes.byref(c), ctypes.c_void_p(4098), 100, fake, None) == 1
    assert L.moe_last_launch_count() == 0


def test_w1_bias_host_rules(lib):
    """w1_bias is 0 or 1; it enlarges the forward pack by G * 2I fp32 and
    leaves the dgrad pack alone; the backward of a biased config requires
    the db1 output, and an unbiased one refuses it, before any device work."""
    import ctypes
    from quantized_grouped_gemm_topk_gb300 import binding as m
    c0 = _cfg(wfmt="mxfp8")
    c1 = _cfg(wfmt="mxfp8", bias=True)
    assert m.moe_config_validate(c1) == 0
    bad = _cfg()
    bad.w1_bias = 2
    assert m.moe_config_validate(bad) == 1
    assert m.moe_packed_weights_size(c1) - m.moe_packed_weights_size(c0) >= 8 * 2 * 128 * 4
    assert m.moe_packed_weights_size(c1, m.MOE_PACK_DGRAD) == m.moe_packed_weights_size(c0, m.MOE_PACK_DGRAD)
    fake = ctypes.c_void_p(4096)
    L = m.load()
    save = m.moe_train_save_t(4096, 4096, 4096, 4096, 4096, 4096, None)
    by = ctypes.byref
    assert L.moe_layer_backward(by(c1), fake, fake, 16, by(save), fake, fake, fake, fake, fake, None, fake,
                                None) == 1                 # bias: db1 required
    assert L.moe_layer_backward(by(c0), fake, fake, 16, by(save), fake, fake, fake, fake, fake, fake, fake,
                                None) == 1                 # no bias: no db1


def test_srelu_host_rules(lib):
    """sReLU: valid; its W1 pack holds I rows (a smaller blob than the gated
    W1's 2I), and so does its dgrad pack's W1 copy (K = I); no bias, no
    fused layer."""
    from quantized_grouped_gemm_topk_gb300 import binding as m
    g = _cfg(wfmt="mxfp8")
    c = _cfg(wfmt="mxfp8", act="srelu")
    assert m.moe_config_validate(c) == 0
    assert m.moe_packed_weights_size(c) < m.moe_packed_weights_size(g)
    assert 0 < m.moe_packed_weights_size(c, m.MOE_PACK_DGRAD) < m.moe_packed_weights_size(g, m.MOE_PACK_DGRAD)
    with pytest.raises(m.MoEError):
        m.moe_packed_weights_size(_cfg(act="srelu"), m.MOE_PACK_DGRAD)   # NVFP4: no dgrad copy
    assert m.moe_config_validate(_cfg(act="srelu", bias=True)) == 2
    assert not m.moe_layer_fused(_cfg(act="srelu"), 1)


def test_dispatch_sms_host_rules(lib):
    """dispatch_sms (the partitioned fused layer's ring CTAs) is 0..64."""
    from quantized_grouped_gemm_topk_gb300 import binding as m
    for nd, want in ((0, 0), (8, 0), (64, 0), (-1, 1), (65, 1)):
        c = _cfg()
        c.dispatch_sms = nd
        assert m.moe_config_validate(c) == want, nd
