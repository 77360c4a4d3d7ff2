"""Thin ctypes binding of libmoe.so (include/moe.h).

Argument marshalling only: each ``moe_*`` function takes torch tensors (on the
current CUDA device) and passes their device pointers, sizes and the current
CUDA stream to the C entry point of the same name. Every step of the layer
runs in the library's CUDA kernels; there is no other implementation here. If
the library is missing or no CUDA device is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libmoe.so")

MOE_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace too small",
                4: "CUDA error", 5: "device status error"}
MOE_DEV_BAD_EXPERT_ID = 0x1
MOE_DEV_NAN_LOGIT = 0x2
MOE_DEV_BAD_PACK = 0x4
MOE_DEV_TIMEOUT = 0x8
MOE_ACT_SWIGLU, MOE_ACT_SWIGLU_CLAMP, MOE_ACT_GEGLU, MOE_ACT_SRELU = 0, 1, 2, 3
ACTS = {"swiglu": MOE_ACT_SWIGLU, "swiglu_clamp": MOE_ACT_SWIGLU_CLAMP, "geglu": MOE_ACT_GEGLU,
        "srelu": MOE_ACT_SRELU}
MOE_WFMT_NVFP4, MOE_WFMT_MXFP8, MOE_WFMT_MXFP4 = 0, 1, 2
WFMTS = {"nvfp4": MOE_WFMT_NVFP4, "mxfp8": MOE_WFMT_MXFP8, "mxfp4": MOE_WFMT_MXFP4}
MOE_PACK_FORWARD, MOE_PACK_DGRAD = 0, 1

# every exported symbol the header declares
EXPORTS = (
    "moe_config_validate", "moe_workspace_size", "moe_workspace_view", "moe_packed_weights_size",
    "moe_train_sizes", "moe_prepack_weights", "moe_router_logits", "moe_route_dispatch", "moe_route_topk",
    "moe_dispatch", "moe_grouped_gemm_w1_swiglu_quant", "moe_grouped_gemm_w2", "moe_combine",
    "moe_layer_forward", "moe_layer_backward", "moe_read_status", "moe_clear_status", "moe_status_string",
    "moe_last_launch_count", "moe_set_phase_events", "moe_router_logits_noalloc", "moe_debug_unpack_weights",
    "moe_layer_fused", "moe_debug_flag_wait",
)
MOE_N_PHASE_EVENTS = 6


class MoEError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {code} ({STATUS_NAMES.get(code, '?')})")
        self.code = code


class moe_config_t(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("T_max", ctypes.c_int32), ("act", ctypes.c_int32),
                ("act_alpha", ctypes.c_float), ("act_limit", ctypes.c_float), ("routed_scale", ctypes.c_float),
                ("weight_fmt", ctypes.c_int32), ("max_sms", ctypes.c_int32), ("w1_bias", ctypes.c_int32),
                ("dispatch_sms", ctypes.c_int32)]


class moe_weights_view_t(ctypes.Structure):
    _fields_ = [("w1_q", ctypes.c_void_p), ("w1_s", ctypes.c_void_p), ("w1_gs", ctypes.c_void_p),
                ("w2_q", ctypes.c_void_p), ("w2_s", ctypes.c_void_p), ("w2_gs", ctypes.c_void_p),
                ("b1", ctypes.c_void_p)]


class moe_dispatch_t(ctypes.Structure):
    _fields_ = [("topk_ids", ctypes.c_void_p), ("topk_w", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("perm_src", ctypes.c_void_p), ("inv", ctypes.c_void_p),
                ("w_row", ctypes.c_void_p), ("xq", ctypes.c_void_p), ("xs", ctypes.c_void_p)]


class moe_train_save_t(ctypes.Structure):
    _fields_ = [("h", ctypes.c_void_p), ("y1t_q", ctypes.c_void_p), ("y1t_s", ctypes.c_void_p),
                ("at_q", ctypes.c_void_p), ("at_s", ctypes.c_void_p), ("poff", ctypes.c_void_p),
                ("amax", ctypes.c_void_p)]


class moe_ws_view_t(ctypes.Structure):
    _fields_ = [("logits", ctypes.c_void_p), ("d", moe_dispatch_t), ("y1_q", ctypes.c_void_p),
                ("y1_s", ctypes.c_void_p), ("z", ctypes.c_void_p), ("status", ctypes.c_void_p)]


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libmoe.so (built by quantized_grouped_gemm_topk_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libmoe.so not built at {p}; run quantized_grouped_gemm_topk_gb300.build.build()")
    lib = ctypes.CDLL(p)
    P = ctypes.c_void_p
    cfgp = ctypes.POINTER(moe_config_t)
    sig = {
        "moe_config_validate": [cfgp],
        "moe_workspace_size": [cfgp, ctypes.POINTER(ctypes.c_size_t)],
        "moe_workspace_view": [cfgp, P, ctypes.POINTER(moe_ws_view_t)],
        "moe_packed_weights_size": [cfgp, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)],
        "moe_train_sizes": [cfgp, ctypes.c_int, ctypes.POINTER(ctypes.c_int64)],
        "moe_prepack_weights": [cfgp, ctypes.POINTER(moe_weights_view_t), ctypes.c_int, P, ctypes.c_size_t, P],
        "moe_router_logits": [cfgp, P, P, ctypes.c_int, P, P, P],
        "moe_route_dispatch": [cfgp, P, P, ctypes.c_int, ctypes.POINTER(moe_dispatch_t), P, P],
        "moe_route_topk": [cfgp, P, ctypes.c_int, P, P, P, P],
        "moe_dispatch": [cfgp, P, ctypes.c_int, ctypes.POINTER(moe_dispatch_t), P, P],
        "moe_grouped_gemm_w1_swiglu_quant": [cfgp, ctypes.POINTER(moe_dispatch_t), ctypes.c_int, P, P, P,
                                             ctypes.POINTER(moe_train_save_t), P, P],
        "moe_grouped_gemm_w2": [cfgp, ctypes.POINTER(moe_dispatch_t), ctypes.c_int, P, P, P, P, P, P],
        "moe_combine": [cfgp, P, P, P, ctypes.c_int, P, P],
        "moe_layer_forward": [cfgp, P, P, P, ctypes.c_int, P, P, ctypes.POINTER(moe_train_save_t), P, P],
        "moe_layer_backward": [cfgp, P, P, ctypes.c_int, ctypes.POINTER(moe_train_save_t), P, P, P, P, P, P, P],
        "moe_read_status": [cfgp, P, ctypes.POINTER(ctypes.c_int32), P],
        "moe_clear_status": [cfgp, P, P],
        "moe_status_string": [ctypes.c_int],
        "moe_last_launch_count": [],
        "moe_set_phase_events": [ctypes.POINTER(ctypes.c_void_p)],
        "moe_layer_fused": [cfgp, ctypes.c_int, ctypes.POINTER(ctypes.c_int32)],
        "moe_debug_flag_wait": [cfgp, P, ctypes.c_int64, P, P],
        "moe_router_logits_noalloc": [cfgp, P, P, ctypes.c_int, P, P],
        "moe_debug_unpack_weights": [cfgp, P, ctypes.c_int, ctypes.c_int, P, P, P],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_char_p if name == "moe_status_string" else ctypes.c_int
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(name, code):
    if code != MOE_OK:
        raise MoEError(name, code)


def _require_cuda():
    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: the routed-MoE library runs only on the GPU")


def make_config(H, I, E, k, n_shared=0, T_max=0, act="swiglu", alpha=1.0, limit=0.0, routed_scale=1.0,
                wfmt="nvfp4", max_sms=0, bias=False, dispatch_sms=0) -> moe_config_t:
    return moe_config_t(H, I, E, k, n_shared, T_max,
                        ACTS[act],
                        float(alpha), float(limit), float(routed_scale),
                        WFMTS[wfmt], max_sms, 1 if bias else 0, dispatch_sms)


def config_from_shape(s, T_max=None, max_sms=0, dispatch_sms=0) -> moe_config_t:
    """moe_config_t from an object with the fields of inputs.MoEShape."""
    return make_config(s.H, s.I, s.E, s.k, s.n_shared, s.T if T_max is None else T_max, s.act, s.alpha,
                       s.limit, s.routed_scale, s.wfmt, max_sms, getattr(s, "bias", False), dispatch_sms)


# ---- sizes / views (host only) -----------------------------------------------
def moe_config_validate(cfg) -> int:
    return load().moe_config_validate(ctypes.byref(cfg))


def moe_workspace_size(cfg) -> int:
    n = ctypes.c_size_t()
    _check("moe_workspace_size", load().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def moe_packed_weights_size(cfg, which=MOE_PACK_FORWARD) -> int:
    n = ctypes.c_size_t()
    _check("moe_packed_weights_size", load().moe_packed_weights_size(ctypes.byref(cfg), which, ctypes.byref(n)))
    return n.value


def moe_train_sizes(cfg, T) -> int:
    n = ctypes.c_int64()
    _check("moe_train_sizes", load().moe_train_sizes(ctypes.byref(cfg), T, ctypes.byref(n)))
    return n.value


def moe_workspace_view(cfg, ws) -> moe_ws_view_t:
    v = moe_ws_view_t()
    _check("moe_workspace_view", load().moe_workspace_view(ctypes.byref(cfg), _ptr(ws), ctypes.byref(v)))
    return v


def moe_status_string(code) -> str:
    return load().moe_status_string(code).decode()


def moe_last_launch_count() -> int:
    return load().moe_last_launch_count()


def moe_debug_flag_wait(cfg, flag, limit_cycles, ws, stream=None):
    """The fused layer's bounded flag wait on its own (flag: int32 device tensor)."""
    _check("moe_debug_flag_wait", load().moe_debug_flag_wait(ctypes.byref(cfg), _ptr(flag), int(limit_cycles),
                                                              _ptr(ws), _stream(stream)))


def moe_layer_fused(cfg, T) -> bool:
    """Whether moe_layer_forward runs W1 -> W2 as one persistent kernel at T."""
    v = ctypes.c_int32(0)
    _check("moe_layer_fused", load().moe_layer_fused(ctypes.byref(cfg), int(T), ctypes.byref(v)))
    return bool(v.value)


def moe_set_phase_events(events):
    """events: MOE_N_PHASE_EVENTS torch.cuda.Event(enable_timing=True) (each
    recorded once beforehand so its handle exists), or None to switch off."""
    if events is None:
        _check("moe_set_phase_events", load().moe_set_phase_events(None))
        return
    if len(events) != MOE_N_PHASE_EVENTS or not all(e.cuda_event for e in events):
        raise ValueError(f"moe_set_phase_events needs {MOE_N_PHASE_EVENTS} events, each recorded once")
    arr = (ctypes.c_void_p * MOE_N_PHASE_EVENTS)(*[e.cuda_event for e in events])
    moe_set_phase_events._keep = arr
    _check("moe_set_phase_events", load().moe_set_phase_events(arr))


# ---- device calls ----------------------------------------------------------------
def moe_prepack_weights(cfg, wts: dict, which=MOE_PACK_FORWARD, dst=None, stream=None):
    """wts: tensors named as in inputs.gen_expert_weights (w1_q, w1_s, w1_gs,
    w2_q, ...; for which=MOE_PACK_DGRAD the w1t_* / w2t_* copies)."""
    _require_cuda()
    n = moe_packed_weights_size(cfg, which)
    if dst is None:
        dst = torch.empty(n, dtype=torch.uint8, device="cuda")
    p = "" if which == MOE_PACK_FORWARD else "t"
    view = moe_weights_view_t(_ptr(wts[f"w1{p}_q"]), _ptr(wts[f"w1{p}_s"]), _ptr(wts.get("w1_gs")),
                              _ptr(wts[f"w2{p}_q"]), _ptr(wts[f"w2{p}_s"]), _ptr(wts.get("w2_gs")),
                              _ptr(wts.get("b1")))
    _check("moe_prepack_weights", load().moe_prepack_weights(ctypes.byref(cfg), ctypes.byref(view), which,
                                                             _ptr(dst), dst.numel(), _stream(stream)))
    return dst


def moe_debug_unpack_weights(cfg, packed, which, mat, q, s, stream=None):
    """Plain-layout copy of matrix `mat` (1 or 2) of a packed blob (tests)."""
    _check("moe_debug_unpack_weights", load().moe_debug_unpack_weights(ctypes.byref(cfg), _ptr(packed), which, mat,
                                                                       _ptr(q), _ptr(s), _stream(stream)))


def moe_router_logits(cfg, x, W_r, T, logits, ws, stream=None):
    _check("moe_router_logits", load().moe_router_logits(ctypes.byref(cfg), _ptr(x), _ptr(W_r), T, _ptr(logits),
                                                         _ptr(ws), _stream(stream)))


def moe_router_logits_noalloc(cfg, x, W_r, T, logits, stream=None):
    """Router logits with no workspace: for callers that cannot allocate
    device memory; the split partials live in the library's static device
    scratch (see include/moe.h for its size limit and sharing rules)."""
    _check("moe_router_logits_noalloc", load().moe_router_logits_noalloc(ctypes.byref(cfg), _ptr(x), _ptr(W_r), T,
                                                                         _ptr(logits), _stream(stream)))


def moe_route_topk(cfg, logits, T, ids, w, ws, stream=None):
    _check("moe_route_topk", load().moe_route_topk(ctypes.byref(cfg), _ptr(logits), T, _ptr(ids), _ptr(w),
                                                   _ptr(ws), _stream(stream)))


def moe_route_dispatch(cfg, logits, x, T, d: moe_dispatch_t, ws, stream=None):
    _check("moe_route_dispatch", load().moe_route_dispatch(ctypes.byref(cfg), _ptr(logits), _ptr(x), T,
                                                           ctypes.byref(d), _ptr(ws), _stream(stream)))


def moe_dispatch(cfg, x, T, d: moe_dispatch_t, ws, stream=None):
    _check("moe_dispatch", load().moe_dispatch(ctypes.byref(cfg), _ptr(x), T, ctypes.byref(d), _ptr(ws),
                                               _stream(stream)))


def moe_grouped_gemm_w1_swiglu_quant(cfg, d, T, packed, y1_q, y1_s, save, ws, stream=None):
    _check("moe_grouped_gemm_w1_swiglu_quant",
           load().moe_grouped_gemm_w1_swiglu_quant(ctypes.byref(cfg), ctypes.byref(d), T, _ptr(packed), _ptr(y1_q),
                                                   _ptr(y1_s), ctypes.byref(save) if save is not None else None,
                                                   _ptr(ws), _stream(stream)))


def moe_grouped_gemm_w2(cfg, d, T, y1_q, y1_s, packed, z, ws, stream=None):
    _check("moe_grouped_gemm_w2", load().moe_grouped_gemm_w2(ctypes.byref(cfg), ctypes.byref(d), T, _ptr(y1_q),
                                                             _ptr(y1_s), _ptr(packed), _ptr(z), _ptr(ws),
                                                             _stream(stream)))


def moe_combine(cfg, z, inv, topk_w, T, out, stream=None):
    _check("moe_combine", load().moe_combine(ctypes.byref(cfg), _ptr(z), _ptr(inv), _ptr(topk_w), T, _ptr(out),
                                             _stream(stream)))


def moe_layer_forward(cfg, x, W_r, logits, T, packed, out, save, ws, stream=None):
    _check("moe_layer_forward",
           load().moe_layer_forward(ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(logits), T, _ptr(packed), _ptr(out),
                                    ctypes.byref(save) if save is not None else None, _ptr(ws), _stream(stream)))


def moe_layer_backward(cfg, dout, x, T, save, packed_dgrad, dx, dW1, dW2, dlogits, ws, stream=None, db1=None):
    """db1: [E, 2I] fp32 W1 bias gradient, required when cfg.w1_bias."""
    _check("moe_layer_backward",
           load().moe_layer_backward(ctypes.byref(cfg), _ptr(dout), _ptr(x), T, ctypes.byref(save),
                                     _ptr(packed_dgrad), _ptr(dx), _ptr(dW1), _ptr(dW2), _ptr(dlogits), _ptr(db1),
                                     _ptr(ws), _stream(stream)))


def moe_read_status(cfg, ws, stream=None) -> int:
    v = ctypes.c_int32()
    code = load().moe_read_status(ctypes.byref(cfg), _ptr(ws), ctypes.byref(v), _stream(stream))
    if code not in (MOE_OK, 5):
        raise MoEError("moe_read_status", code)
    return v.value


def moe_clear_status(cfg, ws, stream=None):
    _check("moe_clear_status", load().moe_clear_status(ctypes.byref(cfg), _ptr(ws), _stream(stream)))


# ---- convenience: torch views of the workspace buffers ------------------------------
def ws_tensor_views(cfg, ws, T):
    """Torch tensors aliasing the workspace buffers that moe_layer_forward fills
    for T tokens (for inspection in tests)."""
    v = moe_workspace_view(cfg, ws)
    kp = cfg.k + cfg.n_shared
    G = cfg.E + cfg.n_shared
    R = T * kp

    def view(ptr, n, dtype):
        base = ws.data_ptr()
        off = ptr - base
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return ws[off:off + nbytes].view(dtype)

    d = v.d
    return {
        "logits": view(v.logits, T * cfg.E, torch.float32).view(T, cfg.E),
        "topk_ids": view(d.topk_ids, T * cfg.k, torch.int32).view(T, cfg.k),
        "topk_w": view(d.topk_w, T * cfg.k, torch.float32).view(T, cfg.k),
        "counts": view(d.counts, G, torch.int32),
        "offsets": view(d.offsets, G + 1, torch.int32),
        "perm_src": view(d.perm_src, R, torch.int32),
        "inv": view(d.inv, R, torch.int32),
        "w_row": view(d.w_row, R, torch.float32),
        "xq": view(d.xq, T * cfg.H, torch.uint8).view(T, cfg.H),
        "xs": view(d.xs, T * cfg.H // 32, torch.uint8).view(T, cfg.H // 32),
        "y1_q": view(v.y1_q, R * cfg.I, torch.uint8).view(R, cfg.I),
        "y1_s": view(v.y1_s, R * cfg.I // 32, torch.uint8).view(R, cfg.I // 32),
        "z": view(v.z, R * cfg.H, torch.int16).view(R, cfg.H),
        "status": view(v.status, 1, torch.int32),
    }


def dispatch_struct(t: dict) -> moe_dispatch_t:
    """moe_dispatch_t over tensors named like ws_tensor_views' keys."""
    return moe_dispatch_t(_ptr(t["topk_ids"]), _ptr(t["topk_w"]), _ptr(t["counts"]), _ptr(t["offsets"]),
                          _ptr(t["perm_src"]), _ptr(t["inv"]), _ptr(t["w_row"]), _ptr(t["xq"]), _ptr(t["xs"]))


def alloc_train_save(cfg, T, device="cuda", amax=False):
    """Caller-side allocation of the training save buffers for T tokens
    (amax=True adds the NVFP4-recipe amax pair)."""
    rp = moe_train_sizes(cfg, T)
    kp = cfg.k + cfg.n_shared
    R = T * kp
    G = cfg.E + cfg.n_shared
    bufs = {
        "h": torch.empty(max(R, 1), (cfg.I if cfg.act == MOE_ACT_SRELU else 2 * cfg.I), dtype=torch.int16,
                         device=device),
        "y1t_q": torch.empty(cfg.I, rp, dtype=torch.uint8, device=device),
        "y1t_s": torch.empty(rp // 128, cfg.I, 4, dtype=torch.uint8, device=device),
        "at_q": torch.empty(cfg.H, rp, dtype=torch.uint8, device=device),
        "at_s": torch.empty(rp // 128, cfg.H, 4, dtype=torch.uint8, device=device),
        "poff": torch.empty(G + 1 + 3, dtype=torch.int32, device=device),
        "amax": torch.empty(4, dtype=torch.float32, device=device) if amax else None,
        "r_pad": rp,
    }
    st = moe_train_save_t(*(_ptr(bufs[k]) for k in ("h", "y1t_q", "y1t_s", "at_q", "at_s", "poff", "amax")))
    return st, bufs
