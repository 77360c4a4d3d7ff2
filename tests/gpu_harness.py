"""Runs the layer through the C ABI on seeded inputs and hands the same inputs
to the oracle (helpers for the -m gpu tests)."""
import numpy as np
import torch

import inputs
from oracle import moe as M

import quantized_grouped_gemm_topk_gb300 as m


class LazyExperts:
    """Per-expert numpy view of a device tensor (copies one expert on demand)."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return self.t[e].cpu().numpy()


def oracle_weights(wts):
    return {k: (v.cpu().numpy() if v.dim() == 1 else LazyExperts(v)) for k, v in wts.items()}


_WCACHE = {}


def weights_for(s, seed, dev):
    key = (s.name, s.H, s.I, s.E, s.n_shared, s.wfmt, s.act == "srelu", getattr(s, "bias", False), seed)
    if key not in _WCACHE:
        _WCACHE.clear()
        torch.cuda.empty_cache()
        _WCACHE[key] = inputs.gen_expert_weights(s, seed, device=dev)
    return _WCACHE[key]


def run_forward(s, T, seed=0, dev="cuda:0", save=False, max_sms=0):
    dev = torch.device(dev)
    x = inputs.gen_x(s, seed, device=dev, T=T)
    if s.logits == "router":
        Wr, lg = inputs.gen_router(s, seed, device=dev), None
    else:
        Wr, lg = None, inputs.gen_logits(s, seed, device=dev, T=T)
    wts = weights_for(s, seed, dev)
    cfg = m.config_from_shape(s, T_max=T, max_sms=max_sms)
    packed = m.moe_prepack_weights(cfg, wts)
    ws = torch.zeros(m.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    out = torch.empty(T, s.H, dtype=torch.bfloat16, device=dev)
    st, bufs = (m.alloc_train_save(cfg, T, dev) if save else (None, None))
    m.moe_layer_forward(cfg, x, Wr, lg, T, packed, out, st, ws)
    torch.cuda.synchronize()
    status = m.moe_read_status(cfg, ws)
    views = m.ws_tensor_views(cfg, ws, T)
    return dict(cfg=cfg, x=x, Wr=Wr, logits_in=lg, wts=wts, packed=packed, ws=ws, out=out, views=views,
                status=status, save=st, save_bufs=bufs)


def oracle_forward(s, r, rows=None):
    """Oracle forward on the GPU run's inputs; routing from the GPU's fp32 logits."""
    logits = r["views"]["logits"].cpu().numpy()
    xb = inputs.bf16_bits(r["x"]).cpu().numpy()
    return M.layer_forward(xb, logits, oracle_weights(r["wts"]), E=s.E, k=s.k, n_shared=s.n_shared,
                           routed_scale=s.routed_scale, act=s.act, alpha=s.alpha, limit=s.limit, wfmt=s.wfmt,
                           rows=rows)
