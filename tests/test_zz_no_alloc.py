"""The workspace-free router-logits entry point gives the same logits as the
workspace one.

moe_router_logits_noalloc exists for callers that cannot allocate device
memory where they need logits; it keeps its split partial sums in a static
device array owned by the library instead of the caller's workspace. Two
calls in a row (different batches, so the second must not see the first
one's leftovers) are compared against moe_router_logits on the same inputs.
This file is collected last on purpose.
"""
import pytest
import torch

import inputs
import quantized_grouped_gemm_topk_gb300 as m

pytestmark = pytest.mark.gpu


def test_noalloc_router_logits_matches_workspace_version():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    dev = torch.device("cuda:0")
    from quantized_grouped_gemm_topk_gb300 import build as b
    b.build()
    s = inputs.workload("dsv3")
    Tmax = 128
    cfg = m.config_from_shape(s, T_max=Tmax)
    ws = torch.zeros(m.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    Wr = inputs.gen_router(s, 0, device=dev)
    for call, T in enumerate((8, 128)):
        x = inputs.gen_x(s, 300 + call, device=dev, T=T)
        ref = torch.empty(T, s.E, dtype=torch.float32, device=dev)
        got = torch.full((T, s.E), float("nan"), dtype=torch.float32, device=dev)
        m.moe_router_logits(cfg, x, Wr, T, ref, ws)
        m.moe_router_logits_noalloc(cfg, x, Wr, T, got)
        torch.cuda.synchronize()
        # same kernels, same split count, same summation order: bit for bit
        assert torch.isfinite(got).all()
        assert torch.equal(got, ref)
