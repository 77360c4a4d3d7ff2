"""Seeded synthetic inputs for the routed-MoE layer workloads.

This module is shared by the tests, the oracle checks and the benchmark. It
holds no step of the layer: it draws token activations, router weights,
router logits, upstream gradients and expert weights from seeded generators,
and it encodes the expert weights into the storage formats the layer consumes
(NVFP4 or MXFP8 bytes), because the workloads hand the layer weights that are
already quantised. The layer itself (and the oracle) only ever decode weights.

Workloads (token count T, hidden H, expert FFN width I, E routed experts,
top-k, S shared experts):

* ``tiny``      T=16, H=256, I=128, E=8, k=2, NVFP4 weights.
* ``dsv3``      DeepSeek-V3-shaped decode: H=7168, I=2048, E=256, k=8,
                T in {1, 8, 32, 128}, NVFP4 weights.
* ``shared``    decode with one always-on shared expert: H=6144, I=1536,
                E=160, k=8, S=1 (width I), routed weights x2.5,
                T in {1, 16, 64}, NVFP4 weights.
* ``train``     training prefill: T=16384, H=2880, I=2880, E=128, k=4,
                MXFP8 weights, SwiGLU clamped at +-7 with alpha 1.702.
* ``skewed``    T=4096, H=4096, I=1536, E=128, k=8, router logits drawn so
                expert popularity is Zipf(1.2) with 30% of experts empty.

Seeds: x uses ``seed``, the router weights ``seed+1``, W1 ``seed+2`` (offset
per expert), W2 ``seed+3`` (offset per expert), the upstream gradient
``seed+4`` and the skewed logits ``seed+5``. Every draw uses a
``torch.Generator`` on the device the tensor is made on, so a given seed gives
the same values on every run of the same device type.
"""
from __future__ import annotations

import dataclasses
import math

import torch

__all__ = [
    "MoEShape", "WORKLOADS", "workload", "gen_x", "gen_router", "gen_logits",
    "gen_dout", "gen_expert_weights", "encode_nvfp4", "encode_mxfp8", "encode_mxfp4",
    "bf16_bits", "expected_touched",
]


@dataclasses.dataclass(frozen=True)
class MoEShape:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    n_shared: int = 0
    routed_scale: float = 1.0
    act: str = "swiglu"          # "swiglu" | "swiglu_clamp" | "geglu" | "srelu"
    alpha: float = 1.0
    limit: float = 0.0
    wfmt: str = "nvfp4"          # "nvfp4" | "mxfp8" | "mxfp4"
    bias: bool = False           # W1 carries a per-expert fp32 bias [2I] (gate b, up c)
    logits: str = "router"       # "router" (x @ W_r) | "zipf" (drawn directly)

    @property
    def kp(self) -> int:
        """Assignment slots per token: k routed plus the shared experts."""
        return self.k + self.n_shared

    @property
    def groups(self) -> int:
        """Expert groups in the grouped GEMMs: routed plus shared."""
        return self.E + self.n_shared

    def with_T(self, T: int) -> "MoEShape":
        return dataclasses.replace(self, T=T)


WORKLOADS = {
    "tiny": MoEShape("tiny", T=16, H=256, I=128, E=8, k=2),
    "dsv3": MoEShape("dsv3", T=128, H=7168, I=2048, E=256, k=8),
    "shared": MoEShape("shared", T=64, H=6144, I=1536, E=160, k=8, n_shared=1,
                       routed_scale=2.5),
    "train": MoEShape("train", T=16384, H=2880, I=2880, E=128, k=4,
                      act="swiglu_clamp", alpha=1.702, limit=7.0, wfmt="mxfp8"),
    "skewed": MoEShape("skewed", T=4096, H=4096, I=1536, E=128, k=8, logits="zipf"),
}

DECODE_T = {"dsv3": (1, 8, 32, 128), "shared": (1, 16, 64)}


def workload(name: str, T: int | None = None, **over) -> MoEShape:
    s = WORKLOADS[name]
    if T is not None:
        s = s.with_T(T)
    if over:
        s = dataclasses.replace(s, **over)
    return s


def expected_touched(s: MoEShape, T: int | None = None) -> float:
    """Expected number of routed experts that receive at least one token
    under uniform routing (used only to size work splits on the host)."""
    T = s.T if T is None else T
    return s.E * (1.0 - (1.0 - s.k / s.E) ** T) + s.n_shared


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def bf16_bits(t: torch.Tensor) -> torch.Tensor:
    """bfloat16 tensor -> its raw 16-bit patterns (int16 view)."""
    return t.contiguous().view(torch.int16)


def gen_x(s: MoEShape, seed: int = 0, device="cpu", T: int | None = None) -> torch.Tensor:
    """Token activations x ~ N(0, 1), rounded to bf16, shape [T, H]."""
    T = s.T if T is None else T
    g = _gen(seed, device)
    return torch.randn(T, s.H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def gen_router(s: MoEShape, seed: int = 0, device="cpu") -> torch.Tensor:
    """Router weights W_r ~ N(0, 0.02), fp32, shape [H, E]."""
    g = _gen(seed + 1, device)
    return torch.randn(s.H, s.E, generator=g, device=device, dtype=torch.float32) * 0.02


def gen_logits(s: MoEShape, seed: int = 0, device="cpu", T: int | None = None,
               empty_frac: float = 0.30, zipf_s: float = 1.2) -> torch.Tensor:
    """Skewed router logits, fp32 [T, E].

    floor(empty_frac * E) experts, chosen at random, get logit -1e30 and so
    never win a top-k slot. The remaining experts get Zipf popularities
    p_r ~ r^-zipf_s over randomly permuted ranks, and
    logit[t, e] = ln p_e + Gumbel(0, 1), so top-k is sampling without
    replacement in proportion to p.
    """
    T = s.T if T is None else T
    g = _gen(seed + 5, device)
    E = s.E
    perm = torch.randperm(E, generator=g, device=device)
    n_empty = int(math.floor(empty_frac * E))
    live = perm[n_empty:]
    ranks = torch.arange(1, live.numel() + 1, device=device, dtype=torch.float64)
    p = ranks.pow(-zipf_s)
    p = p / p.sum()
    base = torch.full((E,), -1e30, dtype=torch.float64, device=device)
    base[live] = torch.log(p)
    u = torch.rand(T, E, generator=g, device=device, dtype=torch.float64)
    u = u.clamp_(min=1e-300)
    gumbel = -torch.log(-torch.log(u))
    logits = base.unsqueeze(0) + gumbel
    logits[:, perm[:n_empty]] = -1e30
    return logits.to(torch.float32)


def gen_dout(s: MoEShape, seed: int = 0, device="cpu", T: int | None = None) -> torch.Tensor:
    """Upstream gradient dOut ~ N(0, 1), bf16 [T, H]."""
    T = s.T if T is None else T
    g = _gen(seed + 4, device)
    return torch.randn(T, s.H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


# ----------------------------------------------------------------------------
# Weight encoders (input preparation only).
# ----------------------------------------------------------------------------
_E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    """Nearest E2M1 code (ties to the even code), saturating at 6."""
    mag = v.abs().clamp(max=6.0)
    grid = torch.tensor(_E2M1_MAG, dtype=v.dtype, device=v.device)
    mids = (grid[1:] + grid[:-1]) * 0.5
    idx = (mag.unsqueeze(-1) > mids).sum(-1)          # ties land on the lower code
    tie = (mag.unsqueeze(-1) == mids).any(-1) & (idx % 2 == 1)
    idx = idx + tie.to(idx.dtype)
    sign = (v < 0) | ((v == 0) & torch.signbit(v))
    return (idx | (sign.to(idx.dtype) << 3)).to(torch.uint8)


def _e4m3_codes(v: torch.Tensor) -> torch.Tensor:
    return v.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)


def encode_nvfp4(w: torch.Tensor):
    """NVFP4-encode one matrix stored [N, K] (K contiguous).

    gs = amax(w) / (6*448) (fp32, one per matrix); per block of 16 along K the
    E4M3 scale s_b = RNE(amax_b / (6*gs)); elements q = RNE_E2M1(w / (s_b*gs)).
    Returns (packed nibbles uint8 [N, K/2] with element 2i in the low nibble,
    scale codes uint8 [N, K/16], gs fp32 scalar tensor).
    """
    N, K = w.shape
    w = w.to(torch.float32)
    amax_t = w.abs().max()
    gs = (amax_t / (6.0 * 448.0)).to(torch.float32)
    if float(gs) == 0.0:
        gs = torch.tensor(1.0, dtype=torch.float32, device=w.device)
    blk = w.view(N, K // 16, 16)
    amax_b = blk.abs().amax(-1)
    sc = _e4m3_codes(amax_b / (6.0 * gs))
    sv = sc.view(torch.float8_e4m3fn).to(torch.float32)
    denom = (sv * gs).unsqueeze(-1)
    safe = torch.where(denom == 0, torch.ones_like(denom), denom)
    q = _e2m1_codes(blk / safe)
    q = torch.where(denom == 0, torch.zeros_like(q), q).view(N, K)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).to(torch.uint8)
    return packed.contiguous(), sc.contiguous(), gs.reshape(())


def _mx_exponent(amax: torch.Tensor) -> torch.Tensor:
    """Smallest integer e with amax <= 448 * 2^e, clamped to [-127, 127];
    amax == 0 gives -127."""
    m, ex = torch.frexp(amax.to(torch.float32))      # amax = m * 2^ex, m in [0.5, 1)
    e = ex.to(torch.int32) - 9 + (m > 0.875).to(torch.int32)
    e = torch.where(amax > 0, e, torch.full_like(e, -127))
    return e.clamp(-127, 127)


def encode_mxfp8(w: torch.Tensor):
    """MXFP8-encode rows of w [N, K]: blocks of 32 along K, E8M0 scale 2^e with
    e the smallest integer such that amax <= 448*2^e, E4M3 elements
    RNE(w / 2^e). Returns (codes uint8 [N, K], scale codes uint8 [N, K/32])."""
    N, K = w.shape
    w = w.to(torch.float32)
    blk = w.view(N, K // 32, 32)
    e = _mx_exponent(blk.abs().amax(-1))
    scaled = blk * torch.pow(2.0, -e.to(torch.float32)).unsqueeze(-1)
    q = _e4m3_codes(scaled).view(N, K)
    return q.contiguous(), (e + 127).to(torch.uint8).contiguous()


def _mx_exponent_fp4(amax: torch.Tensor) -> torch.Tensor:
    """Smallest integer e with amax <= 6 * 2^e, clamped to [-127, 127];
    amax == 0 gives -127."""
    m, ex = torch.frexp(amax.to(torch.float32))      # amax = m * 2^ex, m in [0.5, 1)
    # 6 * 2^e = 0.75 * 2^(e + 3): e = ex - 3 if m <= 0.75, else ex - 2
    e = ex.to(torch.int32) - 3 + (m > 0.75).to(torch.int32)
    e = torch.where(amax > 0, e, torch.full_like(e, -127))
    return e.clamp(-127, 127)


def encode_mxfp4(w: torch.Tensor):
    """MXFP4-encode rows of w [N, K]: blocks of 32 along K, E8M0 scale 2^e
    with e the smallest integer such that amax <= 6 * 2^e, E2M1 elements
    RNE(w / 2^e). Returns (packed nibbles uint8 [N, K/2], element 2i in the
    low nibble, scale codes uint8 [N, K/32])."""
    N, K = w.shape
    w = w.to(torch.float32)
    blk = w.view(N, K // 32, 32)
    e = _mx_exponent_fp4(blk.abs().amax(-1))
    q = _e2m1_codes(blk * torch.pow(2.0, -e.to(torch.float32)).unsqueeze(-1)).view(N, K)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).to(torch.uint8)
    return packed.contiguous(), (e + 127).to(torch.uint8).contiguous()


def gen_one_expert(s: MoEShape, seed: int, e: int, device="cpu", dgrad_copies: bool = False) -> dict:
    """Weights of expert group e, drawn and encoded exactly as in
    gen_expert_weights (per-expert generators, so any expert can be drawn
    alone)."""
    H, I = s.H, s.I
    n1 = I if s.act == "srelu" else 2 * I     # sReLU: a non-gated W1 of I outputs
    w1 = torch.randn(n1, H, generator=_gen((seed + 2) * 65536 + e, device), device=device,
                     dtype=torch.float32) * 0.02
    w2 = torch.randn(H, I, generator=_gen((seed + 3) * 65536 + e, device), device=device,
                     dtype=torch.float32) * 0.02
    out = {}
    if s.wfmt == "nvfp4":
        out["w1_q"], out["w1_s"], out["w1_gs"] = encode_nvfp4(w1)
        out["w2_q"], out["w2_s"], out["w2_gs"] = encode_nvfp4(w2)
    elif s.wfmt == "mxfp4":
        out["w1_q"], out["w1_s"] = encode_mxfp4(w1)
        out["w2_q"], out["w2_s"] = encode_mxfp4(w2)
        out["w1_gs"] = torch.ones((), dtype=torch.float32, device=device)
        out["w2_gs"] = torch.ones((), dtype=torch.float32, device=device)
    elif s.wfmt == "mxfp8":
        w1 = w1.to(torch.bfloat16).to(torch.float32)      # bf16 master weights
        w2 = w2.to(torch.bfloat16).to(torch.float32)
        out["w1_q"], out["w1_s"] = encode_mxfp8(w1)
        out["w2_q"], out["w2_s"] = encode_mxfp8(w2)
        out["w1_gs"] = torch.ones((), dtype=torch.float32, device=device)
        out["w2_gs"] = torch.ones((), dtype=torch.float32, device=device)
        if dgrad_copies:
            out["w1t_q"], out["w1t_s"] = encode_mxfp8(w1.t().contiguous())
            out["w2t_q"], out["w2t_s"] = encode_mxfp8(w2.t().contiguous())
    else:
        raise ValueError(s.wfmt)
    if s.bias:
        # its own generator: the weights' draws do not depend on the bias
        out["b1"] = torch.randn(n1, generator=_gen((seed + 6) * 65536 + e, device), device=device,
                                dtype=torch.float32) * 0.1
    return out


def gen_expert_weights(s: MoEShape, seed: int = 0, device="cpu", dgrad_copies: bool | None = None):
    """Expert weights for every group (routed experts then shared experts).

    W1_e is logically [H, 2I] (gate columns then up columns) and W2_e is
    [I, H]; both are drawn ~N(0, 0.02) and stored transposed, one row per
    output feature with the reduction axis contiguous: W1 as [2I, H], W2 as
    [H, I]. NVFP4: w*_q packed nibbles [N, K/2], w*_s E4M3 scales [N, K/16],
    w*_gs fp32 per (group, matrix). MXFP8 (bf16 master weights): w*_q E4M3
    [N, K], w*_s E8M0 [N, K/32], w*_gs = 1; the dgrad copies w1t_* [H, 2I] and
    w2t_* [I, H] are quantised along the other axis from the same draws.
    With s.bias, b1 [G, 2I] fp32 ~N(0, 0.1) (gate then up).
    """
    G = s.groups
    if dgrad_copies is None:
        dgrad_copies = s.wfmt == "mxfp8"
    out = {}
    for e in range(G):
        one = gen_one_expert(s, seed, e, device, dgrad_copies)
        for name, t in one.items():
            if name not in out:
                out[name] = torch.empty((G,) + tuple(t.shape), dtype=t.dtype, device=device)
            out[name][e] = t
        del one
    return out
