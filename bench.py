"""Benchmark of the routed-MoE layer forward on GB300.

Default workload: DeepSeek-V3-shaped decode (H=7168, I=2048, E=256, top-8,
NVFP4 weights, MXFP8 activations). One step = one layer forward at each of
T = 1, 8, 32 and 128 tokens, every layer on a fresh batch of synthetic tokens
(so routing touches a different set of experts), with the L2 cache flushed
(512 MiB write) before each layer and the flush kept out of the timing.
Each layer call replays a CUDA graph holding one captured moe_layer_forward
(the decode layer is launch-bound without one). The metric is microseconds
per step (lower is better), the sum of the layers' device times; the per-T
layer times are listed in ``config.per_T_us``. The ``e2e`` figure calls the
C ABI directly (no graph) with the tokens copied in from pinned host memory
and the output copied back inside each timed interval.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the same
workload on its own GPU (the layer does not shard across GPUs); the reported
time is the maximum over ranks.
"""
from __future__ import annotations

import os

# the CPU oracle legs run single-threaded so their core count is exact
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import inputs  # noqa: E402

METRIC = "MoE layer us/step (decode T=1-128)"
UNIT = "us/step"
DECODE_TS = (1, 8, 32, 128)
FLUSH_BYTES = 512 << 20


def nvfp4_matrix_bytes(n, k):
    return n * k // 2 + n * k // 16


def w1_bytes_per_expert(s):
    return nvfp4_matrix_bytes(2 * s.I, s.H)


def w2_bytes_per_expert(s):
    return nvfp4_matrix_bytes(s.H, s.I)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_sha():
    """Hash of the GEMM kernel's sources with comments and whitespace
    removed, so a recorded ncu traffic figure stays tied to the code that was
    captured and a comment edit does not void it."""
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "tc.cuh", "common.cuh", "internal.cuh"):
        src = open(os.path.join(ROOT, "quantized_grouped_gemm_topk_gb300", "csrc", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("".join(src.split()).encode())
    return h.hexdigest()[:16]


def traffic_per_launch(kernel_sha):
    """DRAM bytes per W1 launch from the committed ncu summary, if it was taken
    on the kernel source as it is now."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_source_sha") != kernel_sha:
        return None
    return d


def max_over_ranks(value, device):
    """The largest of every rank's value (the job is as slow as its slowest
    replica). Needs an initialised process group when the world has more than
    one rank."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle sample (the cpu_baseline field and the reference arm)
# ---------------------------------------------------------------------------
def oracle_expert_sample(s, x_bits, logits, wts_np, e):
    """Time the oracle's forward of one token through one expert: decode W1/W2
    (NVFP4 -> fp64), both GEMMs, SwiGLU, requantisation. Returns seconds."""
    from oracle import formats as F
    from oracle import moe as M
    t0 = time.perf_counter()
    ids, w = M.topk_route(logits, s.k, s.routed_scale)
    xq, xs = F.mx_quantize(F.bf16_to_f64(x_bits))
    a = F.mx_dequantize(xq, xs)
    W1 = M.expert_w1(wts_np, e, s.wfmt)
    h = a @ W1.T
    y = w[0, 0] * M.act_fwd(h[:, :s.I], h[:, s.I:], s.act, s.alpha, s.limit)
    q, sc = F.mx_quantize(y)
    W2 = M.expert_w2(wts_np, e, s.wfmt)
    z = F.mx_dequantize(q, sc) @ W2.T
    assert np.isfinite(z).all()
    return time.perf_counter() - t0


def cpu_sample_inputs(s, dev):
    """One token of a T=1 batch, its fp32 logits, and its top expert's weights
    on the host (drawn exactly as the GPU run draws that expert)."""
    x = inputs.gen_x(s, 100, device=dev, T=1)
    Wr = inputs.gen_router(s, 0, device=dev)
    logits = (x.float() @ Wr).cpu().numpy().astype(np.float64)
    e = int(np.argmax(logits[0]))
    one = inputs.gen_one_expert(s, 0, e, device=dev)
    wts = {}
    for name, t in one.items():
        t = t.cpu().numpy()
        arr = np.zeros((e + 1,) + t.shape, t.dtype)
        arr[e] = t
        wts[name] = arr
    return inputs.bf16_bits(x).cpu().numpy(), logits, wts, e


def run_reference(args, s, rank, world):
    """Reference arm: the CPU oracle, timed on the host cores, on a bounded
    sample of every step (one token through one expert), scaled to the step's
    (batch, expert) pairs."""
    if rank != 0:
        return
    dev = torch.device("cuda:0") if torch.cuda.is_available() else torch.device("cpu")
    x_bits, logits, wts, e = cpu_sample_inputs(s, dev)
    pairs = float(sum(inputs.expected_touched(s, T) for T in DECODE_TS))
    for _ in range(args.warmup):
        oracle_expert_sample(s, x_bits, logits, wts, e)
    t0 = time.perf_counter()
    per = []
    for _ in range(args.steps):
        per.append(oracle_expert_sample(s, x_bits, logits, wts, e))
    wall = time.perf_counter() - t0
    us_step = statistics.mean(per) * pairs * 1e6
    sample = (f"numpy fp64 oracle, 1 thread: one token through one expert (NVFP4 decode of W1 and W2, both "
              f"GEMMs, SwiGLU, MXFP8 requant) per step, scaled by the expected {pairs:.0f} (batch, expert) "
              f"pairs of a step (T=1,8,32,128)")
    line = {
        "metric": METRIC, "value": us_step, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us_step / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": config_block(s, None),
        "cpu_baseline": {"value": us_step, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": us_step, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }
    print(json.dumps(line), flush=True)


def config_block(s, per_T):
    c = {"workload": f"{s.name}_decode", "H": s.H, "I": s.I, "E": s.E, "k": s.k, "n_shared": s.n_shared,
         "T": list(DECODE_TS), "weights": s.wfmt, "activations": "mxfp8",
         "l2": "flushed by a 512 MiB write before every layer; flush not timed",
         "inputs": "fresh seeded batch per layer call; weights resident in HBM", "parallelism": "replica per GPU",
         "launch": "each layer call is a CUDA graph of one moe_layer_forward; e2e calls the C ABI directly"}
    if per_T is not None:
        c["per_T_us"] = per_T
    return c


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, s, rank, world, local):
    import quantized_grouped_gemm_topk_gb300 as m
    try:
        m.binding.load()
    except RuntimeError:
        from quantized_grouped_gemm_topk_gb300 import build as b
        b.build()
        m.binding.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    Tmax = max(DECODE_TS)
    cfg = m.config_from_shape(s, T_max=Tmax)
    wts = inputs.gen_expert_weights(s, 0, device=dev)
    packed = m.moe_prepack_weights(cfg, wts)
    torch.cuda.synchronize()
    del wts
    torch.cuda.empty_cache()
    ws = torch.zeros(m.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    Wr = inputs.gen_router(s, 0, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    nx = 16
    xs = {T: [inputs.gen_x(s, 100 + 1000 * T + i + 7919 * rank, device=dev, T=T) for i in range(nx)]
          for T in DECODE_TS}
    outs = {T: torch.empty(T, s.H, dtype=torch.bfloat16, device=dev) for T in DECODE_TS}
    # routing is deterministic: learn each batch's touched-expert count once
    touched = {}
    for T in DECODE_TS:
        for i in range(nx):
            m.moe_layer_forward(cfg, xs[T][i], Wr, None, T, packed, outs[T], None, ws)
            v = m.ws_tensor_views(cfg, ws, T)
            touched[(T, i)] = int((v["counts"] > 0).sum())
    torch.cuda.synchronize()
    assert m.moe_read_status(cfg, ws) == 0

    def layer_bytes(T, i):
        n = touched[(T, i)]
        R = T * s.kp
        return n * w1_bytes_per_expert(s), R * (s.H + s.H // 32) + R * (s.I + s.I // 32)

    # One CUDA graph per (T, batch): the whole layer forward captured once,
    # with its phase events as event-record nodes, replayed in the timed loop.
    graphs, gev, glaunch = {}, {}, {}
    for T in DECODE_TS:
        for i in range(nx):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(m.MOE_N_PHASE_EVENTS)]
            for e in evs:
                e.record()      # creates the event's handle
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            m.moe_set_phase_events(evs)
            with torch.cuda.graph(g):
                m.moe_layer_forward(cfg, xs[T][i], Wr, None, T, packed, outs[T], None, ws)
                glaunch[(T, i)] = m.moe_last_launch_count()
            m.moe_set_phase_events(None)
            graphs[(T, i)], gev[(T, i)] = g, evs
    torch.cuda.synchronize()

    # warm-up
    for w in range(args.warmup):
        for T in DECODE_TS:
            flush.zero_()
            graphs[(T, w % nx)].replay()
    torch.cuda.synchronize()
    assert m.moe_read_status(cfg, ws) == 0

    K = args.steps
    launches = 0
    layer_us = []
    w1_us, w1_bytes, w2_us = 0.0, 0, 0.0
    per_T = {T: [] for T in DECODE_TS}
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    with ClockSampler(local) as clk:
        for step in range(K):
            i = step % nx
            for T in DECODE_TS:
                flush.zero_()
                graphs[(T, i)].replay()
                launches += glaunch[(T, i)]
            # the graphs of this step are replayed again nx steps later: read
            # their events now (host-side wait, outside every device interval)
            torch.cuda.synchronize()
            for T in DECODE_TS:
                e = gev[(T, i)]
                t = e[0].elapsed_time(e[5]) * 1e3
                layer_us.append(t)
                per_T[T].append(t)
                w1_us += e[1].elapsed_time(e[2]) * 1e3
                w2_us += e[3].elapsed_time(e[4]) * 1e3
                wb, ab = layer_bytes(T, i)
                w1_bytes += wb + ab
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall_ms = (time.perf_counter() - t_wall) * 1e3 / K
    assert m.moe_read_status(cfg, ws) == 0
    us_step = sum(layer_us) / K
    if world > 1:
        us_step = max_over_ranks(us_step, dev)

    # end to end through the public API with host buffers
    host_x = {T: [xs[T][i].cpu().pin_memory() for i in range(nx)] for T in DECODE_TS}
    host_out = {T: torch.empty(T, s.H, dtype=torch.bfloat16).pin_memory() for T in DECODE_TS}
    dev_x = {T: torch.empty(T, s.H, dtype=torch.bfloat16, device=dev) for T in DECODE_TS}
    ncall = K * len(DECODE_TS)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ncall)]
    torch.cuda.synchronize()
    c = 0
    for step in range(K):
        for T in DECODE_TS:
            flush.zero_()
            a, b = e2e_ev[c]
            a.record()
            dev_x[T].copy_(host_x[T][step % nx], non_blocking=True)
            m.moe_layer_forward(cfg, dev_x[T], Wr, None, T, packed, outs[T], None, ws)
            host_out[T].copy_(outs[T], non_blocking=True)
            b.record()
            c += 1
    torch.cuda.synchronize()
    e2e_us = sum(a.elapsed_time(b) * 1e3 for a, b in e2e_ev) / K
    h2d = sum(T * s.H * 2 for T in DECODE_TS)

    peak, peak_kind = peaks()
    achieved = w1_bytes / (w1_us * 1e-6) / 1e9
    sha = kernel_source_sha()
    tr = traffic_per_launch(sha)
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": None, "kernel": "W1 grouped GEMM (k_gemm_tc)", "peak_source": f"{peak_kind} hbm_gbs",
            "algorithmic_bytes": "touched experts x NVFP4 W1 bytes (2I*H/2 + 2I*H/16) + MXFP8 rows in and out",
            "kernel_us_per_step": w1_us / K, "w2_gemm_us_per_step": w2_us / K}
    if tr is not None:
        # DRAM bytes of one captured W1 launch over its algorithmic bytes,
        # applied to this run's average algorithmic bytes per W1 launch
        roof["traffic"] = tr["dram_over_algorithmic"] * w1_bytes / (K * len(DECODE_TS))
        roof["traffic_note"] = (f"ncu dram__bytes_read+write of one W1 launch ({tr['captured']}) = "
                                f"{tr['dram_over_algorithmic']:.4f} x its algorithmic bytes, scaled to this "
                                f"run's average W1 launch")
    per_T_us = {str(T): statistics.median(v) for T, v in per_T.items()}
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": us_step, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": us_step / 1e3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 x e2m1, f32 accumulate", "data": "synthetic", "config": config_block(s, per_T_us),
        "roofline": roof,
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": h2d},
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_ms_per_step": wall_ms,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        x_bits, logits, wts_np, e = cpu_sample_inputs(s, dev)
        reps = [oracle_expert_sample(s, x_bits, logits, wts_np, e) for _ in range(3)]
        pairs = float(sum(touched[(T, 0)] for T in DECODE_TS))
        line["cpu_baseline"] = {
            "value": statistics.median(reps) * pairs * 1e6, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"numpy fp64 oracle, 1 thread: one token through one expert (W1/W2 NVFP4 decode, GEMMs, "
                      f"SwiGLU, MXFP8 requant), median of 3, scaled by the {pairs:.0f} touched experts of "
                      f"step 0 (T=1,8,32,128)"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dsv3", choices=["dsv3", "shared"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--E", type=int, default=0, help="override the expert count (small profiling cases)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    s = inputs.workload(args.workload)
    if args.E:
        s = inputs.workload(args.workload, E=args.E)
    if args.impl == "reference":
        run_reference(args, s, rank, world)
        return
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, s, rank, world, local)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
