"""Benchmark of the sparse 4-bit MoE block on GB300.

Default workload (one JSON line on rank 0): the Qwen-shaped 40-layer batch-1
decode chain (d=2048, E=256, top-8, I=512, one sigmoid-gated shared expert,
4-bit group-64 weights, RMS normalisation between layers).  One step = one
token through all 40 layers (one kernel launch).  The same line carries the
single-layer prefill case (T=4096 tokens, Zipf-skewed routing) under
"prefill".  ``--workload prefill`` makes the prefill case the headline.

Synthetic seeded inputs (synth/), random-init weights of that architecture.
``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload (host cores).  Under torchrun every rank runs an independent
replica (the path shards into independent batches; no collective on the data
path); value = units of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# workload constants
D, E, K, I = 2048, 256, 8, 512
DECODE_LAYERS = 40
PREFILL_T = 4096
EXPERT_BYTES = 1769472          # 4.5-bit gate/up + down of one expert (codes + fp16 s, beta)
ROUTER_BYTES = E * D * 2
LAYER_BYTES_DECODE = 9 * EXPERT_BYTES + ROUTER_BYTES + D * 2 + 2 * D * 2   # 16,986,112
FLOP_PER_TOKEN = 2 * D * E + K * (2 * D * 2 * I + 2 * I * D) + (2 * D * 2 * I + 2 * I * D) + 2 * D
GATEUP_FLOP_PER_ROW = 2 * D * 2 * I
METRIC = "MoE-layer tokens/s (prefill T=4096; decode T=1) and % of HBM/tensor roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def profiled_traffic(kernel: str):
    """DRAM bytes of `kernel` from profiles/traffic.txt, if the kernel's source
    still has the hash recorded there (else None: the counters are stale)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        kv = dict(tok.split("=", 1) for tok in line.split())
        if kv.get("kernel") != kernel:
            continue
        src = os.path.join(ROOT, kv["source"])
        if not os.path.exists(src):
            return None
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
        return kv if h.startswith(kv["sha256"]) else None
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ ranks
def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend):
    import torch.distributed as dist
    ws, rank, _ = dist_info()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return ws, rank


def max_over_ranks(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and str(device).startswith("cuda"):
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ GPU arm
def l2_flush_buffer(torch, device):
    return torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)


def build_decode(torch, M, sd, gen, device, n_layers=DECODE_LAYERS):
    shape = gen.MoEShape(d=D, E=E, k=K, I=I)
    layers = []
    for l in range(n_layers):
        w = sd.make_layer(0, l, shape, device=device)
        layers.append(M.MoE(M.MoEConfig(d=D, E=E, k=K, I=I, max_tokens=1,
                                        layouts=M.MOE_LAYOUT_DECODE), w))
        del w
    torch.cuda.empty_cache()
    return layers


def decode_traffic(n_layers):
    kv = profiled_traffic("decode_kernel")
    return int(kv["bytes_per_layer"]) * n_layers if kv else None


def gateup_traffic():
    kv = profiled_traffic("grouped_mma_gateup")
    return int(kv["bytes_per_launch"]) if kv else None


def run_decode(args, torch, M, sd, gen, device, peaks):
    layers = build_decode(torch, M, sd, gen, device, args.decode_layers)
    nx = max(args.steps + args.warmup, 8)
    xs = sd.make_x(1, nx, D, device=device)  # a different token every step
    y = torch.empty(D, dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream(device)
    for i in range(args.warmup):
        M.decode(layers, xs[i % nx])
    torch.cuda.synchronize(device)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clk = ClockSampler(device.index)
    clk.start()
    barrier(device)
    torch.cuda.synchronize(device)
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    t_all0.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        M.decode(layers, xs[(args.warmup + i) % nx])
        ends[i].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize(device)
    barrier(device)
    clocks = clk.stop()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_step = t_all0.elapsed_time(t_all1) / args.steps
    ms_step = max_over_ranks(ms_step, device)
    kernel_ms = statistics.mean(per)
    bytes_launch = LAYER_BYTES_DECODE * args.decode_layers
    achieved = bytes_launch / (kernel_ms * 1e-3) / 1e9
    # end to end through the C ABI with host buffers
    xh = xs[:args.steps].cpu().pin_memory()
    yh = torch.empty(D, dtype=torch.bfloat16).pin_memory()
    for i in range(min(3, args.steps)):
        M.decode_host(layers, xh[i], yh)
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for i in range(args.steps):
        M.decode_host(layers, xh[i], yh)
    e2e_s = (time.perf_counter() - t0) / args.steps
    e2e_s = max_over_ranks(e2e_s, device)
    # where a layer's time goes (GPU clock stamps of the first CTA, one traced token)
    _, tr = M.decode(layers, xs[0], trace=True)
    torch.cuda.synchronize(device)
    ts = tr["timestamps"].cpu().numpy().astype("float64") / 1000.0
    phases = {
        "logits_topk_issue": float((ts[:, 1] - ts[:, 0]).mean()),
        "stream_gate_up_down_partials": float((ts[:, 2] - ts[:, 1]).mean()),
        "exchange_and_sum_partials": float((ts[:, 3] - ts[:, 2]).mean()),
        "router_sums_and_next_inputs": float((ts[1:, 0] - ts[:-1, 3]).mean()),
    }
    err = layers[0].device_error()
    return dict(
        ms_per_step=ms_step, value=args.world * 1000.0 / ms_step, unit="tokens/s",
        us_per_layer=ms_step * 1000.0 / args.decode_layers, phase_us=phases,
        roofline={"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                  "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                  "traffic": decode_traffic(args.decode_layers), "kernel": "decode_kernel",
                  "algorithmic_bytes_per_launch": bytes_launch},
        e2e={"value": args.world / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": D * 2,
             "d2h_bytes_per_step": D * 2},
        gpu_launches=args.steps, clocks=clocks, device_error=err)


def run_prefill(args, torch, M, sd, gen, device, peaks):
    shape = gen.MoEShape(d=D, E=E, k=K, I=I)
    w = sd.make_layer(0, 0, shape, device=device)
    layer = M.MoE(M.MoEConfig(d=D, E=E, k=K, I=I, max_tokens=PREFILL_T,
                              layouts=M.MOE_LAYOUT_PREFILL), w)
    del w
    torch.cuda.empty_cache()
    x = sd.make_x(0, PREFILL_T, D, device=device)
    bias = torch.from_numpy(gen.zipf_bias(0, E)).to(device)
    y = torch.empty_like(x)
    flush = l2_flush_buffer(torch, device)
    stream = torch.cuda.current_stream(device)
    # the timed steps replay a CUDA graph of one forward (the library's calls
    # are asynchronous and allocate nothing, so the whole block captures)
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        layer.forward(x, bias, out=y)
    torch.cuda.current_stream(device).wait_stream(side)
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(x, bias, out=y)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(device)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clk = ClockSampler(device.index)
    clk.start()
    barrier(device)
    torch.cuda.synchronize(device)
    for i in range(args.steps):
        flush.zero_()  # L2 flush between timed steps (outside the events)
        starts[i].record(stream)
        graph.replay()
        ends[i].record(stream)
    torch.cuda.synchronize(device)
    barrier(device)
    clocks = clk.stop()
    ms_step = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    ms_step = max_over_ranks(ms_step, device)
    # stage times (and the dominant kernel's duration for the roofline): the
    # same steps launched directly with CUDA events between the stages
    layer.profile(True)
    for i in range(args.steps):
        flush.zero_()
        layer.forward(x, bias, out=y)
    torch.cuda.synchronize(device)
    stages, calls = layer.profile_read()
    layer.profile(False)
    r = layer.route(x, bias)
    counts = r["counts"].cpu()
    rows = PREFILL_T * K + PREFILL_T
    gu_ms = stages["gate_up"] / max(calls, 1)
    gu_tflops = rows * GATEUP_FLOP_PER_ROW / (gu_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    total_flop = FLOP_PER_TOKEN * PREFILL_T
    # end to end through the C ABI with host buffers
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    bh = bias.cpu().pin_memory()
    layer.forward_host(xh, bh, yh)
    t0 = time.perf_counter()
    n_e2e = max(3, min(args.steps, 20))
    for _ in range(n_e2e):
        layer.forward_host(xh, bh, yh)
    e2e_s = (time.perf_counter() - t0) / n_e2e
    e2e_s = max_over_ranks(e2e_s, device)
    err = layer.device_error()
    return dict(
        ms_per_step=ms_step, value=args.world * PREFILL_T * 1000.0 / ms_step, unit="tokens/s",
        us_per_layer=ms_step * 1000.0,
        stage_ms={k: round(v / max(calls, 1), 4) for k, v in stages.items()},
        roofline={"bound": "tensor", "achieved": round(gu_tflops, 1), "peak": peak,
                  "unit": "TFLOP/s", "frac": round(gu_tflops / peak, 4),
                  "traffic": gateup_traffic(),
                  "kernel": "grouped_mma_kernel<gate/up>",
                  "algorithmic_flop_per_launch": rows * GATEUP_FLOP_PER_ROW},
        step_roofline_frac=round((total_flop / (peak * 1e12)) / (ms_step * 1e-3), 4),
        experts_touched=int((counts > 0).sum()), max_expert_rows=int(counts.max()),
        e2e={"value": args.world * PREFILL_T / e2e_s, "unit": "tokens/s",
             "h2d_bytes_per_step": PREFILL_T * D * 2 + E * 4,
             "d2h_bytes_per_step": PREFILL_T * D * 2},
        gpu_launches=5 * args.steps, clocks=clocks, device_error=err)


SWEEP_T = [256, 512, 1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072]
SWEEP_CHUNK = 8192


# Gated DeltaNet prefill scan: one 2K-token prompt through a Qwen-shaped
# linear-attention layer (16 query/key heads, 32 value heads, 128 x 128 fp32
# state per value head).
GDN_T = 2048
GDN_SHAPE = dict(Hk=16, Hv=32, dk=128, dv=128)
SM_MAX_MHZ = 2070.0
FP32_LANES_PER_SM = 128


def gdn_alu_ops(T, Hv, dv, dk):
    """fp32 pipe operations the scan needs at least: per state element and
    token, one multiply-add each for S.k and S.q and two operations for the
    update alpha S + c k."""
    return 4 * T * Hv * dv * dk


def gdn_bytes(T, Hk, Hv, dk, dv):
    """Bytes one scan must move: q, k, v in and o out (bf16), g and beta
    (fp32), the final state out (fp32)."""
    return 2 * T * Hk * dk * 2 + T * Hv * dv * 2 * 2 + T * Hv * 4 * 2 + Hv * dv * dk * 4


def gdn_alu_peak(sm_count):
    """fp32 lane operations per second at the maximum SM clock (T ops/s)."""
    return sm_count * FP32_LANES_PER_SM * SM_MAX_MHZ * 1e6 / 1e12


def run_gdn(args, torch, M, device):
    import numpy as np
    from synth import gdn
    shape = gdn.GdnShape(**GDN_SHAPE)
    inp = gdn.make_inputs(0, [GDN_T], shape)

    def bf16(bits):
        return torch.from_numpy(bits.view(np.int16)).to(device).view(torch.bfloat16)

    q, k, v = bf16(inp.q), bf16(inp.k), bf16(inp.v)
    g = torch.from_numpy(inp.g).to(device)
    beta = torch.from_numpy(inp.beta).to(device)
    o = torch.empty(GDN_T, shape.Hv, shape.dv, dtype=torch.bfloat16, device=device)
    S = torch.empty(1, shape.Hv, shape.dv, shape.dk, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def fn():
        M.gdn_scan(q, k, v, g, beta, o=o, state_out=S, stream=stream)

    flush = l2_flush_buffer(torch, device)
    for _ in range(max(3, args.warmup)):
        fn()
    torch.cuda.synchronize()
    clk = ClockSampler(device.index)
    clk.start()
    us = time_call(torch, fn, flush, max(10, args.steps), stream)
    clocks = clk.stop()
    sm_count = torch.cuda.get_device_properties(device).multi_processor_count
    ops = gdn_alu_ops(GDN_T, shape.Hv, shape.dv, shape.dk)
    achieved = ops / (us * 1e-6) / 1e12
    peak = gdn_alu_peak(sm_count)
    kv = profiled_traffic("gdn_chunk_kernel")
    cpu = None
    if getattr(args, "world", 1) == 1:   # the fp64 oracle on the host, a bounded sample
        try:
            from oracle import gdn_oracle as G
            n = 256
            t_start = time.perf_counter()
            G.gdn_scan(inp.q[:n], inp.k[:n], inp.v[:n], inp.g[:n], inp.beta[:n])
            cpu = {"value": n / (time.perf_counter() - t_start), "unit": "tokens/s", "cores": 1,
                   "kind": "oracle",
                   "sample": f"fp64 oracle, the first {n} tokens of the same prompt, all "
                             f"{shape.Hv} value heads (numpy, one thread)"}
        except Exception as ex:  # informative only; never fail the bench on it
            cpu = {"error": str(ex)}
    return {
        "config": f"one {GDN_T}-token prompt, Hk={shape.Hk} query/key heads, Hv={shape.Hv} "
                  f"value heads, dk=dv={shape.dk}; q, k unit-norm bf16, v bf16, alpha in "
                  "[0.9, 1), beta = sigmoid(N(0,1)); L2 flushed between calls, median",
        "us": us, "tokens_per_s": GDN_T / (us * 1e-6),
        "roofline": {"bound": "alu", "achieved": round(achieved, 3), "peak": round(peak, 3),
                     "unit": "T fp32 lane-ops/s", "frac": round(achieved / peak, 4),
                     "traffic": int(kv["bytes_per_launch"]) if kv else None,
                     "kernel": "gdn_chunk_kernel",
                     "algorithmic_ops_per_launch": ops,
                     "note": "achieved counts the token-by-token rule's 4 fp32 operations per "
                             "state element and token; the kernel evaluates the rule in chunks "
                             "of 32 tokens with its products on the tensor cores",
                     "peak_source": f"{sm_count} SMs x {FP32_LANES_PER_SM} fp32 lanes x "
                                    f"{SM_MAX_MHZ:.0f} MHz"},
        "algorithmic_bytes_per_launch": gdn_bytes(GDN_T, shape.Hk, shape.Hv, shape.dk,
                                                  shape.dv),
        "gpu_launches": 1, "clocks": clocks, "cpu_baseline": cpu,
    }


def point_roofline(T, experts_touched, chunks, peaks):
    """max(FLOP at peak, bytes at HBM bandwidth) for one call: the touched
    experts' 4.5-bit weights (counted per chunk), the router per chunk, x in
    and y out (bf16)."""
    flop = FLOP_PER_TOKEN * T
    nbytes = experts_touched * EXPERT_BYTES + chunks * ROUTER_BYTES + 4 * D * T
    t_flop = flop / (peaks["bf16_tflops"] * 1e12)
    t_bytes = nbytes / (peaks["hbm_gbs"] * 1e9)
    return max(t_flop, t_bytes), ("tensor" if t_flop >= t_bytes else "hbm")


def time_call(torch, fn, flush, reps, stream):
    ts = []
    for _ in range(reps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ts) * 1000.0  # us


def run_sweep(args, torch, M, sd, gen, device, peaks):
    """The prefill length sweep (uniform and Zipf routing, chunks of 8192
    tokens above that) and the T=32768 extreme-imbalance case (one
    unchunked call).  Per point: us per call, tokens/s and the fraction of
    that call's roofline."""
    shape = gen.MoEShape(d=D, E=E, k=K, I=I)
    w = sd.make_layer(0, 0, shape, device=device)
    layer = M.MoE(M.MoEConfig(d=D, E=E, k=K, I=I, max_tokens=SWEEP_CHUNK,
                              layouts=M.MOE_LAYOUT_PREFILL), w)
    stress = M.MoE(M.MoEConfig(d=D, E=E, k=K, I=I, max_tokens=32768,
                               layouts=M.MOE_LAYOUT_PREFILL), w)
    del w
    torch.cuda.empty_cache()
    x = sd.make_x(0, max(SWEEP_T), D, device=device)
    out = torch.empty_like(x)
    flush = l2_flush_buffer(torch, device)
    stream = torch.cuda.current_stream(device)
    zipf = torch.from_numpy(gen.zipf_bias(0, E)).to(device)

    def touched(lay, xs, bias, chunk):
        n = 0
        for t0 in range(0, xs.shape[0], chunk):
            r = lay.route(xs[t0:t0 + chunk], bias)
            n += int((r["counts"] > 0).sum().item()) + 1  # + the shared expert
        return n

    points = []
    for routing, bias in (("uniform", None), ("zipf", zipf)):
        for T in SWEEP_T:
            xs, ys = x[:T], out[:T]
            for _ in range(2):
                layer.forward(xs, bias, out=ys)
            us = time_call(torch, lambda: layer.forward(xs, bias, out=ys), flush,
                           3 if T >= 32768 else 5, stream)
            chunks = (T + SWEEP_CHUNK - 1) // SWEEP_CHUNK
            t_roof, bound = point_roofline(T, touched(layer, xs, bias, SWEEP_CHUNK), chunks, peaks)
            points.append({"routing": routing, "T": T, "us": round(us, 1),
                           "tokens_per_s": round(T / (us * 1e-6), 1), "bound": bound,
                           "roofline_frac": round(t_roof / (us * 1e-6), 4)})
    # extreme imbalance: the 8 top-ranked experts share one bias, set by
    # bisection on this layer's own logits of a 2048-token sample so that they
    # take half of the assignments; the 64 bottom-ranked experts get -1e4
    T = 32768
    rank = torch.from_numpy(gen.expert_ranking(0, E)).to(device)
    hot, cold = rank <= 8, rank > E - 64
    lg = layer.route(x[:2048])["logits"]
    lo, hi = -10.0, 20.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        b = torch.where(hot, torch.tensor(mid, device=device),
                        torch.where(cold, torch.tensor(-1e4, device=device),
                                    torch.tensor(0.0, device=device)))
        share = hot[torch.topk(lg + b, K, dim=1).indices].float().mean().item()
        lo, hi = (mid, hi) if share < 0.5 else (lo, mid)
    bias = torch.where(hot, torch.tensor(0.5 * (lo + hi), device=device),
                       torch.where(cold, torch.tensor(-1e4, device=device),
                                   torch.tensor(0.0, device=device))).float()
    xs, ys = x[:T], out[:T]
    for _ in range(2):
        stress.forward(xs, bias, out=ys)
    us = time_call(torch, lambda: stress.forward(xs, bias, out=ys), flush, 3, stream)
    counts = stress.route(xs, bias)["counts"]
    t_roof, bound = point_roofline(T, int((counts > 0).sum().item()) + 1, 1, peaks)
    hot_share = float(counts[hot].sum().item()) / (T * K)
    stress_pt = {"T": T, "us": round(us, 1), "tokens_per_s": round(T / (us * 1e-6), 1),
                 "bound": bound, "roofline_frac": round(t_roof / (us * 1e-6), 4),
                 "hot_share": round(hot_share, 3),
                 "empty_experts": int((counts == 0).sum().item())}
    layer.close()
    stress.close()
    # a few tokens (speculative-verify shape): a handle with both layouts runs
    # T = 1 on the decode kernel, 2 <= T <= 8 on the few-token kernel (one
    # launch streaming the union of the tokens' experts once), larger T on the
    # tensor-core path
    small = M.MoE(M.MoEConfig(d=D, E=E, k=K, I=I, max_tokens=64), sd.make_layer(0, 0, shape, device=device))
    torch.cuda.empty_cache()
    small_pts = []
    for T in (1, 2, 3, 4, 5, 6, 8, 12, 16):
        xs, ys = x[:T], out[:T]
        for _ in range(2):
            small.forward(xs, None, out=ys)
        us = time_call(torch, lambda: small.forward(xs, None, out=ys), flush, 10, stream)
        t_roof, bound = point_roofline(T, touched(small, xs, None, 64), 1, peaks)
        small_pts.append({"T": T, "us": round(us, 1), "tokens_per_s": round(T / (us * 1e-6), 1),
                          "path": ("decode kernel" if T == 1 else
                                   "few-token kernel" if T <= 8 else "tensor-core"),
                          "bound": bound, "roofline_frac": round(t_roof / (us * 1e-6), 4)})
    small.close()
    return points, stress_pt, small_pts


# ------------------------------------------------------------------ oracle arm
def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info()]
        return max(n) if n else os.cpu_count()
    except Exception:
        return os.cpu_count()


class OracleSample:
    """A bounded sample of the workload for the fp64 oracle on host cores.
    Weights are generated once (outside timing); run() times oracle work only.
      decode : the whole 40-layer chain for one token (router, top-k,
               dequantisation of the 9 experts of every layer, experts,
               combine, RMS normalisation): one step is one full token
      prefill: `n_tok` tokens of the T=4096 Zipf layer (router, top-k,
               dequantisation of every touched expert, experts, combine)."""

    def __init__(self, workload, n_layers=DECODE_LAYERS, n_tok=256):
        import numpy as np
        from oracle import moe_oracle as O
        from synth import gen
        self.O, self.workload = O, workload
        shape = gen.MoEShape(d=D, E=E, k=K, I=I)
        if workload == "decode":
            from concurrent.futures import ThreadPoolExecutor
            self.layers = []
            x = O.bf16_values(gen.make_x(1, 1, D))
            self.x0 = x
            with ThreadPoolExecutor(max_workers=16) as pool:
                for l in range(n_layers):
                    wr = O.bf16_values(gen.bf16_matrix(0, gen.TAG_ROUTER, l, 0, E, D, 0.02))
                    wsg = O.bf16_values(
                        gen.bf16_matrix(0, gen.TAG_SHARED_GATE, l, 0, 1, D, 0.02)[0])
                    idx, _ = O.select_top_k(O.router_logits(x, wr), K)
                    need = [int(e) for e in idx[0]] + [E]
                    ws = pool.map(lambda e, l=l: gen.expert_weights(0, l, e, shape), need)
                    cache = dict(zip(need, ws))
                    vals = dict(E=E, k=K, group=64, has_shared=True, w_router=wr,
                                w_shared_gate=wsg, experts=None, shared=None)
                    self.layers.append((vals, cache))
                    x = O.rms_norm(O.moe_layer(x, vals, expert_source=lambda e: cache[e])["out"])
            self.units = 1
            self.sample = (f"fp64 oracle, the whole {n_layers}-layer decode chain for one token "
                           f"per step")
        else:
            self.x = O.bf16_values(gen.make_x(0, n_tok, D))
            wr = O.bf16_values(gen.bf16_matrix(0, gen.TAG_ROUTER, 0, 0, E, D, 0.02))
            wsg = O.bf16_values(gen.bf16_matrix(0, gen.TAG_SHARED_GATE, 0, 0, 1, D, 0.02)[0])
            self.bias = gen.zipf_bias(0, E)
            idx, _ = O.select_top_k(O.router_logits(self.x, wr, self.bias), K)
            self.cache = {int(e): gen.expert_weights(0, 0, int(e), shape) for e in np.unique(idx)}
            self.cache[E] = gen.expert_weights(0, 0, E, shape)
            self.vals = dict(E=E, k=K, group=64, has_shared=True, w_router=wr,
                             w_shared_gate=wsg, experts=None, shared=None)
            self.units = n_tok
            self.sample = (f"fp64 oracle, {n_tok} tokens of the T=4096 Zipf prefill layer "
                           f"(dequantisation of the {len(self.cache)} touched experts included)")

    def run(self) -> float:
        """One timed step; returns tokens/s."""
        O = self.O
        t0 = time.perf_counter()
        if self.workload == "decode":
            x = self.x0
            for vals, cache in self.layers:
                x = O.rms_norm(O.moe_layer(x, vals, expert_source=lambda e: cache[e])["out"])
            return self.units / (time.perf_counter() - t0)
        O.moe_layer(self.x, self.vals, logit_bias=self.bias, expert_source=lambda e: self.cache[e])
        return self.units / (time.perf_counter() - t0)


_ONE_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                   "BLIS_NUM_THREADS", "VECLIB_MAXIMUM_THREADS")


def single_thread_rate(workload, steps):
    """The same oracle sample in a child process whose BLAS runs one thread
    (the thread count is fixed when numpy loads, hence the process)."""
    env = dict(os.environ, **{k: "1" for k in _ONE_THREAD_ENV})
    code = ("import sys, json, statistics; sys.path.insert(0, %r); import bench; "
            "s = bench.OracleSample(%r); s.run(); "
            "print(json.dumps(statistics.median([s.run() for _ in range(%d)])))"
            % (ROOT, workload, max(1, steps)))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True,
                           text=True, timeout=900)
        v = float(r.stdout.strip().splitlines()[-1])
    except Exception as ex:  # informative only
        return {"error": str(ex)[:200]}
    return {"value": v, "unit": "tokens/s", "cores": 1}


def cpu_baseline(workload, steps=1):
    s = OracleSample(workload)
    v = statistics.median([s.run() for _ in range(max(1, steps))])
    return {"value": v, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
            "sample": s.sample, "single_thread": single_thread_rate(workload, steps)}


# ------------------------------------------------------------------ main
def config_for(workload):
    if workload == "decode":
        return {"workload": "qwen-shaped MoE decode chain: 40 layers, T=1, d=2048, E=256, "
                            "top-8, I=512 + shared expert, 4-bit g64",
                "layers": DECODE_LAYERS, "tokens_per_step": 1,
                "l2": "inputs larger than L2 (679 MB of weights read per step, a new token each step)"}
    return {"workload": "qwen-shaped MoE prefill layer: T=4096, Zipf-skewed routing "
                        "(b_e = 1.5 ln(1/rank_e)), d=2048, E=256, top-8, I=512 + shared, 4-bit g64",
            "tokens_per_step": PREFILL_T, "l2": "flushed between timed steps (256 MB write)",
            "launch": "one CUDA graph of the layer per step (5 kernels)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=["decode", "prefill"])
    ap.add_argument("--no-secondary", action="store_true", help="skip the second workload")
    ap.add_argument("--decode-layers", type=int, default=DECODE_LAYERS,
                    help="layers of the decode chain (profiling captures use fewer)")
    ap.add_argument("--no-gdn", action="store_true",
                    help="skip the Gated DeltaNet prefill scan (one 2K prompt)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the prefill length sweep and the imbalance case")
    args = ap.parse_args()
    ws, rank, local = dist_info()
    args.world = ws

    if args.impl == "reference":
        if rank != 0:
            return 0
        sample = OracleSample(args.workload)
        for _ in range(args.warmup):
            sample.run()
        t0 = time.perf_counter()
        rates = [sample.run() for _ in range(args.steps)]
        ms_step = 1000.0 * (time.perf_counter() - t0) / args.steps  # measured, not scaled
        v = statistics.median(rates)
        cb = {"value": v, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
              "sample": sample.sample,
              "single_thread": single_thread_rate(args.workload, min(2, args.steps))}
        line = {"impl": "reference", "metric": METRIC, "value": v,
                "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic",
                "config": config_for(args.workload),
                "cpu_baseline": cb,
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch
    import sparse_moe_bit_gb300 as M
    from synth import device as sd
    from synth import gen
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist("nccl")
    peaks, peak_src = load_peaks()
    primary = args.workload
    secondary = None if args.no_secondary else ("prefill" if primary == "decode" else "decode")
    runner = {"decode": run_decode, "prefill": run_prefill}
    res = runner[primary](args, torch, M, sd, gen, device, peaks)
    sec = runner[secondary](args, torch, M, sd, gen, device, peaks) if secondary else None
    sweep = None if args.no_sweep else run_sweep(args, torch, M, sd, gen, device, peaks)
    gdn_res = None if args.no_gdn else run_gdn(args, torch, M, device)

    if rank != 0:
        return 0
    line = {
        "metric": METRIC,
        "value": res["value"], "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
        "us_per_layer": res["us_per_layer"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("decode: int16 activations (a power-of-two scale per 64-group) x 4-bit codes, "
                  "exact int32 dot products (dp2a), fp32 scale/bias and sums; prefill: fp16 "
                  "tensor-core operands (per-token power-of-two scaled), fp32 accumulate"),
        "data": "synthetic (seeded counter-based generator; random-init weights)",
        "config": dict(config_for(primary), parallelism=f"replicas x{ws}"),
        "roofline": dict(res["roofline"], peak_source=peak_src),
        "e2e": res["e2e"], "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
        "device_error": res["device_error"],
    }
    for key in ("stage_ms", "phase_us", "step_roofline_frac", "experts_touched",
                "max_expert_rows"):
        if key in res:
            line[key] = res[key]
    if sec is not None:
        line[secondary] = {k: sec[k] for k in ("value", "unit", "ms_per_step", "us_per_layer",
                                               "roofline", "e2e", "gpu_launches")
                           if k in sec}
        for key in ("stage_ms", "phase_us", "step_roofline_frac", "experts_touched",
                    "max_expert_rows"):
            if key in sec:
                line[secondary][key] = sec[key]
    if sweep is not None:
        line["prefill_sweep"] = {
            "config": "same layer as the prefill line; T in 256..128K, uniform and Zipf "
                      "routing, chunks of 8192 tokens above that; one call per point, "
                      "L2 flushed between calls, median of 3-5",
            "points": sweep[0]}
        line["imbalance_T32768"] = dict(
            sweep[1], config="8 hot experts take half of the assignments, 64 experts get "
                             "none; one unchunked call")
        line["small_T"] = {
            "config": "same layer, uniform routing, a handle with both layouts: T = 1 on the "
                      "decode kernel, 2..8 on the few-token kernel (the union of the tokens' "
                      "experts streamed once), more on the tensor-core path; roofline from the "
                      "bytes of the experts touched; L2 flushed, median of 10",
            "points": sweep[2]}
    if gdn_res is not None:
        line["gdn_scan"] = gdn_res
    if ws == 1:
        try:
            line["cpu_baseline"] = cpu_baseline(primary)
        except Exception as ex:  # the baseline is informative; never fail the bench on it
            line["cpu_baseline"] = {"error": str(ex)}
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
