"""Benchmark of the routed NVFP4 MoE decode layer-step on GB300.

Default workload: one layer at serving width -- b = 8 rows (one request
verifying 1 + 7 tokens), hidden 7168, 256 experts, top-8, expert intermediate
2048, NVFP4 experts -- plus the final boundary, replayed as one CUDA graph.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl native|reference]

Prints one JSON line.  value = microseconds per layer-step (lower is better),
timed with CUDA events around K graph replays on device-resident inputs; the
weights of the ~57 activated experts (~1.4 GB per step) exceed L2 (129 MB)
many times over and each step uses a different input draw.  `roofline` is
the gate/up expert kernel (the largest share of the bytes), timed with CUDA
events around its own launches; `e2e` is the same step through the host-buffer
entry point (pinned H2D of the step inputs, D2H of its outputs, inside the
timed region); `cpu_baseline` is the CPU oracle on a bounded sample.
Multi-GPU (torchrun): one independent replica per GPU (the step has no
exchange on one GPU's worth of experts), max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE decode layer-step µs at b=8 and weight-stream HBM GB/s vs GB300 peak"
UNIT = "µs"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# DRAM traffic (read + write) of the experts kernel per active expert, from
# one full ncu capture of that kernel at serving widths with 64 experts
# (dram__bytes_read.sum + dram__bytes_write.sum of one launch, divided by its
# active experts); valid only for the kernel source it was taken on.
EXPERTS_TRAFFIC = {"source": ["speculative_decode_routed_gb300/csrc/experts_tc.cu",
                              "speculative_decode_routed_gb300/csrc/tc_ptx.cuh"],
                   "sha256_prefix": "93a95c69758f057c", "hidden": 7168, "inter": 2048,
                   "bytes_per_active_expert": (1065521920 + 3277568) / 43}


# DRAM traffic (read + write) of one launch of the dense draft layer's
# streamed gate/up projection at 8 rows, from one full ncu capture of that
# launch at the bench's widths; valid only for the kernel source it was taken
# on.
DENSE_GATE_UP_TRAFFIC = {"source": "speculative_decode_routed_gb300/csrc/gemv.cuh",
                         "sha256_prefix": "2557b235656f8a67", "hidden": 7168, "inter": 28672, "rows": 8,
                         "bytes": 822262784 + 3353600}

# The same for one launch of the context-KV projection's streaming kernel at
# 8 rows (hidden 7168, 4 layers of 8 KV heads of 128).
CTXKV_PROJ_TRAFFIC = {"source": "speculative_decode_routed_gb300/csrc/gemv.cuh",
                      "sha256_prefix": "2557b235656f8a67", "shape": (7168, 4, 8, 128, 8),
                      "bytes": 117915392 + 3609088}


def _ctxkv_traffic(hidden: int, layers: int, kv_heads: int, head_dim: int, rows: int):
    """Bytes per launch of the context-KV streaming projection from the ncu
    capture, or None if the kernel changed since or the shape differs."""
    t = CTXKV_PROJ_TRAFFIC
    if not _source_unchanged(t) or (hidden, layers, kv_heads, head_dim, rows) != t["shape"]:
        return None
    return int(t["bytes"])


def _source_unchanged(t) -> bool:
    """True if the kernel's sources (t["source"], one path or several, hashed
    in order as one stream) still hash to those the capture was taken on."""
    import hashlib
    paths = t["source"] if isinstance(t["source"], (list, tuple)) else [t["source"]]
    h = hashlib.sha256()
    try:
        for path in paths:
            with open(os.path.join(ROOT, path), "rb") as f:
                h.update(f.read())
    except OSError:
        return False
    return h.hexdigest().startswith(t["sha256_prefix"])


def _experts_traffic(w: synth.Workload, n_active: float):
    """Bytes per launch of the experts kernel scaled from the ncu capture, or
    None if the kernel changed since or the widths differ."""
    t = EXPERTS_TRAFFIC
    if not _source_unchanged(t) or (w.hidden, w.inter) != (t["hidden"], t["inter"]):
        return None
    return int(round(t["bytes_per_active_expert"] * n_active))


def _dense_traffic(hidden: int, inter: int, rows: int):
    """Bytes per launch of the streamed gate/up projection from the ncu
    capture, or None if the kernel changed since or the shape differs (the
    capture is not scaled: its rows and widths are the bench's)."""
    t = DENSE_GATE_UP_TRAFFIC
    if not _source_unchanged(t) or (hidden, inter, rows) != (t["hidden"], t["inter"], t["rows"]):
        return None
    return int(t["bytes"])


def _algorithmic_bytes(w: synth.Workload, n_active: int, rows: int):
    """Bytes one layer-step must move at minimum (weights read once)."""
    H, I, E, k = w.hidden, w.inter, w.n_experts, w.top_k
    gate_up = n_active * 2 * I * (H // 2 + H // 16) + n_active * 8
    down = n_active * H * (I // 2 + I // 16) + n_active * 4
    router = 2 * E * H + (4 * E if w.zipf_bias else 0)
    acts = rows * H * (4 + 4 + 2)                 # stream read + write, branch / gathered y
    return dict(gate_up=gate_up + rows * H // 2 + rows * k * I * 4, down=down, router=router,
                total=gate_up + down + router + acts)


class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock, throttle reasons)."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        sm.append(float(parts[1]))
                        mx = max(mx, float(parts[2]))
                    except ValueError:
                        continue
                    for n, v in zip(names, parts[5:9]):
                        if v.lower() == "active":
                            reasons.add(n)
        finally:
            os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _max_over_ranks(x: float, ws: int, device):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _expected_active(w: synth.Workload) -> float:
    """Experts a layer-step activates on average under uniform routing:
    E * (1 - (1 - k/E)^b) (the skewed sweep activates fewer)."""
    return w.n_experts * (1.0 - (1.0 - w.top_k / w.n_experts) ** w.rows)


def workload_config(w: synth.Workload, ws: int) -> dict:
    """The `config` both arms print: the workload itself (its shapes, its
    routing, how its inputs relate to L2), not how either arm runs it."""
    H, I = w.hidden, w.inter
    per_expert = 3 * H * I // 2 + 3 * H * I // 16
    gb = _expected_active(w) * per_expert / 1e9
    if gb * 1e9 < 129e6:
        l2 = "L2-resident: the whole layer fits in the 129 MB L2 (a correctness configuration)"
    else:
        l2 = ("inputs larger than L2: each layer-step's activated experts hold about %.2f GB of "
              "weights (uniform-routing estimate), far above the 129 MB L2; 4 input draws cycled" % gb)
    return {"workload": w.name, "rows": w.rows, "hidden": H, "n_experts": w.n_experts,
            "top_k": w.top_k, "inter": I, "n_layers": w.n_layers, "zipf_bias": w.zipf_bias,
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU", "l2": l2}


def moe_cpu_baseline_modules():
    """The CPU oracle and its test-side NVFP4 packing of the generators' raw
    expert weights: the CPU-baseline leg and the reference arm are the only
    parts of the bench that reach them."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from helpers import quantize_expert
    return oracle, quantize_expert


class OracleMoE:
    """The CPU oracle, as it stands, over the workload's layer-steps.  The
    experts a layer-step routes to are quantized by the oracle itself (its
    own NVFP4 packing of the host generator's raw weights) and cached: that
    is input preparation, outside the timed calls.  A probe of the boundary
    and the routing (also untimed) tells which experts a layer-step needs
    before the timed oracle.layer_step runs every stage over every row and
    every activated expert."""

    def __init__(self, w: synth.Workload):
        self.oracle, self.quantize_expert = moe_cpu_baseline_modules()
        self.w = w
        self.experts = {}   # (layer, expert) -> packed tensors
        self.dense = {}     # layer -> (w_post, w_pre, router_w, bias)

    def _weights(self, layer, need):
        quantize_expert = self.quantize_expert
        w, E = self.w, self.w.n_experts
        if layer not in self.dense:
            self.dense[layer] = (*synth.norm_weights(w, layer), synth.router_weights(w, layer),
                                 synth.router_bias(w, layer))
        for e in need:
            if (layer, e) not in self.experts:
                self.experts[(layer, e)] = quantize_expert(w, layer, e)
        w13, w13_sf, w2, w2_sf = {}, {}, {}, {}
        gscale = np.zeros((E, 3), np.float32)
        for e in need:
            w13[e], w13_sf[e], w2[e], w2_sf[e], gscale[e] = self.experts[(layer, e)]
        w_post, w_pre, rw, bias = self.dense[layer]
        return self.oracle.LayerWeights(E, w.hidden, w.inter, w_post, w_pre, rw, bias, w13, w13_sf,
                                        w2, w2_sf, gscale)

    def layer(self, layer, branch, stream):
        """(seconds of the timed oracle.layer_step, its outputs)."""
        o, w = self.oracle, self.w
        if layer not in self.dense:
            self._weights(layer, [])
        w_post, w_pre, rw, bias = self.dense[layer]
        _, x, _ = o.boundary(branch, stream, w_post, w_pre, w.eps)       # probe, untimed
        need = sorted(set(int(e) for e in o.route(x, rw, bias, w.top_k)["ids"].ravel()))
        lw = self._weights(layer, need)
        t0 = time.perf_counter()
        out = o.layer_step(lw, w.top_k, w.eps, branch, stream)
        return time.perf_counter() - t0, out

    def step(self, variant, layers):
        """One step over `layers` (then the final boundary) on input draw
        `variant` -> (seconds of the layers, seconds of the final boundary)."""
        o, w = self.oracle, self.w
        stream, branch = synth.step_inputs(w, variant)
        s, br = stream, o.bf16_to_f64(branch)
        t_layers = 0.0
        for l in layers:
            dt, out = self.layer(l, br, s)
            t_layers += dt
            s, br = out["stream"], o.gather(out["gates"], out["o"], w.top_k)
        wpf, wf = synth.final_norm_weights(w)
        t0 = time.perf_counter()
        o.boundary(br, s, wpf, wf, w.eps)
        return t_layers, time.perf_counter() - t0


def cpu_baseline(w: synth.Workload):
    """The CPU oracle, as it stands, on one whole layer-step (every row, every
    activated expert) of input draw 0, and the final boundary; the weights'
    preparation is not timed.  -> (us per layer-step, info)."""
    om = OracleMoE(w)
    t_layer, t_final = om.step(0, [0])
    info = {"kind": "oracle", "cores": om.oracle.num_threads(),
            "sample": f"one whole layer-step (layer 0, input draw 0: boundary, router, routing, pooler, "
                      f"x quantization, every activated expert, all {w.rows} rows), no extrapolation",
            "final_boundary_us": round(t_final * 1e6, 1)}
    return t_layer * 1e6, info


DENSE_METRIC = "dense draft layer µs at b=8 and weight-stream HBM GB/s vs GB300 peak"


def _dense_bytes(w: synth.Workload, rows: int):
    """Bytes one dense layer must move at minimum: each bf16 weight once, the
    activations of every stage once each way."""
    H, I = w.hidden, w.inter
    w13, w2 = 2 * I * H * 2, H * I * 2
    gate_up = w13 + rows * H * 2 + rows * 2 * I * 2
    down = w2 + rows * I * 2 + rows * H * 2
    norms = 3 * H * 4 + 2 * rows * H * (2 + 4 + 4) + rows * H * 2 + rows * 2 * I * 2 + rows * I * 2
    return dict(gate_up=gate_up, down=down, total=gate_up + down + norms)


def dense_cpu_baseline(w: synth.Workload):
    """The CPU oracle's dense layer, as it stands, on the whole step (all rows,
    both projections); weight generation is not timed.  -> (us, info)."""
    import oracle
    stream, attn = synth.step_inputs(w)
    na, npre, npost = synth.dense_norm_weights(w, 0)
    w13, w2 = synth.dense_weights(w, 0)
    t0 = time.perf_counter()
    oracle.dense_layer(attn, stream, na, npre, w13, w2, npost, w.eps)
    us = (time.perf_counter() - t0) * 1e6
    return us, {"kind": "oracle", "cores": oracle.num_threads(),
                "sample": f"the whole dense layer on all {w.rows} rows (no sampling)"}


CTXKV_METRIC = "draft context-KV projection µs at 8 context rows and weight-stream HBM GB/s vs GB300 peak"


def _ctxkv_bytes(w, n: int):
    """Bytes one projection must move at minimum: the stacked K/V weights once,
    the context, the layer inputs and projections once each way, the keys and
    values into the cache."""
    L, H, KD = w.n_layers, w.hidden, w.n_kv_heads * w.head_dim
    weights = L * 2 * KD * H * 2
    gemm = weights + L * n * H * 2 + L * n * 2 * KD * 2
    rest = n * H * 2 + (H + L * H) * 4 + n * H * 2 + L * n * H * 2 + L * n * 2 * KD * 2 * 3 + n * 16
    return dict(gemm=gemm, total=gemm + rest)


def ctxkv_cpu_baseline(w):
    """The CPU oracle's whole projection (all rows, all layers, the cache write);
    weight generation is not timed.  -> (us, info)."""
    import oracle
    ctx, pos, slots = synth.ctxkv_inputs(w)
    wh, wp = synth.ctxkv_norm_weights(w)
    wkv = synth.ctxkv_weights(w)
    shape = (w.n_layers, w.n_slots, w.n_kv_heads, w.head_dim)
    kc, vc = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    t0 = time.perf_counter()
    o = oracle.context_kv(ctx, pos, wh, wp, wkv, w.n_kv_heads, w.head_dim, w.eps, w.qk_eps, w.rope_theta)
    oracle.kv_cache_write(o["k"], o["v"], slots, w.n_slots, kc, vc)
    us = (time.perf_counter() - t0) * 1e6
    return us, {"kind": "oracle", "cores": oracle.num_threads(),
                "sample": f"the whole projection of all {w.n_ctx} rows into {w.n_layers} layers (no sampling)"}


def run_reference(args, w):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    if isinstance(w, synth.CtxKvWorkload):
        times, info = [], None
        for i in range(args.warmup + args.steps):
            us, info = ctxkv_cpu_baseline(w)
            if i >= args.warmup:
                times.append(us)
        v = float(np.mean(times))
        line = {"impl": "reference", "metric": CTXKV_METRIC, "value": round(v, 1), "unit": UNIT,
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(v / 1000.0, 3), "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": w.name, "n_ctx": w.n_ctx, "hidden": w.hidden,
                           "n_layers": w.n_layers, "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim},
                "cpu_baseline": dict(info, value=round(v, 1), unit=UNIT),
                "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    if w.n_experts == 0:
        times, info = [], None
        for i in range(args.warmup + args.steps):
            us, info = dense_cpu_baseline(w)
            if i >= args.warmup:
                times.append(us)
        v = float(np.mean(times))
        line = {"impl": "reference", "metric": DENSE_METRIC, "value": round(v, 1), "unit": UNIT,
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(v / 1000.0, 3), "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": w.name, "rows": w.rows, "hidden": w.hidden, "inter": w.inter},
                "cpu_baseline": dict(info, value=round(v, 1), unit=UNIT),
                "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    om = OracleMoE(w)
    if args.cpu_cores:
        om.oracle.set_num_threads(args.cpu_cores)
    # a step is the whole step (every layer, then the final boundary) up to 8
    # layers, cycling 4 input draws; a deeper stack is sampled one layer-step
    # per step (layer i mod L) on one draw, so the run ends within minutes
    whole = w.n_layers <= 8
    variants = 4 if w.n_layers == 1 else 1
    lay_s, fin_s, steps_s = [], [], []
    for i in range(args.warmup + args.steps):
        layers = list(range(w.n_layers)) if whole else [i % w.n_layers]
        tl, tf = om.step(i % variants, layers)
        if i >= args.warmup:
            lay_s.append(tl / len(layers))
            fin_s.append(tf)
            steps_s.append(tl + tf)
    v = float(np.mean(lay_s)) * 1e6
    sample = ("the whole step (every layer, every row, every activated expert, the final boundary) "
              if whole else "one layer-step per step (layer i mod %d, every row and activated expert) "
              "and the final boundary " % w.n_layers) + "of %d input draw(s), cycled" % variants
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(float(np.mean(steps_s)) * 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args.gpus),
            "final_boundary_us": round(float(np.mean(fin_s)) * 1e6, 1),
            "cpu_baseline": {"kind": "oracle", "cores": om.oracle.num_threads(), "sample": sample,
                             "value": round(v, 1), "unit": UNIT},
            "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_native(args, w):
    import torch

    import speculative_decode_routed_gb300 as moe
    import synth.gpu as sgpu

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    dec = sgpu.build(w, device=device)
    V = 4                                             # distinct input draws, cycled
    bufs = []
    for v in range(V):
        s, b = sgpu.step_tensors(w, variant=v, device=device)
        bufs.append((s, b, torch.empty_like(b)))
    rows = w.rows
    cs = torch.cuda.current_stream(device)

    # active experts of each draw (for the byte count): one eager layer per draw
    n_active = []
    for s, b, o in bufs:
        st = s.clone()
        dec.layer(0, rows, b, st)
        torch.cuda.synchronize(device)
        n_active.append(int(torch.as_tensor(
            _Cai(dec.debug().n_active, (1,), "<i4"), device=device).item()))
    dec.check()

    for i in range(args.warmup):
        s, b, o = bufs[i % V]
        dec.step_graph(rows, b, s, o)
    torch.cuda.synchronize(device)
    _barrier(ws)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize(device)
        _barrier(ws)
        ev0.record(cs)
        for i in range(args.steps):
            s, b, o = bufs[i % V]
            dec.step_graph(rows, b, s, o)
        ev1.record(cs)
        torch.cuda.synchronize(device)
        _barrier(ws)
    dec.check()
    ms = ev0.elapsed_time(ev1) / args.steps
    ms = _max_over_ranks(ms, ws, device)
    clocks = clk.summary()

    # The layer-step excludes the final boundary (which closes a whole step
    # once): the layers alone and the final boundary alone, each captured in
    # a graph of the library's calls per input draw and timed over K replays
    # with CUDA events on the launching stream.
    side = torch.cuda.Stream(device)
    side.wait_stream(cs)
    layer_graphs, final_graphs = [], []
    for s, b, o in bufs:
        gl, gf = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(gl, stream=side):
            for l in range(w.n_layers):
                dec.layer(l, rows, b if l == 0 else None, s, stream=side)
        with torch.cuda.graph(gf, stream=side):
            dec.final(rows, s, o, stream=side)
        layer_graphs.append(gl)
        final_graphs.append(gf)
    cs.wait_stream(side)

    def timed(graphs):
        for i in range(args.warmup):
            graphs[i % V].replay()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        a.record(cs)
        for i in range(args.steps):
            graphs[i % V].replay()
        z.record(cs)
        torch.cuda.synchronize(device)
        return a.elapsed_time(z) / args.steps

    layers_ms = _max_over_ranks(timed(layer_graphs), ws, device)
    final_ms = _max_over_ranks(timed(final_graphs), ws, device)
    dec.check()
    us_layer = layers_ms * 1000.0 / w.n_layers

    # per-kernel durations (events on the launching stream around each kernel)
    prof, prof_bytes = [], []
    for i in range(max(4, min(args.steps, 20))):
        s, b, o = bufs[i % V]
        prof.append(dec.layer_profile(0, rows, b, s))
        prof_bytes.append(_algorithmic_bytes(w, n_active[i % V], rows))
    prof = np.array(prof)
    k_ms = prof.mean(0)
    na = float(np.mean(n_active))
    byt = _algorithmic_bytes(w, int(round(na)), rows)
    peak, peak_kind = _peaks()
    # the tensor-core build runs gate/up and down in one kernel (slot 3; slot 4 is 0)
    fused = bool(np.all(prof[:, 4] == 0))
    exp_bytes = np.array([pb["gate_up"] + (pb["down"] if fused else 0) for pb in prof_bytes], float)
    exp_gbs = exp_bytes.sum() / (prof[:, 3].sum() * 1e-3) / 1e9
    dn_gbs = None if fused else (sum(pb["down"] for pb in prof_bytes) / (prof[:, 4].sum() * 1e-3) / 1e9)
    step_gbs = byt["total"] * w.n_layers / (layers_ms * 1e-3) / 1e9 * ws

    # the first layer's front (embedded tokens -> stream + input norm), timed
    # alone: CUDA events around 50 launches on the launching stream
    emb_bits, wn = synth.front_inputs(w)
    emb = torch.from_numpy(emb_bits.view(np.int16)).view(torch.bfloat16).to(device)
    wn_t = torch.from_numpy(wn).to(device)
    st_f = torch.empty(rows, w.hidden, dtype=torch.float32, device=device)
    ai_f = torch.empty(rows, w.hidden, dtype=torch.bfloat16, device=device)
    for _ in range(5):
        dec.front(rows, emb, wn_t, st_f, ai_f)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(cs)
    for _ in range(50):
        dec.front(rows, emb, wn_t, st_f, ai_f)
    f1.record(cs)
    torch.cuda.synchronize(device)
    dec.check()
    front_us = f0.elapsed_time(f1) * 1000.0 / 50

    # end to end through the host-buffer entry point
    s_h, b_h = synth.step_inputs(w)
    sh = torch.from_numpy(s_h).pin_memory()
    bh = torch.from_numpy(b_h).view(torch.bfloat16).pin_memory()
    oh = torch.empty_like(bh).pin_memory()
    for _ in range(3):
        dec.step_host(rows, bh, sh, oh)
    _barrier(ws)
    t0 = time.perf_counter()
    n_e2e = max(args.steps, 5)
    for _ in range(n_e2e):
        dec.step_host(rows, bh, sh, oh)
    e2e_ms = (time.perf_counter() - t0) * 1000.0 / n_e2e
    e2e_ms = _max_over_ranks(e2e_ms, ws, device)

    if rank != 0:
        dec.close()
        return
    line = {
        "metric": METRIC, "value": round(us_layer, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "e2m1",
        "data": "synthetic (seeded Philox / Irwin-Hall normals, NVFP4-packed on device)",
        "config": workload_config(w, ws),
        "timing": {"value": "us per layer-step: a graph of the step's layers (no final boundary), "
                            "K replays, divided by the layers",
                   "ms_per_step": "the library's step graph (every layer and the final boundary), K replays",
                   "step_us_per_layer": round(ms * 1000.0 / w.n_layers, 2),
                   "final_boundary_us": round(final_ms * 1000.0, 2),
                   "bytes_per_layer_step_measured": int(byt["total"])},
        "weight_stream_gbs": round(step_gbs, 1),
        "weight_stream_frac_of_peak": round(step_gbs / (peak * ws), 4),
        "bytes_per_layer_step": int(byt["total"]), "n_active_mean": na,
        "roofline": {"kernel": "routed experts (gate/up and down, one kernel)" if fused
                     else "experts gate/up", "bound": "hbm", "achieved": round(exp_gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(exp_gbs / peak, 4),
                     "traffic": _experts_traffic(w, float(np.mean([n_active[i % V] for i in range(len(prof))])))
                     if fused else None, "peak_kind": peak_kind,
                     "launch_us": round(k_ms[3] * 1000, 2),
                     "algorithmic_bytes": int(exp_bytes.mean())},
        "kernels_us": dict({"boundary": round(k_ms[0] * 1000, 2), "router": round(k_ms[1] * 1000, 2),
                            "pool": round(k_ms[2] * 1000, 2), "front": round(front_us, 2),
                            "final_boundary": round(final_ms * 1000.0, 2)},
                           **({"experts": round(k_ms[3] * 1000, 2)} if fused else
                              {"gate_up": round(k_ms[3] * 1000, 2), "down": round(k_ms[4] * 1000, 2),
                               "down_gbs": round(dn_gbs, 1)})),
        "e2e": {"value": round(e2e_ms * 1000.0 / w.n_layers, 2), "unit": UNIT,
                "h2d_bytes_per_step": rows * w.hidden * (2 + 4),
                "d2h_bytes_per_step": rows * w.hidden * (4 + 2),
                "includes": "moe_decode_step_host per call divided by the layers: the host transfers "
                            "and the final boundary are inside"},
        "gpu_launches": moe.moe_decode_step_kernel_count(dec.handle) * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and ws == 1:
        us, info = cpu_baseline(w)
        line["cpu_baseline"] = dict(info, value=round(us, 1), unit=UNIT)
    print(json.dumps(line), flush=True)
    dec.close()
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_dense(args, w):
    """One dense draft layer per step (boundary, gate/up with SiLU * mul, down,
    boundary; the library GEMMs beyond 8 rows), replayed as a CUDA graph per
    input draw."""
    import torch

    import speculative_decode_routed_gb300 as moe

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    H, I, rows = w.hidden, w.inter, w.rows
    w13 = torch.empty(2 * I, H, dtype=torch.bfloat16, device=device)
    w2 = torch.empty(H, I, dtype=torch.bfloat16, device=device)
    synth.dev_dense_weights(w13, w2, w, 0)
    norms = [torch.from_numpy(n).to(device) for n in synth.dense_norm_weights(w, 0)]
    dl = moe.DenseLayer(H, I, rows, norms[0], norms[1], w13, w2, norms[2], eps=w.eps)
    V = 4
    bufs = []
    for v in range(V):
        s, a = synth.step_inputs(w, v)
        bufs.append((torch.from_numpy(s).to(device),
                     torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)))
    cs = torch.cuda.current_stream(device)
    for s, a in bufs:                                 # eager first calls, outside capture
        dl.layer(rows, a, s.clone())
    torch.cuda.synchronize(device)
    graphs = []
    side = torch.cuda.Stream(device)
    side.wait_stream(cs)
    for s, a in bufs:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            dl.layer(rows, a, s, stream=side)
        graphs.append(g)
    cs.wait_stream(side)
    for i in range(args.warmup):
        graphs[i % V].replay()
    torch.cuda.synchronize(device)
    _barrier(ws)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize(device)
        _barrier(ws)
        ev0.record(cs)
        for i in range(args.steps):
            graphs[i % V].replay()
        ev1.record(cs)
        torch.cuda.synchronize(device)
        _barrier(ws)
    ms = ev0.elapsed_time(ev1) / args.steps
    ms = _max_over_ranks(ms, ws, device)
    clocks = clk.summary()

    # per-launch durations: events on the launching stream around each launch
    prof = np.array([dl.layer_profile(rows, *bufs[i % V][::-1]) for i in range(max(4, min(args.steps, 20)))])
    k_ms = prof.mean(0)
    byt = _dense_bytes(w, rows)
    peak, peak_kind = _peaks()
    # up to 8 rows (H and I multiples of 128) the library streams both
    # projections itself: four kernels of its own, SiLU * mul inside gate/up
    streamed = rows <= 8 and H % 128 == 0 and I % 128 == 0
    own = 4                                           # every kernel the library's own
    gu_gbs = byt["gate_up"] / (k_ms[1] * 1e-3) / 1e9
    dn_gbs = byt["down"] / (k_ms[3] * 1e-3) / 1e9
    step_gbs = byt["total"] / (ms * 1e-3) / 1e9 * ws

    # end to end through moe_dense_layer_host: the attention output and the
    # stream in from page-locked host memory, the stream back out
    s_h, a_h = synth.step_inputs(w)
    sh = torch.from_numpy(s_h).pin_memory()
    ah = torch.from_numpy(a_h.view(np.int16)).view(torch.bfloat16).pin_memory()

    def host_step():
        dl.layer_host(rows, ah, sh)

    for _ in range(3):
        host_step()
    _barrier(ws)
    t0 = time.perf_counter()
    n_e2e = max(args.steps, 5)
    for _ in range(n_e2e):
        host_step()
    e2e_ms = (time.perf_counter() - t0) * 1000.0 / n_e2e
    e2e_ms = _max_over_ranks(e2e_ms, ws, device)
    if rank != 0:
        dl.close()
        return
    line = {
        "metric": DENSE_METRIC, "value": round(ms * 1000.0, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Philox / Irwin-Hall normals generated on device)",
        "config": {"workload": w.name, "rows": rows, "hidden": H, "inter": I,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "graph": "one CUDA graph per input draw (the whole layer)",
                   "l2": "inputs larger than L2: %.2f GB of bf16 weights per step, 4 input draws cycled"
                         % ((byt["gate_up"] + byt["down"]) / 1e9)},
        "weight_stream_gbs": round(step_gbs, 1),
        "weight_stream_frac_of_peak": round(step_gbs / (peak * ws), 4),
        "bytes_per_layer_step": int(byt["total"]),
        "roofline": {"kernel": "gate/up projection + SiLU * mul (split-K weight-streaming kernel, bf16 mma.sync)"
                     if streamed else "gate/up projection + SiLU * mul (tcgen05 bf16 projection kernel)",
                     "bound": "hbm",
                     "achieved": round(gu_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gu_gbs / peak, 4),
                     "traffic": _dense_traffic(H, I, rows) if streamed else None, "peak_kind": peak_kind,
                     "launch_us": round(k_ms[1] * 1000, 2), "algorithmic_bytes": int(byt["gate_up"])},
        "kernels_us": {"boundary_attn": round(k_ms[0] * 1000, 2), "gate_up": round(k_ms[1] * 1000, 2),
                       "down": round(k_ms[3] * 1000, 2), "boundary_ffn": round(k_ms[4] * 1000, 2),
                       "down_gbs": round(dn_gbs, 1)},
        "e2e": {"value": round(e2e_ms * 1000.0, 2), "unit": UNIT,
                "h2d_bytes_per_step": rows * H * (4 + 2), "d2h_bytes_per_step": rows * H * 4},
        "gpu_launches": own * args.steps,
        "library_launches": (dl.kernel_count(rows) - own) * args.steps,   # 0: no library kernels
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and ws == 1:
        us, info = dense_cpu_baseline(w)
        line["cpu_baseline"] = dict(info, value=round(us, 1), unit=UNIT)
    print(json.dumps(line), flush=True)
    dl.close()
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_ctxkv(args, w):
    """The draft context-KV projection of n_ctx rows into every draft layer and the
    cache, replayed as a CUDA graph per input draw.  The stacked weights fit in
    L2, so the steps rotate over four copies of them (one handle each): a step's
    copy was last read three steps before, with 352 MB of the other copies
    streamed since, so every step reads its weights from HBM and the steps run
    back to back like the other workloads'.  The per-step figure with L2
    flushed before each step, outside its events, is reported beside it."""
    import torch

    import speculative_decode_routed_gb300 as moe

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    L, H, KVH, D, n = w.n_layers, w.hidden, w.n_kv_heads, w.head_dim, w.n_ctx
    wkv = torch.empty(L, 2 * KVH * D, H, dtype=torch.bfloat16, device=device)
    synth.dev_ctxkv_weights(wkv, w)
    wh, wp = (torch.from_numpy(a).to(device) for a in synth.ctxkv_norm_weights(w))
    V = 4                                           # input draws = weight copies
    ops = [moe.ContextKV(H, L, KVH, D, n, wh, wp, wkv if v == 0 else wkv.clone(), eps=w.eps,
                         qk_eps=w.qk_eps, rope_theta=w.rope_theta, max_position=w.max_position)
           for v in range(V)]
    op = ops[0]
    kc = torch.zeros(L, w.n_slots, KVH, D, dtype=torch.bfloat16, device=device)
    vc = torch.zeros_like(kc)
    bufs = []
    for v in range(V):
        ctx, pos, slots = synth.ctxkv_inputs(w, v)
        bufs.append((torch.from_numpy(ctx.view(np.int16)).view(torch.bfloat16).to(device),
                     torch.from_numpy(pos).to(device), torch.from_numpy(slots).to(device)))
    cs = torch.cuda.current_stream(device)
    for o, (c, p, s_) in zip(ops, bufs):
        o.project(n, c, p, s_, kc, vc)
    torch.cuda.synchronize(device)
    for o in ops:
        o.check()
    side = torch.cuda.Stream(device)
    side.wait_stream(cs)
    graphs = []
    for o, (c, p, s_) in zip(ops, bufs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            o.project(n, c, p, s_, kc, vc, stream=side)
        graphs.append(g)
    cs.wait_stream(side)
    # the flushed figure: before each step, write a buffer twice the L2, then
    # read another one, so the weights are not resident and L2 holds clean
    # lines (the flush's own write-backs are not charged to the step)
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    flush_r = torch.ones(64 << 20, dtype=torch.int32, device=device)

    def flush():
        flush_w.zero_()
        return flush_r.sum()

    for i in range(args.warmup):
        graphs[i % V].replay()
    torch.cuda.synchronize(device)
    _barrier(ws)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize(device)
        _barrier(ws)
        ev0.record(cs)
        for i in range(args.steps):
            graphs[i % V].replay()
        ev1.record(cs)
        torch.cuda.synchronize(device)
        _barrier(ws)
    ms = ev0.elapsed_time(ev1) / args.steps
    ms = _max_over_ranks(ms, ws, device)
    clocks = clk.summary()

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.warmup):
        flush()
        graphs[i % V].replay()
    for i in range(args.steps):
        flush()
        evs[i][0].record(cs)
        graphs[i % V].replay()
        evs[i][1].record(cs)
    torch.cuda.synchronize(device)
    flushed_ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    flushed_ms = _max_over_ranks(flushed_ms, ws, device)
    for o in ops:
        o.check()

    prof = []
    for i in range(max(4, min(args.steps, 20))):
        c, p, s_ = bufs[i % V]
        flush()
        prof.append(op.profile(n, c, p, s_, kc, vc))
    k_ms = np.array(prof).mean(0)
    byt = _ctxkv_bytes(w, n)
    # the library streams the projection itself up to 8 rows when H is a multiple of 128
    streamed = n <= 8 and H % 128 == 0
    peak, peak_kind = _peaks()
    gemm_gbs = byt["gemm"] / (k_ms[1] * 1e-3) / 1e9
    step_gbs = byt["total"] / (ms * 1e-3) / 1e9 * ws

    # end to end through moe_ctxkv_project_host: context, positions and slots
    # in from page-locked host memory, the keys and values out (the caches are
    # device memory)
    ctx_h, pos_h, slots_h = synth.ctxkv_inputs(w)
    ch = torch.from_numpy(ctx_h.view(np.int16)).view(torch.bfloat16).pin_memory()
    ph, sh = torch.from_numpy(pos_h).pin_memory(), torch.from_numpy(slots_h).pin_memory()
    kh = torch.empty(L, n, KVH, D, dtype=torch.bfloat16).pin_memory()
    vh = torch.empty_like(kh).pin_memory()

    def host_step(i):                # the weight copies in rotation, as above
        ops[i % V].project_host(n, ch, ph, kh, vh, slots=sh, k_cache=kc, v_cache=vc)

    for i in range(3):
        host_step(i)
    _barrier(ws)
    t0 = time.perf_counter()
    n_e2e = max(args.steps, 5)
    for i in range(n_e2e):
        host_step(i)
    e2e_ms = (time.perf_counter() - t0) * 1000.0 / n_e2e
    e2e_ms = _max_over_ranks(e2e_ms, ws, device)
    for o in ops:
        o.check()
    if rank != 0:
        for o in ops:
            o.close()
        return
    line = {
        "metric": CTXKV_METRIC, "value": round(ms * 1000.0, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Philox / Irwin-Hall normals generated on device)",
        "config": {"workload": w.name, "n_ctx": n, "hidden": H, "n_layers": L, "n_kv_heads": KVH,
                   "head_dim": D, "rope_theta": w.rope_theta,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "graph": "one CUDA graph per input draw, K replays back to back",
                   "l2": "inputs larger than L2: the steps rotate over %d copies of the %.1f MB of "
                         "K/V weights (%.0f MB streamed between two reads of a copy)"
                         % (V, L * 2 * KVH * D * H * 2 / 1e6, (V - 1) * L * 2 * KVH * D * H * 2 / 1e6)},
        "flushed": {"value": round(flushed_ms * 1000.0, 2), "unit": UNIT,
                    "how": "CUDA events around each replay; before each, outside the events, a 256 MB "
                           "write, then a 256 MB read so L2 holds clean lines"},
        "weight_stream_gbs": round(step_gbs, 1),
        "weight_stream_frac_of_peak": round(step_gbs / (peak * ws), 4),
        "bytes_per_step": int(byt["total"]),
        "roofline": {"kernel": "K/V projection (split-K weight-streaming kernel, bf16 mma.sync)" if streamed
                     else "K/V projection (tcgen05 bf16 projection kernel)", "bound": "hbm",
                     "achieved": round(gemm_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gemm_gbs / peak, 4), "traffic": _ctxkv_traffic(H, L, KVH, D, n) if streamed
                     else None, "peak_kind": peak_kind,
                     "launch_us": round(k_ms[1] * 1000, 2), "algorithmic_bytes": int(byt["gemm"])},
        "kernels_us": {"norms": round(k_ms[0] * 1000, 2), "projection": round(k_ms[1] * 1000, 2),
                       "key_norm_rope_cache": round(k_ms[2] * 1000, 2)},
        "e2e": {"value": round(e2e_ms * 1000.0, 2), "unit": UNIT,
                "h2d_bytes_per_step": n * H * 2 + n * 8 * 2,
                "d2h_bytes_per_step": 2 * L * n * KVH * D * 2},
        "gpu_launches": 3 * args.steps,
        "library_launches": (op.kernel_count(n) - 3) * args.steps,   # 0: no library kernels
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and ws == 1:
        us, info = ctxkv_cpu_baseline(w)
        line["cpu_baseline"] = dict(info, value=round(us, 1), unit=UNIT)
    print(json.dumps(line), flush=True)
    for o in ops:
        o.close()
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


class _Cai:
    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": shape, "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3, "strides": None}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="serving",
                    choices=sorted(synth.WORKLOADS) + sorted(synth.DENSE_WORKLOADS)
                    + sorted(synth.CTXKV_WORKLOADS))
    ap.add_argument("--rows", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-cores", type=int, default=0,
                    help="host threads of the oracle in the reference arm (default: all)")
    args = ap.parse_args()
    w = (synth.WORKLOADS.get(args.workload) or synth.DENSE_WORKLOADS.get(args.workload)
         or synth.CTXKV_WORKLOADS[args.workload])
    if args.rows:
        w = w.with_ctx(args.rows) if isinstance(w, synth.CtxKvWorkload) else w.with_rows(args.rows)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args, w)
    elif isinstance(w, synth.CtxKvWorkload):
        run_ctxkv(args, w)
    elif w.n_experts == 0:
        run_dense(args, w)
    else:
        run_native(args, w)


if __name__ == "__main__":
    main()
