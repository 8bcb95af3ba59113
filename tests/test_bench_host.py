"""bench.py's multi-process bookkeeping without a GPU: the max over ranks and
the barrier on a two-rank gloo group, and the reference arm's rank-0-only
output under a two-rank launch."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, values, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    bench._barrier(world)
    out[rank] = bench._max_over_ranks(values[rank], world, "cpu")
    bench._barrier(world)
    dist.destroy_process_group()


def test_max_over_ranks_on_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    values = [0.25, 1.75]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, values, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 1.75, 1: 1.75}


def test_reference_arm_prints_once_under_two_ranks():
    lines = {}
    for rank in (1, 0):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2")
        r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                            "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        lines[rank] = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert lines[1] == []
    assert len(lines[0]) == 1
    rec = json.loads(lines[0][0])
    assert rec["impl"] == "reference" and rec["unit"] == "µs" and rec["higher_is_better"] is False
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_figures_are_gated_on_their_capture(monkeypatch):
    """The ncu traffic figures are reported only for the kernel source and the
    shape they were captured on, and each sits just above its kernel's
    algorithmic bytes (every weight byte read once)."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    wd = synth.DENSE_WORKLOADS["draft_dense"]
    traffic = bench._dense_traffic(wd.hidden, wd.inter, 8)
    if traffic is not None:   # the projection source is the captured one
        ratio = traffic / bench._dense_bytes(wd, 8)["gate_up"]
        assert 1.0 <= ratio < 1.01
    assert bench._dense_traffic(wd.hidden, wd.inter, 4) is None
    assert bench._dense_traffic(256, 384, 8) is None
    monkeypatch.setitem(bench.DENSE_GATE_UP_TRAFFIC, "sha256_prefix", "0" * 16)
    assert bench._dense_traffic(wd.hidden, wd.inter, 8) is None
    monkeypatch.setitem(bench.EXPERTS_TRAFFIC, "sha256_prefix", "0" * 16)
    assert bench._experts_traffic(synth.WORKLOADS["serving"], 60.0) is None
    # the context-KV projection's: the fp32 partials and the per-head counts
    # come on top of the weights and activations
    wc = synth.CTXKV_WORKLOADS["draft_ctx_kv"]
    shape = (wc.hidden, wc.n_layers, wc.n_kv_heads, wc.head_dim, 8)
    traffic = bench._ctxkv_traffic(*shape)
    if traffic is not None:
        ratio = traffic / bench._ctxkv_bytes(wc, 8)["gemm"]
        assert 1.0 <= ratio < 1.04
    assert bench._ctxkv_traffic(*shape[:4], 128) is None
    monkeypatch.setitem(bench.CTXKV_PROJ_TRAFFIC, "sha256_prefix", "0" * 16)
    assert bench._ctxkv_traffic(*shape) is None


@pytest.mark.parametrize("workload", ["tiny", "draft_dense_small", "draft_ctx_kv_small"])
def test_reference_arm_line_keeps_the_contract(workload):
    """The oracle arm's one JSON line, for each kind of workload, carries the
    keys the bench contract names, with a cpu_baseline describing the run
    and an e2e of zero host bytes."""
    import time
    t0 = time.perf_counter()
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload,
                        "--steps", "2", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    wall = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in rec, key
    assert rec["impl"] == "reference" and rec["n_gpus"] == 1 and rec["steps"] == 2 and rec["warmup"] == 3
    # the steps it claims to have timed fit inside the run (nothing extrapolated)
    assert rec["steps"] * rec["ms_per_step"] / 1000.0 <= wall
    assert rec["value"] > 0 and rec["unit"] == "µs" and rec["higher_is_better"] is False
    assert rec["config"]["workload"] == workload
    cb = rec["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == rec["value"]
    assert rec["e2e"] == {"value": rec["value"], "unit": rec["unit"], "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}


def test_both_arms_print_the_same_config():
    """The native arm's config and the reference arm's are one function of the
    workload, so the two lines compare; the reference arm's line carries it."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    w = synth.WORKLOADS["tiny"]
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    rec = json.loads([ln for ln in r.stdout.splitlines() if ln.strip()][0])
    assert rec["config"] == bench.workload_config(w, 1)
    src = open(os.path.join(ROOT, "bench.py")).read()
    native = src[src.index("def run_native("):src.index("def run_dense(")]
    assert '"config": workload_config(w, ws)' in native
    serving = bench.workload_config(synth.WORKLOADS["serving"], 1)
    assert serving["l2"].startswith("inputs larger than L2")
    assert bench.workload_config(w, 1)["l2"].startswith("L2-resident")
