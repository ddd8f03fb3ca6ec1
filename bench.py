"""Benchmark: causal GQA + RoPE attention, forward + backward, TFLOP/s.

One step = forward + backward of every layer of the GPU-pipeline workload (B=16,
T=512, Hq=12, Hkv=4, D=64, bf16, 16 layers with distinct buffers, so the 16 x 115 MB
working set is far larger than L2 and every step reads from HBM).  FLOPs per layer
count exact causal pairs: 14 * D * T(T+1)/2 * B * Hq (4 D forward, 10 D backward).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --decode     # the decode step over a KV cache instead: cache-read GB/s

Beside the headline, the default line carries points measured outside its timed region:
the long-sequence sweep (T 2048, 8192, 16384), the fused prologue and the decode step.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the
attention of independent sequences needs no exchange); the timed region is bracketed
by a barrier and the max over ranks is reported.  `--impl reference` times the fp64
CPU oracle on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal GQA+RoPE attn fwd+bwd TFLOP/s (B16 T512 Hq12/Hkv4 D64 bf16), % of peak"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", type=int, default=2, help="workload id (see synthetic.WORKLOADS)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-sweep", action="store_true",
                   help="leave out the long-sequence sweep points and the TF32 peak measurement")
    p.add_argument("--bare", action="store_true",
                   help="only the warm-up and the K timed steps of one workload (layer 0 only), then a short "
                        "line: the command profilers run")
    p.add_argument("--decode", action="store_true",
                   help="time the decode step over a KV cache instead (cache-read GB/s)")
    p.add_argument("--prologue", action="store_true",
                   help="only the fused RMSNorm -> QKV -> RoPE prologue at the GPU-pipeline shape (K steps of 16 "
                        "layers), then a short line")
    p.add_argument("--phase-timing", choices=["timed", "separate"], default="separate",
                   help="per-kernel CUDA events inside the timed region, or (default) in as many profiled "
                        "steps right after it: events between kernels cost ~20%% and disable the overlap of "
                        "dependent launches, so the timed region itself runs bare")
    return p.parse_args()


# ------------------------------------------------------------------ distributed harness
class Harness:
    """Rank bookkeeping.  Collectives here only synchronise the timing (barrier, max
    of the step time); the attention itself never communicates."""

    def __init__(self, backend: str):
        import torch.distributed as dist
        self.dist = dist
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        if self.world > 1 and not dist.is_initialized():
            dist.init_process_group(backend)

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def max(self, x: float, device=None) -> float:
        if self.world == 1:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1 and self.dist.is_initialized():
            self.dist.destroy_process_group()


def shard_layers(layers: int, world: int, rank: int):
    """Replicas: every rank runs all layers on its own copy (weak scaling)."""
    return list(range(layers))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, timeout_s: float = 5.0):
        """Block until nvidia-smi has produced its first sample (it starts slowly)."""
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < timeout_s:
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ peaks / profile data
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": d.get("bf16_tflops"), "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d.get("hbm_gbs"), "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def profiled_traffic(kernel_source: str, key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current source of the kernel (matched by the source file's sha256)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(key)
    if not ent:
        return None
    with open(kernel_source, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    return ent["dram_bytes_per_launch"] if ent.get("source_sha256") == sha else None


# ------------------------------------------------------------------ CPU oracle baseline
def oracle_sample(w, rows: int = 4):
    """A bounded sample of the workload for the CPU oracle: the first `rows` batch rows
    of layer 0, every head (so the oracle's OpenMP loops over (batch, head) and
    (batch, kv head) have 48 and 16 independent units)."""
    from causal_gqa_flash_attention_gb300 import synthetic
    q, k, v, dO = synthetic.make_inputs(w, layer=0, batch=slice(0, rows))
    arrs = [t.double().numpy() for t in (q, k, v, dO)]
    flops = 14 * w.D * w.pairs * rows * w.Hq
    desc = f"layer 0, batch rows 0..{rows - 1}, all {w.Hq} query / {w.Hkv} kv heads, T={w.T}, D={w.D}, fp64"
    return arrs, flops, desc


def cpu_baseline(w, seconds_target=10.0):
    """The fp64 oracle, as it stands, on a bounded sample (forward + backward),
    repeated until ~seconds_target of host time."""
    import oracle
    oracle.build()
    (qn, kn, vn, dn), flops, desc = oracle_sample(w)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.attn_fwd(qn, kn, vn, w.theta)
        oracle.attn_bwd(qn, kn, vn, dn, w.theta)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds_target or n >= 1000:
            break
    return {"value": flops * n / el / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{desc}; fwd+bwd x{n} in {el:.1f} s"}


def run_reference(args, w):
    """--impl reference: the fp64 CPU oracle on the host cores, timed per step on a
    bounded sample of the workload (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    (q, k, v, dO), flops, sample = oracle_sample(w)
    for _ in range(args.warmup):
        oracle.attn_fwd(q, k, v, w.theta)
        oracle.attn_bwd(q, k, v, dO, w.theta)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attn_fwd(q, k, v, w.theta)
        oracle.attn_bwd(q, k, v, dO, w.theta)
    el = time.perf_counter() - t0
    val = flops * args.steps / el / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": sample},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------ our arm
def tf32_peak(dev, n=8192, reps=10):
    """Dense TF32 tensor-core throughput of this GPU, measured here: a torch fp32
    n x n x n matmul with TF32 allowed, best of `reps` (burst), 2 n^3 FLOPs each."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.randn((n, n), device=dev, dtype=torch.float32)
        b = torch.randn((n, n), device=dev, dtype=torch.float32)
        c = torch.empty((n, n), device=dev, dtype=torch.float32)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            torch.cuda.synchronize(dev)
            best = min(best, e0.elapsed_time(e1))
        del a, b, c
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def kernel_work(w):
    """Algorithmic FLOPs per launch of each tensor-core kernel, P = T(T+1)/2 B Hq causal
    pairs: the forward 4 D P, the backward main kernel 10 D P (S recomputed, dP, dV, dK,
    dQ)."""
    P = w.pairs * w.B * w.Hq
    return {"attn_fwd": 4 * w.D * P, "attn_bwd": 10 * w.D * P}


def step_times(step, steps, stream):
    """Runs `steps` steps with a CUDA event between consecutive steps (on the launching
    stream) and returns the per-step milliseconds."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]


def dist_stats(ms):
    """Median and 10th / 90th percentiles of per-step times (ms)."""
    xs = sorted(ms)
    q = lambda f: xs[min(len(xs) - 1, max(0, int(round(f * (len(xs) - 1)))))]
    return {"median_ms": statistics.median(xs), "p10_ms": q(0.10), "p90_ms": q(0.90), "n": len(xs)}


def flat_views(shapes, dtype, device, pinned=False):
    """One contiguous allocation holding tensors of the given shapes, each starting on a
    256-byte boundary, so that a layer's inputs (or gradients) move in one copy."""
    import math

    import torch
    al = 256 // torch.empty((), dtype=dtype).element_size()
    offs, n = [], 0
    for sh in shapes:
        offs.append(n)
        n += (math.prod(sh) + al - 1) // al * al
    buf = torch.empty(n, dtype=dtype, device=device, pin_memory=pinned)
    return buf, [buf[o:o + math.prod(sh)].view(sh) for o, sh in zip(offs, shapes)]


class LayerSet:
    """Device (and pinned host) buffers of every layer of a workload: inputs, outputs
    and one shared backward workspace, as a training step would hold them.  A layer's
    q, k, v, dO share one allocation, as do its dq, dk, dv (on the device and, for the
    end-to-end step, in pinned host memory): one copy moves each set."""

    def __init__(self, w, layers, dev, pinned: bool):
        import torch

        import causal_gqa_flash_attention_gb300 as ne
        from causal_gqa_flash_attention_gb300 import synthetic
        self.w = w
        self.host, self.devs, self.grads_host = [], [], []
        self.host_flat, self.dev_flat, self.grads_flat, self.grads_host_flat = [], [], [], []
        ws = ne.alloc_workspace(w.B, w.T, w.Hq, w.Hkv, w.D, dev)
        for L in layers:
            src = [t.contiguous() for t in synthetic.make_inputs(w, layer=L)]   # q, k, v, dO
            shapes, dt = [t.shape for t in src], src[0].dtype
            dflat, d = flat_views(shapes, dt, dev)
            for x, t in zip(d, src):
                x.copy_(t)
            self.dev_flat.append(dflat)
            if pinned:
                hflat, hq = flat_views(shapes, dt, "cpu", pinned=True)
                for x, t in zip(hq, src):
                    x.copy_(t)
                self.host.append(hq)
                self.host_flat.append(hflat)
                ghflat, gh = flat_views(shapes[:3], dt, "cpu", pinned=True)
                self.grads_host.append(gh)
                self.grads_host_flat.append(ghflat)
            o = torch.empty_like(d[0])
            lse = torch.empty((w.B, w.Hq, w.T), dtype=torch.float32, device=dev)
            gflat, (dq, dk, dv) = flat_views(shapes[:3], dt, dev)
            self.grads_flat.append(gflat)
            self.devs.append(dict(q=d[0], k=d[1], v=d[2], dO=d[3], o=o, lse=lse, ws=ws, dq=dq, dk=dk, dv=dv))

    def run_layer(self, b):
        """One layer's forward and backward: the training pair, whose forward also fills
        the layer's backward workspace (rotated queries, zeroed dQ accumulator)."""
        import causal_gqa_flash_attention_gb300 as ne
        ne.attn_fwd_train(b["q"], b["k"], b["v"], b["ws"], self.w.theta, o=b["o"], lse=b["lse"])
        ne.attn_bwd_train(b["q"], b["k"], b["v"], b["o"], b["lse"], b["dO"], b["ws"], self.w.theta,
                          dq=b["dq"], dk=b["dk"], dv=b["dv"])

    def step(self):
        for b in self.devs:
            self.run_layer(b)

    def step_l2_hot(self):
        """The same number of layers, all on layer 0's buffers (L2-resident inputs)."""
        for _ in self.devs:
            self.run_layer(self.devs[0])


def graph_step_ms(ls, stream, steps):
    """One step captured into a CUDA graph and replayed: per-replay milliseconds."""
    import torch
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        ls.step()                     # warm the side stream (no first-call work inside capture)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=side):
        ls.step()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    return step_times(g.replay, steps, torch.cuda.current_stream())


def sweep_point(wid, dev, steps, peak):
    """TFLOP/s of one sequence-sweep workload (one layer per step, inputs resident),
    with the per-kernel split from the library's phase timing."""
    import torch

    import causal_gqa_flash_attention_gb300 as ne
    from causal_gqa_flash_attention_gb300 import synthetic
    w = synthetic.WORKLOADS[wid]
    ls = LayerSet(w, [0], dev, pinned=False)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        ls.step()
    torch.cuda.synchronize(dev)
    ms = step_times(ls.step, steps, stream)
    ne.profile_enable(True)
    for _ in range(steps):
        ls.step()
    ph = ne.profile_totals()
    ne.profile_enable(False)
    st = dist_stats(ms)
    tf = w.flops() / (st["median_ms"] * 1e-3) / 1e12
    avg = lambda k: ph[k][0] / ph[k][1] if ph[k][1] else None
    kw = kernel_work(w)
    tfl = lambda k: kw[k] / (avg(k) * 1e-3) / 1e12 if avg(k) else None
    out = {"workload": w.name, "tflops": tf, "pct_of_peak": tf / peak, **st,
           "fwd_ms": avg("attn_fwd"), "bwd_main_ms": avg("attn_bwd"),
           "bwd_pre_ms": avg("bwd_pre"), "bwd_post_ms": avg("bwd_post"),
           "fwd_tflops": tfl("attn_fwd"), "bwd_main_tflops": tfl("attn_bwd")}
    del ls
    torch.cuda.empty_cache()
    return out


def prologue_point(dev, steps, peak, layers=16):
    """The fused RMSNorm -> QKV projection -> RoPE prologue at the GPU-pipeline shape
    (x [16, 512, 768] bf16, 12/4 heads of 64), one call per layer on distinct buffers:
    2 M N K FLOPs per call, M = 8192 tokens, N = 1280 features, K = 768 (the call includes
    its two small passes: the gain folded into the weights, each row's 1/rms)."""
    import torch

    import causal_gqa_flash_attention_gb300 as ne
    from causal_gqa_flash_attention_gb300 import synthetic
    B, T, dim, Hq, Hkv, D = 16, 512, 768, 12, 4, 64
    bufs = []
    for L in range(layers):
        x, g, wt = (t.to(dev) for t in synthetic.make_prologue(B, T, dim, Hq, Hkv, D, seed=200 + L))
        bufs.append((x, g, wt, torch.empty((B, T, Hq, D), dtype=torch.bfloat16, device=dev),
                     torch.empty((B, T, Hkv, D), dtype=torch.bfloat16, device=dev),
                     torch.empty((B, T, Hkv, D), dtype=torch.bfloat16, device=dev)))

    n_ws = int(ne.load().ne_qkv_prologue_workspace_size(B, T, dim, Hq, Hkv, D))
    ws = torch.empty(n_ws, dtype=torch.uint8, device=dev)      # W diag(gamma) and 1/rms, rewritten by each call

    def step():
        for x, g, wt, q, k, v in bufs:
            ne.qkv_prologue(x, g, wt, Hq, Hkv, D, rotate=True, q=q, k=k, v=v, workspace=ws)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    st = dist_stats(step_times(step, steps, torch.cuda.current_stream(dev)))
    flops = 2.0 * B * T * (Hq + 2 * Hkv) * D * dim * layers
    tf = flops / (st["median_ms"] * 1e-3) / 1e12
    del bufs
    torch.cuda.empty_cache()
    return {"workload": f"RMSNorm->QKV->RoPE prologue B{B} T{T} dim{dim} Hq{Hq} Hkv{Hkv} D{D} bf16 x{layers} layers",
            "tflops": tf, "pct_of_peak": tf / peak, "us_per_call": st["median_ms"] * 1e3 / layers, **st}


def decode_point(dev, steps, hbm_peak, layers=4):
    """The decode step of `--decode` (B8, every sequence's cache 16384 positions, Hq12/Hkv4
    D64 bf16, distinct 134 MB caches per layer), device-timed only, so that every default
    run also measures the decode kernel: cache-read GB/s against the HBM copy peak."""
    import torch

    import causal_gqa_flash_attention_gb300 as ne
    from causal_gqa_flash_attention_gb300 import synthetic
    B, T, Hq, Hkv, D = 8, 16384, 12, 4, 64
    bufs = []
    for i in range(layers):
        q, k, v, lens = synthetic.make_decode(B, T, Hq, Hkv, D, torch.bfloat16, seed=100 + i, lens=[T] * B)
        bufs.append((q.to(dev), k.to(dev), v.to(dev), lens.to(dev), torch.empty_like(q, device=dev),
                     torch.empty((B, Hq), dtype=torch.float32, device=dev)))
    ws = torch.empty(max(ne.decode_workspace_size(B, T, Hq, Hkv, D), 256), dtype=torch.uint8, device=dev)

    def step():
        for q, k, v, lens, o, lse in bufs:
            ne.attn_decode(q, k, v, lens, o=o, lse=lse, workspace=ws)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    st = dist_stats(step_times(step, steps, torch.cuda.current_stream(dev)))
    per_layer = B * T * Hkv * D * 2 * 2 + 2 * B * Hq * D * 2 + B * Hq * 4
    gbs = per_layer * layers / (st["median_ms"] * 1e-3) / 1e9
    del bufs
    torch.cuda.empty_cache()
    return {"workload": f"decode B{B} T_max{T} Hq{Hq} Hkv{Hkv} D{D} bf16 x{layers} layers",
            "gbs": gbs, "pct_of_hbm": gbs / hbm_peak, "us_per_layer": st["median_ms"] * 1e3 / layers, **st}


def run_ours(args, w):
    import torch

    import causal_gqa_flash_attention_gb300 as ne
    from causal_gqa_flash_attention_gb300 import _build

    hz = Harness("nccl")
    torch.cuda.set_device(hz.local_rank)
    dev = torch.device("cuda", hz.local_rank)
    if hz.local_rank == 0:
        _build.build()
    hz.barrier()
    ne.load()
    layers = shard_layers(w.layers, hz.world, hz.rank)
    if args.bare:
        run_bare(args, w, dev)
        hz.close()
        return

    # Inputs resident in HBM (device arm) and pinned host copies (end-to-end arm).  The
    # backward scratch (Delta and the fp32 dQ accumulator) is one buffer for all layers,
    # as a training step would allocate it; every layer has its own inputs and outputs.
    ls = LayerSet(w, layers, dev, pinned=True)
    devs, host, grads_host = ls.devs, ls.host, ls.grads_host
    stream = torch.cuda.current_stream(dev)
    step = ls.step

    # End-to-end step: every layer's inputs go host -> device on a copy stream (one copy:
    # q, k, v, dO share an allocation), its forward and backward run on the compute
    # stream, and its gradients go device -> host on a third stream (one copy), so the
    # copies of one layer overlap the kernels of its neighbours.
    # Events keep each layer's buffers safe: an input is overwritten only after the
    # previous step's kernels of that layer consumed it, a gradient only after the previous
    # step's copy-out of it finished.
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in devs]
    ev_comp = [torch.cuda.Event() for _ in devs]
    ev_out = [torch.cuda.Event() for _ in devs]
    for e in ev_comp + ev_out:
        e.record(stream)

    def step_e2e():
        for i, b in enumerate(devs):
            with torch.cuda.stream(h2d_s):
                h2d_s.wait_event(ev_comp[i])
                ls.dev_flat[i].copy_(ls.host_flat[i], non_blocking=True)
                ev_in[i].record(h2d_s)
            stream.wait_event(ev_in[i])
            stream.wait_event(ev_out[i])
            ls.run_layer(b)
            ev_comp[i].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_comp[i])
                ls.grads_host_flat[i].copy_(ls.grads_flat[i], non_blocking=True)
                ev_out[i].record(d2h_s)

    # Clocks are sampled from the warm-up through the last extra measurement, so the
    # timed region lies inside the sampled window.
    clocks = ClockSampler(hz.local_rank)
    clocks.start()
    clocks.wait_first()
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if ne.get_device_error() != ne.NE_OK:
        raise RuntimeError("device error during warm-up: " + ne.last_error())

    # Per-kernel durations come from the library's phase timing (CUDA events recorded on
    # the launching stream around each kernel).  With --phase-timing timed they cover the
    # timed region itself; with "separate" the timed region runs bare and the same
    # number of profiled steps follows it.  One profiled step first grows the event pool,
    # so profiled regions only record events.
    ne.profile_enable(True)
    step()
    torch.cuda.synchronize(dev)
    ne.profile_enable(args.phase_timing == "timed")
    hz.barrier()
    torch.cuda.synchronize(dev)
    # The timed region: exactly K steps, one CUDA event between consecutive steps, so the
    # per-step distribution comes from the same run as the mean.
    per_step = step_times(step, args.steps, stream)
    hz.barrier()
    ms_local = sum(per_step) / args.steps
    if args.phase_timing == "separate":
        ne.profile_enable(True)
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize(dev)
    phases = ne.profile_totals()
    ne.profile_enable(False)
    if ne.get_device_error() != ne.NE_OK:
        raise RuntimeError("device error during timing: " + ne.last_error())
    ms = hz.max(ms_local, dev)

    # Beside the eager number: the same step replayed from a CUDA graph, and an L2-hot
    # step whose layers all reuse layer 0's buffers (labelled: not the headline).
    extra_steps = max(args.steps, 50)
    graph_ms = graph_step_ms(ls, stream, extra_steps)
    for _ in range(3):
        ls.step_l2_hot()
    hot_ms = step_times(ls.step_l2_hot, extra_steps, stream)

    # End-to-end: host buffers, H2D of the inputs and D2H of the gradients inside the step.
    for _ in range(2):
        step_e2e()
    torch.cuda.synchronize(dev)
    hz.barrier()
    e2 = max(2, args.steps // 2)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    h2d_s.wait_stream(stream)
    d2h_s.wait_stream(stream)
    for _ in range(e2):
        step_e2e()
    stream.wait_stream(h2d_s)
    stream.wait_stream(d2h_s)
    g1.record(stream)
    torch.cuda.synchronize(dev)
    hz.barrier()
    e2e_ms = hz.max(g0.elapsed_time(g1) / e2, dev)

    peaks = measured_peaks()
    tf32 = tf32_peak(dev) if w.dtype == "f32" or not args.no_sweep else None
    # The sequence-length sweep points at T >= 2048 (one layer per step, resident inputs)
    # ride along in the default line so that a long-sequence number exists for every run.
    sweep = {}
    if not args.no_sweep and w.wid == 2:
        for wid in (52, 53, 54):
            sweep[f"T{synthetic_T(wid)}"] = sweep_point(wid, dev, 10, peaks["bf16_tflops"])
    # The step before attention (not part of the headline step): the fused prologue.
    prologue = prologue_point(dev, 20, peaks["bf16_tflops"]) if not args.no_sweep and w.wid == 2 else None
    decode = decode_point(dev, 20, peaks["hbm_gbs"]) if not args.no_sweep and w.wid == 2 else None
    clk = clocks.stop()

    flops_step = w.flops() * len(layers)
    total_flops = flops_step * hz.world
    value = total_flops / (ms * 1e-3) / 1e12
    e2e_val = total_flops / (e2e_ms * 1e-3) / 1e12
    es = 2 if w.dtype == "bf16" else 4
    h2d = sum(f.numel() * es for f in ls.host_flat)
    d2h = sum(f.numel() * es for f in ls.grads_host_flat)

    # The peak of the path's own dtype: bf16 for bf16 tensors, the TF32 rate measured
    # above for fp32 tensors (they run on TF32 tensor cores).
    peak = peaks["bf16_tflops"] if w.dtype == "bf16" else tf32
    peak_name = "bf16 burst" if w.dtype == "bf16" else "tf32 burst (torch fp32 matmul 8192^3, TF32 on, measured here)"
    # Per-kernel averages over the timed region; the dominant kernel is the one with the
    # largest share.  Algorithmic FLOPs per launch: forward 4 D P, backward main 10 D P
    # with P = T(T+1)/2 B Hq; bytes per launch (HBM-bound preprocess/epilogue) from
    # compulsory_bytes().
    avg = {k: (v[0] / v[1] if v[1] else 0.0) for k, v in phases.items()}
    total = sum(v[0] for v in phases.values()) or 1.0
    share = {k: v[0] / total for k, v in phases.items()}
    cb = w.compulsory_bytes()
    acc_bytes = w.B * w.T * w.Hq * w.D * 4
    # The preprocess pass of the training pair: Delta from O and dO; for bf16 head_dim <= 64
    # the training forward already stored R Q and zeroed the dQ accumulator, otherwise the
    # pass zeroes the accumulator (and, bf16, reads Q and writes fp16 R Q) itself.
    prepared = w.dtype == "bf16" and w.D <= 64
    pre_bytes = cb["pre"] + (0 if prepared else acc_bytes + (2 * w.B * w.T * w.Hq * w.D * es if w.dtype == "bf16" else 0))
    kw = kernel_work(w)
    tfl = lambda k: kw[k] / (avg[k] * 1e-3) / 1e12 if avg[k] else None
    kernels = {
        "attn_fwd": {"ms": avg["attn_fwd"], "share": share["attn_fwd"], "bound": "tensor",
                     "achieved": tfl("attn_fwd"), "unit": "TFLOP/s"},
        "attn_bwd": {"ms": avg["attn_bwd"], "share": share["attn_bwd"], "bound": "tensor",
                     "achieved": tfl("attn_bwd"), "unit": "TFLOP/s"},
        "bwd_pre": {"ms": avg["bwd_pre"], "share": share["bwd_pre"], "bound": "hbm",
                    "achieved": pre_bytes / (avg["bwd_pre"] * 1e-3) / 1e9 if avg["bwd_pre"] else None,
                    "unit": "GB/s"},
        "bwd_post": {"ms": avg["bwd_post"], "share": share["bwd_post"], "bound": "hbm",
                     "achieved": (acc_bytes + w.B * w.T * w.Hq * w.D * es) / (avg["bwd_post"] * 1e-3) / 1e9
                     if avg["bwd_post"] else None, "unit": "GB/s"},
    }
    kernels = {k: v for k, v in kernels.items() if phases[k][1]}   # the kernels this path launches
    for k in kernels:
        kernels[k]["launches"] = phases[k][1]
    dom = max(kernels, key=lambda k: kernels[k]["share"])
    dk = kernels[dom]
    dom_peak = peak if dk["unit"] == "TFLOP/s" else peaks["hbm_gbs"]
    bwd_main_src = "attn_bwd_d64.cu" if (w.dtype == "bf16" and w.D == 64) else \
        ("attn_bwd_tf32.cu" if w.dtype == "f32" else "attn_bwd.cu")
    src = {"attn_fwd": "attn_fwd.cu", "attn_bwd": bwd_main_src, "bwd_pre": "attn_bwd.cu", "bwd_post": "attn_bwd.cu"}[dom]
    traffic = profiled_traffic(os.path.join(ROOT, "causal_gqa_flash_attention_gb300", "csrc", src), f"{dom}:{w.name}")
    st = dist_stats(per_step)
    gst, hst = dist_stats(graph_ms), dist_stats(hot_ms)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": hz.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded N(0,1), layer-distinct buffers)",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "layers_per_step": len(layers), "rope_theta": w.theta,
                   "l2": f"inputs larger than L2: {len(layers)} distinct layer buffer sets "
                         f"({sum(b['q'].numel() + b['k'].numel() * 2 + b['dO'].numel() for b in devs) * es / 1e6:.0f} MB of inputs); "
                         f"one shared backward workspace",
                   "parallelism": f"replicas x{hz.world}"},
        "pct_of_peak": value / hz.world / peak,
        "timing": {
            "eager": {**st, "tflops_at_median": flops_step / (st["median_ms"] * 1e-3) / 1e12,
                      "what": "the timed region: per-step CUDA events, layer-distinct buffers"},
            "graph": {**gst, "tflops_at_median": flops_step / (gst["median_ms"] * 1e-3) / 1e12,
                      "what": "one step captured in a CUDA graph, replayed"},
            "l2_hot": {**hst, "tflops_at_median": flops_step / (hst["median_ms"] * 1e-3) / 1e12,
                       "what": "L2-HOT, not the headline: every layer on layer 0's buffers"},
        },
        "roofline": {"kernel": dom, "bound": dk["bound"], "achieved": dk["achieved"], "peak": dom_peak,
                     "unit": dk["unit"], "frac": dk["achieved"] / dom_peak,
                     "peak_source": (f"{peaks['source']} " + peak_name) if dk["unit"] == "TFLOP/s"
                     else f"{peaks['source']} HBM copy",
                     "traffic": traffic, "per_launch_ms": dk["ms"],
                     "timing": ("CUDA events around every launch over the timed region" if args.phase_timing == "timed"
                                else f"CUDA events around every launch over {args.steps} steps run right after "
                                     "the timed region (same work, same stream)")},
        "kernels": kernels,
        "peaks": {"bf16_tflops": peaks["bf16_tflops"], "hbm_gbs": peaks["hbm_gbs"], "tf32_tflops_measured": tf32,
                  "source": peaks["source"]},
        "sweep": sweep,
        "prologue": prologue,
        "decode": decode,
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "gpu_launches": sum(v[1] for v in phases.values()),
        "clocks": clk,
    }
    if hz.rank == 0 and not args.no_cpu_baseline and hz.world == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    elif hz.rank == 0 and hz.world == 1:
        line["cpu_baseline"] = None
    if hz.rank == 0:
        print(json.dumps(line), flush=True)
    hz.close()


def run_bare(args, w, dev):
    """--bare: warm-up, then K steps of layer 0 of the workload, and one short line.
    This is the command the ncu captures run (few launches, nothing else)."""
    import torch

    import causal_gqa_flash_attention_gb300 as ne
    ls = LayerSet(w, [0], dev, pinned=False)
    for _ in range(args.warmup):
        ls.step()
    torch.cuda.synchronize(dev)
    ms = step_times(ls.step, args.steps, torch.cuda.current_stream(dev))
    ne.profile_enable(True)
    for _ in range(args.steps):
        ls.step()
    ph = ne.profile_totals()
    ne.profile_enable(False)
    if ne.get_device_error() != ne.NE_OK:
        raise RuntimeError("device error: " + ne.last_error())
    st = dist_stats(ms)
    per_kernel = {k: v[0] / v[1] for k, v in ph.items() if v[1]}
    print(json.dumps({"bare": True, "workload": w.name, **st,
                      "tflops_at_median": w.flops() / (st["median_ms"] * 1e-3) / 1e12,
                      "kernel_ms": per_kernel}), flush=True)


def synthetic_T(wid):
    from causal_gqa_flash_attention_gb300 import synthetic
    return synthetic.WORKLOADS[wid].T


# ------------------------------------------------------------------ decode step
DECODE_METRIC = "decode over a KV cache: cache-read GB/s (B8 T16384 Hq12/Hkv4 D64 bf16, 4 layers)"


def run_decode(args):
    """--decode: one decode step per layer (each sequence's newest token attends to its
    whole cache) over 4 layers with distinct caches of 134 MB each, so a step streams
    537 MB from HBM (more than L2).  Algorithmic bytes: the cache rows each step must
    read (sum of lengths x Hkv x D x 2 tensors) plus q, o and lse.  The kernel time is
    that of the chunk kernel and the merge of the chunks together (the merge moves
    under 2% of the bytes)."""
    import torch

    import causal_gqa_flash_attention_gb300 as ne
    from causal_gqa_flash_attention_gb300 import _build

    B, T, Hq, Hkv, D, L = 8, 16384, 12, 4, 64, 4
    hz = Harness("nccl")
    torch.cuda.set_device(hz.local_rank)
    dev = torch.device("cuda", hz.local_rank)
    if hz.local_rank == 0:
        _build.build()
    hz.barrier()
    ne.load()
    from causal_gqa_flash_attention_gb300 import synthetic
    layers, host = [], []
    for i in range(L):
        q, k, v, lens = synthetic.make_decode(B, T, Hq, Hkv, D, torch.bfloat16, seed=100 + i, lens=[T] * B)
        hq = q.pin_memory()
        host.append((hq, lens.pin_memory(), torch.empty_like(q).pin_memory(),
                     torch.empty((B, Hq), dtype=torch.float32).pin_memory()))
        layers.append(dict(q=q.to(dev), k=k.to(dev), v=v.to(dev), lens=lens.to(dev), o=torch.empty_like(q, device=dev),
                           lse=torch.empty((B, Hq), dtype=torch.float32, device=dev)))
    ws = torch.empty(max(ne.decode_workspace_size(B, T, Hq, Hkv, D), 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        for b in layers:
            ne.attn_decode(b["q"], b["k"], b["v"], b["lens"], o=b["o"], lse=b["lse"], workspace=ws)

    def step_e2e():
        for b, (hq, hl, ho, hlse) in zip(layers, host):
            b["q"].copy_(hq, non_blocking=True)
            b["lens"].copy_(hl, non_blocking=True)
            ne.attn_decode(b["q"], b["k"], b["v"], b["lens"], o=b["o"], lse=b["lse"], workspace=ws)
            ho.copy_(b["o"], non_blocking=True)
            hlse.copy_(b["lse"], non_blocking=True)

    clocks = ClockSampler(hz.local_rank)
    clocks.start()
    clocks.wait_first()
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if ne.get_device_error() != ne.NE_OK:
        raise RuntimeError("device error during warm-up: " + ne.last_error())
    hz.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    hz.barrier()
    ms = hz.max(e0.elapsed_time(e1) / args.steps, dev)
    for _ in range(2):
        step_e2e()
    torch.cuda.synchronize(dev)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        step_e2e()
    g1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    e2e_ms = hz.max(g0.elapsed_time(g1) / args.steps, dev)
    if ne.get_device_error() != ne.NE_OK:
        raise RuntimeError("device error during timing: " + ne.last_error())

    es = 2
    per_layer = B * T * Hkv * D * es * 2 + 2 * B * Hq * D * es + B * Hq * 4
    byts = per_layer * L * hz.world
    value = byts / (ms * 1e-3) / 1e9
    peaks = measured_peaks()
    plan_ws = ne.decode_workspace_size(B, T, Hq, Hkv, D)
    line = {
        "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": hz.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in, f32 arithmetic", "data": "synthetic (seeded N(0,1) caches, every sequence full)",
        "config": {"workload": f"decode B{B} T_max{T} Hq{Hq} Hkv{Hkv} D{D} bf16 x{L} layers", "seq_lens": T,
                   "l2": f"inputs larger than L2: {L} distinct caches of {per_layer / 1e6:.0f} MB",
                   "workspace_bytes": plan_ws, "parallelism": f"replicas x{hz.world}"},
        "roofline": {"kernel": "attn_decode (chunk kernel + merge)", "bound": "hbm",
                     "achieved": per_layer / (ms / L * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": per_layer / (ms / L * 1e-3) / 1e9 / peaks["hbm_gbs"],
                     "peak_source": f"{peaks['source']} HBM copy", "traffic": None,
                     "per_launch_ms": ms / L, "timing": "CUDA events around the timed steps (2 launches per layer)"},
        "e2e": {"value": byts / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": L * (B * Hq * D * es + B * 4),
                "d2h_bytes_per_step": L * (B * Hq * D * es + B * Hq * 4), "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * L * (2 if plan_ws else 1),
        "clocks": clk,
    }
    if hz.rank == 0:
        print(json.dumps(line), flush=True)
    hz.close()


def main():
    args = parse()
    from causal_gqa_flash_attention_gb300 import synthetic
    w = synthetic.WORKLOADS[args.workload]
    if args.decode and args.impl == "ours":
        run_decode(args)
        return
    if args.prologue and args.impl == "ours":
        import torch

        import causal_gqa_flash_attention_gb300 as ne
        from causal_gqa_flash_attention_gb300 import _build
        _build.build()
        ne.load()
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
        torch.cuda.set_device(dev)
        line = prologue_point(dev, args.steps, measured_peaks()["bf16_tflops"])
        if ne.get_device_error() != ne.NE_OK:
            raise RuntimeError("device error: " + ne.last_error())
        print(json.dumps({"prologue": True, **line}), flush=True)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
