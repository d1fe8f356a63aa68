"""Benchmark of the fused MoE layer on GB300.

One step = one moe_forward (align, Gate-Up, SiLU-and-mul, Down, combine) over
one batch of the Mixtral-8x7B-shaped bf16 layer (H=4096, I=14336, E=8, k=2)
at T tokens (default 64, the top of the decode range), inputs resident in HBM.
L2 is flushed (a write of 2x the L2 size) before every timed step and every
step is timed with CUDA events on the launching stream, as the SGLang MoE
tuning guide (section 2.5) does.  Steps replay a CUDA graph of one
moe_forward so that host launch cost is not measured.

The JSON line reports the layer latency (us), the roofline fractions, the
dominant kernel's achieved HBM bandwidth (per-stage CUDA events), the sweep
over the workload's other token counts, an end-to-end number through host
buffers, the oracle timed on the host cores, and the SM clocks sampled during
the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--T 64] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "MoE layer µs & HBM GB/s vs 8 TB/s at T=1–64; TFLOP/s vs peak at T≥1024"
CFG = 2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_SOURCES = ("k_gemm.cuh", "k_gemm_bf16.cu", "k_gemm_bf16_direct.cu", "ptx.cuh")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def gemm_source_hash() -> str:
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        h.update(open(os.path.join(ROOT, "moe_expert_layer_align_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, T: int):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(f"{kernel}@T={T}")
    if not e or e.get("source_hash") != gemm_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        pw = np.array([r[2] for r in rows])
        load = [r for r in rows if r[2] >= np.percentile(pw, 50)] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3][1:5]) if v == "Active"})
        return {"sm_mhz": float(np.median([r[0] for r in load])),
                "sm_max_mhz": float(max(r[1] for r in rows)), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(load)}


# ---------------------------------------------------------------- workload

def layer_numbers(wl):
    """Algorithmic bytes and FLOPs of one layer invocation (routed work only)."""
    ids = wl.topk_ids.cpu().numpy()
    U = len(np.unique(ids))
    T, H, I, k = wl.T, wl.H, wl.I, wl.k
    wbytes = 3 * H * I * 2 * U
    io = T * H * 2 + T * k * 8 + T * H * 2
    return dict(U=U, weight_bytes=wbytes, bytes=wbytes + io, flops=6 * T * k * H * I,
                gateup_bytes=2 * I * H * 2 * U + T * H * 2,
                down_bytes=H * I * 2 * U + T * H * 2)


def make_workload(T, device, weights=None):
    from moe_expert_layer_align_gb300 import workloads
    if weights is None:
        return workloads.make(CFG, T, device)
    c = workloads.CONFIGS[CFG]
    g = torch.Generator(device=device)
    g.manual_seed(1000 * CFG + T)
    x = torch.randn((T, c["H"]), generator=g, device=device).bfloat16()
    ids, w = workloads.synth_routing(T, c["E"], c["k"], c["routing"], c["scale"], g, device)
    return workloads.Workload(name=c["name"], T=T, H=c["H"], I=c["I"], E=c["E"], k=c["k"],
                              mode="bf16", out="bf16", x=x, w13=weights[0], w2=weights[1],
                              topk_ids=ids, topk_w=w, meta=dict(config=CFG))


class Layer:
    """One moe_forward on fixed buffers, captured in a CUDA graph."""

    def __init__(self, wl, stream, opts=None, graph=True):
        import moe_expert_layer_align_gb300 as moe
        self.moe, self.wl, self.stream, self.opts = moe, wl, stream, opts
        shape = moe.layer_shape(wl.x, wl.w13, wl.topk_ids, 0, torch.bfloat16)
        self.ws = torch.empty(moe.moe_workspace_bytes(shape, opts), dtype=torch.uint8, device="cuda")
        self.out = torch.empty(wl.x.shape, dtype=torch.bfloat16, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.graph = None
        if graph:
            with torch.cuda.stream(stream):
                self.call()                       # warm the launch path before capture
            stream.synchronize()
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=stream):
                self.call()
            stream.synchronize()

    def call(self):
        wl = self.wl
        self.moe.moe_forward(wl.x, wl.w13, wl.w2, wl.topk_ids, wl.topk_w, out=self.out,
                             workspace=self.ws, dev_status=self.status, stream=self.stream,
                             opts=self.opts)

    def run(self):
        # replay() launches on the current stream: make it ours
        with torch.cuda.stream(self.stream):
            if self.graph is not None:
                self.graph.replay()
            else:
                self.call()


def time_layer(layer, stream, flush, steps, warmup):
    for _ in range(warmup):
        with torch.cuda.stream(stream):
            flush.zero_()
        layer.run()
    stream.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    t0 = time.perf_counter()
    for s, e in evs:
        with torch.cuda.stream(stream):
            flush.zero_()
            s.record(stream)
        layer.run()
        e.record(stream)
    stream.synchronize()
    wall = time.perf_counter() - t0
    return np.array([s.elapsed_time(e) * 1e3 for s, e in evs]), wall  # us


def stage_times(wl, stream, flush, steps):
    """Per-stage device time (us) from events recorded between the stages,
    captured with the layer in a CUDA graph (recording events between stages
    serialises them: PDL overlap is lost in this pass)."""
    import moe_expert_layer_align_gb300 as moe
    n = len(moe.STAGES) + 1
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for ev in evs:                  # torch creates the CUDA event on first record
        ev.record(stream)
    layer = Layer(wl, stream, opts=moe.make_opts(stage_events=evs), graph=True)
    acc = np.zeros(n - 1)
    for _ in range(steps):
        with torch.cuda.stream(stream):
            flush.zero_()
        layer.run()
        stream.synchronize()
        for i in range(n - 1):
            acc[i] += evs[i].elapsed_time(evs[i + 1]) * 1e3
    return dict(zip(moe.STAGES, (acc / steps).tolist()))


def e2e_time(wl, stream, steps, warmup):
    """moe_forward through the public API with host (pinned) inputs and result:
    H2D of x / topk ids / topk weights, the layer, D2H of the output."""
    import moe_expert_layer_align_gb300 as moe
    hx = wl.x.cpu().pin_memory()
    hid = wl.topk_ids.cpu().pin_memory()
    hw = wl.topk_w.cpu().pin_memory()
    hout = torch.empty(wl.x.shape, dtype=torch.bfloat16).pin_memory()
    dx, did, dw = torch.empty_like(wl.x), torch.empty_like(wl.topk_ids), torch.empty_like(wl.topk_w)
    shape = moe.layer_shape(wl.x, wl.w13, wl.topk_ids, 0, torch.bfloat16)
    ws = torch.empty(moe.moe_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    out = torch.empty(wl.x.shape, dtype=torch.bfloat16, device="cuda")

    def step():
        with torch.cuda.stream(stream):
            dx.copy_(hx, non_blocking=True)
            did.copy_(hid, non_blocking=True)
            dw.copy_(hw, non_blocking=True)
            moe.moe_forward(dx, wl.w13, wl.w2, did, dw, out=out, workspace=ws, stream=stream)
            hout.copy_(out, non_blocking=True)

    for _ in range(warmup):
        step()
    stream.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        step()
    e.record(stream)
    stream.synchronize()
    us = s.elapsed_time(e) * 1e3 / steps
    return {"value": us, "unit": "us",
            "h2d_bytes_per_step": hx.numel() * 2 + hid.numel() * 4 + hw.numel() * 4,
            "d2h_bytes_per_step": hout.numel() * 2}


def oracle_baseline(wl, budget_s=15.0, max_tokens=None):
    """The oracle on the host cores over a bounded sample of the batch's
    tokens; latency scaled to the whole batch."""
    import oracle
    from tests.helpers import bits16
    x = bits16(wl.x)
    w13 = bits16(wl.w13)
    w2 = bits16(wl.w2)
    ids = wl.topk_ids.cpu().numpy()
    w = wl.topk_w.cpu().numpy()
    t0 = time.perf_counter()
    oracle.moe_bf16(x, w13, w2, ids, w, np.array([0], np.int32))
    one = time.perf_counter() - t0
    n = int(max(1, min(wl.T, budget_s // max(one, 1e-6))))
    if max_tokens:
        n = min(n, max_tokens)
    sel = np.linspace(0, wl.T - 1, n).astype(np.int32)
    t0 = time.perf_counter()
    oracle.moe_bf16(x, w13, w2, ids, w, sel)
    dt = time.perf_counter() - t0
    return {"value": dt / n * wl.T * 1e6, "unit": "us", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{n} of {wl.T} tokens of the T={wl.T} batch (fp64 C oracle, OpenMP); "
                      f"measured {dt:.2f} s, scaled x{wl.T}/{n}"}


# ---------------------------------------------------------------- arms

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    wl = make_workload(args.T, "cpu")
    for _ in range(args.warmup):
        oracle_baseline(wl, budget_s=0, max_tokens=1)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(oracle_baseline(wl, budget_s=5.0)["value"])
    wall = time.perf_counter() - t0
    cb = oracle_baseline(wl, budget_s=5.0)
    v = float(np.mean(vals))
    import oracle
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "us", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"mixtral-8x7b-bf16 MoE layer T={args.T}", "T": args.T,
                       "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k, "l2": "n/a (host)"},
            "cpu_baseline": {"value": v, "unit": "us", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": cb["sample"]},
            "e2e": {"value": v, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)


def run_cuda(args):
    import moe_expert_layer_align_gb300 as moe  # noqa: F401  (loads the CUDA library)
    ws_, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws_ > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pk, pk_kind = peaks()
    stream = torch.cuda.Stream()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device="cuda")

    wl = make_workload(args.T, "cuda")
    weights = (wl.w13, wl.w2)
    nums = layer_numbers(wl)
    layer = Layer(wl, stream)

    def barrier():
        if ws_ > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    clk = ClockSampler(local).__enter__()
    barrier()
    times, wall = time_layer(layer, stream, flush, args.steps, args.warmup)
    barrier()
    us = float(np.mean(times))
    if ws_ > 1:
        t = torch.tensor([us], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        us = float(t.item())
    st = int(layer.status.item())

    result = None
    if rank == 0:
        stg = stage_times(wl, stream, flush, max(3, min(args.steps, 10)))
        t_bytes = nums["bytes"] / (pk["hbm_gbs"] * 1e9) * 1e6
        t_flops = nums["flops"] / (pk["bf16_tflops"] * 1e12) * 1e6
        gu_us = stg["gateup"]
        achieved = nums["gateup_bytes"] / (gu_us * 1e-6) / 1e9
        roof = {"bound": "hbm", "kernel": "moe_gemm_kernel<bf16, gather> (Gate-Up)",
                "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "peak_kind": f"{pk_kind} burst copy",
                "traffic": ncu_traffic("gateup", args.T),
                "algorithmic_bytes_per_launch": nums["gateup_bytes"],
                "launch_us": gu_us}
        sweep = []
        if not args.no_sweep:
            for T in (1, 2, 4, 8, 16, 32, 64, 128, 512, 2048):
                w2l = make_workload(T, "cuda", weights)
                n2 = layer_numbers(w2l)
                L2 = Layer(w2l, stream)
                tt, _ = time_layer(L2, stream, flush, 20, 3)
                u = float(np.median(tt))
                tb = n2["bytes"] / (pk["hbm_gbs"] * 1e9) * 1e6
                tf = n2["flops"] / (pk["bf16_tflops"] * 1e12) * 1e6
                sweep.append({"T": T, "us": u, "active_experts": n2["U"],
                              "hbm_gbs": n2["bytes"] / (u * 1e-6) / 1e9,
                              "tflops": n2["flops"] / (u * 1e-6) / 1e12,
                              "bound": "hbm" if tb >= tf else "tensor",
                              "roofline_frac": max(tb, tf) / u})
                del L2, w2l
        e2e = e2e_time(wl, stream, max(args.steps, 5), args.warmup)
        clk.__exit__()
        clocks = clk.summary()
        clocks["window"] = "timed region, stage pass, sweep and e2e pass"
        cpu = None if args.no_cpu else oracle_baseline(wl.to("cpu"))
        result = {
            "metric": METRIC, "value": us, "unit": "us", "n_gpus": ws_, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; random-init Mixtral-8x7B-shaped experts)",
            "config": {"workload": f"mixtral-8x7b-bf16 MoE layer T={args.T}", "T": args.T,
                       "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                       "active_experts": nums["U"], "replicas": ws_,
                       "l2": f"flushed before every step ({flush.numel() >> 20} MiB write)",
                       "timing": "CUDA graph of one moe_forward, CUDA events per step"},
            "layer": {"us_median": float(np.median(times)), "us_p10": float(np.percentile(times, 10)),
                      "us_p90": float(np.percentile(times, 90)),
                      "hbm_gbs": nums["bytes"] / (us * 1e-6) / 1e9,
                      "tflops": nums["flops"] / (us * 1e-6) / 1e12,
                      "roofline_frac": max(t_bytes, t_flops) / us,
                      "bound": "hbm" if t_bytes >= t_flops else "tensor",
                      "algorithmic_bytes": nums["bytes"], "flops": nums["flops"],
                      "dev_status": st},
            "stages_us": stg,
            "roofline": roof,
            "sweep": sweep,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "gpu_launches": 5 * args.steps,
            "wall_s_timed_region": wall,
        }
        print(json.dumps(result), flush=True)
    else:
        clk.__exit__()
    if ws_ > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return result


def run_ncu(args):
    """Profiler mode: W + K plain moe_forward calls on the workload, nothing
    else on the GPU (no graphs, flush, sweep or oracle).  Not a bench line."""
    import moe_expert_layer_align_gb300 as moe  # noqa: F401
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    wl = make_workload(args.T, "cuda")
    layer = Layer(wl, stream, graph=False)
    for _ in range(args.warmup + args.steps):
        layer.run()
    stream.synchronize()
    print(json.dumps({"ncu_mode": True, "T": args.T, "calls": args.warmup + args.steps,
                      "dev_status": int(layer.status.item())}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--T", type=int, default=64)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--ncu", action="store_true", help="profiler mode (no bench line)")
    args = ap.parse_args()
    if args.ncu:
        return run_ncu(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
