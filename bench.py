"""Benchmark of the fused MoE layer on GB300.

One step = one pass of the layer (align, [x-quant], Gate-Up, SiLU-and-mul,
Down, combine; the router first where it is in the path) over one batch of a
workload of moe_expert_layer_align_gb300.workloads, inputs resident in HBM.
Default: the Mixtral-8x7B-shaped bf16 layer (H=4096, I=14336, E=8, k=2) at
T=64, the top of the decode range; --config/--T pick another.
L2 is flushed (a write of 2x the L2 size) before every timed step and every
step is timed with CUDA events on the launching stream, as the SGLang MoE
tuning guide (section 2.5) does.  Steps replay a CUDA graph of one
moe_forward so that host launch cost is not measured.

The JSON line reports the layer latency (us), the roofline fractions, the
dominant kernel's achieved HBM bandwidth (per-stage CUDA events), the sweep
over the workload's other token counts, the other workloads at their first
decode size and largest token count ("workloads": latency, roofline
fraction, Gate-Up bandwidth, oracle baseline each), an end-to-end number
through host buffers, the oracle timed on the host cores, and the SM clocks
sampled during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 2] [--T 64]
                  [--impl reference] [--no-sweep] [--no-workloads] [--no-cpu] [--ncu]
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
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_SOURCES = ("k_gemm.cuh", "k_gemm_bf16.cu", "k_gemm_bf16_direct.cu", "k_gemm_fp8.cu",
                "ptx.cuh", "index_build.cuh")


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


def record_traffic(csv_path: str, cfg: int, T: int, command: str):
    """Store the DRAM bytes per launch of the expert GEMMs from an ncu capture
    (exported with `ncu -i <report> --page raw --csv > <csv_path>`) in
    profiles/traffic.json, keyed by workload and stage and stamped with the
    hash of the GEMM sources it was taken on."""
    import csv
    rows = list(csv.reader(open(csv_path)))
    hdr, data = rows[0], rows[2:]
    col = {h: i for i, h in enumerate(hdr)}
    stage_of = {"0": "gateup", "1": "down", "2": "router"}
    p = os.path.join(ROOT, "profiles", "traffic.json")
    d = json.load(open(p)) if os.path.exists(p) else {}
    d["_what"] = ("DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the "
                  "expert GEMMs from ncu --set full captures; source_hash covers the GEMM "
                  "sources each was taken on (bench.py reports null for a stale one).")
    for r in data:
        name = r[col["Kernel Name"]]
        if "moe_gemm_kernel" not in name:
            continue
        targs = name[name.index("<") + 1: name.index(">")].replace(" ", "").split(",")
        stage = stage_of.get(targs[2], "gemm")
        rd = float(r[col["dram__bytes_read.sum"]].replace(",", ""))
        wr = float(r[col["dram__bytes_write.sum"]].replace(",", ""))
        unit_r, unit_w = rows[1][col["dram__bytes_read.sum"]], rows[1][col["dram__bytes_write.sum"]]
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
        rd *= scale.get(unit_r, 1)
        wr *= scale.get(unit_w, 1)
        dur = float(r[col["gpu__time_duration.sum"]].replace(",", ""))
        dur *= {"ns": 1, "nsecond": 1, "us": 1e3, "usecond": 1e3, "ms": 1e6,
                "msecond": 1e6}.get(rows[1][col["gpu__time_duration.sum"]], 1)
        d[f"c{cfg}:{stage}@T={T}"] = {
            "kernel": name.split("(")[0].replace("void ", ""),
            "source_hash": gemm_source_hash(), "duration_ns": dur,
            "dram_bytes_read": int(rd), "dram_bytes_write": int(wr),
            "dram_bytes_per_launch": int(rd + wr), "command": command}
    json.dump(d, open(p, "w"), indent=1, sort_keys=True)
    print(json.dumps({k: v for k, v in d.items() if k.startswith(f"c{cfg}:")}, indent=1))


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float) -> float:
    """The largest of every rank's `x` (each rank times its own replica; the
    step takes as long as the slowest).  One process: `x` itself."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


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

def layer_numbers(wl, topk_ids):
    """Algorithmic bytes and FLOPs of one layer invocation (routed work only;
    the method's own intermediates are overhead, not credited)."""
    ids = topk_ids.cpu().numpy()
    U = len(np.unique(ids))
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    bw = 2 if wl.mode == "bf16" else 1
    scales13 = 0 if wl.mode == "bf16" else 4 * (2 * I // 128) * (H // 128)
    scales2 = 0 if wl.mode == "bf16" else 4 * (H // 128) * (I // 128)
    w13_bytes = U * (2 * I * H * bw + scales13)
    w2_bytes = U * (H * I * bw + scales2)
    router_bytes = 2 * E * H * 2 if wl.wr is not None else 0
    io = T * H * 2 + T * k * 8 + T * H * 2
    flops = 6 * T * k * H * I + (2 * T * H * 2 * E if wl.wr is not None else 0)
    return dict(U=U, weight_bytes=w13_bytes + w2_bytes,
                bytes=w13_bytes + w2_bytes + router_bytes + io, flops=flops,
                gateup_bytes=w13_bytes + T * H * bw, down_bytes=w2_bytes)


def workloads_module():
    """moe_expert_layer_align_gb300/workloads.py (the seeded input generators)
    loaded by path, without importing the package, whose __init__ loads the
    CUDA library: the reference arm draws its inputs with it and runs the
    oracle alone."""
    import importlib.util
    name = "_moe_workloads"
    if name not in sys.modules:
        path = os.path.join(ROOT, "moe_expert_layer_align_gb300", "workloads.py")
        spec = importlib.util.spec_from_file_location(name, path)
        mod = importlib.util.module_from_spec(spec)
        sys.modules[name] = mod
        spec.loader.exec_module(mod)
    return sys.modules[name]


def make_workload(cfg, T, device, base=None, **kw):
    return workloads_module().make(cfg, T, device, base=base, **kw)


class Layer:
    """One step on fixed buffers — moe_router_topk (in-path router only) then
    moe_forward — captured in a CUDA graph.  Router weights are split into
    their two bf16 parts once, before any timing."""

    def __init__(self, wl, stream, opts=None, graph=True, w8a16=False, block_m=0):
        import moe_expert_layer_align_gb300 as moe
        self.moe, self.wl, self.stream, self.opts = moe, wl, stream, opts
        self.block_m = block_m      # 0: the planner's row tile
        self.w8a16 = w8a16          # FP8 workload's weights with bf16 activations
        dev = wl.x.device
        # The inputs were drawn on the current stream, whose freed blocks the
        # allocations below may reuse: order the layer's stream after it.
        stream.wait_stream(torch.cuda.current_stream(dev))
        self.fp8 = wl.mode == "fp8"
        self.w13 = wl.w13q if self.fp8 else wl.w13
        self.w2 = wl.w2q if self.fp8 else wl.w2
        self.scales = (wl.w13s, wl.w2s) if self.fp8 else None
        if wl.wr is not None:
            self.hi_lo = moe.moe_router_prepare(wl.wr, stream=stream)
            self.ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device=dev)
            self.w = torch.empty((wl.T, wl.k), dtype=torch.float32, device=dev)
            self.scores = torch.empty((wl.T, wl.E), dtype=torch.float32, device=dev)
            self.rws = torch.empty(max(16, moe.moe_router_workspace_bytes(wl.T, wl.H, wl.E)),
                                   dtype=torch.uint8, device=dev)
        else:
            self.hi_lo = None
            self.ids, self.w = wl.topk_ids, wl.topk_w
        out_dtype = torch.float32 if wl.out == "f32" else torch.bfloat16
        shape = moe.layer_shape(wl.x, self.w13, self.ids, block_m, out_dtype, 0, w8a16)
        self.shape = shape
        if self.hi_lo is not None:
            self.plan = moe.moe_plan_routed(shape, opts)
            ws_bytes = moe.moe_routed_workspace_bytes(shape, opts)
        else:
            self.plan = moe.moe_plan(shape, opts)
            ws_bytes = moe.moe_workspace_bytes(shape, opts)
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        self.out = torch.empty(wl.x.shape, dtype=out_dtype, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.graph = None
        # launches per step: [router GEMM + (fused routing | top-k, align[, x-quant])]
        # or align[, x-quant]; Gate-Up; [act]; Down; combine
        L = self.plan
        quant = 1 if (self.fp8 and not w8a16) else 0
        front = (1 if L.route_fused else 3 + quant) if self.hi_lo is not None \
            else (0 if L.smem_index else 1) + quant
        self.kernels_per_step = front + 3 + (0 if L.fused_act else 1)
        if graph:
            with torch.cuda.stream(stream):
                self.call()                       # warm the launch path before capture
            stream.synchronize()
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=stream):
                self.call()
            stream.synchronize()

    def route(self):
        wl = self.wl
        self.moe.moe_router_topk(wl.x, self.hi_lo, wl.k, wl.router_fn, wl.router_scale,
                                 scores=self.scores, topk_ids=self.ids, topk_w=self.w,
                                 workspace=self.rws, stream=self.stream)

    def call(self):
        wl = self.wl
        if self.hi_lo is not None:
            # router in the path: one chain (router GEMM, then routing + index)
            self.moe.moe_forward_routed(wl.x, self.hi_lo, wl.k, self.w13, self.w2,
                                        score_fn=wl.router_fn, scale=wl.router_scale,
                                        scales=self.scales, out=self.out, scores=self.scores,
                                        topk_ids=self.ids, topk_w=self.w, workspace=self.ws,
                                        block_m=self.block_m, dev_status=self.status,
                                        stream=self.stream, opts=self.opts)
            return
        self.moe.moe_forward(wl.x, self.w13, self.w2, self.ids, self.w, scales=self.scales,
                             out=self.out, workspace=self.ws, block_m=self.block_m,
                             dev_status=self.status, stream=self.stream, opts=self.opts,
                             w8a16=self.w8a16)

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


def stage_times(wl, stream, flush, steps, w8a16=False):
    """Per-stage device time (us) from events recorded between the stages,
    captured with the layer in a CUDA graph (recording events between stages
    serialises them: PDL overlap is lost in this pass).  With the router in
    the path, "router" is the fused routing launch (router GEMM, top-k, x-quant
    and index; "align" and "quant_x" are then empty) or, with separate
    kernels, the router GEMM alone ("align" then holds the top-k too)."""
    import moe_expert_layer_align_gb300 as moe
    n = len(moe.STAGES) + 1
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ev_router = torch.cuda.Event(enable_timing=True)
    for ev in evs + [ev_router]:    # torch creates the CUDA event on first record
        ev.record(stream)
    routed = wl.wr is not None
    opts = moe.make_opts(stage_events=evs)
    if routed:
        opts.stage_events[7] = ev_router.cuda_event
    layer = Layer(wl, stream, opts=opts, graph=True, w8a16=w8a16)
    acc = np.zeros(n - 1)
    router = 0.0
    for _ in range(steps):
        with torch.cuda.stream(stream):
            flush.zero_()
        layer.run()
        stream.synchronize()
        for i in range(n - 1):
            acc[i] += evs[i].elapsed_time(evs[i + 1]) * 1e3
        if routed:
            router += ev_router.elapsed_time(evs[0]) * 1e3
    out = dict(zip(moe.STAGES, (acc / steps).tolist()))
    if routed:
        out = {"router": router / steps, **out}
    return out


def e2e_time(wl, stream, steps, warmup, w8a16=False):
    """The public API with host (pinned) inputs and result: H2D of x (and of
    the top-k ids and weights when the router is outside the path), the step,
    D2H of the output.  The inputs are staged the way a caller would batch
    them: one pinned host buffer and one device buffer holding x, ids and
    weights back to back (16-byte aligned parts), so each step is one H2D
    copy, the layer, one D2H copy."""
    import copy
    routed = wl.wr is not None
    parts = [wl.x] if routed else [wl.x, wl.topk_ids, wl.topk_w]
    offs, n = [], 0
    for t in parts:
        offs.append(n)
        n += (t.numel() * t.element_size() + 15) // 16 * 16
    dbuf = torch.empty(n, dtype=torch.uint8, device=wl.x.device)
    hbuf = torch.empty(n, dtype=torch.uint8).pin_memory()
    views = []
    for t, o in zip(parts, offs):
        nb = t.numel() * t.element_size()
        dv = dbuf[o:o + nb].view(t.dtype).view(t.shape)
        dv.copy_(t)
        hbuf[o:o + nb].copy_(t.cpu().contiguous().view(torch.uint8).view(-1))
        views.append(dv)
    wl2 = copy.copy(wl)
    wl2.x = views[0]
    if not routed:
        wl2.topk_ids, wl2.topk_w = views[1], views[2]
    torch.cuda.synchronize()
    dev_layer = Layer(wl2, stream, graph=False, w8a16=w8a16)
    hout = torch.empty(wl.x.shape, dtype=dev_layer.out.dtype).pin_memory()

    def step():
        with torch.cuda.stream(stream):
            dbuf.copy_(hbuf, non_blocking=True)
            dev_layer.call()
            hout.copy_(dev_layer.out, non_blocking=True)

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
    return {"value": us, "unit": "us", "h2d_bytes_per_step": n,
            "d2h_bytes_per_step": hout.numel() * hout.element_size()}


def _oracle_call(wl, ids, w, sel, w8a16=False):
    """The oracle's layer over the tokens `sel`: it is fed the sampled x rows
    and only the experts they route to, ids renumbered into that subset (a
    selection of inputs, no arithmetic; a token's output depends on nothing
    else).  Returns a thunk that runs it."""
    import oracle
    from tests.helpers import bits16, u8
    sel = np.asarray(sel)
    ids_s = ids[sel]
    used, inv = np.unique(ids_s, return_inverse=True)
    ids_c = inv.reshape(ids_s.shape).astype(np.int32)
    w_s = np.ascontiguousarray(w[sel])
    dev = wl.x.device
    rows = torch.from_numpy(sel).long().to(dev)
    ex = torch.from_numpy(used).long().to(dev)
    x = bits16(wl.x[rows])
    if w8a16:
        args = (x, u8(wl.w13q[ex]), wl.w13s[ex].cpu().numpy(), u8(wl.w2q[ex]),
                wl.w2s[ex].cpu().numpy(), ids_c, w_s)
        return lambda: oracle.moe_w8a16(*args)
    if wl.mode == "bf16":
        args = (x, bits16(wl.w13[ex]), bits16(wl.w2[ex]), ids_c, w_s)
        return lambda: oracle.moe_bf16(*args)
    wq = (u8(wl.w13q[ex]), wl.w13s[ex].cpu().numpy(), u8(wl.w2q[ex]), wl.w2s[ex].cpu().numpy())

    def run():
        xq, xs = oracle.quant_x(x)          # the layer's own x quantisation, timed
        return oracle.moe_fp8(xq, xs, *wq, ids_c, w_s)
    return run


def oracle_baseline(wl, topk_ids, topk_w, budget_s=15.0, max_tokens=None, w8a16=False):
    """The oracle on the host cores over a bounded sample of the batch's
    tokens (evenly spaced), fed those tokens' rows and experts; latency scaled
    to the whole batch.  (In-path router: its fp64 scores over the whole batch
    are timed and added.)"""
    import oracle
    from tests.helpers import bits16
    ids = topk_ids.cpu().numpy()
    w = topk_w.cpu().numpy()
    run = _oracle_call(wl, ids, w, [0], w8a16)
    t0 = time.perf_counter()
    run()
    one = time.perf_counter() - t0
    n = int(max(1, min(wl.T, budget_s // max(one, 1e-6))))
    if max_tokens:
        n = min(n, max_tokens)
    sel = np.unique(np.linspace(0, wl.T - 1, n).astype(np.int64))
    n = len(sel)
    run = _oracle_call(wl, ids, w, sel, w8a16)
    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    us = dt / n * wl.T * 1e6
    extra = ""
    if wl.wr is not None:
        t0 = time.perf_counter()
        oracle.router_scores(bits16(wl.x), wl.wr.cpu().numpy())
        r = time.perf_counter() - t0
        us += r * 1e6
        extra = f"; fp64 router scores of all {wl.T} tokens {r:.3f} s added"
    return {"value": us, "unit": "us", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} of {wl.T} tokens of the T={wl.T} batch (fp64 C oracle, OpenMP, fed "
                      f"those tokens' rows and experts); measured {dt:.2f} s, scaled "
                      f"x{wl.T}/{n}{extra}"}


# ---------------------------------------------------------------- arms

def workload_config(cfg, T, wl, nums, extra=None):
    c = workloads_module().CONFIGS[cfg]
    d = {"workload": f"{c['name']} MoE layer T={T}", "T": T, "H": wl.H, "I": wl.I, "E": wl.E,
         "k": wl.k, "weights": "e4m3 + fp32 128x128 block scales" if wl.mode == "fp8" else "bf16",
         "routing": "in-path router (two-bf16 split), Zipf(1.2) bias" if wl.wr is not None
         else f"{c['routing']} top-{wl.k}" + (f" x{c['scale']}" if c["scale"] != 1.0 else ""),
         "active_experts": nums["U"]}
    d.update(extra or {})
    return d


def oracle_routing(wl):
    """Top-k ids and weights of the in-path router computed by the oracle."""
    import oracle
    from tests.helpers import bits16
    s = oracle.router_scores(bits16(wl.x), wl.wr.cpu().numpy())
    ids, w = oracle.router_topk(s, wl.k, wl.router_fn, wl.router_scale)
    return torch.from_numpy(ids), torch.from_numpy(w.astype(np.float32))


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    # The inputs are drawn exactly as the CUDA arm draws them (the same seeded
    # generators on the same device, so the same values), then moved to the
    # host; nothing of the CUDA library is loaded.
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = make_workload(args.config, args.T, gen_dev).to("cpu")
    if gen_dev == "cuda":
        torch.cuda.empty_cache()
    if wl.wr is not None:
        ids, w = oracle_routing(wl)
    else:
        ids, w = wl.topk_ids, wl.topk_w
    nums = layer_numbers(wl, ids)
    for _ in range(args.warmup):
        oracle_baseline(wl, ids, w, budget_s=0, max_tokens=1)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(oracle_baseline(wl, ids, w, budget_s=5.0)["value"])
    wall = time.perf_counter() - t0
    cb = oracle_baseline(wl, ids, w, budget_s=5.0)
    v = float(np.mean(vals))
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "us", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": workload_config(args.config, args.T, wl, nums, {"l2": "n/a (host)"}),
            "cpu_baseline": {"value": v, "unit": "us", "cores": cb["cores"], "kind": "oracle",
                             "sample": cb["sample"]},
            "e2e": {"value": v, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)


def roofline_times(nums, pk, fp8):
    t_bytes = nums["bytes"] / (pk["hbm_gbs"] * 1e9) * 1e6
    peak = pk["bf16_tflops"] * (2.0 if fp8 else 1.0)   # e4m3 dense = 2x bf16 (nominal ratio)
    t_flops = nums["flops"] / (peak * 1e12) * 1e6
    return t_bytes, t_flops


# The other workloads, each at its first decode size and its largest token
# count (workload 4 also with bf16 activations, w8a16), reported beside the
# headline line.
WORKLOAD_POINTS = [(1, 8, False), (3, 1, False), (3, 4096, False), (4, 1, False),
                   (4, 4096, False), (4, 1, True), (4, 4096, True), (5, 4, False),
                   (5, 256, False)]


def workload_points(stream, flush, pk, points, steps=20, warmup=3, cpu_budget_s=2.0):
    """One entry per (workload, T, w8a16): layer latency, its roofline
    fraction, the Gate-Up GEMM's event-timed duration and bandwidth (the
    dominant kernel), and the oracle on the host cores over a bounded token
    sample.  One full-size weight set is held on the device at a time."""
    import moe_expert_layer_align_gb300 as moe
    out = []
    base_cfg, base = None, None
    for cfg, T, w8 in points:
        if cfg != base_cfg:
            base = None
            torch.cuda.empty_cache()
            base = make_workload(cfg, T, "cuda")
            base_cfg = cfg
        wl = make_workload(cfg, T, "cuda", base=base)
        fp8 = wl.mode == "fp8" and not w8
        L = Layer(wl, stream, w8a16=w8)
        stream.synchronize()
        nums = layer_numbers(wl, L.ids)
        tt, _ = time_layer(L, stream, flush, steps, warmup)
        us = float(np.mean(tt))
        tb, tf = roofline_times(nums, pk, fp8)
        stg = stage_times(wl, stream, flush, 3, w8)
        gu = stg["gateup"]
        gu_gbs = nums["gateup_bytes"] / (gu * 1e-6) / 1e9
        plan = moe.moe_plan(L.shape)
        cpu = oracle_baseline(wl, L.ids, L.w, budget_s=cpu_budget_s, w8a16=w8)
        c = workloads_module().CONFIGS[cfg]
        out.append({
            "workload": f"{c['name']}{' w8a16' if w8 else ''} MoE layer T={T}", "config": cfg,
            "T": T, "dtype": "e4m3" if fp8 else ("w8a16" if w8 else "bf16"),
            "us": us, "us_median": float(np.median(tt)), "active_experts": nums["U"],
            "block_m": int(plan.block_m), "split_k": [plan.split_gateup, plan.split_down],
            "hbm_gbs": nums["bytes"] / (us * 1e-6) / 1e9,
            "tflops": nums["flops"] / (us * 1e-6) / 1e12,
            "bound": "hbm" if tb >= tf else "tensor", "roofline_us": max(tb, tf),
            "roofline_frac": max(tb, tf) / us,
            "gateup_us": gu, "gateup_gbs": gu_gbs, "gateup_frac_of_hbm": gu_gbs / pk["hbm_gbs"],
            "stages_us": stg, "dev_status": int(L.status.item()),
            "cpu_baseline": cpu})
        del L, wl
    del base
    torch.cuda.empty_cache()
    return out


# The router-GEMM table of the "HPC-Ops × SGLang" post (section "Router GEMM",
# Table 2: H20, K = 4096, N = 192, BF16 x FP32 -> FP32, their kernel), us per
# call: context for the router line, measured on other hardware.
ROUTER_TABLE_H20_US = {1: 11.200, 16: 11.744, 48: 12.144, 96: 13.904, 208: 17.088,
                       512: 26.992, 1024: 50.640, 2048: 76.688, 4096: 141.120}


class _Replay:
    """A captured CUDA graph of one call, replayed on `stream` (time_layer's
    step)."""

    def __init__(self, fn, stream):
        self.stream = stream
        with torch.cuda.stream(stream):
            fn()                                  # warm the launch path before capture
        stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            fn()
        stream.synchronize()

    def run(self):
        with torch.cuda.stream(self.stream):
            self.graph.replay()


def router_points(stream, flush, pk, steps=20, warmup=3):
    """The router alone (moe_router_topk: the two-bf16 GEMM on the tensor cores
    and the softmax top-k) at the router-GEMM table shape over its token
    counts: latency, roofline fraction, the pages' H20 figure for context."""
    import moe_expert_layer_align_gb300 as moe
    W = workloads_module()
    H, E, k = W.ROUTER_SHAPE["H"], W.ROUTER_SHAPE["E"], W.ROUTER_SHAPE["k"]
    _, wr = W.router_inputs(1, "cuda")
    hi_lo = moe.moe_router_prepare(wr, stream=stream)
    stream.synchronize()
    out = []
    for M in W.ROUTER_SHAPE["sweep"]:
        x, _ = W.router_inputs(M, "cuda")
        stream.wait_stream(torch.cuda.current_stream())
        sc = torch.empty((M, E), dtype=torch.float32, device="cuda")
        ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
        w = torch.empty((M, k), dtype=torch.float32, device="cuda")
        ws = torch.empty(max(16, moe.moe_router_workspace_bytes(M, H, E)), dtype=torch.uint8,
                         device="cuda")
        r = _Replay(lambda: moe.moe_router_topk(x, hi_lo, k, scores=sc, topk_ids=ids, topk_w=w,
                                                workspace=ws, stream=stream), stream)
        tt, _ = time_layer(r, stream, flush, steps, warmup)
        us = float(np.median(tt))
        nbytes = 2 * E * H * 2 + M * H * 2 + M * E * 4 + M * k * 8
        flops = 2 * M * 2 * E * H
        tb = nbytes / (pk["hbm_gbs"] * 1e9) * 1e6
        tf = flops / (pk["bf16_tflops"] * 1e12) * 1e6
        out.append({"M": M, "K": H, "N": E, "k": k, "us": us,
                    "tflops": flops / (us * 1e-6) / 1e12, "hbm_gbs": nbytes / (us * 1e-6) / 1e9,
                    "roofline_frac": max(tb, tf) / us, "page_table_h20_us": ROUTER_TABLE_H20_US[M]})
        del r, x, sc, ids, w, ws
    return out


def run_cuda(args):
    import moe_expert_layer_align_gb300 as moe  # noqa: F401  (loads the CUDA library)
    workloads = workloads_module()
    ws_, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws_ > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pk, pk_kind = peaks()
    stream = torch.cuda.Stream()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device="cuda")

    cfg = args.config
    wl = make_workload(cfg, args.T, "cuda")
    w8 = bool(args.w8a16)
    if w8 and wl.mode != "fp8":
        raise SystemExit("--w8a16 needs a workload with e4m3 weights (--config 4 or 5)")
    fp8 = wl.mode == "fp8" and not w8      # e4m3 activations and tensor rate
    layer = Layer(wl, stream, w8a16=w8)
    stream.synchronize()
    nums = layer_numbers(wl, layer.ids)

    def barrier():
        if ws_ > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    clk = ClockSampler(local).__enter__()
    barrier()
    times, wall = time_layer(layer, stream, flush, args.steps, args.warmup)
    barrier()
    us = max_over_ranks(float(np.mean(times)))
    st = int(layer.status.item())

    result = None
    if rank == 0:
        stg = stage_times(wl, stream, flush, max(3, min(args.steps, 10)), w8)
        t_bytes, t_flops = roofline_times(nums, pk, fp8)
        gu_us = stg["gateup"]
        achieved = nums["gateup_bytes"] / (gu_us * 1e-6) / 1e9
        kname = ("moe_gemm_w8_kernel<gather> (Gate-Up, e4m3 weights dequantised to bf16)" if w8
                 else f"moe_gemm_kernel<{'e4m3' if fp8 else 'bf16'}, gather> (Gate-Up)")
        roof = {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                "peak_kind": f"{pk_kind} burst copy (MEASURED_PEAKS.json hbm_gbs)",
                "traffic": ncu_traffic(f"c{cfg}:gateup", args.T),
                "algorithmic_bytes_per_launch": nums["gateup_bytes"], "launch_us": gu_us}
        sweep = []
        if not args.no_sweep:
            for T in workloads.CONFIGS[cfg]["sweep"]:
                w2l = make_workload(cfg, T, "cuda", base=wl)
                L2 = Layer(w2l, stream, w8a16=w8)
                stream.synchronize()
                n2 = layer_numbers(w2l, L2.ids)
                tt, _ = time_layer(L2, stream, flush, 20, 3)
                u = float(np.median(tt))
                tb, tf = roofline_times(n2, pk, fp8)
                sweep.append({"T": T, "us": u, "active_experts": n2["U"],
                              "block_m": int(moe.moe_plan(L2.shape).block_m),
                              "hbm_gbs": n2["bytes"] / (u * 1e-6) / 1e9,
                              "tflops": n2["flops"] / (u * 1e-6) / 1e12,
                              "bound": "hbm" if tb >= tf else "tensor",
                              "roofline_frac": max(tb, tf) / u})
                del L2, w2l
        e2e = e2e_time(wl, stream, max(args.steps, 5), args.warmup, w8)
        others, router = [], []
        if not args.no_workloads:
            points = [pt for pt in WORKLOAD_POINTS if (pt[0], pt[1], pt[2]) != (cfg, args.T, w8)]
            others = workload_points(stream, flush, pk, points)
            router = router_points(stream, flush, pk)
        clk.__exit__()
        clocks = clk.summary()
        clocks["window"] = "timed region, stage pass, sweep, e2e pass and other workloads"
        cpu = None if args.no_cpu else oracle_baseline(wl, layer.ids, layer.w, w8a16=w8)
        plan = moe.moe_plan(layer.shape)
        result = {
            "metric": METRIC, "value": us, "unit": "us", "n_gpus": ws_, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3" if fp8 else ("w8a16 (e4m3 weights, bf16 activations)" if w8 else "bf16"),
            "data": "synthetic (seeded; random-init experts of the named shape)",
            "config": workload_config(cfg, args.T, wl, nums, {
                **({"precision": "w8a16: the workload's e4m3 weights, bf16 activations"} if w8 else {}),
                "replicas": ws_, "block_m": plan.block_m,
                "split_k": [plan.split_gateup, plan.split_down],
                "l2": f"flushed before every step ({flush.numel() >> 20} MiB write)",
                "timing": "CUDA graph of one step, CUDA events per step"}),
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
            "workloads": others,
            "router": {"what": "moe_router_topk (two-bf16 router GEMM + softmax top-8) at the "
                               "router-GEMM table shape K=4096, N=192; page_table_h20_us: the "
                               "pages' H20 figure (GEMM alone), context only",
                       "points": router},
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "gpu_launches": layer.kernels_per_step * args.steps,
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
    """Profiler mode: W + K plain steps on the workload, nothing else on the
    GPU (no graphs, flush, sweep or oracle).  Not a bench line."""
    import moe_expert_layer_align_gb300 as moe  # noqa: F401
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    if args.experts:
        # a small case of the same recipe for multi-pass captures: E experts,
        # the same rows per expert at T * E / E_config tokens
        wl = make_workload(args.config, args.T, "cuda", E=args.experts)
    else:
        wl = make_workload(args.config, args.T, "cuda")
    layer = Layer(wl, stream, graph=False, w8a16=args.w8a16)
    for _ in range(args.warmup + args.steps):
        layer.run()
    stream.synchronize()
    print(json.dumps({"ncu_mode": True, "config": args.config, "T": args.T, "E": wl.E,
                      "calls": args.warmup + args.steps, "dev_status": int(layer.status.item())}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5],
                    help="workload (moe_expert_layer_align_gb300.workloads.CONFIGS)")
    ap.add_argument("--T", type=int, default=64)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads' lines (the 'workloads' key)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--ncu", action="store_true", help="profiler mode (no bench line)")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiler mode: draw the workload with this many experts (small case)")
    ap.add_argument("--w8a16", action="store_true",
                    help="e4m3-weight workloads (4, 5) with bf16 activations (MOE_W8A16)")
    ap.add_argument("--record-traffic", metavar="CSV",
                    help="store DRAM bytes per GEMM launch of --config/--T from an ncu raw-page "
                         "CSV export in profiles/traffic.json (no GPU needed)")
    ap.add_argument("--traffic-command", default="",
                    help="the ncu command the CSV came from (recorded beside the numbers)")
    args = ap.parse_args()
    if args.record_traffic:
        return record_traffic(args.record_traffic, args.config, args.T, args.traffic_command)
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
