"""Benchmark of the fused CG tensor-product graph convolution on GB300.

Workload: the MACE-like fused convolution -- N = 10,000 atoms in a periodic
box (density 0.1 / A^3, cutoff 5 A, ~525k directed edges), node features
64x(0e,1o,2e), edge spherical harmonics l <= 3, 24 'uvu' paths to
64x(0e,1o,1e,2o,2e,3o,3e), per-edge weights from a random radial MLP, fp32
(seeded synthetic inputs from ``workloads.config2``).

One step = the whole hot path on one batch: spherical harmonics of the edge
vectors -> fused conv forward -> conv backward (dL/dx, dL/dY, dL/dW for a fixed
output cotangent) -> spherical-harmonic backward (dL/dr).  ``value`` is edges
per second of that forward+backward step; the forward alone is reported under
``fwd``.  All inputs are resident in HBM before the timed region; the weight
stream (3.2 GB) is far larger than L2, so no flush is needed between steps.

``--impl reference`` times the CPU oracle (the reference arm of this build) on
a bounded subgraph of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CG-TP conv edges/sec (fwd, fwd+bwd) at 1 GB300 and % of HBM/FP-pipe roofline"
WORKLOAD = ("fused CG-TP conv: N=10000 atoms, density 0.1/A^3, cutoff 5 A, "
            "64x(0e,1o,2e) (x) Y(l<=3) -> 64x(0e,1o,1e,2o,2e,3o,3e), 24 uvu paths, fp32")
SM_COUNT = 152
FP32_LANES_PER_SM = 128  # FMA lanes per SM per clock


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), sm_max_mhz=float(d.get("sm_max_mhz", 2070.0)),
                    src="measured")
    return dict(hbm=6800.0, sm_max_mhz=2070.0, src="fallback")


# ------------------------------------------------------------ work counts

def algorithmic_counts(prob, N, E, esize=4):
    """Algorithmic bytes and FLOPs per launch of each kernel of the step.

    FLOPs per edge of the tensor product: mul * sum_p 2 (nnz_p + d_l3) (the
    sparse CG multiply-adds plus the weight multiply per output component).
    Bytes count every tensor read or written once (gathered node rows assumed
    to hit L2)."""
    import oracle as O  # only for the CG nonzero counts

    mul = prob.paths[0][6]
    nnz = sum(int((np.abs(O.cg_real(l1, l2, l3)) > 0).sum())
              for (_, _, _, l1, l2, l3, *_r) in prob.paths)
    d3 = sum(2 * p[5] + 1 for p in prob.paths)
    flop_edge = mul * 2 * (nnz + d3)
    dx, dy, do, dw = prob.dim1, prob.dim2, prob.dimo, prob.wdim
    fwd_bytes = E * (dw + dy) * esize + 4 * E + 4 * (N + 1) + N * (dx + do) * esize
    bwd_bytes = (E * (dw + dy) * esize  # read w, y
                 + N * (dx + do + dx) * esize  # read x, g; write gx
                 + E * (dw + dy) * esize  # write gw, gy
                 + 12 * E + 4 * (N + 1))  # s_perm, s_recv, s_rowptr
    return dict(
        sh_fwd=dict(bytes=E * (3 + dy) * esize, flops=None),
        conv_fwd=dict(bytes=fwd_bytes, flops=E * flop_edge),
        conv_bwd=dict(bytes=bwd_bytes, flops=3 * E * flop_edge),
        sh_bwd=dict(bytes=E * (3 + dy + 3) * esize, flops=None),
        flop_edge=flop_edge, nnz=nnz)


# --------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [s.strip() for s in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ GPU arm

def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("gloo")
        return dist, int(os.environ.get("RANK", "0")), ws
    return None, 0, 1


def run_gpu(args):
    import torch

    import clebsch_gordan_tensor_gb300 as cg
    import workloads as W

    dist, rank, world = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    cfg = W.config2(N=args.atoms)
    gr = cfg["graph"]
    N, E = gr.N, gr.E
    plan = cg.Plan(*cfg["irreps"])
    G = cg.Graph.from_numpy(gr)
    x = torch.from_numpy(cfg["x"]).cuda()
    vec = torch.from_numpy(cfg["vec"]).cuda()
    w = torch.from_numpy(cfg["w"]).cuda()
    g = torch.from_numpy(np.random.default_rng(7).standard_normal(
        (N, plan.dim_out)).astype(np.float32)).cuda()
    scale = cfg["scale"]
    y = torch.empty(E, plan.dim_in2, device="cuda")
    out = torch.empty(N, plan.dim_out, device="cuda")
    gx, gy, gw = torch.empty_like(x), torch.empty_like(y), torch.empty_like(w)
    gvec = torch.empty_like(vec)
    names = ["sh_fwd", "conv_fwd", "conv_bwd", "sh_bwd"]

    def step(ev=None):
        if ev is not None:
            ev[0].record()
        cg.sh_forward(vec, 3, out=y)
        if ev is not None:
            ev[1].record()
        plan.conv_forward(G, x, y, w, scale, out=out)
        if ev is not None:
            ev[2].record()
        plan.conv_backward(G, x, y, w, scale, g, out=(gx, gy, gw))
        if ev is not None:
            ev[3].record()
        cg.sh_backward(vec, gy, 3, out=gvec)
        if ev is not None:
            ev[4].record()

    plan.compile()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = cg.launch_count()
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        start.record()
        for k in range(args.steps):
            step(evs[k])
        stop.record()
        torch.cuda.synchronize()
    launches = cg.launch_count() - launches0
    if dist:
        dist.barrier()
    ms_total = start.elapsed_time(stop)
    per = {n: float(np.mean([evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(args.steps)]))
           for i, n in enumerate(names)}
    if dist:
        t = torch.tensor([ms_total], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_total = float(t.item())
    ms_step = ms_total / args.steps

    # ---- e2e: host buffers, copies inside the timed region
    e2e = None if args.no_e2e else run_e2e(args, plan, G, cfg, g, scale, N, E)

    if rank != 0:
        return None
    import oracle as O
    prob = O.make_problem(*cfg["irreps"])
    counts = algorithmic_counts(prob, N, E)
    peaks = _peaks()
    fp32_peak = SM_COUNT * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12  # TFLOP/s
    kernels = {}
    for n in names:
        c = counts[n]
        t = per[n] * 1e-3
        gbs = c["bytes"] / t / 1e9
        ent = {"ms": per[n], "hbm_gbs": gbs, "hbm_frac": gbs / peaks["hbm"]}
        if c["flops"]:
            tf = c["flops"] / t / 1e12
            ent.update(tflops=tf, alu_frac=tf / fp32_peak)
            t_hbm = c["bytes"] / (peaks["hbm"] * 1e9)
            t_alu = c["flops"] / (fp32_peak * 1e12)
            ent["bound"] = "hbm" if t_hbm >= t_alu else "alu"
            ent["roofline_frac"] = max(t_hbm, t_alu) / t
        else:
            ent["bound"] = "hbm"
            ent["roofline_frac"] = gbs / peaks["hbm"]
        kernels[n] = ent
    dom = max(names, key=lambda n: per[n])
    kd = kernels[dom]
    if kd["bound"] == "alu":
        roof = {"bound": "alu", "achieved": kd["tflops"], "peak": fp32_peak, "unit": "TFLOP/s",
                "frac": kd["tflops"] / fp32_peak}
    else:
        roof = {"bound": "hbm", "achieved": kd["hbm_gbs"], "peak": peaks["hbm"], "unit": "GB/s",
                "frac": kd["hbm_gbs"] / peaks["hbm"]}
    roof.update(kernel=dom, traffic=_traffic(dom, plan),
                peak_source=f"{peaks['src']} (HBM copy; FP32 = 152 SM x 128 FMA x 2 x "
                            f"{peaks['sm_max_mhz']:.0f} MHz)")
    line = {
        "metric": METRIC, "value": E * world / (ms_step * 1e-3), "unit": "edges/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded periodic atom cloud, random radial-MLP weights)",
        "config": {"workload": WORKLOAD if N == 10_000 else WORKLOAD.replace("N=10000", f"N={N}"),
                   "N": N, "E": E, "mul": 64, "paths": plan.n_paths,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (3.2 GB weight stream per step)"},
        "fwd": {"value": E * world / (per["conv_fwd"] * 1e-3 + per["sh_fwd"] * 1e-3),
                "unit": "edges/s", "conv_fwd_ms": per["conv_fwd"]},
        "roofline": roof,
        "kernels": kernels,
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": e2e,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, budget_s=args.cpu_seconds)
    return line


def _traffic(kernel, plan):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else null)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d:
        return None
    h = hashlib.sha256(plan.source().encode()).hexdigest()[:16]
    return d.get("bytes") if d.get("source_sha") == h else None


def run_e2e(args, plan, G, cfg, g, scale, N, E):
    """Same step through the public API with host buffers: every step copies
    its inputs (x, edge vectors, weights) from pinned host memory and reads the
    results (output features and dL/dx) back."""
    import torch

    import clebsch_gordan_tensor_gb300 as cg
    hx = torch.from_numpy(cfg["x"]).pin_memory()
    hv = torch.from_numpy(cfg["vec"]).pin_memory()
    hw = torch.from_numpy(cfg["w"]).pin_memory()
    ho = torch.empty(N, plan.dim_out).pin_memory()
    hgx = torch.empty(N, plan.dim_in1).pin_memory()
    x, vec, w = (torch.empty_like(t, device="cuda") for t in (hx, hv, hw))
    y = torch.empty(E, plan.dim_in2, device="cuda")
    out = torch.empty(N, plan.dim_out, device="cuda")
    gx, gy, gw = torch.empty_like(x), torch.empty_like(y), torch.empty_like(w)
    gvec = torch.empty_like(vec)

    def step():
        x.copy_(hx, non_blocking=True)
        vec.copy_(hv, non_blocking=True)
        w.copy_(hw, non_blocking=True)
        cg.sh_forward(vec, 3, out=y)
        plan.conv_forward(G, x, y, w, scale, out=out)
        plan.conv_backward(G, x, y, w, scale, g, out=(gx, gy, gw))
        cg.sh_backward(vec, gy, 3, out=gvec)
        ho.copy_(out, non_blocking=True)
        hgx.copy_(gx, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(1, min(args.steps, 10))
    a.record()
    for _ in range(steps):
        step()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d = sum(t.numel() * t.element_size() for t in (hx, hv, hw))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hgx))
    return {"value": E / (ms * 1e-3), "unit": "edges/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


# ------------------------------------------------------------ CPU oracle

def _oracle_subgraph_step(prob, cfg, R):
    """Oracle forward + backward of the receivers [0, R) and their edges."""
    import oracle as O
    gr = cfg["graph"]
    e1 = int(gr.rowptr[R])
    # receivers R.. keep no edges; senders still index all N nodes
    rowptr = np.concatenate([gr.rowptr[:R + 1], np.full(gr.N - R, e1, dtype=gr.rowptr.dtype)])
    sender = gr.sender[:e1]
    vec, w = cfg["vec"][:e1], cfg["w"][:e1]
    y = O.sh(3, vec)
    out = O.conv_forward(prob, rowptr, sender, cfg["x"], y, w, cfg["scale"])
    g = np.ones_like(out)
    _, gy, _ = O.conv_backward(prob, rowptr, sender, cfg["x"], y, w, cfg["scale"], g)
    O.sh_vjp(3, vec, gy)
    return e1


def cpu_baseline(cfg, budget_s: float = 15.0, R0: int = 4):
    """Time the oracle as it stands (single thread) on a bounded subgraph sized
    to about ``budget_s`` seconds, reported in edges/s."""
    import oracle as O
    prob = O.make_problem(*cfg["irreps"])
    t = time.perf_counter()
    e = _oracle_subgraph_step(prob, cfg, R0)
    dt = time.perf_counter() - t
    R = int(max(R0, min(cfg["graph"].N, R0 * budget_s / max(dt, 1e-3))))
    t = time.perf_counter()
    e = _oracle_subgraph_step(prob, cfg, R)
    dt = time.perf_counter() - t
    return {"value": e / dt, "unit": "edges/s", "cores": 1, "kind": "oracle",
            "sample": f"fwd+bwd (SH, conv fwd, conv bwd, SH bwd) of receivers 0..{R - 1} "
                      f"({e} edges) of the same workload, {dt:.1f} s on 1 host thread"}


def run_reference(args):
    dist, rank, world = _dist()
    if rank != 0:
        return None
    import oracle as O
    import workloads as W
    cfg = W.config2()
    prob = O.make_problem(*cfg["irreps"])
    R = 24
    for _ in range(args.warmup):
        _oracle_subgraph_step(prob, cfg, 4)
    t = time.perf_counter()
    edges = 0
    for _ in range(args.steps):
        edges += _oracle_subgraph_step(prob, cfg, R)
    dt = time.perf_counter() - t
    v = edges / dt
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "edges/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "N": cfg["graph"].N, "E": cfg["graph"].E},
            "cpu_baseline": {"value": v, "unit": "edges/s", "cores": 1, "kind": "oracle",
                             "sample": f"per step: receivers 0..{R - 1} and their edges"},
            "e2e": {"value": v, "unit": "edges/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--atoms", type=int, default=10_000,
                    help="atom count (10000 is the benchmark workload; smaller for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    line = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
