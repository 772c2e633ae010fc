"""Benchmark of the CG tensor-product hot path on GB300.

Default workload (the headline): the MACE-like fused convolution -- N = 10,000
atoms in a periodic box (density 0.1 / A^3, cutoff 5 A, ~525k directed edges),
node features 64x(0e,1o,2e), edge spherical harmonics l <= 3, 24 'uvu' paths
to 64x(0e,1o,1e,2o,2e,3o,3e), per-edge weights from a random radial MLP, fp32
(seeded synthetic inputs from ``workloads.conv64_cloud10k``).

One step = the whole hot path on one batch: spherical harmonics of the edge
vectors -> fused conv forward -> conv backward (dL/dx, dL/dY, dL/dW for a fixed
output cotangent) -> spherical-harmonic backward (dL/dr).  ``value`` is edges
per second of that forward+backward step; the forward alone is reported under
``fwd``.  All inputs are resident in HBM before the timed region; the weight
stream (3.2 GB) is far larger than L2, so no flush is needed between steps.

Other workloads (``--workload``): ``tp`` standalone product, B = 200,000
samples, 128 channels (fwd+bwd, samples/s); ``conv64`` the fp64 fused conv,
N = 5,000, 128 channels (forward, edges/s); ``tfn`` the TFN layer on 1000
molecules (forward, backward, forces and the double backward, edges/s); ``kv``
the same molecules at 64 channels, keys and values of an SE(3)-Transformer layer
from one TFN (fwd+bwd, edges/s); ``uvw`` the 200,000 samples of ``tp`` under a 'uvw'
product (one shared 128x128 matrix per path; channel mixing on tcgen05).

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
FP32_LANES_PER_SM = 128  # FP32 FMA lanes per SM per clock (for the derived figure only)


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), sm_max_mhz=float(d.get("sm_max_mhz", 2070.0)),
                    bf16=float(d["bf16_tflops"]) if "bf16_tflops" in d else None,
                    src="measured")
    return dict(hbm=6800.0, sm_max_mhz=2070.0, bf16=1900.0, src="fallback")


# nominal dense tensor rates per GPU: tf32 1.1 PFLOP/s against bf16 2.25 PFLOP/s
TF32_PER_BF16 = 1.1 / 2.25

# ------------------------------------------------------------ work counts

class Dims:
    """Row widths and FLOPs per row of a plan, read from the library's own plan
    (path list and CG tables); the oracle is not involved."""

    def __init__(self, plan):
        self.dim1, self.dim2, self.dimo, self.wdim = (plan.dim_in1, plan.dim_in2, plan.dim_out,
                                                      plan.weight_numel)
        mul = plan.weight_numel // plan.n_paths
        nnz = d3 = nT = dmin = d1s = 0
        for p in range(plan.n_paths):
            C = plan.coefficients(p)
            l1, _, l3 = plan.path(p)[:3]
            nz = np.abs(C) > 0
            nnz += int(nz.sum())
            nT += int(nz.any(axis=1).sum())  # (m1, m3) pairs with a CG term
            d3 += 2 * l3 + 1
            d1s += 2 * l1 + 1
            dmin += min(2 * l1 + 1, 2 * l3 + 1)
        # FLOPs of one tensor product (one edge or sample): mul * sum_p 2 (nnz_p
        # + d_l3) -- the sparse CG multiply-adds plus the weight multiply per
        # output component
        self.flops = mul * 2 * (nnz + d3)
        # FLOPs the kernels execute (the y-first form: T_p[m1, m3] = sum_m2 C
        # y[m2] once per edge, then per channel one multiply-add per T entry
        # and min(d1, d3) weight products per path).  Backward per channel: h =
        # T g, grad_x, grad_w, the weight products and one dot per T entry;
        # the grad_y spread over the CG terms runs once per lane (cpt channels).
        f64 = plan.dtype == torch_f64()
        cpt = 2 if (not f64 and mul % 64 == 0) else 1
        self.exec_fwd = 2 * mul * (nT + dmin) + 2 * nnz
        self.exec_bwd = 2 * mul * (2 * nT + 2 * d1s + dmin) + 2 * (mul // cpt) * nnz + 2 * nnz


def torch_f64():
    import torch
    return torch.float64


def conv_counts(d: Dims, N, E, es):
    """Algorithmic bytes and FLOPs per launch: every tensor read or written
    once, gathered node rows assumed to hit L2."""
    dx, dy, do, dw = d.dim1, d.dim2, d.dimo, d.wdim
    f = d.flops
    fwd = E * (dw + dy) * es + 4 * E + 4 * (N + 1) + N * (dx + do) * es
    bwd = (E * (dw + dy) * es + N * (dx + do + dx) * es + E * (dw + dy) * es
           + 12 * E + 4 * (N + 1))
    return dict(conv_fwd=(fwd, E * f), conv_bwd=(bwd, 3 * E * f),
                sh_fwd=(E * (3 + dy) * es, None), sh_bwd=(E * (6 + dy) * es, None))


def exec_counts(d: Dims, E):
    """FLOPs the forward and backward kernels execute per launch."""
    return dict(conv_fwd=E * d.exec_fwd, conv_bwd=E * d.exec_bwd, tp_fwd=E * d.exec_fwd,
                tp_bwd=E * d.exec_bwd)


def measure_fma_peaks(torch, cg, dev: int):
    """FMA-pipe throughput of this device, measured with the library's probe
    (cgtp_fma_probe: 8 independent dependent chains per thread, 64 warps per
    SM), best of three launches per precision; clocks sampled meanwhile."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    threads, blocks = 256, sms * 8
    sink = torch.empty(blocks * threads, dtype=torch.int64, device="cuda")
    out = {"sms": sms}
    cases = (("fp32_scalar", torch.float32, False, 40000), ("fp32_packed", torch.float32, True, 20000),
             ("fp64", torch.float64, False, 1500))
    with ClockSampler(dev) as clk:
        for name, dt, packed, iters in cases:
            best = 0.0
            for _ in range(3):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fl = cg.fma_probe(dt, packed, blocks, threads, iters, sink)
                b.record()
                torch.cuda.synchronize()
                best = max(best, fl / (a.elapsed_time(b) * 1e-3) / 1e12)
            out[name] = best
    c = clk.summary()
    out["fp32"] = max(out["fp32_scalar"], out["fp32_packed"])
    out["sm_mhz"] = c.get("sm_mhz")
    out["clock_reasons"] = c.get("reasons")
    mhz = c.get("sm_max_mhz") or 2070.0
    out["fp32_derived"] = sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
    out["how"] = (f"cgtp_fma_probe: {blocks} CTAs x {threads} threads, 8 dependent FMA chains "
                  "per thread, best of 3 launches (CUDA events)")
    return out


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
                 "--format=csv,noheader,nounits", "-lms", "100"],
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


# ------------------------------------------------------ multi-process

def dist_setup():
    """(dist, rank, world): one process per GPU under torchrun; the ranks run
    independent replicas of the workload (no collective on the data path)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("gloo")
        return dist, int(os.environ.get("RANK", "0")), ws
    return None, 0, 1


def max_over_ranks(dist, value: float) -> float:
    """Slowest rank's time (the whole job waits for it)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ workloads

class Workload:
    """A named sequence of launches forming one step, with work counts."""

    def __init__(self, name, desc, units, unit, dtype, kernels, counts, fwd_names, cfg,
                 e2e=None, oracle_step=None, oracle_prep=None, side=None):
        self.name, self.desc, self.units, self.unit, self.dtype = name, desc, units, unit, dtype
        self.kernels, self.counts, self.fwd_names, self.cfg = kernels, counts, fwd_names, cfg
        self.e2e, self.oracle_step, self.oracle_prep = e2e, oracle_step, oracle_prep
        # kernels outside the step, timed on their own: name -> (call, bytes, flops)
        self.side = side or {}
        self.e2e_note = None
        self.exec_flops = {}  # kernel -> FLOPs it executes per launch (y-first form)
        self.fma_peaks = None


def make_conv(args, cg, W, torch):
    cfg = W.conv64_cloud10k(N=args.atoms or 10_000)
    gr = cfg["graph"]
    N, E = gr.N, gr.E
    plan = cg.Plan(*cfg["irreps"])
    G = cg.Graph.from_numpy(gr)
    x, vec, W1, W2 = (torch.from_numpy(cfg[k]).cuda() for k in ("x", "vec", "W1", "W2"))
    # per-edge weights from the radial network, on the device
    w = cg.radial_forward(vec, W1, W2, cfg["cutoff"])
    g = torch.from_numpy(np.random.default_rng(7).standard_normal(
        (N, plan.dim_out)).astype(np.float32)).cuda()
    scale = cfg["scale"]
    y = torch.empty(E, plan.dim_in2, device="cuda")
    out = torch.empty(N, plan.dim_out, device="cuda")
    gx, gy, gw = torch.empty_like(x), torch.empty_like(y), torch.empty_like(w)
    gvec = torch.empty_like(vec)
    plan.compile()
    kernels = [
        ("sh_fwd", lambda: cg.sh_forward(vec, 3, out=y)),
        ("conv_fwd", lambda: plan.conv_forward(G, x, y, w, scale, out=out)),
        ("conv_bwd", lambda: plan.conv_backward(G, x, y, w, scale, g, out=(gx, gy, gw))),
        ("sh_bwd", lambda: cg.sh_backward(vec, gy, 3, out=gvec)),
    ]
    desc = (f"fused CG-TP conv: N={N} atoms, density 0.1/A^3, cutoff 5 A, 64x(0e,1o,2e) (x) "
            "Y(l<=3) -> 64x(0e,1o,1e,2o,2e,3o,3e), 24 uvu paths, fp32")

    def e2e_step_factory():
        # the step's inputs are what a model layer holds: node features, edge
        # vectors and the radial network's parameters; the per-edge weights
        # are computed on the device every step.  Two device buffer sets
        # alternate between steps so that step k's read-back (and step k+1's
        # upload) overlap step k's compute on separate copy streams.
        hx, hv, h1, h2 = (torch.from_numpy(cfg[k]).pin_memory() for k in ("x", "vec", "W1", "W2"))
        ho = [torch.empty(N, plan.dim_out).pin_memory() for _ in range(2)]
        hgx = [torch.empty(N, plan.dim_in1).pin_memory() for _ in range(2)]
        sets = [dict(x=x, vec=vec, W1=W1, W2=W2, w=w, y=y, out=out, gx=gx, gy=gy, gw=gw,
                     gvec=gvec)]
        sets.append({k: torch.empty_like(v) for k, v in sets[0].items()})
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        comp = torch.cuda.current_stream()
        done = [None, None]  # compute-finished event of the step that last used each set
        read = [None, None]  # read-back-finished event of each set
        state = {"k": 0}

        def step():
            k = state["k"]
            b = sets[k % 2]
            with torch.cuda.stream(up):
                if done[k % 2] is not None:
                    up.wait_event(done[k % 2])  # the set's previous step has finished
                for name, h in (("x", hx), ("vec", hv), ("W1", h1), ("W2", h2)):
                    b[name].copy_(h, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(up)
            comp.wait_event(ready)
            if read[k % 2] is not None:
                comp.wait_event(read[k % 2])  # outputs of two steps ago were read back
            cg.radial_forward(b["vec"], b["W1"], b["W2"], cfg["cutoff"], out=b["w"])
            cg.sh_forward(b["vec"], 3, out=b["y"])
            plan.conv_forward(G, b["x"], b["y"], b["w"], scale, out=b["out"])
            plan.conv_backward(G, b["x"], b["y"], b["w"], scale, g, out=(b["gx"], b["gy"], b["gw"]))
            cg.sh_backward(b["vec"], b["gy"], 3, out=b["gvec"])
            fin = torch.cuda.Event()
            fin.record(comp)
            done[k % 2] = fin
            with torch.cuda.stream(down):
                down.wait_event(fin)
                ho[k % 2].copy_(b["out"], non_blocking=True)
                hgx[k % 2].copy_(b["gx"], non_blocking=True)
                r = torch.cuda.Event()
                r.record(down)
            read[k % 2] = r
            state["k"] = k + 1

        def finish():
            comp.wait_stream(up)
            comp.wait_stream(down)

        nb = lambda ts: sum(t.numel() * t.element_size() for t in ts)
        return step, nb((hx, hv, h1, h2)), nb((ho[0], hgx[0])), finish

    hidden, n_out = W2.shape
    side = {"radial_fwd": (lambda: cg.radial_forward(vec, W1, W2, cfg["cutoff"], out=w),
                           E * (3 + n_out) * 4 + (8 + n_out) * hidden * 4,
                           2 * E * (8 * hidden + hidden * n_out)),
            # gradient of the radial network for the conv gradient's grad_w:
            # grad_w is read twice (gh = grad_w W2^T; grad_W2 = h^T grad_w)
            "radial_bwd": (lambda: cg.radial_backward(vec, W1, W2, gw, cfg["cutoff"]),
                           2 * E * n_out * 4 + E * 3 * 8 + (8 + n_out) * hidden * 4,
                           4 * E * hidden * n_out + 4 * E * 8 * hidden)}
    wl = Workload("conv", desc, E, "edges/s", "f32", kernels,
                  conv_counts(Dims(plan), N, E, 4), ["sh_fwd", "conv_fwd"],
                  dict(N=N, E=E, mul=64, paths=plan.n_paths),
                  e2e_step_factory, lambda r0, r1: _oracle_conv_range(cfg, r0, r1),
                  oracle_prep=lambda: _oracle_weights(cfg), side=side)
    wl.exec_flops = exec_counts(Dims(plan), E)
    wl.e2e_note = ("every step: H2D of x, edge vectors and the radial network's parameters "
                   "(pinned), radial network on the device (per-edge weights), SH, conv fwd, "
                   "conv bwd, SH bwd, D2H of out and grad_x; two device buffer sets, copies on "
                   "their own streams overlap the neighbouring steps' compute")
    return wl


def make_conv64(args, cg, W, torch):
    cfg = W.conv128_f64_cloud5k(N=args.atoms or 5_000)
    gr = cfg["graph"]
    N, E = gr.N, gr.E
    plan = cg.Plan(*cfg["irreps"], dtype=torch.float64)
    G = cg.Graph.from_numpy(gr)
    x, vec, W1, W2 = (torch.from_numpy(cfg[k]).cuda() for k in ("x", "vec", "W1", "W2"))
    w = cg.radial_forward(vec, W1, W2, cfg["cutoff"])
    y = torch.empty(E, plan.dim_in2, device="cuda", dtype=torch.float64)
    out = torch.empty(N, plan.dim_out, device="cuda", dtype=torch.float64)
    plan.compile()
    kernels = [("sh_fwd", lambda: cg.sh_forward(vec, 3, out=y)),
               ("conv_fwd", lambda: plan.conv_forward(G, x, y, w, cfg["scale"], out=out))]
    c = conv_counts(Dims(plan), N, E, 8)
    counts = {k: c[k] for k in ("sh_fwd", "conv_fwd")}
    desc = (f"fused CG-TP conv fp64: N={N} atoms, 128x(0e,1o,2e) (x) Y(l<=3) -> "
            "128x(0e,1o,1e,2o,2e,3o,3e), 24 uvu paths, forward only")
    wl = Workload("conv64", desc, E, "edges/s", "f64", kernels, counts, ["sh_fwd", "conv_fwd"],
                  dict(N=N, E=E, mul=128, paths=plan.n_paths), None,
                  lambda r0, r1: _oracle_conv_range(cfg, r0, r1, bwd=False),
                  oracle_prep=lambda: _oracle_weights(cfg))
    wl.exec_flops = exec_counts(Dims(plan), E)
    return wl


def make_tp(args, cg, W, torch):
    cfg = W.mace128_b200k(args.samples)
    B = cfg["B"]
    plan = cg.Plan(*cfg["irreps"])
    x, vec, w = (torch.from_numpy(cfg[k]).cuda() for k in ("x", "vec", "w"))
    g = torch.randn(B, plan.dim_out, device="cuda",
                    generator=torch.Generator("cuda").manual_seed(7))
    y = torch.empty(B, plan.dim_in2, device="cuda")
    gvec = torch.empty_like(vec)
    out = torch.empty(B, plan.dim_out, device="cuda")
    res = {}
    plan.compile()

    def bwd():
        res["g"] = plan.backward(x, y, w, g)

    kernels = [("sh_fwd", lambda: cg.sh_forward(vec, 3, out=y)),
               ("tp_fwd", lambda: plan.forward(x, y, w, out=out)),
               ("tp_bwd", bwd),
               ("sh_bwd", lambda: cg.sh_backward(vec, res["g"][1], 3, out=gvec))]
    prob = Dims(plan)
    f = prob.flops
    rowb = (prob.dim1 + prob.dim2 + prob.wdim) * 4
    counts = {"sh_fwd": (B * (3 + prob.dim2) * 4, None),
              "tp_fwd": (B * (rowb + prob.dimo * 4), B * f),
              "tp_bwd": (B * (rowb + prob.dimo * 4 + rowb), 3 * B * f),
              "sh_bwd": (B * (6 + prob.dim2) * 4, None)}
    desc = (f"standalone CG-TP: B={B}, 128x(0e,1o,2e) (x) Y(l<=3) -> "
            "128x(0e,1o,1e,2o,2e,3o,3e), 24 uvu paths, fp32")
    wl = Workload("tp", desc, B, "samples/s", "f32", kernels, counts, ["sh_fwd", "tp_fwd"],
                  dict(B=B, mul=128, paths=plan.n_paths), None,
                  lambda r0, r1: _oracle_tp_range(cfg, r0, r1))
    wl.exec_flops = exec_counts(prob, B)
    return wl


def make_tfn(args, cg, W, torch):
    cfg = W.tfn32_mol1000()
    gr = cfg["graph"]
    N, E = gr.N, gr.E
    plan = cg.Plan(*cfg["irreps"])
    G = cg.Graph.from_numpy(gr)
    x, vec, w, c, gF = (torch.from_numpy(cfg[k]).cuda() for k in ("x", "vec", "w", "c", "gF"))
    y = torch.empty(E, plan.dim_in2, device="cuda")
    out = torch.empty(N, plan.dim_out, device="cuda")
    gx, gy, gw = torch.empty_like(x), torch.empty_like(y), torch.empty_like(w)
    dEdr, q = torch.empty_like(vec), torch.empty_like(vec)
    F = torch.empty(N, 3, device="cuda")
    ggy = torch.empty_like(y)
    dLdr, FL = torch.empty_like(vec), torch.empty(N, 3, device="cuda")
    plan.compile()
    kernels = [
        ("sh_fwd", lambda: cg.sh_forward(vec, 3, out=y)),
        ("conv_fwd", lambda: plan.conv_forward(G, x, y, w, 1.0, out=out)),
        ("conv_bwd", lambda: plan.conv_backward(G, x, y, w, 1.0, c, out=(gx, gy, gw))),
        ("sh_bwd", lambda: cg.sh_backward(vec, gy, 3, out=dEdr)),
        ("forces", lambda: cg.edge_forces(G, dEdr, out=F)),
        ("forces_adj", lambda: cg.edge_forces_adjoint(G, gF, out=q)),
        ("sh_jvp", lambda: cg.sh_jvp(vec, q, 3, out=ggy)),
        ("conv_dbl", lambda: plan.conv_double_backward(G, x, y, w, 1.0, c, None, ggy, None,
                                                       need=(True, False, True, False))),
        ("sh_hvp", lambda: cg.sh_hvp(vec, gy, q, 3, out=dLdr)),
        ("forces_pos", lambda: cg.edge_forces(G, dLdr, out=FL)),
    ]
    prob = Dims(plan)
    cc = conv_counts(prob, N, E, 4)
    counts = {"sh_fwd": cc["sh_fwd"], "conv_fwd": cc["conv_fwd"], "conv_bwd": cc["conv_bwd"],
              "sh_bwd": cc["sh_bwd"], "forces": (E * 12 + N * 12, None),
              "forces_adj": (E * 12 + N * 12, None), "sh_jvp": (E * (6 + 16) * 4, None),
              "conv_dbl": (cc["conv_bwd"][0] - E * prob.dim2 * 4, cc["conv_bwd"][1] * 2 // 3),
              "sh_hvp": (E * (3 + 16 + 3 + 3) * 4, None), "forces_pos": (E * 12 + N * 12, None)}
    desc = ("TFN layer: 1000 molecules of 9-29 atoms, fully connected, 32x(0e,1o,2e,3o) (x) "
            "Y(l<=3) -> 32x(0e,1o,2e,3o), 23 paths, fp32: fwd, bwd, forces, double backward, "
            "force-loss gradient in the positions")
    wl = Workload("tfn", desc, E, "edges/s", "f32", kernels, counts, ["sh_fwd", "conv_fwd"],
                  dict(N=N, E=E, mul=32, paths=plan.n_paths), None, None)
    wl.exec_flops = exec_counts(prob, E)
    return wl


def make_kv(args, cg, W, torch):
    """SE(3)-Transformer keys and values from one TFN with doubled channels:
    the molecule graph of the TFN workload at 64 channels per irrep."""
    cfg = W.tfn_kv64_mol1000()
    gr = cfg["graph"]
    N, E = gr.N, gr.E
    plan = cg.Plan(*cfg["irreps"])
    G = cg.Graph.from_numpy(gr)
    x, vec, w, g = (torch.from_numpy(cfg[k]).cuda() for k in ("x", "vec", "w", "g"))
    y = torch.empty(E, plan.dim_in2, device="cuda")
    out = torch.empty(N, plan.dim_out, device="cuda")
    gx, gy, gw = torch.empty_like(x), torch.empty_like(y), torch.empty_like(w)
    gvec = torch.empty_like(vec)
    plan.compile()
    kernels = [
        ("sh_fwd", lambda: cg.sh_forward(vec, 3, out=y)),
        ("conv_fwd", lambda: plan.conv_forward(G, x, y, w, 1.0, out=out)),
        ("conv_bwd", lambda: plan.conv_backward(G, x, y, w, 1.0, g, out=(gx, gy, gw))),
        ("sh_bwd", lambda: cg.sh_backward(vec, gy, 3, out=gvec)),
    ]
    desc = ("fused keys/values (one TFN, doubled channels): 1000 molecules of 9-29 atoms, "
            "fully connected, 64x(0e,1o,2e,3o) (x) Y(l<=3) -> 64x(0e,1o,2e,3o), 23 paths, fp32")
    d = Dims(plan)
    wl = Workload("kv", desc, E, "edges/s", "f32", kernels, conv_counts(d, N, E, 4),
                  ["sh_fwd", "conv_fwd"], dict(N=N, E=E, mul=64, paths=plan.n_paths), None, None)
    wl.exec_flops = exec_counts(d, E)
    return wl


def make_uvw(args, cg, W, torch):
    """'uvw' product on the 200,000-sample, 128-channel inputs of ``tp``:
    per-path 'uvu' blocks (unit shared weights), then the channel mixing on the
    tensor cores."""
    cfg = W.mace128_uvw_b200k(args.samples)
    B = cfg["B"]
    uvw = cg.UVWProduct(*W.IRREPS_MACE128)
    x, vec, Wm = (torch.from_numpy(cfg[k]).cuda() for k in ("x", "vec", "W"))
    y = torch.empty(B, uvw.dim_in2, device="cuda")
    mid = torch.empty(B, uvw.dim_mid, device="cuda")
    out = torch.empty(B, uvw.dim_out, device="cuda")
    ones = torch.ones(uvw.plan.weight_numel, device="cuda")
    fwb, bwb = uvw.linear.workspace_bytes(B)
    ws = torch.empty(fwb, dtype=torch.uint8, device="cuda")
    wsb = torch.empty(bwb, dtype=torch.uint8, device="cuda")
    g = torch.randn(B, uvw.dim_out, device="cuda", generator=torch.Generator("cuda").manual_seed(7))
    res = {}
    uvw.plan.compile()

    def mix_bwd_x():
        res["gmid"] = uvw.linear.backward(mid, Wm, g, need=(True, False), workspace=wsb)[0]

    wsu = torch.empty(uvw.workspace_bytes(B)[0], dtype=torch.uint8, device="cuda")
    # forward: the fused kernel (per-path blocks computed inside the mixing);
    # the gradient recomputes the blocks it needs (tp_paths) and runs the
    # mixing's two gradients and the per-path gradient
    kernels = [("sh_fwd", lambda: cg.sh_forward(vec, 3, out=y)),
               ("uvw_fwd", lambda: uvw.forward(x, y, Wm, out=out, workspace=wsu)),
               ("tp_paths", lambda: uvw.plan.forward(x, y, ones, out=mid)),
               ("linear_bwd_x", mix_bwd_x),
               ("linear_bwd_w", lambda: uvw.linear.backward(mid, Wm, g, need=(False, True),
                                                            workspace=wsb)),
               ("tp_paths_bwd", lambda: uvw.plan.backward(x, y, ones, res["gmid"],
                                                          need=(True, True, False)))]
    d = Dims(uvw.plan)
    mix = 0
    for j in range(uvw.linear.n_instr):
        i, o, _ = uvw.linear.instruction(j)
        mix += uvw.plan.path(j)[2] * 2 + 1
    mix_flops = 2 * B * mix * 128 * 128
    counts = {"sh_fwd": (B * (3 + d.dim2) * 4, None),
              "tp_paths": (B * (d.dim1 + d.dim2 + d.dimo) * 4 + d.wdim * 4, B * d.flops),
              "uvw_fwd": (B * (d.dim1 + d.dim2 + uvw.dim_out) * 4 + uvw.weight_numel * 4,
                          mix_flops, "tensor3"),
              "linear_bwd_x": (B * (uvw.dim_mid + uvw.dim_out) * 4 + uvw.weight_numel * 4,
                               mix_flops, "tensor3"),
              "linear_bwd_w": (B * (uvw.dim_mid + uvw.dim_out) * 4 + uvw.weight_numel * 4,
                               mix_flops, "tensor3"),
              "tp_paths_bwd": (B * (2 * d.dim1 + 2 * d.dim2 + d.dimo) * 4, 2 * B * d.flops)}
    desc = (f"'uvw' CG-TP: B={B}, 128x(0e,1o,2e) (x) Y(l<=3) -> 128x(0e,1o,1e,2o,2e,3o,3e), "
            "24 paths, one shared 128x128 matrix per path, fp32, forward (fused: per-path blocks "
            "computed inside the tcgen05 channel mixing) and gradient (blocks recomputed, mixing "
            "gradients on tcgen05, TF32 split in three products)")
    return Workload("uvw", desc, B, "samples/s", "f32", kernels, counts,
                    ["sh_fwd", "uvw_fwd"], dict(B=B, mul=128, paths=uvw.n_paths),
                    None, None)


WORKLOADS = {"conv": make_conv, "conv64": make_conv64, "tp": make_tp, "tfn": make_tfn,
             "kv": make_kv, "uvw": make_uvw}


# ------------------------------------------------------------ GPU arm

def analyze(wl, per, fma, peaks):
    """Per-kernel rates and roofline fractions of a workload's step, and the
    roofline of its dominant kernel.  per: kernel -> mean ms."""
    names = [n for n, _ in wl.kernels]
    # the CUDA-core kernels' ALU peak: the FMA-pipe throughput measured in this
    # run by the library's probe (FP32: the better of scalar and packed FMA)
    if wl.dtype == "f64":
        fp32_peak, alu_src = fma["fp64"], "FP64 pipe: measured by cgtp_fma_probe in this run"
    else:
        fp32_peak, alu_src = fma["fp32"], "FP32 pipe: measured by cgtp_fma_probe in this run"
    # fp32 products as three TF32 products on the tensor cores: the effective
    # peak is the measured bf16 GEMM rate x the nominal tf32/bf16 ratio / 3
    tc_peak = peaks["bf16"] * TF32_PER_BF16 / 3 if peaks.get("bf16") else None
    kernels = {}
    for n in names:
        nbytes, flops, *kind = wl.counts[n]
        t = per[n] * 1e-3
        gbs = nbytes / t / 1e9
        ent = {"ms": per[n], "hbm_gbs": gbs, "hbm_frac": gbs / peaks["hbm"]}
        if flops and kind and kind[0] == "tensor3" and tc_peak:
            tf = flops / t / 1e12
            t_hbm, t_tc = nbytes / (peaks["hbm"] * 1e9), flops / (tc_peak * 1e12)
            ent.update(tflops=tf, tensor_frac=tf / tc_peak,
                       bound="tensor" if t_tc >= t_hbm else "hbm",
                       roofline_frac=max(t_hbm, t_tc) / t)
        elif flops:
            tf = flops / t / 1e12
            ent.update(tflops=tf, alu_frac=tf / fp32_peak)
            t_hbm, t_alu = nbytes / (peaks["hbm"] * 1e9), flops / (fp32_peak * 1e12)
            ent["bound"] = "hbm" if t_hbm >= t_alu else "alu"
            ent["roofline_frac"] = max(t_hbm, t_alu) / t
            ex = wl.exec_flops.get(n)
            if ex:  # the FLOPs the kernel executes (y-first form)
                ent.update(exec_tflops=ex / t / 1e12, exec_alu_frac=ex / t / 1e12 / fp32_peak)
        else:
            ent["bound"] = "hbm"
            ent["roofline_frac"] = gbs / peaks["hbm"]
        kernels[n] = ent
    dom = max(names, key=lambda n: per[n])
    kd = kernels[dom]
    if kd["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": kd["tflops"], "peak": tc_peak, "unit": "TFLOP/s",
                "frac": kd["tflops"] / tc_peak,
                "note": "fp32 products as three TF32 tensor-core products: peak = measured bf16 "
                        "x nominal tf32/bf16 / 3"}
    elif kd["bound"] == "alu":
        roof = {"bound": "alu", "achieved": kd["tflops"], "peak": fp32_peak, "unit": "TFLOP/s",
                "frac": kd["tflops"] / fp32_peak}
        if "exec_tflops" in kd:
            roof.update(achieved_exec=kd["exec_tflops"], frac_exec=kd["exec_alu_frac"])
    else:
        roof = {"bound": "hbm", "achieved": kd["hbm_gbs"], "peak": peaks["hbm"], "unit": "GB/s",
                "frac": kd["hbm_gbs"] / peaks["hbm"]}
    roof.update(kernel=dom, traffic=_traffic(wl.name, dom),
                peak_source=f"HBM: {peaks['src']} copy bandwidth (MEASURED_PEAKS.json); {alu_src}")
    return kernels, roof, fp32_peak, alu_src


def run_workloads(args, cg, W, torch, fma, peaks):
    """The other workloads of the benchmark set, each timed briefly in the same
    process after the main measurement (3 warm-up steps, 20 timed steps, CUDA
    events per kernel): their step time, rate and the roofline of their
    dominant kernel.  A workload that fails is reported with its error."""
    out = {}
    for name in ("tp", "conv64", "tfn", "kv", "uvw"):
        if name == args.workload:
            continue
        try:
            wl = WORKLOADS[name](args, cg, W, torch)
            names = [n for n, _ in wl.kernels]
            for _ in range(3):
                for _, k in wl.kernels:
                    k()
            torch.cuda.synchronize()
            steps = 20
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
                   for _ in range(steps)]
            for k in range(steps):
                for i, (_, fn) in enumerate(wl.kernels):
                    evs[k][i].record()
                    fn()
                evs[k][-1].record()
            torch.cuda.synchronize()
            per = {n: float(np.mean([evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(steps)]))
                   for i, n in enumerate(names)}
            ms_step = float(np.mean([evs[k][0].elapsed_time(evs[k][-1]) for k in range(steps)]))
            kernels, roof, _, _ = analyze(wl, per, fma, peaks)
            fwd_ms = sum(per[n] for n in wl.fwd_names)
            out[name] = {
                "workload": wl.desc, "steps": steps, "warmup": 3, "ms_per_step": ms_step,
                "value": wl.units / (ms_step * 1e-3), "unit": wl.unit, "dtype": wl.dtype,
                "fwd": {"value": wl.units / (fwd_ms * 1e-3), "ms": fwd_ms},
                "roofline": roof,
                "kernels": {n: {"ms": e["ms"], "bound": e.get("bound"),
                                "roofline_frac": e.get("roofline_frac")}
                            for n, e in kernels.items()},
            }
            del wl
        except Exception as e:  # reported, the main line stands
            out[name] = {"error": f"{type(e).__name__}: {e}"[:200]}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def run_gpu(args):
    import torch

    import clebsch_gordan_tensor_gb300 as cg
    import workloads as W

    dist, rank, world = dist_setup()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    wl = WORKLOADS[args.workload](args, cg, W, torch)
    names = [n for n, _ in wl.kernels]

    def step(ev=None):
        for i, (_, k) in enumerate(wl.kernels):
            if ev is not None:
                ev[i].record()
            k()
        if ev is not None:
            ev[-1].record()

    wl.fma_peaks = measure_fma_peaks(torch, cg, local) if rank == 0 else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    nk = len(wl.kernels)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
           for _ in range(args.steps)]
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
    ms_step = max_over_ranks(dist, start.elapsed_time(stop)) / args.steps
    per = {n: float(np.mean([evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(args.steps)]))
           for i, n in enumerate(names)}
    e2e = None
    if wl.e2e is not None and not args.no_e2e:
        e2e = run_e2e(args, wl)
    side = {n: time_side(torch, fn) for n, (fn, _, _) in wl.side.items()}
    if rank != 0:
        return None
    others = None
    # with the benchmark sizes only (profiling runs shrink --atoms / --samples)
    if world == 1 and not args.no_workloads and args.atoms is None and args.samples == 200_000:
        others = run_workloads(args, cg, W, torch, wl.fma_peaks, _peaks())

    peaks = _peaks()
    fma = wl.fma_peaks
    kernels, roof, fp32_peak, alu_src = analyze(wl, per, fma, peaks)
    side_out = {}
    for n, ms in side.items():
        _, nbytes, flops = wl.side[n]
        gbs = nbytes / (ms * 1e-3) / 1e9
        tf = flops / (ms * 1e-3) / 1e12
        if n == "radial_fwd":
            # tensor-core rate of the split TF32 products (three per multiply-add)
            # against the measured bf16 GEMM peak scaled by the nominal tf32/bf16 ratio
            tf32_peak = peaks["bf16"] * TF32_PER_BF16 if peaks.get("bf16") else None
            side_out[n] = {"ms": ms, "hbm_gbs": gbs, "hbm_frac": gbs / peaks["hbm"],
                           "tflops": tf, "tf32_issued_tflops": 3 * tf,
                           "tf32_frac": 3 * tf / tf32_peak if tf32_peak else None,
                           "bound": "hbm", "roofline_frac": gbs / peaks["hbm"],
                           "note": "outside the step: per-edge weights from the radial network, "
                                   "recomputed every step of the e2e leg"}
        else:
            side_out[n] = {"ms": ms, "hbm_gbs": gbs, "hbm_frac": gbs / peaks["hbm"],
                           "tflops": tf, "alu_frac": tf / fp32_peak,
                           "roofline_frac": max(gbs / peaks["hbm"], tf / fp32_peak),
                           "note": "outside the step: radial-network gradient for the conv "
                                   "gradient's grad_w (gh = grad_w W2^T and grad_W2 on the "
                                   "tensor cores, the rest on the CUDA cores)"}
    config = {"workload": wl.desc, **wl.cfg,
              "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
              "l2": "inputs larger than L2 (weight stream per step >> 129 MB)"}
    fwd_ms = sum(per[n] for n in wl.fwd_names)
    line = {
        "metric": METRIC, "value": wl.units * world / (ms_step * 1e-3), "unit": wl.unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded; see workloads/)", "config": config,
        "fwd": {"value": wl.units * world / (fwd_ms * 1e-3), "unit": wl.unit, "ms": fwd_ms},
        "roofline": roof, "kernels": kernels, "side_kernels": side_out or None,
        "fma_peaks": fma, "gpu_launches": launches,
        "clocks": clk.summary(), "e2e": e2e,
    }
    if others:
        # measured after the timed region above, outside it
        line["workloads"] = others
    if not args.no_cpu_baseline and wl.oracle_step is not None:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_seconds)
    return line


def _traffic(workload, kernel):
    """DRAM bytes per launch from the committed ncu summary for this workload
    and kernel, if recorded on the current kernel source (else null)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(f"{workload}/{kernel}")
    if not d:
        return None
    import hashlib
    src = os.path.join(ROOT, "clebsch_gordan_tensor_gb300", "csrc")
    h = hashlib.sha256()
    for f in d.get("sources", ("tp_kernels.cuh", "plan.cpp")):
        h.update(open(os.path.join(src, f), "rb").read())
    return d.get("bytes") if d.get("kernel_sha") == h.hexdigest()[:16] else None


def time_side(torch, fn, reps: int = 10) -> float:
    """Mean CUDA-event time (ms) of a kernel run on its own, after warm-up."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def run_e2e(args, wl):
    """The same step through the public API with host buffers: every step
    copies its inputs from pinned host memory and reads its results back."""
    import torch
    step, h2d, d2h, *rest = wl.e2e()
    finish = rest[0] if rest else (lambda: None)
    for _ in range(max(1, min(args.warmup, 3))):
        step()
    finish()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(1, min(args.steps, 10))
    a.record()
    for _ in range(steps):
        step()
    finish()  # the last step's read-back is inside the timed region
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    line = {"value": wl.units / (ms * 1e-3), "unit": wl.unit, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    if wl.e2e_note:
        line["note"] = wl.e2e_note
    return line


# ------------------------------------------------------------ CPU oracle

def _oracle_weights(cfg):
    """The oracle's per-edge weights of a conv workload (computed once, before
    any timing: they are an input of the timed oracle step)."""
    import oracle as O
    if "w" not in cfg:
        cfg["w"] = O.radial_forward(cfg["vec"], cfg["W1"], cfg["W2"], cfg["cutoff"],
                                    out_dtype=cfg["dtype"])[0]


def _oracle_problem(cfg):
    import oracle as O
    if "prob" not in cfg:
        cfg["prob"] = O.make_problem(*cfg["irreps"])
    return cfg["prob"]


def _oracle_conv_range(cfg, r0, r1, bwd=True):
    """Oracle forward (+ backward) of the receivers [r0, r1) and their edges;
    returns the edge count."""
    import oracle as O
    prob = _oracle_problem(cfg)
    gr = cfg["graph"]
    e0, e1 = int(gr.rowptr[r0]), int(gr.rowptr[r1])
    # only receivers r0..r1-1 keep edges; senders still index all N nodes
    rowptr = np.clip(gr.rowptr.astype(np.int64) - e0, 0, e1 - e0)
    rowptr[:r0 + 1] = 0
    rowptr[r1:] = e1 - e0
    sender = gr.sender[e0:e1]
    vec, w = cfg["vec"][e0:e1], cfg["w"][e0:e1]
    y = O.sh(3, vec)
    out = O.conv_forward(prob, rowptr, sender, cfg["x"], y, w, cfg["scale"])
    if bwd:
        _, gy, _ = O.conv_backward(prob, rowptr, sender, cfg["x"], y, w, cfg["scale"],
                                   np.ones_like(out))
        O.sh_vjp(3, vec, gy)
    return e1 - e0


def _oracle_tp_range(cfg, r0, r1):
    import oracle as O
    prob = _oracle_problem(cfg)
    x, vec, w = cfg["x"][r0:r1], cfg["vec"][r0:r1], cfg["w"][r0:r1]
    y = O.sh(3, vec)
    out = O.tp_forward(prob, x, y, w)
    _, gy, _ = O.tp_backward(prob, x, y, w, np.ones_like(out))
    O.sh_vjp(3, vec, gy)
    return r1 - r0


def _oracle_all_cores(run_range, n_items, per_thread, threads, offset=0):
    """The oracle on `threads` host threads at once, each on its own contiguous
    item range of `per_thread` items (the oracle's C loops run outside the
    Python lock, so the threads use separate cores).  Returns (units, seconds)."""
    from concurrent.futures import ThreadPoolExecutor
    span = max(1, min(per_thread, n_items // threads))
    starts = [(offset + i * span) % max(1, n_items - span + 1) for i in range(threads)]
    ranges = [(a, a + span) for a in starts]
    with ThreadPoolExecutor(threads) as ex:
        t = time.perf_counter()
        units = sum(ex.map(lambda r: run_range(*r), ranges))
        dt = time.perf_counter() - t
    return units, dt


def cpu_baseline(wl, budget_s: float = 15.0, R0: int = 4):
    """The oracle as it stands on a bounded sample of the same workload, about
    ``budget_s`` seconds in all: first on one host thread, then on every host
    core (one thread per core, disjoint item ranges)."""
    if wl.oracle_prep is not None:
        wl.oracle_prep()
    n_items = wl.cfg.get("N", wl.cfg.get("B"))
    t = time.perf_counter()
    u0 = wl.oracle_step(0, R0)
    dt = time.perf_counter() - t
    per_item = max(dt, 1e-4) / R0
    R = int(min(n_items, max(R0, 0.35 * budget_s / per_item)))
    t = time.perf_counter()
    units = wl.oracle_step(0, R)
    dt1 = time.perf_counter() - t
    cores = os.cpu_count() or 1
    Rc = int(max(R0, 0.5 * budget_s / per_item))
    uc, dtc = _oracle_all_cores(wl.oracle_step, n_items, Rc, cores)
    what = wl.unit.split("/")[0]
    return {"value": uc / dtc, "unit": wl.unit, "cores": cores, "kind": "oracle",
            "sample": f"{cores} host threads at once, each on its own {min(Rc, n_items // cores)} "
                      f"consecutive items of the workload ({uc} {what} in {dtc:.1f} s)",
            "single_thread": {"value": units / dt1, "unit": wl.unit, "cores": 1,
                              "sample": f"items 0..{R - 1} ({units} {what}) in {dt1:.1f} s"},
            "nproc": cores}


def run_reference(args):
    dist, rank, world = dist_setup()
    if rank != 0:
        return None
    import workloads as W
    cfg = W.conv64_cloud10k()
    _oracle_problem(cfg)
    _oracle_weights(cfg)
    N = cfg["graph"].N
    cores = os.cpu_count() or 1
    step = lambda r0, r1: _oracle_conv_range(cfg, r0, r1)
    R = 8  # receivers per host thread per step (about 420 edges, fwd + bwd)
    for k in range(args.warmup):
        _oracle_all_cores(step, N, 2, cores, offset=k * 97)
    edges, dt = 0, 0.0
    for k in range(args.steps):
        u, t = _oracle_all_cores(step, N, R, cores, offset=k * 131)
        edges += u
        dt += t
    v = edges / dt
    desc = ("fused CG-TP conv: N=10000 atoms, density 0.1/A^3, cutoff 5 A, 64x(0e,1o,2e) (x) "
            "Y(l<=3) -> 64x(0e,1o,1e,2o,2e,3o,3e), 24 uvu paths, fp32")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "edges/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; see workloads/)",
            "config": {"workload": desc, "N": N, "E": cfg["graph"].E},
            "cpu_baseline": {"value": v, "unit": "edges/s", "cores": cores, "kind": "oracle",
                             "sample": f"per step: {cores} host threads at once, each on {R} "
                                       f"receivers and their edges (fwd + bwd)"},
            "e2e": {"value": v, "unit": "edges/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="conv", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--atoms", type=int, default=None,
                    help="atom count of the conv (10000) and conv64 (5000) workloads; smaller "
                         "for profiling")
    ap.add_argument("--samples", type=int, default=200_000,
                    help="sample count of the tp and uvw workloads (200000 is the benchmark; "
                         "smaller for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the brief runs of the other workloads after the main one")
    args = ap.parse_args()
    line = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
