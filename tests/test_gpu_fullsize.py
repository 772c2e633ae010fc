"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times.  The GPU computes every output; the oracle computes sampled
rows (receivers, senders, edges or samples) one by one.

Workloads (seeded recipes in ``workloads``):
  tp16_b1000           standalone TP, B = 1000, fp32               (compared in full)
  mace128_b200k        standalone TP, B = 200,000, 128 channels    (sampled rows)
  conv64_cloud10k      fused conv, N = 10,000 atoms, ~525k edges   (sampled rows)
  conv128_f64_cloud5k  fused conv, N = 5,000 atoms, 128 ch., fp64  (forward, sampled)
  tfn32_mol1000        TFN layer on 1000 molecules, fwd + bwd + double backward
                       and forces, fp32; with 64 channels for fused keys/values
  mace128_uvw_b200k    the 'uvw' channel mixing on the 200,000 samples
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests.gpu_util import assert_close, conv_weights, dev, host, need_gpu, torch

pytestmark = pytest.mark.gpu


def _cg():
    import clebsch_gordan_tensor_gb300 as cg
    return cg


def _sample(rng, n, k):
    idx = rng.choice(n, size=min(k, n), replace=False)
    return np.unique(np.concatenate([idx, [0, n - 1]]))


def test_tp16_full():
    need_gpu()
    cg = _cg()
    cfg = W.tp16_b1000()
    prob = O.make_problem(*cfg["irreps"])
    plan = cg.Plan(*cfg["irreps"])
    x, v, w = cfg["x"], cfg["vec"], cfg["w"]
    y = cg.sh_forward(dev(v), 2)
    out = plan.forward(dev(x), y, dev(w))
    yr = O.sh(2, v)
    assert_close(host(y), yr, np.float32, "Y")
    assert_close(host(out), O.tp_forward(prob, x, yr, w), np.float32, "out")
    g = np.random.default_rng(0).standard_normal(out.shape).astype(np.float32)
    gx, gy, gw = plan.backward(dev(x), y, dev(w), dev(g))
    rx, ry, rw = O.tp_backward(prob, x, yr, w, g)
    for a, b, n in ((gx, rx, "gx"), (gy, ry, "gy"), (gw, rw, "gw")):
        assert_close(host(a), b, np.float32, n)


def test_mace128_b200k_sampled():
    need_gpu()
    cg = _cg()
    cfg = W.mace128_b200k()
    prob = O.make_problem(*cfg["irreps"])
    plan = cg.Plan(*cfg["irreps"])
    B = cfg["B"]
    x, v, w = dev(cfg["x"]), dev(cfg["vec"]), dev(cfg["w"])
    y = cg.sh_forward(v, 3)
    out = plan.forward(x, y, w)
    rng = np.random.default_rng(1)
    idx = _sample(rng, B, 256)
    yr = O.sh(3, cfg["vec"][idx])
    ref = O.tp_forward(prob, cfg["x"][idx], yr, cfg["w"][idx])
    assert_close(host(out[torch.from_numpy(idx).cuda()]), ref, np.float32, "out rows")
    g = torch.randn(B, plan.dim_out, device="cuda", generator=torch.Generator("cuda").manual_seed(1))
    gx, gy, gw = plan.backward(x, y, w, g)
    ti = torch.from_numpy(idx).cuda()
    rx, ry, rw = O.tp_backward(prob, cfg["x"][idx], yr, cfg["w"][idx], host(g[ti]))
    assert_close(host(gx[ti]), rx, np.float32, "gx rows")
    assert_close(host(gy[ti]), ry, np.float32, "gy rows")
    assert_close(host(gw[ti]), rw, np.float32, "gw rows")


def _conv_sampled(cfg, dt, do_bwd: bool):
    cg = _cg()
    gr = cfg["graph"]
    prob = O.make_problem(*cfg["irreps"])
    plan = cg.Plan(*cfg["irreps"], dtype=torch.float64 if dt == np.float64 else torch.float32)
    G = cg.Graph.from_numpy(gr)
    conv_weights(cfg)
    x, v, w = dev(cfg["x"]), dev(cfg["vec"]), dev(cfg["w"])
    y = cg.sh_forward(v, 3)
    out = plan.conv_forward(G, x, y, w, cfg["scale"])
    yr = O.sh(3, cfg["vec"])
    assert_close(host(y), yr, dt, "Y")
    rng = np.random.default_rng(2)
    nodes = _sample(rng, gr.N, 120)
    ref = O.conv_forward(prob, gr.rowptr, gr.sender, cfg["x"], yr, cfg["w"], cfg["scale"],
                         receivers=nodes)
    assert_close(host(out)[nodes], ref[nodes], dt, "conv out rows")
    if not do_bwd:
        return
    g = np.random.default_rng(3).standard_normal((gr.N, prob.dimo)).astype(dt)
    gx, gy, gw = plan.conv_backward(G, x, y, w, cfg["scale"], dev(g))
    edges = _sample(rng, gr.E, 400)
    rx, ry, rw = O.conv_backward(prob, gr.rowptr, gr.sender, cfg["x"], yr, cfg["w"],
                                 cfg["scale"], g, nodes=nodes, edges=edges)
    assert_close(host(gx)[nodes], rx[nodes], dt, "gx rows")
    assert_close(host(gy)[edges], ry[edges], dt, "gy rows")
    assert_close(host(gw)[edges], rw[edges], dt, "gw rows")


def test_conv64_cloud10k_sampled():
    need_gpu()
    _conv_sampled(W.conv64_cloud10k(), np.float32, True)


def test_conv128_cloud5k_sampled_fp64():
    need_gpu()
    _conv_sampled(W.conv128_f64_cloud5k(), np.float64, False)


def test_tfn32_chain_sampled():
    need_gpu()
    cg = _cg()
    from tests.test_gpu_conv import tfn_chain_gpu

    cfg = W.tfn32_mol1000()
    gr = cfg["graph"]
    prob = O.make_problem(*W.IRREPS_TFN32)
    plan = cg.Plan(*W.IRREPS_TFN32)
    G = cg.Graph.from_numpy(gr)
    res = tfn_chain_gpu(cg, plan, G, dev(cfg["x"]), dev(cfg["vec"]), dev(cfg["w"]),
                        dev(cfg["c"]), dev(cfg["gF"]))
    res = {k: host(t) for k, t in res.items()}
    rng = np.random.default_rng(4)
    x, w, c, gF, vec = cfg["x"], cfg["w"], cfg["c"], cfg["gF"], cfg["vec"]
    yr = O.sh(3, vec)
    assert_close(res["y"], yr, np.float32, "Y")
    nodes = _sample(rng, gr.N, 100)
    assert_close(res["out"][nodes],
                 O.conv_forward(prob, gr.rowptr, gr.sender, x, yr, w, 1.0, receivers=nodes)[nodes],
                 np.float32, "out rows")
    # edges incident to the sampled nodes (for the forces there)
    inc = np.zeros(gr.E, dtype=bool)
    inc[np.isin(gr.receiver, nodes) | np.isin(gr.sender, nodes)] = True
    edges = np.nonzero(inc)[0]
    rx, ry, rw = O.conv_backward(prob, gr.rowptr, gr.sender, x, yr, w, 1.0, c, nodes=nodes,
                                 edges=edges)
    assert_close(res["gx"][nodes], rx[nodes], np.float32, "gx rows")
    assert_close(res["gy"][edges], ry[edges], np.float32, "gy rows")
    assert_close(res["gw"][edges], rw[edges], np.float32, "gw rows")
    dEdr = np.zeros((gr.E, 3))
    dEdr[edges] = O.sh_vjp(3, vec[edges], ry[edges])
    assert_close(res["dEdr"][edges], dEdr[edges], np.float32, "dE/dr rows")
    F = O.edge_forces(gr.rowptr, gr.sender, dEdr)
    assert_close(res["F"][nodes], F[nodes], np.float32, "forces rows")
    q = gF[gr.sender].astype(np.float64) - gF[gr.receiver]
    ggy = O.sh_jvp(3, vec, q)
    assert_close(res["ggy"], ggy, np.float32, "ggY")
    dx, _, dw = O.conv_backward(prob, gr.rowptr, gr.sender, x, ggy, w, 1.0, c, nodes=nodes,
                                edges=edges)
    assert_close(res["d_x"][nodes], dx[nodes], np.float32, "dL/dx rows")
    assert_close(res["d_w"][edges], dw[edges], np.float32, "dL/dw rows")
    dLdr = np.zeros((gr.E, 3))
    dLdr[edges] = O.sh_hvp(3, vec[edges], ry[edges], q[edges])
    FL = O.edge_forces(gr.rowptr, gr.sender, dLdr)
    assert_close(res["FL"][nodes], FL[nodes], np.float32, "-dL/dpos rows")


def test_tfn_kv64_fused_sampled():
    """Keys and values from one TFN (the 1000-molecule graph at 64 channels): forward
    and gradient at full size, sampled receivers / senders / edges."""
    need_gpu()
    cfg = W.tfn_kv64_mol1000()
    conv_weights(cfg)  # the workload carries its own w
    _conv_sampled(cfg, np.float32, True)


def test_uvw_mixing_full_size():
    """The 'uvw' workload's channel mixing at full size (200,000 samples; 24
    path blocks of 128 channels into 128x(0e,1o,1e,2o,2e,3o,3e); its 24 shared
    [128, 128] matrices): forward, x-gradient and W-gradient through the
    calls the benchmark times.  The input is a 1000-sample block repeated 200
    times and copy k of the cotangent carries a sign s_k (107 plus, 93 minus,
    shuffled), so the oracle's results on the block give every output row and
    the W-gradient, a sum over 1.8 million rows per matrix set, is
    (sum_k s_k) = 14 times the block's."""
    need_gpu()
    cg = _cg()
    B, P = 200_000, 1000
    uvw = cg.UVWProduct(*W.IRREPS_MACE128)
    lin = uvw.linear
    assert lin.tensor_cores
    instr = [lin.instruction(j)[:2] for j in range(lin.n_instr)]
    Wm = W.mace128_uvw_b200k(P)["W"]
    rng = np.random.default_rng(23)
    X0 = rng.standard_normal((P, uvw.dim_mid)).astype(np.float32)
    G0 = rng.standard_normal((P, uvw.dim_out)).astype(np.float32)
    s = np.array([1.0] * 107 + [-1.0] * 93, dtype=np.float32)
    rng.shuffle(s)
    x = dev(X0).repeat(B // P, 1)
    g = (dev(G0).unsqueeze(0) * dev(s)[:, None, None]).reshape(B, uvw.dim_out)
    out = lin.forward(x, dev(Wm))
    gx, _ = lin.backward(x, dev(Wm), g, need=(True, False))
    _, gW = lin.backward(x, dev(Wm), g, need=(False, True))
    rout = O.linear_forward(uvw.mid, W.IRREPS_MACE128[2], instr, X0, Wm)
    rx, rW = O.linear_backward(uvw.mid, W.IRREPS_MACE128[2], instr, X0, Wm, G0)
    idx = _sample(rng, B, 3000)
    ti = torch.from_numpy(idx).cuda()
    assert_close(host(out[ti]), rout[idx % P], np.float32, "out rows")
    assert_close(host(gx[ti]), s[idx // P, None].astype(np.float64) * rx[idx % P], np.float32,
                 "grad_x rows")
    assert_close(host(gW), float(s.sum()) * rW, np.float32, "grad_W")
    assert cg.linear_device_status() == 0


def test_mace128_uvw_b200k_fused_forward_sampled():
    """The fused 'uvw' forward at full size (200,000 samples, 24 paths of 128
    channels into 128x(0e,1o,1e,2o,2e,3o,3e), the benchmark's call): every
    output row computed on the GPU, sampled rows by the oracle."""
    need_gpu()
    cg = _cg()
    cfg = W.mace128_uvw_b200k()
    B = cfg["B"]
    uvw = cg.UVWProduct(*W.IRREPS_MACE128)
    x = dev(cfg["x"])
    y = cg.sh_forward(dev(cfg["vec"]), 3)
    out = uvw.forward(x, y, dev(cfg["W"]))
    rng = np.random.default_rng(29)
    idx = _sample(rng, B, 2000)
    ti = torch.from_numpy(idx).cuda()
    ref = O.tp_uvw_forward(*W.IRREPS_MACE128, cfg["x"][idx], host(y[ti]), cfg["W"])
    assert_close(host(out[ti]), ref, np.float32, "uvw out rows")
    assert cg.linear_device_status() == 0
