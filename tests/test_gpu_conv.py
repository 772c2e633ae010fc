"""GPU parity of the fused graph convolution (forward, gradient, double
backward), spherical harmonics and force kernels against the oracle.

Small graphs include receivers without edges, a node that never sends, and an
edgeless graph; sizes span several CTAs with a ragged tail.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests.gpu_util import assert_close, dev, host, need_gpu, torch

pytestmark = pytest.mark.gpu


def _cg():
    import clebsch_gordan_tensor_gb300 as cg
    return cg


def _graph(rng, N, max_deg=9, isolated=(3,), silent=(5,)):
    recv, send = [], []
    for n in range(N):
        if n in isolated:
            continue
        k = int(rng.integers(0, max_deg + 1))
        cand = [s for s in range(N) if s not in silent]
        for s in rng.choice(cand, size=min(k, len(cand)), replace=False):
            recv.append(n)
            send.append(int(s))
    vec = rng.standard_normal((len(recv), 3))
    return W.make_graph(N, np.array(recv, dtype=np.int64), np.array(send, dtype=np.int64), vec)


CASES = [
    (W.IRREPS_CONV64[0].replace("64x", "8x"), W.IRREPS_CONV64[1], W.IRREPS_CONV64[2].replace("64x", "8x"), np.float32),
    W.IRREPS_CONV64 + (np.float32,),
    W.IRREPS_TFN32 + (np.float32,),
    (W.IRREPS_MACE128[0], W.IRREPS_MACE128[1], W.IRREPS_MACE128[2], np.float32),
    ("3x0e+3x1o", "0e+1o+2e", "3x0e+3x1o+3x2e", np.float32),
    (W.IRREPS_CONV128[0].replace("128x", "16x"), W.IRREPS_CONV128[1], W.IRREPS_CONV128[2].replace("128x", "16x"), np.float64),
    W.IRREPS_CONV128 + (np.float64,),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0][:12]}-{np.dtype(c[3]).name}")
def test_conv_forward_backward(case):
    need_gpu()
    cg = _cg()
    a, b, c, dt = case
    prob = O.make_problem(a, b, c)
    plan = cg.Plan(a, b, c, dtype=torch.float64 if dt == np.float64 else torch.float32)
    rng = np.random.default_rng(1)
    gr = _graph(rng, 41)
    G = cg.Graph.from_numpy(gr)
    x = rng.standard_normal((gr.N, prob.dim1)).astype(dt)
    y = rng.standard_normal((gr.E, prob.dim2)).astype(dt)
    w = rng.standard_normal((gr.E, prob.wdim)).astype(dt)
    g = rng.standard_normal((gr.N, prob.dimo)).astype(dt)
    scale = 0.37
    out = plan.conv_forward(G, dev(x), dev(y), dev(w), scale)
    ref = O.conv_forward(prob, gr.rowptr, gr.sender, x, y, w, scale)
    assert_close(host(out), ref, dt, "conv forward")
    assert not host(out)[3].any()
    gx, gy, gw = plan.conv_backward(G, dev(x), dev(y), dev(w), scale, dev(g))
    rx, ry, rw = O.conv_backward(prob, gr.rowptr, gr.sender, x, y, w, scale, g)
    assert_close(host(gx), rx, dt, "conv grad_x")
    assert not host(gx)[5].any()
    assert_close(host(gy), ry, dt, "conv grad_y")
    assert_close(host(gw), rw, dt, "conv grad_w")


@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[5]],
                         ids=lambda c: f"{c[0][:12]}-{np.dtype(c[3]).name}")
@pytest.mark.parametrize("which", ["all", "y"])
def test_conv_double_backward(case, which):
    need_gpu()
    cg = _cg()
    a, b, c, dt = case
    prob = O.make_problem(a, b, c)
    plan = cg.Plan(a, b, c, dtype=torch.float64 if dt == np.float64 else torch.float32)
    rng = np.random.default_rng(2)
    gr = _graph(rng, 23)
    G = cg.Graph.from_numpy(gr)
    x = rng.standard_normal((gr.N, prob.dim1)).astype(dt)
    y = rng.standard_normal((gr.E, prob.dim2)).astype(dt)
    w = rng.standard_normal((gr.E, prob.wdim)).astype(dt)
    g = rng.standard_normal((gr.N, prob.dimo)).astype(dt)
    ggy = rng.standard_normal(y.shape).astype(dt)
    ggx = rng.standard_normal(x.shape).astype(dt) if which == "all" else None
    ggw = rng.standard_normal(w.shape).astype(dt) if which == "all" else None
    d = plan.conv_double_backward(G, dev(x), dev(y), dev(w), 0.5, dev(g),
                                  None if ggx is None else dev(ggx), dev(ggy),
                                  None if ggw is None else dev(ggw))
    r = O.conv_double_backward(prob, gr.rowptr, gr.sender, x, y, w, 0.5, g, ggx, ggy, ggw)
    for k, name in enumerate(("d_x", "d_y", "d_w", "d_grad_out")):
        assert_close(host(d[k]), r[k], dt, name)


def test_edgeless_graph_writes_zeros():
    need_gpu()
    cg = _cg()
    plan = cg.Plan(*W.IRREPS_CONV64)
    gr = W.make_graph(6, np.zeros(0, np.int64), np.zeros(0, np.int64), np.zeros((0, 3)))
    G = cg.Graph.from_numpy(gr)
    x = torch.randn(6, plan.dim_in1, device="cuda")
    y = torch.zeros(0, plan.dim_in2, device="cuda")
    w = torch.zeros(0, plan.weight_numel, device="cuda")
    out = torch.full((6, plan.dim_out), 7.0, device="cuda")
    plan.conv_forward(G, x, y, w, 1.0, out=out)
    assert not host(out).any()
    gx, gy, gw = plan.conv_backward(G, x, y, w, 1.0, torch.randn(6, plan.dim_out, device="cuda"))
    assert not host(gx).any() and gy.numel() == 0 and gw.numel() == 0


@pytest.mark.parametrize("lmax", range(7))
@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_spherical_harmonics(lmax, dt):
    need_gpu()
    cg = _cg()
    rng = np.random.default_rng(lmax)
    v = (rng.standard_normal((1000, 3)) * rng.uniform(0.1, 5, (1000, 1))).astype(dt)
    gy = rng.standard_normal((1000, (lmax + 1) ** 2)).astype(dt)
    t = rng.standard_normal((1000, 3)).astype(dt)
    assert_close(host(cg.sh_forward(dev(v), lmax)), O.sh(lmax, v), dt, "sh")
    assert_close(host(cg.sh_backward(dev(v), dev(gy), lmax)), O.sh_vjp(lmax, v, gy), dt, "vjp")
    assert_close(host(cg.sh_jvp(dev(v), dev(t), lmax)), O.sh_jvp(lmax, v, t), dt, "jvp")
    assert_close(host(cg.sh_hvp(dev(v), dev(gy), dev(t), lmax)), O.sh_hvp(lmax, v, gy, t), dt,
                 "hvp")


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_edge_forces_and_adjoint(dt):
    need_gpu()
    cg = _cg()
    rng = np.random.default_rng(3)
    gr = _graph(rng, 57)
    G = cg.Graph.from_numpy(gr)
    d = rng.standard_normal((gr.E, 3)).astype(dt)
    F = cg.edge_forces(G, dev(d))
    Fr = O.edge_forces(gr.rowptr, gr.sender, d)
    assert_close(host(F), Fr, dt, "forces")
    gF = rng.standard_normal((gr.N, 3)).astype(dt)
    q = host(cg.edge_forces_adjoint(G, dev(gF)))
    # adjoint identity with the oracle's forces: <q, d> = <gF, F(d)>
    for _ in range(3):
        d2 = rng.standard_normal((gr.E, 3))
        lhs, rhs = (q * d2).sum(), (gF * O.edge_forces(gr.rowptr, gr.sender, d2)).sum()
        assert abs(lhs - rhs) <= 1e-5 * max(1.0, abs(rhs))


def tfn_chain_gpu(cg, plan, G, x, vec, w, c, gF, lmax=3):
    """TFN-layer step (1000 molecules): energy E = sum c * conv(x, Y(vec), w); gradients dE/dx,
    dE/dw, dE/dvec; forces; force loss L = sum gF * F; dL/dx, dL/dw, and
    FL = edge_forces(dL/dr) = -dL/dpos."""
    y = cg.sh_forward(vec, lmax)
    out = plan.conv_forward(G, x, y, w, 1.0)
    gx, gy, gw = plan.conv_backward(G, x, y, w, 1.0, c)
    dEdr = cg.sh_backward(vec, gy, lmax)
    F = cg.edge_forces(G, dEdr)
    q = cg.edge_forces_adjoint(G, gF)
    ggy = cg.sh_jvp(vec, q, lmax)
    d_x, _, d_w, _ = plan.conv_double_backward(G, x, y, w, 1.0, c, None, ggy, None,
                                               need=(True, False, True, False))
    FL = cg.edge_forces(G, cg.sh_hvp(vec, gy, q, lmax))
    return dict(y=y, out=out, gx=gx, gy=gy, gw=gw, dEdr=dEdr, F=F, ggy=ggy, d_x=d_x, d_w=d_w,
                FL=FL)


def tfn_chain_oracle(prob, gr, x, vec, w, c, gF, lmax=3, nodes=None, edges=None):
    y = O.sh(lmax, vec)
    res = dict(y=y)
    res["out"] = O.conv_forward(prob, gr.rowptr, gr.sender, x, y, w, 1.0, receivers=nodes)
    gx, gy, gw = O.conv_backward(prob, gr.rowptr, gr.sender, x, y, w, 1.0, c)
    res.update(gx=gx, gy=gy, gw=gw)
    res["dEdr"] = O.sh_vjp(lmax, vec, gy)
    res["F"] = O.edge_forces(gr.rowptr, gr.sender, res["dEdr"])
    q = gF[gr.sender] - gF[gr.receiver]  # adjoint of edge_forces (pinned above)
    res["ggy"] = O.sh_jvp(lmax, vec, q)
    d = O.conv_double_backward(prob, gr.rowptr, gr.sender, x, y, w, 1.0, c, None, res["ggy"], None)
    res.update(d_x=d[0], d_w=d[2])
    res["FL"] = O.edge_forces(gr.rowptr, gr.sender, O.sh_hvp(lmax, vec, gy, q))
    return res


def test_tfn_force_chain_small():
    need_gpu()
    cg = _cg()
    cfg = W.tfn32_mol1000(n_mol=40)
    gr = cfg["graph"]
    prob = O.make_problem(*W.IRREPS_TFN32)
    plan = cg.Plan(*W.IRREPS_TFN32)
    G = cg.Graph.from_numpy(gr)
    gpu = tfn_chain_gpu(cg, plan, G, dev(cfg["x"]), dev(cfg["vec"]), dev(cfg["w"]),
                        dev(cfg["c"]), dev(cfg["gF"]))
    ref = tfn_chain_oracle(prob, gr, cfg["x"], cfg["vec"], cfg["w"], cfg["c"], cfg["gF"])
    for k in ("y", "out", "gx", "gy", "gw", "dEdr", "F", "ggy", "d_x", "d_w", "FL"):
        assert_close(host(gpu[k]), ref[k], np.float32, k)


def _offset_view(a, dtype):
    """Device copy of a whose data pointer is 8 but not 16 bytes aligned, so
    the library takes its direct-load kernels instead of the staged ones."""
    t = torch.from_numpy(np.ascontiguousarray(a)).to(dtype)
    k = 8 // t.element_size()
    buf = torch.zeros(t.numel() + k, dtype=dtype, device="cuda")
    v = buf[k:].view(t.shape)
    v.copy_(t.cuda())
    assert v.data_ptr() % 16 == 8
    return v


@pytest.mark.parametrize("case", [CASES[1], CASES[3], CASES[6]],
                         ids=lambda c: f"{c[0][:12]}-{np.dtype(c[3]).name}")
def test_staged_and_direct_paths_agree(case):
    """The staged (TMA) and direct kernels give the oracle's result; the
    direct ones are selected by 16-byte-misaligned inputs."""
    need_gpu()
    cg = _cg()
    a, b, c, dt = case
    tdt = torch.float64 if dt == np.float64 else torch.float32
    prob = O.make_problem(a, b, c)
    plan = cg.Plan(a, b, c, dtype=tdt)
    rng = np.random.default_rng(11)
    gr = _graph(rng, 70, max_deg=12)
    G = cg.Graph.from_numpy(gr)
    x = rng.standard_normal((gr.N, prob.dim1)).astype(dt)
    y = rng.standard_normal((gr.E, prob.dim2)).astype(dt)
    w = rng.standard_normal((gr.E, prob.wdim)).astype(dt)
    g = rng.standard_normal((gr.N, prob.dimo)).astype(dt)
    ref = O.conv_forward(prob, gr.rowptr, gr.sender, x, y, w, 0.5)
    rx, ry, rw = O.conv_backward(prob, gr.rowptr, gr.sender, x, y, w, 0.5, g)
    for mk in (dev, lambda arr: _offset_view(arr, tdt)):
        xs, ys, ws, gs = mk(x), mk(y), mk(w), mk(g)
        out = plan.conv_forward(G, xs, ys, ws, 0.5)
        assert_close(host(out), ref, dt, "forward")
        gx, gy, gw = plan.conv_backward(G, xs, ys, ws, 0.5, gs)
        assert_close(host(gx), rx, dt, "grad_x")
        assert_close(host(gy), ry, dt, "grad_y")
        assert_close(host(gw), rw, dt, "grad_w")
    code = __import__("ctypes").c_int(-1)
    assert cg.lib().cgtp_plan_device_status(plan._h, __import__("ctypes").byref(code)) == 0
    assert code.value == 0


@pytest.mark.parametrize("case", [CASES[1], CASES[5]], ids=lambda c: f"{c[0][:12]}-{np.dtype(c[3]).name}")
def test_conv_shared_weight_gradient(case):
    """Fused convolution with one weight row shared by every edge: grad_w sums
    over all edges (per-CTA partial rows, ordered reduction)."""
    need_gpu()
    cg = _cg()
    a, b, c, dt = case
    prob = O.make_problem(a, b, c)
    plan = cg.Plan(a, b, c, dtype=torch.float64 if dt == np.float64 else torch.float32,
                   shared_weights=True)
    rng = np.random.default_rng(21)
    gr = _graph(rng, 300, max_deg=12)
    G = cg.Graph.from_numpy(gr)
    x = rng.standard_normal((gr.N, prob.dim1)).astype(dt)
    y = rng.standard_normal((gr.E, prob.dim2)).astype(dt)
    w = rng.standard_normal(prob.wdim).astype(dt)
    g = rng.standard_normal((gr.N, prob.dimo)).astype(dt)
    out = plan.conv_forward(G, dev(x), dev(y), dev(w), 0.25)
    assert_close(host(out), O.conv_forward(prob, gr.rowptr, gr.sender, x, y, w, 0.25), dt, "fwd")
    gx, gy, gw = plan.conv_backward(G, dev(x), dev(y), dev(w), 0.25, dev(g))
    rx, ry, rw = O.conv_backward(prob, gr.rowptr, gr.sender, x, y, w, 0.25, g)
    assert_close(host(gx), rx, dt, "grad_x")
    assert_close(host(gy), ry, dt, "grad_y")
    assert_close(host(gw), rw, dt, "grad_w")
    # double backward: d_w sums both terms over all edges
    ggx, ggy, ggw = (rng.standard_normal(a.shape).astype(dt) for a in (x, y, w))
    got = plan.conv_double_backward(G, dev(x), dev(y), dev(w), 0.25, dev(g), dev(ggx), dev(ggy),
                                    dev(ggw))
    ref = O.conv_double_backward(prob, gr.rowptr, gr.sender, x, y, w, 0.25, g, ggx, ggy, ggw)
    for a, r, n in zip(got, ref, ("d_x", "d_y", "d_w", "d_g")):
        assert_close(host(a), r, dt, "double backward " + n)
