"""GPU parity of plans whose weights are stored in a 16-bit format, bfloat16
or IEEE binary16 (fp32 arithmetic, features and gradients): standalone and
fused-conv forward and backward, the staged and the direct kernels, per-edge
and shared weights, and the radial network writing 16-bit weights.  The oracle
receives the same 16-bit values widened to fp64, so the comparison keeps the
fp32 tolerance."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests.gpu_util import assert_close, dev, host, need_gpu, torch

pytestmark = pytest.mark.gpu


WDT = ["bfloat16", "float16"]


def _w16(a, wdt):
    """16-bit device tensor and the exact fp64 values it holds."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(getattr(torch, wdt)).cuda()
    return t, t.float().cpu().numpy().astype(np.float64)


CASES = [
    W.IRREPS_CONV64,                                                   # mul 64: two channels per lane, staged
    ("3x0e+3x1o", "0e+1o+2e", "3x0e+3x1o+3x2e"),              # masked lanes, direct
    ("5x0e+5x1o", "0e+1o+2e", "5x0e+5x1o+5x2e"),              # odd mul: one channel per lane
    (W.IRREPS_MACE128[0], W.IRREPS_MACE128[1], W.IRREPS_MACE128[2]),                        # mul 128: two warps per item
]


@pytest.mark.parametrize("irreps", CASES, ids=lambda c: c[0][:10])
@pytest.mark.parametrize("B", [1, 333])
@pytest.mark.parametrize("wdt", WDT)
def test_standalone_16bit_weights(irreps, B, wdt):
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    prob = O.make_problem(*irreps)
    plan = cg.Plan(*irreps, weight_dtype=getattr(torch, wdt))
    rng = np.random.default_rng(B)
    x = rng.standard_normal((B, prob.dim1)).astype(np.float32)
    y = rng.standard_normal((B, prob.dim2)).astype(np.float32)
    wd, wr = _w16(rng.standard_normal((B, prob.wdim)), wdt)
    g = rng.standard_normal((B, prob.dimo)).astype(np.float32)
    out = plan.forward(dev(x), dev(y), wd)
    assert_close(host(out), O.tp_forward(prob, x, y, wr), np.float32, "forward")
    gx, gy, gw = plan.backward(dev(x), dev(y), wd, dev(g))
    assert gw.dtype == torch.float32
    rx, ry, rw = O.tp_backward(prob, x, y, wr, g)
    assert_close(host(gx), rx, np.float32, "grad_x")
    assert_close(host(gy), ry, np.float32, "grad_y")
    assert_close(host(gw), rw, np.float32, "grad_w")
    with pytest.raises(cg.CgtpError, match="unsupported"):
        plan.double_backward(dev(x), dev(y), wd, dev(g), gg_x=dev(x))


def _cloud(n):
    rng = np.random.default_rng(n)
    _, _, gr = W.periodic_cloud(rng, n)
    return gr, rng


@pytest.mark.parametrize("misaligned", [False, True], ids=["staged", "direct"])
@pytest.mark.parametrize("wdt", WDT)
def test_conv_16bit_weights(misaligned, wdt):
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    gr, rng = _cloud(600)
    irreps = W.IRREPS_CONV64
    prob = O.make_problem(*irreps)
    plan = cg.Plan(*irreps, weight_dtype=getattr(torch, wdt))
    G = cg.Graph.from_numpy(gr)
    x = rng.standard_normal((gr.N, prob.dim1)).astype(np.float32)
    y = rng.standard_normal((gr.E, prob.dim2)).astype(np.float32)
    wd, wr = _w16(rng.standard_normal((gr.E, prob.wdim)), wdt)
    if misaligned:  # a 4-byte offset view: not 16-byte aligned, so the direct kernels run
        buf = torch.empty(gr.E * prob.wdim + 2, dtype=getattr(torch, wdt), device="cuda")
        view = buf[2:].view(gr.E, prob.wdim)
        view.copy_(wd)
        wd = view
    g = rng.standard_normal((gr.N, prob.dimo)).astype(np.float32)
    out = plan.conv_forward(G, dev(x), dev(y), wd, 0.02)
    ref = O.conv_forward(prob, gr.rowptr, gr.sender, x, y, wr, 0.02)
    assert_close(host(out), ref, np.float32, "conv out")
    gx, gy, gw = plan.conv_backward(G, dev(x), dev(y), wd, 0.02, dev(g))
    rx, ry, rw = O.conv_backward(prob, gr.rowptr, gr.sender, x, y, wr, 0.02, g)
    assert_close(host(gx), rx, np.float32, "conv grad_x")
    assert_close(host(gy), ry, np.float32, "conv grad_y")
    assert_close(host(gw), rw, np.float32, "conv grad_w")
    assert plan.device_status() == 0


@pytest.mark.parametrize("wdt", WDT)
def test_shared_16bit_weights(wdt):
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    irreps = ("8x0e+8x1o", "0e+1o+2e", "8x0e+8x1o+8x2e")
    prob = O.make_problem(*irreps)
    plan = cg.Plan(*irreps, shared_weights=True, weight_dtype=getattr(torch, wdt))
    rng = np.random.default_rng(4)
    B = 700
    x = rng.standard_normal((B, prob.dim1)).astype(np.float32)
    y = rng.standard_normal((B, prob.dim2)).astype(np.float32)
    wd, wr = _w16(rng.standard_normal(prob.wdim), wdt)
    g = rng.standard_normal((B, prob.dimo)).astype(np.float32)
    out = plan.forward(dev(x), dev(y), wd)
    assert_close(host(out), O.tp_forward(prob, x, y, wr), np.float32, "shared forward")
    _, _, gw = plan.backward(dev(x), dev(y), wd, dev(g), need=(False, False, True))
    assert_close(host(gw), O.tp_backward(prob, x, y, wr, g)[2], np.float32, "shared grad_w")


@pytest.mark.parametrize("cuda_cores", [False, True])
@pytest.mark.parametrize("wdt", WDT)
def test_radial_writes_16bit(cuda_cores, wdt):
    """16-bit output: each element is the fp32 result rounded to nearest (p = 8
    significant bits for bfloat16, 11 for binary16), so it lies within half a
    unit (at most 2^-p relative) of the fp32 result, which is itself within the
    fp32 normwise tolerance (1e-5 of the largest value) of the oracle; and it is
    exactly torch's rounding of the fp32 path's output."""
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    rng = np.random.default_rng(8)
    E, nb, hidden, n_out = 1111, 8, 64, 1536
    d = rng.standard_normal((E, 3))
    vec = (d / np.linalg.norm(d, axis=1, keepdims=True) * rng.uniform(0.5, 5, (E, 1))).astype(np.float32)
    W1 = (rng.standard_normal((nb, hidden)) / np.sqrt(nb)).astype(np.float32)
    W2 = (rng.standard_normal((hidden, n_out)) / 8).astype(np.float32)
    odt = getattr(torch, wdt)
    p = 8 if wdt == "bfloat16" else 11
    w = cg.radial_forward(dev(vec), dev(W1), dev(W2), out_dtype=odt, cuda_cores=cuda_cores)
    assert w.dtype == odt
    rw, _ = O.radial_forward(vec, W1, W2)
    got = w.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - rw)
    assert np.all(err <= 2.0 ** -p * np.abs(rw) * (1 + 1e-3) + 1e-5 * np.abs(rw).max())
    # rounding is to nearest: the typical error is a quarter of a unit or less
    assert np.median(err / np.maximum(np.abs(rw), 1e-30)) < 2.0 ** -(p + 1)
    wf = cg.radial_forward(dev(vec), dev(W1), dev(W2), cuda_cores=cuda_cores)
    assert torch.equal(w, wf.to(odt))
    assert cg.radial_device_status() == 0
    # and it feeds a plan with the same weight storage directly
    plan = cg.Plan(*W.IRREPS_CONV64, weight_dtype=odt)
    assert w.shape[1] == plan.weight_numel
