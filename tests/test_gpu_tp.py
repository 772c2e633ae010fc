"""GPU parity of the standalone tensor product, its gradient and double
backward against the oracle, through the C ABI (via the ctypes binding).

Irreps cover the launch geometries the generator picks: one lane per channel
pair with several slots per warp (mul 16), a full warp (64), two warps per
slot (128), masked lanes (mul 3, 96), odd multiplicity (scalar path) and fp64.
Batch sizes are ragged (1, 7, 333).
"""
import numpy as np
import pytest

import oracle as O
from tests.gpu_util import assert_close, dev, host, need_gpu, torch

pytestmark = pytest.mark.gpu

CASES = [
    ("16x0e+16x1o", "0e+1o+2e", "16x0e+16x1o+16x2e", np.float32),
    ("3x0e+3x1o+3x2e", "0e+1o+2e+3o", "3x0e+3x1o+3x1e+3x2o+3x2e+3x3o+3x3e", np.float32),
    ("64x0e+64x1o+64x2e", "0e+1o+2e+3o", "64x0e+64x1o+64x1e+64x2o+64x2e+64x3o+64x3e",
     np.float32),
    ("128x0e+128x1o", "0e+1o+2e", "128x0e+128x1o+128x1e+128x2e", np.float32),
    ("96x1o+96x2e", "1o+2e", "96x0e+96x1e+96x2e+96x3o", np.float32),
    ("2x0e+2x1o+2x2e+2x3o", "0e+1o+2e+3o", "2x0e+2x1o+2x2e+2x3o", np.float32),
    ("5x0e+5x1o+5x2e", "0e+1o+2e+3o", "5x0e+5x1o+5x2e+5x3o", np.float64),
    ("32x0e+32x1o+32x2e", "0e+1o+2e+3o", "32x0e+32x1o+32x2e+32x3o", np.float64),
]


def _plan(a, b, c, dt):
    import clebsch_gordan_tensor_gb300 as cg
    return cg.Plan(a, b, c, dtype=torch.float64 if dt == np.float64 else torch.float32)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{np.dtype(c[3]).name}")
@pytest.mark.parametrize("B", [1, 7, 333])
def test_forward_backward(case, B):
    need_gpu()
    a, b, c, dt = case
    prob = O.make_problem(a, b, c)
    plan = _plan(a, b, c, dt)
    rng = np.random.default_rng(B)
    x = rng.standard_normal((B, prob.dim1)).astype(dt)
    y = rng.standard_normal((B, prob.dim2)).astype(dt)
    w = rng.standard_normal((B, prob.wdim)).astype(dt)
    g = rng.standard_normal((B, prob.dimo)).astype(dt)
    out = plan.forward(dev(x), dev(y), dev(w))
    assert_close(host(out), O.tp_forward(prob, x, y, w), dt, "forward")
    gx, gy, gw = plan.backward(dev(x), dev(y), dev(w), dev(g))
    rx, ry, rw = O.tp_backward(prob, x, y, w, g)
    assert_close(host(gx), rx, dt, "grad_x")
    assert_close(host(gy), ry, dt, "grad_y")
    assert_close(host(gw), rw, dt, "grad_w")
    # subsets of outputs
    gx2, gy2, gw2 = plan.backward(dev(x), dev(y), dev(w), dev(g), need=(False, True, False))
    assert gx2 is None and gw2 is None
    assert_close(host(gy2), ry, dt, "grad_y alone")
    _, _, gw3 = plan.backward(dev(x), dev(y), dev(w), dev(g), need=(False, False, True))
    assert_close(host(gw3), rw, dt, "grad_w alone")


@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[3], CASES[6]],
                         ids=lambda c: f"{c[0]}-{np.dtype(c[3]).name}")
@pytest.mark.parametrize("which", ["all", "y", "x", "w"])
def test_double_backward(case, which):
    need_gpu()
    a, b, c, dt = case
    prob = O.make_problem(a, b, c)
    plan = _plan(a, b, c, dt)
    B = 37
    rng = np.random.default_rng(5)
    x, y, w, g = (rng.standard_normal((B, d)).astype(dt)
                  for d in (prob.dim1, prob.dim2, prob.wdim, prob.dimo))
    ggx = rng.standard_normal(x.shape).astype(dt) if which in ("all", "x") else None
    ggy = rng.standard_normal(y.shape).astype(dt) if which in ("all", "y") else None
    ggw = rng.standard_normal(w.shape).astype(dt) if which in ("all", "w") else None
    d = plan.double_backward(dev(x), dev(y), dev(w), dev(g),
                             None if ggx is None else dev(ggx), None if ggy is None else dev(ggy),
                             None if ggw is None else dev(ggw))
    r = O.tp_double_backward(prob, x, y, w, g, ggx, ggy, ggw)
    for k, name in enumerate(("d_x", "d_y", "d_w", "d_grad_out")):
        assert_close(host(d[k]), r[k], dt, name)


def test_shared_weights_forward():
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    a, b, c = "8x0e+8x1o", "0e+1o+2e", "8x0e+8x1o+8x2e"
    prob = O.make_problem(a, b, c)
    plan = cg.Plan(a, b, c, shared_weights=True)
    rng = np.random.default_rng(9)
    x = rng.standard_normal((50, prob.dim1)).astype(np.float32)
    y = rng.standard_normal((50, prob.dim2)).astype(np.float32)
    w = rng.standard_normal(prob.wdim).astype(np.float32)
    out = plan.forward(dev(x), dev(y), dev(w))
    assert_close(host(out), O.tp_forward(prob, x, y, w), np.float32, "shared forward")
    g = rng.standard_normal((50, prob.dimo)).astype(np.float32)
    gx, gy, gw = plan.backward(dev(x), dev(y), dev(w), dev(g))
    rx, ry, rw = O.tp_backward(prob, x, y, w, g)
    assert_close(host(gx), rx, np.float32, "shared grad_x")
    assert_close(host(gy), ry, np.float32, "shared grad_y")
    assert gw.shape == (prob.wdim,)
    assert_close(host(gw), rw, np.float32, "shared grad_w (sum over samples)")


@pytest.mark.parametrize("B", [1, 3, 5000])
@pytest.mark.parametrize("irreps,dt", [(("64x0e+64x1o+64x2e", "0e+1o+2e+3o",
                                         "64x0e+64x1o+64x1e+64x2o+64x2e+64x3o+64x3e"), np.float32),
                                       (("3x0e+3x1o", "0e+1o", "3x0e+3x1o"), np.float32),
                                       (("8x0e+8x1o", "0e+1o+2e", "8x0e+8x1o+8x2e"), np.float64)])
def test_shared_weight_gradient(B, irreps, dt):
    """grad_w of a shared weight row: per-CTA partial rows reduced in order."""
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    prob = O.make_problem(*irreps)
    plan = cg.Plan(*irreps, dtype=torch.float64 if dt == np.float64 else torch.float32,
                   shared_weights=True)
    rng = np.random.default_rng(B)
    x = rng.standard_normal((B, prob.dim1)).astype(dt)
    y = rng.standard_normal((B, prob.dim2)).astype(dt)
    w = rng.standard_normal(prob.wdim).astype(dt)
    g = rng.standard_normal((B, prob.dimo)).astype(dt)
    _, _, gw = plan.backward(dev(x), dev(y), dev(w), dev(g), need=(False, False, True))
    _, _, rw = O.tp_backward(prob, x, y, w, g)
    assert_close(host(gw), rw, dt, "shared grad_w")
    with pytest.raises(cg.CgtpError, match="workspace"):
        cg._check(cg.lib().cgtp_backward(plan._h, B, cg._ptr(dev(x)), cg._ptr(dev(y)),
                                         cg._ptr(dev(w)), cg._ptr(dev(g)), None, None,
                                         cg._ptr(torch.empty_like(dev(w))), cg._stream()))


@pytest.mark.parametrize("B", [1, 3, 5000])
@pytest.mark.parametrize("irreps,dt", [(("64x0e+64x1o+64x2e", "0e+1o+2e+3o",
                                         "64x0e+64x1o+64x1e+64x2o+64x2e+64x3o+64x3e"), np.float32),
                                       (("8x0e+8x1o", "0e+1o+2e", "8x0e+8x1o+8x2e"), np.float64)])
def test_shared_weight_double_backward(B, irreps, dt):
    """Double backward of a shared weight row: d_w sums both terms over all
    samples (partial rows of the two terms side by side, one ordered sum)."""
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    prob = O.make_problem(*irreps)
    plan = cg.Plan(*irreps, dtype=torch.float64 if dt == np.float64 else torch.float32,
                   shared_weights=True)
    rng = np.random.default_rng(B + 1)
    x = rng.standard_normal((B, prob.dim1)).astype(dt)
    y = rng.standard_normal((B, prob.dim2)).astype(dt)
    w = rng.standard_normal(prob.wdim).astype(dt)
    g = rng.standard_normal((B, prob.dimo)).astype(dt)
    ggx, ggy, ggw = (rng.standard_normal(a.shape).astype(dt) for a in (x, y, w))
    got = plan.double_backward(dev(x), dev(y), dev(w), dev(g), dev(ggx), dev(ggy), dev(ggw))
    ref = O.tp_double_backward(prob, x, y, w, g, ggx, ggy, ggw)
    for a, r, n in zip(got, ref, ("d_x", "d_y", "d_w", "d_g")):
        assert_close(host(a), r, dt, n)
    # d_w from the gg_y term alone
    _, _, dw, _ = plan.double_backward(dev(x), dev(y), dev(w), dev(g), None, dev(ggy), None,
                                       need=(False, False, True, False))
    assert_close(host(dw), O.tp_double_backward(prob, x, y, w, g, None, ggy, None)[2], dt,
                 "d_w (gg_y only)")
    # without the workspace the entry point refuses a shared d_w
    with pytest.raises(cg.CgtpError, match="workspace"):
        cg._check(cg.lib().cgtp_double_backward(
            plan._h, B, cg._ptr(dev(x)), cg._ptr(dev(y)), cg._ptr(dev(w)), cg._ptr(dev(g)),
            cg._ptr(dev(ggx)), None, None, None, None, cg._ptr(torch.empty_like(dev(w))), None,
            cg._stream()))


def test_empty_batch_is_noop():
    need_gpu()
    plan = _plan(*CASES[0])
    x = torch.zeros(0, plan.dim_in1, device="cuda")
    y = torch.zeros(0, plan.dim_in2, device="cuda")
    w = torch.zeros(0, plan.weight_numel, device="cuda")
    assert plan.forward(x, y, w).shape == (0, plan.dim_out)
