"""Failure detection without a GPU fault: the staged kernels' bounded waits.

Every wait of the staged tensor-product kernels on a bulk copy is bounded;
when one runs out the kernel records a code in the plan's device error flag,
waits (bounded) for the copies it still has in flight and returns, so the
context stays usable.  The test-only plan flag CGTP_PLAN_TEST_WAIT_TIMEOUT
makes the first wait of every CTA give up at once, which runs that path with
no real stall: nothing faults, traps or hangs.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests.gpu_util import assert_close, dev, host, need_gpu, torch

pytestmark = pytest.mark.gpu


def _status(plan):
    """(status code of cgtp_plan_device_status, device error code)."""
    import ctypes
    import clebsch_gordan_tensor_gb300 as cg
    code = ctypes.c_int(-1)
    st = cg.lib().cgtp_plan_device_status(plan._h, ctypes.byref(code))
    return st, code.value


def test_bounded_wait_timeout_reports_and_context_survives():
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg

    rng = np.random.default_rng(11)
    _, _, gr = W.periodic_cloud(rng, 300)
    G = cg.Graph.from_numpy(gr)
    bad = cg.Plan(*W.IRREPS_CONV64, flags=cg.TEST_WAIT_TIMEOUT)
    good = cg.Plan(*W.IRREPS_CONV64)
    prob = O.make_problem(*W.IRREPS_CONV64)
    xh = rng.standard_normal((gr.N, good.dim_in1)).astype(np.float32)
    yh = rng.standard_normal((gr.E, good.dim_in2)).astype(np.float32)
    wh = rng.standard_normal((gr.E, good.weight_numel)).astype(np.float32)
    gh = rng.standard_normal((gr.N, good.dim_out)).astype(np.float32)
    x, y, w, g = dev(xh), dev(yh), dev(wh), dev(gh)
    # forward: the stage wait of the first edge gives up (code 1)
    bad.conv_forward(G, x, y, w, 0.5)
    torch.cuda.synchronize()
    assert _status(bad) == (9, 1)  # CGTP_E_DEVICE, code 1
    assert _status(bad) == (0, 0)   # read once, then cleared
    # backward: the wait for the first sender's x row gives up (code 2)
    bad.conv_backward(G, x, y, w, 0.5, g)
    torch.cuda.synchronize()
    assert _status(bad) == (9, 2)
    assert _status(bad) == (0, 0)
    # the context is still usable: a normal plan gives the oracle's results
    out = good.conv_forward(G, x, y, w, 0.5)
    gx, gy, gw = good.conv_backward(G, x, y, w, 0.5, g)
    assert_close(host(out), O.conv_forward(prob, gr.rowptr, gr.sender, xh, yh, wh, 0.5),
                 np.float32, "out after the timed-out launches")
    rx, ry, rw = O.conv_backward(prob, gr.rowptr, gr.sender, xh, yh, wh, 0.5, gh)
    assert_close(host(gx), rx, np.float32, "grad_x")
    assert_close(host(gy), ry, np.float32, "grad_y")
    assert_close(host(gw), rw, np.float32, "grad_w")
    assert _status(good) == (0, 0)


def test_radial_tensor_core_timeout_reports_and_context_survives():
    """The radial network's tensor-core kernel with its first bounded wait
    giving up (CGTP_RADIAL_TEST_WAIT_TIMEOUT): the flag is reported once, the
    tensor memory is released (the next launch allocates it again) and a
    normal call matches the oracle."""
    need_gpu()
    import ctypes
    import clebsch_gordan_tensor_gb300 as cg

    rng = np.random.default_rng(12)
    E = 1000
    vec = rng.standard_normal((E, 3)).astype(np.float32)
    W1, W2 = W.radial_params(rng, 256)
    v, a, b = dev(vec), dev(W1), dev(W2)
    out = torch.empty(E, 256, device="cuda")
    n = ctypes.c_size_t()
    L = cg.lib()
    assert L.cgtp_radial_workspace(0, 8, 64, 256, ctypes.byref(n)) == 0 and n.value > 0
    ws = torch.empty(n.value, dtype=torch.uint8, device="cuda")
    cg._check(L.cgtp_radial_forward(0, E, 8, 5.0, 64, 256, cg._ptr(v), cg._ptr(a), cg._ptr(b),
                                    cg._ptr(out), None, cg._ptr(ws), n.value, 8, cg._stream()))
    torch.cuda.synchronize()
    assert cg.radial_device_status() == 1
    assert cg.radial_device_status() == 0
    w = cg.radial_forward(v, a, b, 5.0)
    ref, _ = O.radial_forward(vec, W1, W2, 5.0)
    assert_close(host(w), ref, np.float32, "radial w after the timed-out launch")
    assert cg.radial_device_status() == 0


def test_mixing_tensor_core_timeout_reports_and_context_survives():
    """The channel-mixing tensor-core kernel with its first bounded wait giving
    up (CGTP_LINEAR_TEST_WAIT_TIMEOUT): reported once, then a normal call
    matches the oracle."""
    need_gpu()
    import ctypes
    import clebsch_gordan_tensor_gb300 as cg

    irreps = ("64x0e+64x1o", "64x0e+32x1o")
    rng = np.random.default_rng(13)
    lin = cg.Linear(*irreps)
    assert lin.tensor_cores
    n = 700
    x = rng.standard_normal((n, lin.dim_in)).astype(np.float32)
    Wm = (rng.standard_normal(lin.weight_numel) / 8).astype(np.float32)
    xd, Wd = dev(x), dev(Wm)
    out = torch.empty(n, lin.dim_out, device="cuda")
    fb, _ = lin.workspace_bytes(n)
    ws = torch.empty(max(fb, 16), dtype=torch.uint8, device="cuda")
    cg._check(cg.lib().cgtp_linear_forward(lin._h, n, cg._ptr(xd), cg._ptr(Wd), cg._ptr(out),
                                           cg._ptr(ws), fb, 2, cg._stream()))
    torch.cuda.synchronize()
    assert cg.linear_device_status() == 1
    assert cg.linear_device_status() == 0
    good = lin.forward(xd, Wd)
    instr = [lin.instruction(j)[:2] for j in range(lin.n_instr)]
    ref = O.linear_forward(*irreps, instr, x, Wm)
    assert_close(host(good), ref, np.float32, "mixing out after the timed-out launch")
    assert cg.linear_device_status() == 0
