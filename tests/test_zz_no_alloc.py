"""The fused-convolution gradient entry point that allocates nothing.

Callers that cannot allocate device memory when they need the gradient -- a
framework whose own pool owns all device memory, a plugin under a fixed memory
budget, a loop that cannot take cudaMalloc's implicit synchronisation -- call
``cgtp_conv_backward_noalloc``.  It gives the same results as
``cgtp_conv_backward_ws`` but takes its scratch (the per-CTA partial rows of a
shared weight row's gradient) from a fixed array inside the library instead of
from the caller.  These tests check it against that entry point and against
the oracle, on two calls in a row, and check that calls after the first on a
device leave the device's free memory unchanged.

This file is collected last so that a run stopping at its first failure has
already run every other test; it passes alone in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest

import oracle as O
import workloads as W
from tests.gpu_util import assert_close, dev, host, need_gpu, torch

pytestmark = pytest.mark.gpu


def _noalloc(cg, plan, G, x, y, w, scale, g, gx, gy, gw):
    L = cg.lib()
    f = L.cgtp_conv_backward_noalloc
    vp = ctypes.c_void_p
    f.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, vp, vp, vp, vp, vp, vp, vp, vp,
                  ctypes.c_double, vp, vp, vp, vp, vp]
    f.restype = ctypes.c_int
    p = cg._ptr
    cg._check(f(plan._h, G.N, G.E, p(G.rowptr), p(G.sender), p(G.s_rowptr), p(G.s_perm),
                p(G.s_recv), p(x), p(y), p(w), float(scale), p(g), p(gx), p(gy), p(gw),
                cg._stream()))


@pytest.mark.parametrize("shared", [True, False])
def test_noalloc_conv_backward_matches_workspace_entry_point_and_oracle(shared):
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg

    rng = np.random.default_rng(5)
    _, _, gr = W.periodic_cloud(rng, 800)
    G = cg.Graph.from_numpy(gr)
    plan = cg.Plan(*W.IRREPS_CONV64, shared_weights=shared)
    prob = O.make_problem(*W.IRREPS_CONV64)
    xh = rng.standard_normal((gr.N, plan.dim_in1)).astype(np.float32)
    yh = rng.standard_normal((gr.E, plan.dim_in2)).astype(np.float32)
    wshape = (plan.weight_numel,) if shared else (gr.E, plan.weight_numel)
    wh = rng.standard_normal(wshape).astype(np.float32)
    x, y, w = dev(xh), dev(yh), dev(wh)
    for call in range(2):  # two calls in a row, different gradients each time
        gh = rng.standard_normal((gr.N, plan.dim_out)).astype(np.float32)
        g = dev(gh)
        # the existing entry point (caller-provided workspace) is the reference;
        # its first call also loads the plan's kernels on this device
        rx, ry, rw = plan.conv_backward(G, x, y, w, 0.3, g)
        gx, gy, gw = torch.full_like(rx, 7.0), torch.full_like(ry, 7.0), torch.full_like(rw, 7.0)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        _noalloc(cg, plan, G, x, y, w, 0.3, g, gx, gy, gw)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        if call > 0:  # the first call on a device may load kernels (set-up)
            assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
        assert_close(host(gx), host(rx), np.float32, f"grad_x vs _ws, call {call}")
        assert_close(host(gy), host(ry), np.float32, f"grad_y vs _ws, call {call}")
        assert_close(host(gw), host(rw), np.float32, f"grad_w vs _ws, call {call}")
        ox, oy, ow = O.conv_backward(prob, gr.rowptr, gr.sender, xh, yh, wh, 0.3, gh)
        assert_close(host(gx), ox, np.float32, f"grad_x vs oracle, call {call}")
        assert_close(host(gy), oy, np.float32, f"grad_y vs oracle, call {call}")
        assert_close(host(gw), ow, np.float32, f"grad_w vs oracle, call {call}")
    assert plan.device_status() == 0
