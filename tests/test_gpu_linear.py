"""GPU parity of the per-irrep channel mixing (tcgen05 and CUDA-core kernels)
and of the 'uvw' tensor product built on it, against the oracle."""
import numpy as np
import pytest

import oracle as O
from tests.gpu_util import assert_close, dev, host, need_gpu, torch

pytestmark = pytest.mark.gpu

# several 128-row tiles with a ragged tail; an input irrep used twice, an
# output irrep reached by two instructions and one reached by none
LIN = ("32x0e+32x1o+64x1o+32x2e", "64x0e+32x1o+32x2e+32x3o")
LIN_WIDE = ("128x0e+128x1o+256x2e", "256x0e+128x1o+128x2e")


def _cg():
    import clebsch_gordan_tensor_gb300 as cg
    return cg


def _problem(rng, irreps, n, dt):
    instr = O.linear_instructions(*irreps)
    a, b = O.parse_irreps(irreps[0]), O.parse_irreps(irreps[1])
    nw = sum(a[i][0] * b[o][0] for i, o in instr)
    x = rng.standard_normal((n, O.irreps_dim(a))).astype(dt)
    W = (rng.standard_normal(nw) / 8).astype(dt)
    g = rng.standard_normal((n, O.irreps_dim(b))).astype(dt)
    return instr, x, W, g


@pytest.mark.parametrize("irreps", [LIN, LIN_WIDE], ids=["mixed", "wide"])
@pytest.mark.parametrize("n", [1, 333])
@pytest.mark.parametrize("path", ["tensor", "cuda", "fp64"])
def test_linear_forward_backward(irreps, n, path):
    need_gpu()
    cg = _cg()
    dt = np.float64 if path == "fp64" else np.float32
    tdt = torch.float64 if path == "fp64" else torch.float32
    rng = np.random.default_rng(n)
    instr, x, W, g = _problem(rng, irreps, n, dt)
    lin = cg.Linear(*irreps, dtype=tdt)
    assert lin.tensor_cores == (path != "fp64")
    cc = path == "cuda"
    out = lin.forward(dev(x), dev(W), cuda_cores=cc)
    assert_close(host(out), O.linear_forward(*irreps, instr, x, W), dt, "out")
    gx, gW = lin.backward(dev(x), dev(W), dev(g), cuda_cores=cc)
    rx, rW = O.linear_backward(*irreps, instr, x, W, g)
    assert_close(host(gx), rx, dt, "grad_x")
    assert_close(host(gW), rW, dt, "grad_W")
    assert cg.linear_device_status() == 0


def test_linear_unaligned_input_takes_cuda_cores():
    """An 8-byte (not 16-byte) aligned x is served by the CUDA-core kernel."""
    need_gpu()
    cg = _cg()
    rng = np.random.default_rng(5)
    instr, x, W, _ = _problem(rng, LIN, 200, np.float32)
    buf = torch.zeros(x.size + 2, device="cuda")
    xv = buf[2:].view(x.shape)
    xv.copy_(dev(x))
    assert xv.data_ptr() % 16 == 8
    lin = cg.Linear(*LIN)
    assert_close(host(lin.forward(xv, dev(W))), O.linear_forward(*LIN, instr, x, W), np.float32,
                 "out")


def test_linear_empty_and_repeat():
    need_gpu()
    cg = _cg()
    lin = cg.Linear(*LIN)
    x = torch.zeros(0, lin.dim_in, device="cuda")
    W = torch.randn(lin.weight_numel, device="cuda")
    assert lin.forward(x, W).shape == (0, lin.dim_out)
    gx, gW = lin.backward(x, W, torch.zeros(0, lin.dim_out, device="cuda"))
    assert gx.shape == x.shape and not host(gW).any()
    # the same workspace reused by consecutive calls gives identical results
    rng = np.random.default_rng(6)
    instr, xn, Wn, _ = _problem(rng, LIN, 1000, np.float32)
    ws = torch.empty(lin.workspace_bytes(1000)[0], dtype=torch.uint8, device="cuda")
    a = lin.forward(dev(xn), dev(Wn), workspace=ws).clone()
    b = lin.forward(dev(xn), dev(Wn), workspace=ws)
    assert torch.equal(a, b)


UVW_SMALL = ("32x0e+32x1o+32x2e", "0e+1o+2e+3o", "64x0e+32x1o+32x1e+32x2o+32x2e+32x3o+32x3e")


def test_uvw_product_matches_oracle():
    """'uvw' = per-path 'uvu' blocks (unit shared weights) + channel mixing,
    against the oracle's direct definition."""
    need_gpu()
    cg = _cg()
    rng = np.random.default_rng(7)
    B = 300
    uvw = cg.UVWProduct(*UVW_SMALL)
    x = rng.standard_normal((B, uvw.dim_in1)).astype(np.float32)
    v = rng.standard_normal((B, 3)).astype(np.float32)
    W = (rng.standard_normal(uvw.weight_numel) / 16).astype(np.float32)
    y = cg.sh_forward(dev(v), 3)
    out = uvw.forward(dev(x), y, dev(W))
    ref = O.tp_uvw_forward(*UVW_SMALL, x, O.sh(3, v), W)
    assert_close(host(out), ref, np.float32, "uvw out")


def test_uvw_fused_forward_matches_two_step_and_oracle():
    """The fused forward (the mixing kernel's producers compute each path's
    block from x and y) against the two-step forward (blocks written to an
    intermediate, then mixed) and the oracle, on a ragged row count."""
    need_gpu()
    cg = _cg()
    rng = np.random.default_rng(17)
    B = 1037
    uvw = cg.UVWProduct(*UVW_SMALL)
    x = rng.standard_normal((B, uvw.dim_in1)).astype(np.float32)
    v = rng.standard_normal((B, 3)).astype(np.float32)
    W = (rng.standard_normal(uvw.weight_numel) / 16).astype(np.float32)
    y = cg.sh_forward(dev(v), 3)
    n0 = cg.launch_count()
    fused = uvw.forward(dev(x), y, dev(W))
    n1 = cg.launch_count()
    mid = torch.empty(B, uvw.dim_mid, device="cuda")
    two = uvw.forward(dev(x), y, dev(W), mid=mid)
    n2 = cg.launch_count()
    assert n1 - n0 == 3 and n2 - n1 == 4  # fused: T rows, weight pack, mixing; else unit row, blocks, pack, mixing
    ref = O.tp_uvw_forward(*UVW_SMALL, x, host(y), W)
    assert_close(host(fused), ref, np.float32, "fused uvw out")
    assert_close(host(two), ref, np.float32, "two-step uvw out")
    assert_close(host(fused), host(two), np.float32, "fused vs two-step")
    assert cg.linear_device_status() == 0


def test_uvw_backward_matches_oracle():
    need_gpu()
    cg = _cg()
    rng = np.random.default_rng(8)
    B = 257
    uvw = cg.UVWProduct(*UVW_SMALL)
    x = rng.standard_normal((B, uvw.dim_in1)).astype(np.float32)
    v = rng.standard_normal((B, 3)).astype(np.float32)
    W = (rng.standard_normal(uvw.weight_numel) / 16).astype(np.float32)
    g = rng.standard_normal((B, uvw.dim_out)).astype(np.float32)
    y = cg.sh_forward(dev(v), 3)
    gx, gy, gW = uvw.backward(dev(x), y, dev(W), dev(g))
    rx, ry, rW = O.tp_uvw_backward(*UVW_SMALL, x, host(y), W, g)
    assert_close(host(gx), rx, np.float32, "uvw grad_x")
    assert_close(host(gy), ry, np.float32, "uvw grad_y")
    assert_close(host(gW), rW, np.float32, "uvw grad_W")


def test_uvw_convolution_matches_oracle():
    """Fused convolution with 'uvw' paths: the standalone 'uvw' product of each
    edge, summed per receiver (and its gradient), on a random graph."""
    need_gpu()
    cg = _cg()
    from tests.test_gpu_conv import _graph
    rng = np.random.default_rng(9)
    gr = _graph(rng, 120, max_deg=9)
    G = cg.Graph.from_numpy(gr)
    uvw = cg.UVWProduct(*UVW_SMALL)
    x = rng.standard_normal((gr.N, uvw.dim_in1)).astype(np.float32)
    y = O.sh(3, rng.standard_normal((gr.E, 3))).astype(np.float32)
    W = (rng.standard_normal(uvw.weight_numel) / 16).astype(np.float32)
    g = rng.standard_normal((gr.N, uvw.dim_out)).astype(np.float32)
    scale = 0.5
    out = uvw.conv_forward(G, dev(x), dev(y), dev(W), scale)
    per_edge = O.tp_uvw_forward(*UVW_SMALL, x[gr.sender], y, W)
    ref = np.zeros((gr.N, uvw.dim_out))
    np.add.at(ref, gr.receiver, scale * per_edge)
    assert_close(host(out), ref, np.float32, "uvw conv out")
    gx, gy, gW = uvw.conv_backward(G, dev(x), dev(y), dev(W), scale, dev(g))
    ex, ey, eW = O.tp_uvw_backward(*UVW_SMALL, x[gr.sender], y, W, scale * g[gr.receiver])
    rx = np.zeros((gr.N, uvw.dim_in1))
    np.add.at(rx, gr.sender, ex)
    assert_close(host(gx), rx, np.float32, "uvw conv grad_x")
    assert_close(host(gy), ey, np.float32, "uvw conv grad_y")
    assert_close(host(gW), eW, np.float32, "uvw conv grad_W")


def test_linear_weight_gradient_long_sums():
    """grad_W summed over many rows (20,000 items x (1 + 3 + 5) rows per
    matrix): the tensor-core reduction and the CUDA-core one against the oracle."""
    need_gpu()
    cg = _cg()
    irreps = ("128x0e+128x1o+128x2e", "128x0e+128x1o+64x2e")
    rng = np.random.default_rng(11)
    instr, x, W, g = _problem(rng, irreps, 20000, np.float32)
    lin = cg.Linear(*irreps)
    rx, rW = O.linear_backward(*irreps, instr, x, W, g)
    for cc in (False, True):
        _, gW = lin.backward(dev(x), dev(W), dev(g), need=(False, True), cuda_cores=cc)
        assert_close(host(gW), rW, np.float32, f"grad_W (cuda cores: {cc})")
    assert cg.linear_device_status() == 0


@pytest.mark.parametrize("n", [5, 3001])
def test_linear_128_channel_layer_ragged(n):
    """A layer whose instructions all take 128 input and 128 output channels
    (the 'uvw' mixing's shape): the W-gradient stages chunks of whole items
    with 3D tensor-map copies (items per chunk 32 / d, a ragged last chunk and
    split tails at these n), and the forward and x-gradient, one 128-channel
    source per block, run the three split products into two alternating
    accumulators; all against the oracle."""
    need_gpu()
    cg = _cg()
    irreps = ("128x0e+128x1o+128x2e+128x3o", "128x0e+128x1o+128x2e+128x3o")
    rng = np.random.default_rng(40 + n)
    instr, x, W, g = _problem(rng, irreps, n, np.float32)
    lin = cg.Linear(*irreps)
    out = lin.forward(dev(x), dev(W))
    assert_close(host(out), O.linear_forward(*irreps, instr, x, W), np.float32, "forward")
    rx, rW = O.linear_backward(*irreps, instr, x, W, g)
    gx, gW = lin.backward(dev(x), dev(W), dev(g))
    assert_close(host(gx), rx, np.float32, "grad_x")
    assert_close(host(gW), rW, np.float32, "grad_W")
    assert cg.linear_device_status() == 0
