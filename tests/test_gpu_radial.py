"""GPU parity of the radial network (Bessel basis -> Linear -> SiLU -> Linear)
against the oracle, through the C ABI: the tensor-core path (fp32, TF32 split
in three products) and the CUDA-core path (fp32, fp64), ragged edge counts,
a zero-length edge, the stored hidden activations, and the benchmark
workload's full size on sampled edges."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests.gpu_util import assert_close, dev, host, need_gpu, torch

pytestmark = pytest.mark.gpu


def _inputs(rng, E, nb, hidden, n_out, dt):
    d = rng.standard_normal((E, 3))
    d /= np.linalg.norm(d, axis=1, keepdims=True)
    vec = (d * rng.uniform(0.5, 5.0, size=(E, 1))).astype(dt)
    W1 = (rng.standard_normal((nb, hidden)) / np.sqrt(nb)).astype(dt)
    W2 = (rng.standard_normal((hidden, n_out)) / np.sqrt(hidden)).astype(dt)
    return vec, W1, W2


CASES = [  # E, n_basis, hidden, n_out, dtype
    (1000, 8, 64, 1536, np.float32),
    (1, 8, 64, 1536, np.float32),
    (128, 8, 64, 256, np.float32),
    (129, 8, 32, 128, np.float32),
    (5000, 8, 64, 384, np.float32),
    (333, 5, 40, 256, np.float32),
    (300, 8, 12, 100, np.float32),
    (200, 8, 64, 192, np.float32),
    (257, 16, 8, 64, np.float32),
    (300, 32, 256, 96, np.float32),
    (777, 8, 64, 1536, np.float64),
    (50, 3, 7, 5, np.float64),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"E{c[0]}-nb{c[1]}-h{c[2]}-o{c[3]}-{np.dtype(c[4]).name}")
@pytest.mark.parametrize("cuda_cores", [False, True])
def test_radial_forward_matches_oracle(case, cuda_cores):
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    E, nb, hidden, n_out, dt = case
    rng = np.random.default_rng(E + hidden)
    vec, W1, W2 = _inputs(rng, E, nb, hidden, n_out, dt)
    vec[0] = 0.0  # a zero-length edge takes the basis' limit
    tdt = torch.float64 if dt == np.float64 else torch.float32
    hid = torch.full((E, hidden), 7.0, dtype=tdt, device="cuda")
    w = cg.radial_forward(dev(vec), dev(W1), dev(W2), 5.0, hidden_out=hid, cuda_cores=cuda_cores)
    rw, rh = O.radial_forward(vec, W1, W2, 5.0)
    assert_close(host(w), rw, dt, "w")
    assert_close(host(hid), rh, dt, "hidden")
    assert cg.radial_device_status() == 0
    if not cuda_cores and dt == np.float32:
        expect_tc = nb <= 16 and hidden % 8 == 0 and hidden <= 64 and n_out % 128 == 0
        assert cg.radial_uses_tensor_cores(tdt, nb, hidden, n_out) == expect_tc


def test_radial_tensor_cores_agree_with_cuda_cores_to_fp32_rounding():
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    rng = np.random.default_rng(3)
    vec, W1, W2 = _inputs(rng, 4096, 8, 64, 1536, np.float32)
    a = cg.radial_forward(dev(vec), dev(W1), dev(W2))
    b = cg.radial_forward(dev(vec), dev(W1), dev(W2), cuda_cores=True)
    rel = float((a - b).abs().max() / b.abs().max())
    assert rel < 2e-6, rel


def test_radial_empty_and_errors():
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    W1 = torch.zeros(8, 64, device="cuda")
    W2 = torch.zeros(64, 128, device="cuda")
    w = cg.radial_forward(torch.zeros(0, 3, device="cuda"), W1, W2)
    assert w.shape == (0, 128)
    with pytest.raises(cg.CgtpError):
        cg.radial_forward(torch.zeros(4, 3, device="cuda"), torch.zeros(40, 64, device="cuda"), W2)


def test_radial_benchmark_workload_sampled():
    """The benchmark workload at full size (~525k edges, 8 -> 64 -> 1536):
    the GPU computes every row, the oracle sampled rows."""
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    cfg = W.conv64_cloud10k()
    E = cfg["graph"].E
    w = cg.radial_forward(dev(cfg["vec"]), dev(cfg["W1"]), dev(cfg["W2"]), cfg["cutoff"])
    assert cg.radial_uses_tensor_cores(torch.float32, 8, 64, 1536)
    rng = np.random.default_rng(4)
    idx = np.unique(np.concatenate([rng.choice(E, 2000, replace=False), [0, E - 1]]))
    rw, _ = O.radial_forward(cfg["vec"][idx], cfg["W1"], cfg["W2"], cfg["cutoff"])
    assert_close(host(w[torch.from_numpy(idx).cuda()]), rw, np.float32, "w rows")
    assert cg.radial_device_status() == 0


BWD_CASES = [  # E, n_basis, hidden, n_out, dtype
    (1000, 8, 64, 1536, np.float32),
    (1, 8, 64, 256, np.float32),
    (300, 16, 32, 128, np.float32),
    (4000, 8, 64, 384, np.float32),
    (333, 5, 40, 200, np.float32),
    (129, 32, 256, 96, np.float32),
    (700, 8, 64, 384, np.float64),
    (50, 3, 7, 5, np.float64),
]


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: f"E{c[0]}-nb{c[1]}-h{c[2]}-o{c[3]}-{np.dtype(c[4]).name}")
@pytest.mark.parametrize("cuda_cores", [False, True])
def test_radial_backward_matches_oracle(case, cuda_cores):
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    E, nb, hidden, n_out, dt = case
    rng = np.random.default_rng(E + 7 * hidden)
    vec, W1, W2 = _inputs(rng, E, nb, hidden, n_out, dt)
    vec[0] = 0.0  # zero-length edge: no gradient
    g = rng.standard_normal((E, n_out)).astype(dt)
    gv, g1, g2 = cg.radial_backward(dev(vec), dev(W1), dev(W2), dev(g), 5.0, cuda_cores=cuda_cores)
    rv, r1, r2 = O.radial_backward(vec, W1, W2, g, 5.0)
    assert_close(host(gv), rv, dt, "grad_vec")
    assert_close(host(g1), r1, dt, "grad_W1")
    assert_close(host(g2), r2, dt, "grad_W2")
    assert np.all(host(gv)[0] == 0.0)
    # subsets, and a second call gives the same bits (ordered reductions)
    _, g1b, g2b = cg.radial_backward(dev(vec), dev(W1), dev(W2), dev(g), 5.0,
                                     need=(False, True, True), cuda_cores=cuda_cores)
    assert torch.equal(g1b, g1) and torch.equal(g2b, g2)
    gvb, n1, n2 = cg.radial_backward(dev(vec), dev(W1), dev(W2), dev(g), 5.0,
                                     need=(True, False, False), cuda_cores=cuda_cores)
    assert n1 is None and n2 is None and torch.equal(gvb, gv)


def test_radial_backward_empty():
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    W1 = torch.ones(8, 16, device="cuda")
    W2 = torch.ones(16, 32, device="cuda")
    gv, g1, g2 = cg.radial_backward(torch.zeros(0, 3, device="cuda"), W1, W2,
                                    torch.zeros(0, 32, device="cuda"))
    assert gv.shape == (0, 3)
    assert float(g1.abs().max()) == 0.0 and float(g2.abs().max()) == 0.0


def test_radial_backward_benchmark_workload():
    """Full size (525k edges, 8 -> 64 -> 1536): the oracle's grad_W1 / grad_W2
    over all edges (fp64 matmuls) and grad_vec on sampled edges."""
    need_gpu()
    import clebsch_gordan_tensor_gb300 as cg
    cfg = W.conv64_cloud10k()
    E = cfg["graph"].E
    g = np.random.default_rng(5).standard_normal((E, 1536)).astype(np.float32)
    gv, g1, g2 = cg.radial_backward(dev(cfg["vec"]), dev(cfg["W1"]), dev(cfg["W2"]), dev(g),
                                    cfg["cutoff"])
    rv, r1, r2 = O.radial_backward(cfg["vec"], cfg["W1"], cfg["W2"], g, cfg["cutoff"])
    assert_close(host(g1), r1, np.float32, "grad_W1")
    assert_close(host(g2), r2, np.float32, "grad_W2")
    idx = np.unique(np.concatenate([np.random.default_rng(6).choice(E, 3000, replace=False), [0, E - 1]]))
    assert_close(host(gv)[idx], rv[idx], np.float32, "grad_vec rows")
