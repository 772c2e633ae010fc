"""Shared helpers of the GPU parity tests (test code only)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

# Normwise tolerance: max |gpu - oracle| / max |oracle| per output tensor.
# fp32: 1e-5, fp64: 1e-11 (the accuracy targets stated for this path).
TOL = {np.dtype(np.float32): 1e-5, np.dtype(np.float64): 1e-11}


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy().astype(np.float64)


def relerr(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    scale = np.abs(ref).max() if ref.size else 0.0
    diff = np.abs(got - ref).max() if ref.size else 0.0
    if scale == 0.0:
        return float(diff)
    return float(diff / scale)


def assert_close(got, ref, dtype, what=""):
    e = relerr(got, ref)
    assert e <= TOL[np.dtype(dtype)], f"{what}: normwise relative error {e:.3e}"
    return e


def conv_weights(cfg):
    """The per-edge weights of a conv workload: the oracle's radial network on
    the workload's edge vectors and parameters, rounded to the workload dtype
    (an input shared by both sides of a parity test)."""
    import oracle as O
    if "w" not in cfg:
        cfg["w"] = O.radial_forward(cfg["vec"], cfg["W1"], cfg["W2"], cfg["cutoff"],
                                    out_dtype=cfg["dtype"])[0]
    return cfg["w"]
