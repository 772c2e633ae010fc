"""Host logic of bench.py: the per-kernel rates and roofline fractions it
reports, checked on a synthetic step with hand-computed numbers (no GPU)."""
import math

import pytest

import bench


def _wl(dtype="f32"):
    noop = lambda: None  # noqa: E731
    kernels = [("k_hbm", noop), ("k_alu", noop), ("k_tc", noop)]
    counts = {
        "k_hbm": (6.0e9, None),             # bytes only
        "k_alu": (1.0e9, 8.0e10),           # ALU-heavy
        "k_tc": (2.0e9, 3.0e11, "tensor3"),  # three-TF32 tensor products
    }
    wl = bench.Workload("syn", "synthetic", 1000, "edges/s", dtype, kernels, counts,
                        ["k_hbm"], {})
    wl.exec_flops = {"k_alu": 6.0e10}
    return wl


PEAKS = {"hbm": 6000.0, "bf16": 2000.0, "src": "test"}
FMA = {"fp32": 80.0, "fp64": 1.25}


def test_rates_and_bounds():
    per = {"k_hbm": 1.5, "k_alu": 2.0, "k_tc": 1.0}  # ms
    kernels, roof, peak, src = bench.analyze(_wl(), per, FMA, PEAKS)
    # k_hbm: 6 GB in 1.5 ms = 4000 GB/s, 2/3 of the HBM peak
    assert kernels["k_hbm"]["bound"] == "hbm"
    assert math.isclose(kernels["k_hbm"]["hbm_gbs"], 4000.0)
    assert math.isclose(kernels["k_hbm"]["roofline_frac"], 4000.0 / 6000.0)
    # k_alu: 8e10 FLOP in 2 ms = 40 TFLOP/s = half of the FP32 peak; its bytes
    # at HBM speed take 0.167 ms < 1 ms of FLOPs at peak, so ALU-bound
    ka = kernels["k_alu"]
    assert ka["bound"] == "alu"
    assert math.isclose(ka["tflops"], 40.0) and math.isclose(ka["alu_frac"], 0.5)
    assert math.isclose(ka["roofline_frac"], 0.5)
    assert math.isclose(ka["exec_tflops"], 30.0) and math.isclose(ka["exec_alu_frac"], 0.375)
    # k_tc: the three-TF32 peak = bf16 x tf32/bf16 / 3
    tc_peak = 2000.0 * bench.TF32_PER_BF16 / 3
    kt = kernels["k_tc"]
    assert kt["bound"] == "tensor"
    assert math.isclose(kt["tflops"], 300.0)
    assert math.isclose(kt["tensor_frac"], 300.0 / tc_peak)
    # the dominant kernel (longest) is k_alu: its roofline is the line's
    assert roof["kernel"] == "k_alu" and roof["bound"] == "alu"
    assert math.isclose(roof["achieved"], 40.0) and math.isclose(roof["frac"], 0.5)
    assert math.isclose(roof["frac_exec"], 0.375)
    assert roof["peak"] == 80.0 and peak == 80.0 and "FP32" in src


def test_fp64_uses_the_dfma_peak_and_hbm_dominant():
    per = {"k_hbm": 5.0, "k_alu": 2.0, "k_tc": 1.0}
    kernels, roof, peak, src = bench.analyze(_wl("f64"), per, FMA, PEAKS)
    assert peak == 1.25 and "FP64" in src
    # 8e10 FLOP in 2 ms = 40 TFLOP/s against a 1.25 TFLOP/s pipe
    assert math.isclose(kernels["k_alu"]["alu_frac"], 32.0)
    assert roof["kernel"] == "k_hbm" and roof["bound"] == "hbm"
    assert roof["unit"] == "GB/s" and math.isclose(roof["achieved"], 1200.0)
    assert math.isclose(roof["frac"], 0.2)


@pytest.mark.parametrize("ms", [0.5, 4.0])
def test_roofline_fraction_is_the_slower_bound_over_time(ms):
    """roofline_frac = max(bytes / HBM, FLOPs / peak) / time for a kernel with
    both counts."""
    per = {"k_hbm": 1.0, "k_alu": ms, "k_tc": 1.0}
    kernels, *_ = bench.analyze(_wl(), per, FMA, PEAKS)
    t = ms * 1e-3
    want = max(1.0e9 / (6000.0e9), 8.0e10 / 80.0e12) / t
    assert math.isclose(kernels["k_alu"]["roofline_frac"], want)


def test_algorithmic_flop_counts_of_the_configs():
    """bench's per-unit FLOP count, mul * sum_p 2 (nnz_p + d_l3), from the
    planner's CG tables: 58,496 per edge for the 64-channel conv layer (config
    2) and 116,992 per sample for the 128-channel one (configs 1 and 3)."""
    import clebsch_gordan_tensor_gb300 as cg
    import workloads as W
    assert bench.Dims(cg.Plan(*W.IRREPS_CONV64)).flops == 58_496
    assert bench.Dims(cg.Plan(*W.IRREPS_MACE128)).flops == 116_992
