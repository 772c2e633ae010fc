"""Host-side checks of the C-ABI library (no GPU needed).

The library loads, exports every symbol declared in include/cgtp.h, plans the
five workloads, computes CG coefficients that agree with the oracle's (an
independent route: ladder recursion vs Racah's sum), reports bad arguments with
status codes, and its generated kernels compile for sm_103a with NVRTC.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O
import workloads as W
import clebsch_gordan_tensor_gb300 as cg
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ALL_CFGS = [W.IRREPS_TP16, W.IRREPS_MACE128, W.IRREPS_CONV64, W.IRREPS_CONV128, W.IRREPS_TFN32]


def _declared():
    text = open(os.path.join(ROOT, "include", "cgtp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cgtp_\w+)\s*\(", text)))


def test_exports_every_declared_symbol():
    L = cg.lib()
    names = _declared()
    assert len(names) >= 20
    for n in names:
        assert hasattr(L, n), n


@pytest.mark.parametrize("irreps", ALL_CFGS)
def test_plan_matches_oracle_problem(irreps):
    plan = cg.Plan(*irreps)
    prob = O.make_problem(*irreps)
    assert (plan.dim_in1, plan.dim_in2, plan.dim_out, plan.weight_numel, plan.n_paths) == (
        prob.dim1, prob.dim2, prob.dimo, prob.wdim, len(prob.paths))
    for p, path in enumerate(prob.paths):
        i1, i2, i3, l1, l2, l3 = path[:6]
        assert plan.path(p) == (l1, l2, l3, i1, i2, i3)
        assert np.abs(plan.coefficients(p) - O.cg_real(l1, l2, l3)).max() < 1e-14


def test_planner_cg_agrees_with_racah_up_to_l6():
    """Ladder recursion (library) vs Racah's closed form (oracle) for every
    triple with l <= 6; the error grows with l (1e-14 at l <= 3)."""
    worst = {}
    for l1 in range(7):
        for l2 in range(7):
            outs = list(range(abs(l1 - l2), min(6, l1 + l2) + 1))
            par = "e" if l2 % 2 == 0 else "o"  # in1 is even: p3 = p2
            out = "+".join(f"1x{l3}{par}" for l3 in outs)
            plan = cg.Plan(f"1x{l1}e", f"{l2}{'e' if l2 % 2 == 0 else 'o'}", out)
            assert plan.n_paths == len(outs)
            for p in range(plan.n_paths):
                a, b, c = plan.path(p)[:3]
                err = np.abs(plan.coefficients(p) - O.cg_real(a, b, c)).max()
                key = max(a, b, c)
                worst[key] = max(worst.get(key, 0.0), err)
    assert max(v for k, v in worst.items() if k <= 3) < 1e-14
    assert max(worst.values()) < 1e-12


def test_explicit_instructions_and_errors():
    plan = cg.Plan("4x0e+4x1o", "0e+1o", "4x1o", instructions=[(0, 1, 0), (1, 0, 0)])
    assert plan.n_paths == 2 and plan.weight_numel == 8
    with pytest.raises(cg.CgtpError, match="allowed path"):
        cg.Plan("4x0e", "0e", "4x1o", instructions=[(0, 0, 0)])
    with pytest.raises(cg.CgtpError, match="allowed path"):
        cg.Plan("4x0e", "0e", "4x0e", instructions=[(0, 3, 0)])
    with pytest.raises(cg.CgtpError, match="irreps"):
        cg.Plan("4x1q", "0e", "4x1o")
    with pytest.raises(cg.CgtpError, match="irreps"):
        cg.Plan("", "0e", "4x1o")
    with pytest.raises(cg.CgtpError, match="irreps"):
        cg.Plan("4x7e", "0e", "4x7e")
    with pytest.raises(cg.CgtpError, match="unsupported"):
        cg.Plan("4x0e+8x1o", "0e", "4x0e")
    with pytest.raises(cg.CgtpError, match="unsupported"):
        cg.Plan("4x0e", "2x0e", "4x0e")


def test_c_abi_argument_errors():
    L = cg.lib()
    h = ctypes.c_void_p()
    assert L.cgtp_plan_create(None, b"1x0e", b"0e", b"1x0e", None, 0, 0, 0, 0) == 1
    assert L.cgtp_plan_create(ctypes.byref(h), b"1x0e", b"0e", b"1x0e", None, 0, 7, 0, 0) == 1
    assert L.cgtp_plan_create(ctypes.byref(h), b"4x0e", b"0e", b"4x0e", None, 0, 0, 0, 0) == 0
    null = ctypes.c_void_p()
    # size and pointer checks return before any CUDA call
    assert L.cgtp_forward(h, -1, null, null, null, null, null) == 1
    assert L.cgtp_forward(h, 0, null, null, null, null, null) == 0
    assert L.cgtp_forward(h, 5, null, null, null, null, null) == 1
    misaligned = ctypes.c_void_p(0x1004)
    assert L.cgtp_forward(h, 5, misaligned, misaligned, misaligned, misaligned, null) == 1
    assert L.cgtp_conv_forward(h, -1, 0, null, null, null, null, null, 1.0, null, null) == 5
    assert L.cgtp_conv_forward(h, 3, 4, null, null, null, null, null, 1.0, null, null) == 5
    assert L.cgtp_conv_forward(h, 0, 0, null, null, null, null, null, 1.0, null, null) == 0
    assert L.cgtp_sh_forward(9, 0, 4, null, null, null) == 4
    assert L.cgtp_sh_forward(3, 0, 0, null, null, null) == 0
    assert L.cgtp_sh_forward(3, 0, 4, null, null, null) == 1
    assert L.cgtp_forward(None, 1, null, null, null, null, null) == 1
    assert L.cgtp_status_str(7) == b"CUDA error"
    err = ctypes.c_int(-1)
    assert L.cgtp_last_cuda_error(ctypes.byref(err)) == 0
    assert L.cgtp_plan_destroy(h) == 0
    # bfloat16 weights: fp32 plans only; their weight rows need 4-byte alignment
    assert L.cgtp_plan_create(ctypes.byref(h), b"64x0e", b"0e", b"64x0e", None, 0, 1, 0,
                              1 << 24) == 4
    assert L.cgtp_plan_create(ctypes.byref(h), b"64x0e", b"0e", b"64x0e", None, 0, 0, 0,
                              1 << 24) == 0
    a8, a2 = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1002)
    assert L.cgtp_forward(h, 5, a8, a8, a2, a8, null) == 1
    assert b"weight pointer" in L.cgtp_last_error_message()
    assert L.cgtp_plan_destroy(h) == 0
    # binary16 weights: the same rules; one 16-bit format at a time
    assert L.cgtp_plan_create(ctypes.byref(h), b"64x0e", b"0e", b"64x0e", None, 0, 1, 0,
                              1 << 25) == 4
    assert L.cgtp_plan_create(ctypes.byref(h), b"64x0e", b"0e", b"64x0e", None, 0, 0, 0,
                              (1 << 24) | (1 << 25)) == 1
    assert L.cgtp_plan_create(ctypes.byref(h), b"64x0e", b"0e", b"64x0e", None, 0, 0, 0,
                              1 << 25) == 0
    assert L.cgtp_forward(h, 5, a8, a8, a2, a8, null) == 1
    assert L.cgtp_plan_destroy(h) == 0
    s = cg.Plan("2x0e", "0e", "2x0e", shared_weights=True)
    gx = ctypes.c_void_p(0x1000)
    # shared-weight gradient: needs the workspace variant, and enough scratch
    assert L.cgtp_backward(s._h, 1, gx, gx, gx, gx, null, null, gx, null) == 1
    n = ctypes.c_size_t()
    assert L.cgtp_weight_grad_workspace(s._h, ctypes.byref(n)) == 0 and n.value == 2048 * 2 * 4
    assert L.cgtp_backward_ws(s._h, 1, gx, gx, gx, gx, null, null, gx, gx, ctypes.c_size_t(8),
                              null) == 1
    pe = cg.Plan("2x0e", "0e", "2x0e")
    assert L.cgtp_weight_grad_workspace(pe._h, ctypes.byref(n)) == 0 and n.value == 0


def test_radial_argument_errors_and_path():
    L = cg.lib()
    null = ctypes.c_void_p()
    # sizes and pointers are checked before any CUDA call
    args = lambda E, nb, rc, hid, no, p=null: (0, E, nb, rc, hid, no, p, p, p, p, null, null,
                                                0, 0, null)
    assert L.cgtp_radial_forward(*args(0, 8, 5.0, 64, 1536)) == 0
    assert L.cgtp_radial_forward(*args(-1, 8, 5.0, 64, 1536)) == 1
    assert L.cgtp_radial_forward(*args(4, 0, 5.0, 64, 1536)) == 1
    assert L.cgtp_radial_forward(*args(4, 33, 5.0, 64, 1536)) == 1
    assert L.cgtp_radial_forward(*args(4, 8, 0.0, 64, 1536)) == 1
    assert L.cgtp_radial_forward(*args(4, 8, 5.0, 257, 1536)) == 1
    assert L.cgtp_radial_forward(*args(4, 8, 5.0, 64, 0)) == 1
    assert L.cgtp_radial_forward(*args(4, 8, 5.0, 64, 1536)) == 1  # NULL tensors
    assert L.cgtp_radial_forward(*args(4, 8, 5.0, 64, 1536, ctypes.c_void_p(0x1002))) == 1
    assert cg.radial_uses_tensor_cores(torch.float32, 8, 64, 1536)
    assert cg.radial_uses_tensor_cores(torch.float32, 8, 32, 256)
    assert not cg.radial_uses_tensor_cores(torch.float32, 8, 12, 1536)   # hidden % 8
    assert not cg.radial_uses_tensor_cores(torch.float32, 8, 128, 1536)  # hidden > 64
    assert not cg.radial_uses_tensor_cores(torch.float32, 8, 64, 100)    # n_out % 128
    assert not cg.radial_uses_tensor_cores(torch.float32, 8, 64, 192)
    assert not cg.radial_uses_tensor_cores(torch.float64, 8, 64, 1536)
    assert not cg.radial_uses_tensor_cores(torch.float32, 17, 64, 1536)  # n_basis > 16
    n = ctypes.c_size_t()
    assert L.cgtp_radial_workspace(0, 8, 64, 1536, ctypes.byref(n)) == 0 and n.value == 1536 * 64 * 8
    assert L.cgtp_radial_workspace(1, 8, 64, 1536, ctypes.byref(n)) == 0 and n.value == 0
    assert L.cgtp_radial_workspace(0, 8, 12, 1536, ctypes.byref(n)) == 0 and n.value == 0
    # 16-bit outputs: fp32 inputs only, one format at a time (checked before any launch)
    fake = ctypes.c_void_p(0x1000)
    assert L.cgtp_radial_forward(1, 4, 8, ctypes.c_double(5.0), 64, 1536, fake, fake, fake, fake,
                                 None, None, ctypes.c_size_t(0), 4, None) == 4
    assert L.cgtp_radial_forward(0, 4, 8, ctypes.c_double(5.0), 64, 1536, fake, fake, fake, fake,
                                 None, None, ctypes.c_size_t(0), 2 | 4, None) == 1
    v = ctypes.c_int()
    assert L.cgtp_radial_path(0, 8, 64, 1536, None) == 1
    assert L.cgtp_radial_path(0, 40, 64, 1536, ctypes.byref(v)) == 1


@pytest.mark.parametrize("wdtype", ["bfloat16", "float16"])
def test_16bit_weight_kernels_compile_for_sm103a(wdtype):
    """The generated kernels with 16-bit weight storage (widened to fp32 on
    load) compile for sm_103a, the forward kernels without spills."""
    import torch
    plan = cg.Plan(*W.IRREPS_CONV64, weight_dtype=getattr(torch, wdtype))
    log = plan.compile()
    assert "sm_103a" in log
    assert "#define W_STORE " + ("1" if wdtype == "bfloat16" else "2") in plan.source()
    spills = {k: int(v) for k, v in
              re.findall(r"Function properties for (cgtp_\w+)\n.*?(\d+) bytes spill stores", log)}
    for k in ("cgtp_fwd_conv", "cgtp_fwd_single", "cgtp_fwd_conv_tma", "cgtp_fwd_single_tma"):
        assert spills.get(k, 0) == 0, log


@pytest.mark.parametrize("irreps,dtype", [(W.IRREPS_TP16, "f32"), (W.IRREPS_CONV64, "f32"), (W.IRREPS_TFN32, "f32"),
                                          (W.IRREPS_MACE128, "f32"), (W.IRREPS_CONV128, "f64")])
def test_generated_kernels_compile_for_sm103a(irreps, dtype):
    import torch
    plan = cg.Plan(*irreps, dtype=torch.float64 if dtype == "f64" else torch.float32)
    log = plan.compile()
    assert "sm_103a" in log
    spills = {k: int(v) for k, v in
              re.findall(r"Function properties for (cgtp_\w+)\n.*?(\d+) bytes spill stores", log)}
    direct = {"cgtp_fwd_conv", "cgtp_fwd_single", "cgtp_bwd_conv", "cgtp_bwd_conv_nogy",
              "cgtp_bwd_single", "cgtp_bwd_single_nogy"}
    assert direct <= set(spills)
    staged = set(spills) - direct
    assert staged in (set(), {k + "_tma" for k in direct}), staged
    if irreps is not W.IRREPS_TP16:
        assert staged, "the workload plans use the staged (TMA) kernels"
    for k in ("cgtp_fwd_conv", "cgtp_fwd_single", "cgtp_fwd_conv_tma", "cgtp_fwd_single_tma"):
        assert spills.get(k, 0) == 0, log
    assert max(spills.values()) <= 256, log
    src = plan.source()
    assert "fma.rn.f32x2" in src or dtype == "f64"


def test_linear_layer_host_side():
    """Instruction list, weight offsets, workspace sizes and argument errors
    of the channel-mixing layer (host only) agree with the oracle's layout."""
    ins, outs = "32x0e+32x1o+64x1o+32x2e", "64x0e+32x1o+32x2e+32x3o"
    lin = cg.Linear(ins, outs)
    ref = O.linear_instructions(ins, outs)
    assert lin.n_instr == len(ref)
    a, b = O.parse_irreps(ins), O.parse_irreps(outs)
    off = 0
    for j, (i, o) in enumerate(ref):
        assert lin.instruction(j) == (i, o, off)
        off += a[i][0] * b[o][0]
    assert lin.weight_numel == off
    assert (lin.dim_in, lin.dim_out) == (O.irreps_dim(a), O.irreps_dim(b))
    assert lin.tensor_cores
    fb, bb = lin.workspace_bytes(1000)
    assert fb > 0 and bb >= 4 * off
    assert not cg.Linear("16x0e", "16x0e").tensor_cores
    assert not cg.Linear("32x0e", "32x0e", dtype=torch.float64).tensor_cores
    with pytest.raises(cg.CgtpError):
        cg.Linear("4x0e", "4x1o", instr=[(0, 0)])
    with pytest.raises(cg.CgtpError):
        cg.Linear("4x0e", "4x0e", instr=[(0, 1)])
    with pytest.raises(cg.CgtpError):
        cg.Linear("4x0q", "4x0e")


def test_noalloc_entry_point_host_errors():
    """The no-allocation gradient rejects, before any CUDA call, a plan whose
    kernels never ran (their first load allocates) and a shared weight row
    too large for the fixed scratch (64 KiB at most)."""
    L = cg.lib()
    vp = ctypes.c_void_p
    f = L.cgtp_conv_backward_noalloc
    f.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, vp, vp, vp, vp, vp, vp, vp, vp,
                  ctypes.c_double, vp, vp, vp, vp, vp]
    f.restype = ctypes.c_int
    a = vp(0x1000)
    args = lambda plan: (plan._h, 3, 4, a, a, a, a, a, a, a, a, 1.0, a, a, a, a, None)
    fresh = cg.Plan(*W.IRREPS_CONV64)
    assert f(*args(fresh)) == 1
    assert b"have not run" in L.cgtp_last_error_message()
    fresh_shared = cg.Plan(*W.IRREPS_CONV64, shared_weights=True)
    assert f(*args(fresh_shared)) == 1
    assert b"have not run" in L.cgtp_last_error_message()
    # 24 paths x 1024 channels x 4 bytes = 96 KiB per weight row
    big = cg.Plan("1024x0e+1024x1o+1024x2e", "0e+1o+2e+3o",
                  "1024x0e+1024x1o+1024x1e+1024x2o+1024x2e+1024x3o+1024x3e", shared_weights=True)
    assert big.weight_numel * 4 > 64 * 1024
    assert f(*args(big)) == 1
    assert b"no-allocation limit" in L.cgtp_last_error_message()
    # the same row without a weight gradient needs no scratch: the size check passes
    no_gw = (big._h, 3, 4, a, a, a, a, a, a, a, a, 1.0, a, a, a, None, None)
    assert f(*no_gw) == 1
    assert b"have not run" in L.cgtp_last_error_message()
    assert f(None, 3, 4, a, a, a, a, a, a, a, a, 1.0, a, a, a, a, None) == 1


def test_uvw_product_host_side():
    """The 'uvw' product's path list (planner) is the oracle's parity-allowed
    list, its matrices lie one after another, and bad arguments are refused
    before any CUDA call."""
    a, b, c = "16x0e+16x1o+16x2e", "0e+1o+2e+3o", "8x0e+8x1o+8x1e+8x2o+8x2e"
    u = cg.UVWProduct(a, b, c)
    ref = O.make_problem(a, b, c.replace("8x", "16x"))
    assert u.n_paths == len(ref.paths)
    for p, q in enumerate(ref.paths):
        l1, l2, l3, i1, i2, io, off = u.path(p)
        assert (i1, i2, io, l1, l2, l3) == q[:6]
        assert off == p * 16 * 8
    assert u.weight_numel == u.n_paths * 16 * 8
    assert u.dim_in1 == 16 * 9 and u.dim_in2 == 16 and u.dim_out == 8 * (1 + 3 + 3 + 5 + 5)
    assert u.dim_mid == 16 * sum(2 * q[5] + 1 for q in ref.paths)
    f, bwd = u.workspace_bytes(1000)
    assert f >= 1000 * u.dim_mid * 4 and bwd >= 2 * 1000 * u.dim_mid * 4
    L = cg.lib()
    h = ctypes.c_void_p()
    assert L.cgtp_uvw_create(ctypes.byref(h), b"16x0e+8x1o", b"0e", b"16x0e", 0) == 2
    assert L.cgtp_uvw_create(ctypes.byref(h), b"16x0e", b"2x0e", b"16x0e", 0) == 2
    assert L.cgtp_uvw_create(ctypes.byref(h), b"16x0e", b"0e", b"16x1o", 0) == 3
    assert L.cgtp_uvw_create(None, b"16x0e", b"0e", b"16x0e", 0) == 1
    null = ctypes.c_void_p()
    # a workspace that is missing or too small is refused
    assert L.cgtp_uvw_forward(u._h, 4, null, null, null, null, null, null, 0, null) == 1
    assert b"workspace" in L.cgtp_last_error_message()


def _defines(src):
    return dict(re.findall(r"#define (W_DIRECT_B|W_DIRECT_F|GB|GF|STAGES_B|STAGES_F|CPT|LANES) (\w+)",
                           src))


def test_planner_automatic_launch_shapes():
    """The automatic launch shapes the measurements chose (no GPU needed: the
    generated source carries them): one warp group and a 2-deep ring each way;
    backward weights loaded by the lanes with two channels per lane, through
    the ring with one (32-channel irreps) and in fp64; forward weights through
    the ring.  Flags override them."""
    conv = _defines(cg.Plan(*W.IRREPS_CONV64).source())
    assert conv == {"CPT": "2", "LANES": "32", "STAGES_F": "2", "STAGES_B": "2",
                    "W_DIRECT_F": "0", "W_DIRECT_B": "1", "GF": "1", "GB": "1"}
    tfn = _defines(cg.Plan(*W.tfn32_mol1000()["irreps"]).source())
    assert (tfn["CPT"], tfn["W_DIRECT_B"], tfn["GB"], tfn["STAGES_B"]) == ("1", "0", "1", "2")
    f64 = _defines(cg.Plan(*W.IRREPS_CONV64, dtype=torch.float64).source())
    assert f64["W_DIRECT_B"] == "0"
    # overrides: backward weights through the ring, 3-deep backward ring, two
    # forward warp groups
    ovr = _defines(cg.Plan(*W.IRREPS_CONV64, flags=(1 << 17) | (3 << 12) | 2).source())
    assert (ovr["W_DIRECT_B"], ovr["STAGES_B"], ovr["GF"]) == ("0", "3", "2")
