"""Clebsch-Gordan tensor products on GB300 (sm_103a): Python binding.

A thin ctypes layer over the C ABI of ``libcgtp.so`` (declared in
``include/cgtp.h``).  It marshals torch CUDA tensors into pointers and the
current torch stream; every step of the computation runs in the library's own
kernels.  If the library has not been built, every entry point raises -- there
is no CPU fallback.

Operations (see "An Efficient Sparse Kernel Generator for O(3)-Equivariant
Deep Networks", abstract): the CG tensor product of irrep features x and
spherical harmonics y under per-edge 'uvu' weights, standalone and fused with
the graph convolution, with gradients and higher derivatives; spherical
harmonics of edge vectors (NVIDIA SE(3)-Transformer blog, "Basis
precomputation") and interatomic forces from edge gradients.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libcgtp.so")

_lock = threading.Lock()
_lib = None

F32, F64 = 0, 1
W_PER_EDGE, W_SHARED = 0, 1
WEIGHTS_BF16 = 1 << 24  # plan flag: weights stored as bfloat16
WEIGHTS_F16 = 1 << 25  # plan flag: weights stored as IEEE binary16
TEST_WAIT_TIMEOUT = 1 << 26  # plan flag, tests only: the first bounded wait of each CTA gives up
GY_WARP = 1 << 19  # plan flag: grad_y on a second warp per backward CTA


class CgtpError(RuntimeError):
    pass


class _LinInstr(ctypes.Structure):
    _fields_ = [("i_in", ctypes.c_int), ("i_out", ctypes.c_int)]


class _Instr(ctypes.Structure):
    _fields_ = [("i_in1", ctypes.c_int), ("i_in2", ctypes.c_int), ("i_out", ctypes.c_int),
                ("mode", ctypes.c_char * 4)]


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise CgtpError(f"{LIB_PATH} is missing: build it with "
                                "`python -m clebsch_gordan_tensor_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            P = ctypes.POINTER
            sig = {
                "cgtp_plan_create": [P(vp), ctypes.c_char_p, ctypes.c_char_p, ctypes.c_char_p,
                                     P(_Instr), i32, i32, i32, ctypes.c_uint],
                "cgtp_plan_destroy": [vp],
                "cgtp_plan_info": [vp, P(i64), P(i64), P(i64), P(i64), P(i32)],
                "cgtp_plan_path": [vp, i32, P(i32), P(i32), P(i32), P(i32), P(i32), P(i32)],
                "cgtp_plan_coefficients": [vp, i32, P(ctypes.c_double)],
                "cgtp_plan_compile": [vp, ctypes.c_char_p, ctypes.c_size_t],
                "cgtp_plan_source": [vp, ctypes.c_char_p, ctypes.c_size_t, P(ctypes.c_size_t)],
                "cgtp_forward": [vp, i64, vp, vp, vp, vp, vp],
                "cgtp_backward": [vp, i64, vp, vp, vp, vp, vp, vp, vp, vp],
                "cgtp_double_backward": [vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp],
                "cgtp_double_backward_ws": [vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                            vp, ctypes.c_size_t, vp],
                "cgtp_conv_forward": [vp, i64, i64, vp, vp, vp, vp, vp, ctypes.c_double, vp, vp],
                "cgtp_conv_backward": [vp, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp,
                                       ctypes.c_double, vp, vp, vp, vp, vp],
                "cgtp_conv_double_backward": [vp, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp,
                                              ctypes.c_double, vp, vp, vp, vp, vp, vp, vp, vp,
                                              vp],
                "cgtp_conv_double_backward_ws": [vp, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp,
                                                 ctypes.c_double, vp, vp, vp, vp, vp, vp, vp, vp,
                                                 vp, ctypes.c_size_t, vp],
                "cgtp_sh_forward": [i32, i32, i64, vp, vp, vp],
                "cgtp_sh_backward": [i32, i32, i64, vp, vp, vp, vp],
                "cgtp_sh_jvp": [i32, i32, i64, vp, vp, vp, vp],
                "cgtp_sh_hvp": [i32, i32, i64, vp, vp, vp, vp, vp],
                "cgtp_edge_forces": [i32, i64, i64, vp, vp, vp, vp, vp, vp],
                "cgtp_edge_forces_adjoint": [i32, i64, i64, vp, vp, vp, vp, vp],
                "cgtp_last_cuda_error": [P(i32)],
                "cgtp_plan_device_status": [vp, P(i32)],
                "cgtp_weight_grad_workspace": [vp, P(ctypes.c_size_t)],
                "cgtp_backward_ws": [vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp],
                "cgtp_conv_backward_ws": [vp, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp,
                                          ctypes.c_double, vp, vp, vp, vp, vp, ctypes.c_size_t,
                                          vp],
                "cgtp_conv_backward_noalloc": [vp, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp,
                                               ctypes.c_double, vp, vp, vp, vp, vp],
                "cgtp_radial_forward": [i32, i64, i32, ctypes.c_double, i32, i64, vp, vp, vp,
                                        vp, vp, vp, ctypes.c_size_t, ctypes.c_uint, vp],
                "cgtp_radial_workspace": [i32, i32, i32, i64, P(ctypes.c_size_t)],
                "cgtp_radial_backward": [i32, i64, i32, ctypes.c_double, i32, i64, vp, vp, vp, vp,
                                         vp, vp, vp, vp, ctypes.c_size_t, ctypes.c_uint, vp],
                "cgtp_radial_backward_workspace": [i32, i64, i32, i32, i64, P(ctypes.c_size_t)],
                "cgtp_radial_path": [i32, i32, i32, i64, P(i32)],
                "cgtp_radial_device_status": [P(i32)],
                "cgtp_linear_create": [P(vp), ctypes.c_char_p, ctypes.c_char_p, P(_LinInstr),
                                       i32, i32],
                "cgtp_linear_destroy": [vp],
                "cgtp_linear_info": [vp, P(i64), P(i64), P(i64), P(i32)],
                "cgtp_linear_instruction": [vp, i32, P(i32), P(i32), P(i64)],
                "cgtp_linear_workspace": [vp, i64, P(ctypes.c_size_t), P(ctypes.c_size_t)],
                "cgtp_linear_path": [vp, P(i32)],
                "cgtp_linear_forward": [vp, i64, vp, vp, vp, vp, ctypes.c_size_t, ctypes.c_uint,
                                        vp],
                "cgtp_linear_backward": [vp, i64, vp, vp, vp, vp, vp, vp, ctypes.c_size_t,
                                         ctypes.c_uint, vp],
                "cgtp_linear_device_status": [P(i32)],
                "cgtp_fma_probe": [i32, i32, i64, i32, i64, vp, P(i64), vp],
                "cgtp_uvw_create": [P(vp), ctypes.c_char_p, ctypes.c_char_p, ctypes.c_char_p,
                                    i32],
                "cgtp_uvw_destroy": [vp],
                "cgtp_uvw_info": [vp, P(i64), P(i64), P(i64), P(i64), P(i64), P(i32)],
                "cgtp_uvw_path": [vp, i32, P(i32), P(i32), P(i32), P(i32), P(i32), P(i32),
                                  P(i64)],
                "cgtp_uvw_parts": [vp, P(vp), P(vp)],
                "cgtp_uvw_workspace": [vp, i64, P(ctypes.c_size_t), P(ctypes.c_size_t)],
                "cgtp_uvw_forward": [vp, i64, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp],
                "cgtp_uvw_backward": [vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      ctypes.c_size_t, vp],
                "cgtp_uvw_conv_forward": [vp, i64, i64, vp, vp, vp, vp, vp, ctypes.c_double, vp,
                                          vp, vp, ctypes.c_size_t, vp],
                "cgtp_uvw_conv_backward": [vp, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp,
                                           ctypes.c_double, vp, vp, vp, vp, vp, vp,
                                           ctypes.c_size_t, vp],
            }
            for name, args in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = ctypes.c_int
            L.cgtp_status_str.argtypes = [ctypes.c_int]
            L.cgtp_status_str.restype = ctypes.c_char_p
            L.cgtp_last_error_message.argtypes = []
            L.cgtp_last_error_message.restype = ctypes.c_char_p
            L.cgtp_launch_count.argtypes = []
            L.cgtp_launch_count.restype = ctypes.c_int64
            _lib = L
    return _lib


def _check(st: int) -> None:
    if st != 0:
        L = lib()
        msg = L.cgtp_last_error_message().decode(errors="replace")
        raise CgtpError(f"{L.cgtp_status_str(st).decode()} (status {st}): {msg}")


def launch_count() -> int:
    """Kernel launches issued through the library by this process."""
    return int(lib().cgtp_launch_count())


def fma_probe(dtype, packed: bool, blocks: int, threads: int, iters: int, sink) -> int:
    """Launch the FMA-pipe throughput probe on the current stream (see
    cgtp_fma_probe); returns the floating-point operations it performs.  sink:
    a device tensor of at least blocks * threads 8-byte words."""
    assert sink.numel() * sink.element_size() >= blocks * threads * 8
    fl = ctypes.c_int64()
    _check(lib().cgtp_fma_probe(_dt(dtype), int(packed), blocks, threads, iters, _ptr(sink),
                                ctypes.byref(fl), _stream()))
    return fl.value


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dt(dtype) -> int:
    if dtype == torch.float32:
        return F32
    if dtype == torch.float64:
        return F64
    raise CgtpError(f"unsupported dtype {dtype}")


def _need(t, name, dtype, shape=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise CgtpError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise CgtpError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise CgtpError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise CgtpError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


class Graph:
    """Receiver-sorted CSR (rowptr, sender) plus the sender-grouped view
    (s_rowptr, s_perm, s_recv), as int32 CUDA tensors."""

    def __init__(self, N, rowptr, sender, s_rowptr=None, s_perm=None, s_recv=None):
        self.N = int(N)
        self.rowptr, self.sender = rowptr, sender
        self.s_rowptr, self.s_perm, self.s_recv = s_rowptr, s_perm, s_recv
        self.E = int(sender.shape[0])
        for n, t in (("rowptr", rowptr), ("sender", sender), ("s_rowptr", s_rowptr),
                     ("s_perm", s_perm), ("s_recv", s_recv)):
            _need(t, n, torch.int32)
        if rowptr.shape[0] != self.N + 1:
            raise CgtpError("rowptr must have N+1 entries")

    @classmethod
    def from_numpy(cls, g, device="cuda"):
        """From a workloads.Graph-like object with numpy int32 arrays."""
        t = lambda a: torch.from_numpy(a).to(device=device, dtype=torch.int32).contiguous()
        return cls(g.N, t(g.rowptr), t(g.sender), t(g.s_rowptr), t(g.s_perm), t(g.s_recv))


class Plan:
    """A tensor-product plan: irreps, 'uvu' paths and the real CG tables, with
    its kernels compiled for sm_103a on first use."""

    def __init__(self, irreps_in1: str, irreps_in2: str, irreps_out: str,
                 dtype=torch.float32, shared_weights: bool = False, instructions=None,
                 weight_dtype=None, flags: int = 0):
        """weight_dtype=torch.bfloat16 or torch.float16 stores the weights in that
        16-bit format (fp32 plans; arithmetic, features and grad_w stay fp32).
        flags: further cgtp_plan_create flags (launch-shape overrides, tests)."""
        L = lib()
        self.dtype = dtype
        self.wdtype = dtype if weight_dtype is None else weight_dtype
        if self.wdtype not in (dtype, torch.bfloat16, torch.float16):
            raise CgtpError(f"weight_dtype {weight_dtype} is not supported")
        flags = int(flags) | {torch.bfloat16: WEIGHTS_BF16,
                              torch.float16: WEIGHTS_F16}.get(self.wdtype, 0)
        self.irreps = (irreps_in1, irreps_in2, irreps_out)
        h = ctypes.c_void_p()
        arr, n = None, 0
        if instructions is not None:
            n = len(instructions)
            arr = (_Instr * max(1, n))()
            for k, (a, b, c) in enumerate(instructions):
                arr[k] = _Instr(a, b, c, b"uvu")
        _check(L.cgtp_plan_create(ctypes.byref(h), irreps_in1.encode(), irreps_in2.encode(),
                                  irreps_out.encode(), arr, n, _dt(dtype),
                                  W_SHARED if shared_weights else W_PER_EDGE, flags))
        self._h = h
        d1, d2, do, wn = (ctypes.c_int64() for _ in range(4))
        npth = ctypes.c_int()
        _check(L.cgtp_plan_info(h, ctypes.byref(d1), ctypes.byref(d2), ctypes.byref(do),
                                ctypes.byref(wn), ctypes.byref(npth)))
        self.dim_in1, self.dim_in2, self.dim_out = d1.value, d2.value, do.value
        self.weight_numel, self.n_paths = wn.value, npth.value
        self.shared_weights = shared_weights

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None and not getattr(self, "_borrowed", False):
            _lib.cgtp_plan_destroy(h)
            self._h = None

    # ---- host queries
    def path(self, p: int):
        vals = [ctypes.c_int() for _ in range(6)]
        _check(lib().cgtp_plan_path(self._h, p, *[ctypes.byref(v) for v in vals]))
        return tuple(v.value for v in vals)

    def coefficients(self, p: int):
        import numpy as np
        l1, l2, l3 = self.path(p)[:3]
        out = np.zeros((2 * l1 + 1) * (2 * l2 + 1) * (2 * l3 + 1))
        _check(lib().cgtp_plan_coefficients(self._h, p, out.ctypes.data_as(
            ctypes.POINTER(ctypes.c_double))))
        return out.reshape(2 * l1 + 1, 2 * l2 + 1, 2 * l3 + 1)

    def device_status(self) -> int:
        """Raise if a staged kernel of this plan reported a device-side error
        (bounded wait timed out); synchronises with the device."""
        code = ctypes.c_int(0)
        _check(lib().cgtp_plan_device_status(self._h, ctypes.byref(code)))
        return code.value

    def compile(self) -> str:
        buf = ctypes.create_string_buffer(1 << 16)
        _check(lib().cgtp_plan_compile(self._h, buf, len(buf)))
        return buf.value.decode(errors="replace")

    def source(self) -> str:
        need = ctypes.c_size_t()
        _check(lib().cgtp_plan_source(self._h, None, 0, ctypes.byref(need)))
        buf = ctypes.create_string_buffer(need.value)
        _check(lib().cgtp_plan_source(self._h, buf, need.value, None))
        return buf.value.decode()

    def _workspace(self, device, gw, copies: int = 1):
        """Scratch for the shared-weight gradient (torch-allocated), or None;
        the double backward takes two copies."""
        if not self.shared_weights or gw is None:
            return None, 0
        n = ctypes.c_size_t()
        _check(lib().cgtp_weight_grad_workspace(self._h, ctypes.byref(n)))
        nb = copies * n.value
        return torch.empty(nb, dtype=torch.uint8, device=device), nb

    def _wshape(self, rows):
        return (self.weight_numel,) if self.shared_weights else (rows, self.weight_numel)

    # ---- standalone
    def forward(self, x, y, w, out=None):
        B = x.shape[0]
        _need(x, "x", self.dtype, (B, self.dim_in1))
        _need(y, "y", self.dtype, (B, self.dim_in2))
        _need(w, "w", self.wdtype, self._wshape(B))
        if out is None:
            out = torch.empty(B, self.dim_out, dtype=self.dtype, device=x.device)
        _need(out, "out", self.dtype, (B, self.dim_out))
        _check(lib().cgtp_forward(self._h, B, _ptr(x), _ptr(y), _ptr(w), _ptr(out), _stream()))
        return out

    def backward(self, x, y, w, grad_out, need=(True, True, True)):
        B = x.shape[0]
        _need(x, "x", self.dtype, (B, self.dim_in1))
        _need(y, "y", self.dtype, (B, self.dim_in2))
        _need(w, "w", self.wdtype, self._wshape(B))
        _need(grad_out, "grad_out", self.dtype, (B, self.dim_out))
        gx = torch.empty_like(x) if need[0] else None
        gy = torch.empty_like(y) if need[1] else None
        gw = torch.empty(w.shape, dtype=self.dtype, device=w.device) if need[2] else None
        ws, nws = self._workspace(x.device, gw)
        _check(lib().cgtp_backward_ws(self._h, B, _ptr(x), _ptr(y), _ptr(w), _ptr(grad_out),
                                      _ptr(gx), _ptr(gy), _ptr(gw), _ptr(ws), nws, _stream()))
        return gx, gy, gw

    def double_backward(self, x, y, w, grad_out, gg_x=None, gg_y=None, gg_w=None,
                        need=(True, True, True, True)):
        B = x.shape[0]
        for n, t, s in (("x", x, (B, self.dim_in1)), ("y", y, (B, self.dim_in2)),
                        ("w", w, self._wshape(B)), ("grad_out", grad_out, (B, self.dim_out)),
                        ("gg_x", gg_x, (B, self.dim_in1)), ("gg_y", gg_y, (B, self.dim_in2)),
                        ("gg_w", gg_w, self._wshape(B))):
            _need(t, n, self.wdtype if n in ("w", "gg_w") else self.dtype, s)
        dx = torch.empty_like(x) if need[0] else None
        dy = torch.empty_like(y) if need[1] else None
        dw = torch.empty_like(w) if need[2] else None
        dg = torch.empty_like(grad_out) if need[3] else None
        ws, nws = self._workspace(x.device, dw, 2)
        _check(lib().cgtp_double_backward_ws(self._h, B, _ptr(x), _ptr(y), _ptr(w), _ptr(grad_out),
                                             _ptr(gg_x), _ptr(gg_y), _ptr(gg_w), _ptr(dx), _ptr(dy),
                                             _ptr(dw), _ptr(dg), _ptr(ws), nws, _stream()))
        return dx, dy, dw, dg

    # ---- fused convolution
    def _conv_check(self, g: Graph, x, y, w):
        _need(x, "x", self.dtype, (g.N, self.dim_in1))
        _need(y, "y", self.dtype, (g.E, self.dim_in2))
        _need(w, "w", self.wdtype, self._wshape(g.E))

    def conv_forward(self, g: Graph, x, y, w, scale: float = 1.0, out=None):
        self._conv_check(g, x, y, w)
        if out is None:
            out = torch.empty(g.N, self.dim_out, dtype=self.dtype, device=x.device)
        _need(out, "out", self.dtype, (g.N, self.dim_out))
        _check(lib().cgtp_conv_forward(self._h, g.N, g.E, _ptr(g.rowptr), _ptr(g.sender),
                                       _ptr(x), _ptr(y), _ptr(w), float(scale), _ptr(out),
                                       _stream()))
        return out

    def conv_backward(self, g: Graph, x, y, w, scale, grad_out, need=(True, True, True),
                      out=None):
        self._conv_check(g, x, y, w)
        _need(grad_out, "grad_out", self.dtype, (g.N, self.dim_out))
        if out is not None:
            gx, gy, gw = out
        else:
            gx = torch.empty_like(x) if need[0] else None
            gy = torch.empty_like(y) if need[1] else None
            gw = torch.empty(w.shape, dtype=self.dtype, device=w.device) if need[2] else None
        ws, nws = self._workspace(x.device, gw)
        _check(lib().cgtp_conv_backward_ws(self._h, g.N, g.E, _ptr(g.rowptr), _ptr(g.sender),
                                           _ptr(g.s_rowptr), _ptr(g.s_perm), _ptr(g.s_recv),
                                           _ptr(x), _ptr(y), _ptr(w), float(scale),
                                           _ptr(grad_out), _ptr(gx), _ptr(gy), _ptr(gw), _ptr(ws),
                                           nws, _stream()))
        return gx, gy, gw

    def conv_double_backward(self, g: Graph, x, y, w, scale, grad_out, gg_x=None, gg_y=None,
                             gg_w=None, need=(True, True, True, True)):
        self._conv_check(g, x, y, w)
        _need(grad_out, "grad_out", self.dtype, (g.N, self.dim_out))
        _need(gg_x, "gg_x", self.dtype, (g.N, self.dim_in1))
        _need(gg_y, "gg_y", self.dtype, (g.E, self.dim_in2))
        _need(gg_w, "gg_w", self.wdtype, self._wshape(g.E))
        dx = torch.empty_like(x) if need[0] else None
        dy = torch.empty_like(y) if need[1] else None
        dw = torch.empty_like(w) if need[2] else None
        dg = torch.empty_like(grad_out) if need[3] else None
        ws, nws = self._workspace(x.device, dw, 2)
        _check(lib().cgtp_conv_double_backward_ws(
            self._h, g.N, g.E, _ptr(g.rowptr), _ptr(g.sender), _ptr(g.s_rowptr), _ptr(g.s_perm),
            _ptr(g.s_recv), _ptr(x), _ptr(y), _ptr(w), float(scale), _ptr(grad_out), _ptr(gg_x),
            _ptr(gg_y), _ptr(gg_w), _ptr(dx), _ptr(dy), _ptr(dw), _ptr(dg), _ptr(ws), nws,
            _stream()))
        return dx, dy, dw, dg


# ------------------------------------------------------ spherical harmonics

def sh_forward(vec, lmax: int, out=None):
    E = vec.shape[0]
    _need(vec, "vec", vec.dtype, (E, 3))
    if out is None:
        out = torch.empty(E, (lmax + 1) ** 2, dtype=vec.dtype, device=vec.device)
    _need(out, "out", vec.dtype, (E, (lmax + 1) ** 2))
    _check(lib().cgtp_sh_forward(lmax, _dt(vec.dtype), E, _ptr(vec), _ptr(out), _stream()))
    return out


def sh_backward(vec, grad_y, lmax: int, out=None):
    E = vec.shape[0]
    _need(vec, "vec", vec.dtype, (E, 3))
    _need(grad_y, "grad_y", vec.dtype, (E, (lmax + 1) ** 2))
    if out is None:
        out = torch.empty_like(vec)
    _check(lib().cgtp_sh_backward(lmax, _dt(vec.dtype), E, _ptr(vec), _ptr(grad_y), _ptr(out),
                                  _stream()))
    return out


def sh_jvp(vec, tangent_vec, lmax: int, out=None):
    E = vec.shape[0]
    _need(vec, "vec", vec.dtype, (E, 3))
    _need(tangent_vec, "tangent_vec", vec.dtype, (E, 3))
    if out is None:
        out = torch.empty(E, (lmax + 1) ** 2, dtype=vec.dtype, device=vec.device)
    _check(lib().cgtp_sh_jvp(lmax, _dt(vec.dtype), E, _ptr(vec), _ptr(tangent_vec), _ptr(out),
                             _stream()))
    return out


def sh_hvp(vec, grad_y, tangent_vec, lmax: int, out=None):
    """Hessian of grad_y . Y(vec) in vec applied to tangent_vec, per edge."""
    E = vec.shape[0]
    _need(vec, "vec", vec.dtype, (E, 3))
    _need(grad_y, "grad_y", vec.dtype, (E, (lmax + 1) ** 2))
    _need(tangent_vec, "tangent_vec", vec.dtype, (E, 3))
    if out is None:
        out = torch.empty_like(vec)
    _need(out, "out", vec.dtype, (E, 3))
    _check(lib().cgtp_sh_hvp(lmax, _dt(vec.dtype), E, _ptr(vec), _ptr(grad_y), _ptr(tangent_vec),
                             _ptr(out), _stream()))
    return out


def radial_forward(vec, W1, W2, cutoff: float = 5.0, out=None, hidden_out=None,
                   cuda_cores: bool = False, out_dtype=None):
    """Per-edge weights of the radial network: w[e] = silu(b(|vec[e]|) W1) W2
    with the Bessel basis b_n(r) = sqrt(2/rc) sin(n pi r / rc) / r.  Returns w
    [E, n_out]; ``hidden_out`` [E, hidden], if given, receives silu(b W1)."""
    E = vec.shape[0]
    _need(vec, "vec", vec.dtype, (E, 3))
    nb, hidden = W1.shape
    _need(W1, "W1", vec.dtype, (nb, hidden))
    n_out = W2.shape[1]
    _need(W2, "W2", vec.dtype, (hidden, n_out))
    odt = vec.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty(E, n_out, dtype=odt, device=vec.device)
    _need(out, "out", odt, (E, n_out))
    _need(hidden_out, "hidden_out", vec.dtype, (E, hidden))
    n = ctypes.c_size_t(0)
    _check(lib().cgtp_radial_workspace(_dt(vec.dtype), nb, hidden, n_out, ctypes.byref(n)))
    ws = torch.empty(n.value, dtype=torch.uint8, device=vec.device) if n.value else None
    _check(lib().cgtp_radial_forward(_dt(vec.dtype), E, nb, float(cutoff), hidden, n_out,
                                     _ptr(vec), _ptr(W1), _ptr(W2), _ptr(out), _ptr(hidden_out),
                                     _ptr(ws), n.value,
                                     (1 if cuda_cores else 0) | (2 if odt == torch.bfloat16 else 0)
                                     | (4 if odt == torch.float16 else 0),
                                     _stream()))
    return out


def radial_backward(vec, W1, W2, grad_w, cutoff: float = 5.0, need=(True, True, True),
                    cuda_cores: bool = False):
    """Gradients of radial_forward's output for the cotangent grad_w: returns
    (grad_vec, grad_W1, grad_W2); entries not in `need` are None."""
    E = vec.shape[0]
    _need(vec, "vec", vec.dtype, (E, 3))
    nb, hidden = W1.shape
    n_out = W2.shape[1]
    _need(W1, "W1", vec.dtype, (nb, hidden))
    _need(W2, "W2", vec.dtype, (hidden, n_out))
    _need(grad_w, "grad_w", vec.dtype, (E, n_out))
    gv = torch.empty_like(vec) if need[0] else None
    g1 = torch.empty_like(W1) if need[1] else None
    g2 = torch.empty_like(W2) if need[2] else None
    n = ctypes.c_size_t(0)
    _check(lib().cgtp_radial_backward_workspace(_dt(vec.dtype), E, nb, hidden, n_out,
                                                ctypes.byref(n)))
    ws = torch.empty(n.value, dtype=torch.uint8, device=vec.device) if n.value else None
    _check(lib().cgtp_radial_backward(_dt(vec.dtype), E, nb, float(cutoff), hidden, n_out,
                                      _ptr(vec), _ptr(W1), _ptr(W2), _ptr(grad_w), _ptr(gv),
                                      _ptr(g1), _ptr(g2), _ptr(ws), n.value,
                                      1 if cuda_cores else 0, _stream()))
    return gv, g1, g2


def radial_uses_tensor_cores(dtype, n_basis: int, hidden: int, n_out: int) -> bool:
    """Whether radial_forward takes the tensor-core path for these sizes (with
    16-byte aligned tensors)."""
    v = ctypes.c_int(0)
    _check(lib().cgtp_radial_path(_dt(dtype), n_basis, hidden, n_out, ctypes.byref(v)))
    return bool(v.value)


def radial_device_status() -> int:
    """Reads and clears the radial kernels' device error flag (synchronous)."""
    v = ctypes.c_int(0)
    _check(lib().cgtp_radial_device_status(ctypes.byref(v)))
    return int(v.value)


def edge_forces(g: Graph, dEdr, out=None):
    _need(dEdr, "dEdr", dEdr.dtype, (g.E, 3))
    if out is None:
        out = torch.empty(g.N, 3, dtype=dEdr.dtype, device=dEdr.device)
    _check(lib().cgtp_edge_forces(_dt(dEdr.dtype), g.N, g.E, _ptr(g.rowptr), _ptr(g.s_rowptr),
                                  _ptr(g.s_perm), _ptr(dEdr), _ptr(out), _stream()))
    return out


def edge_forces_adjoint(g: Graph, grad_forces, out=None):
    _need(grad_forces, "grad_forces", grad_forces.dtype, (g.N, 3))
    if out is None:
        out = torch.empty(g.E, 3, dtype=grad_forces.dtype, device=grad_forces.device)
    _check(lib().cgtp_edge_forces_adjoint(_dt(grad_forces.dtype), g.N, g.E, _ptr(g.rowptr),
                                          _ptr(g.sender), _ptr(grad_forces), _ptr(out),
                                          _stream()))
    return out


class Linear:
    """Per-irrep channel mixing: out[n, o, m, w] = sum over instructions (i, o)
    of sum_u x[n, i, m, u] W_j[u, w] (the layer of ``cgtp_linear_forward``).
    ``instr`` lists (i_in, i_out) pairs; None takes every pair of equal irreps."""

    def __init__(self, irreps_in: str, irreps_out: str, instr=None, dtype=torch.float32):
        self.dtype = dtype
        h = ctypes.c_void_p()
        if instr is None:
            arr, n = None, 0
        else:
            arr = (_LinInstr * max(1, len(instr)))(*[_LinInstr(i, o) for i, o in instr])
            n = len(instr)
        _check(lib().cgtp_linear_create(ctypes.byref(h), irreps_in.encode(), irreps_out.encode(),
                                        arr, n, _dt(dtype)))
        self._h = h
        a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        k = ctypes.c_int()
        _check(lib().cgtp_linear_info(h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c),
                                      ctypes.byref(k)))
        self.dim_in, self.dim_out, self.weight_numel, self.n_instr = a.value, b.value, c.value, k.value
        t = ctypes.c_int()
        _check(lib().cgtp_linear_path(h, ctypes.byref(t)))
        self.tensor_cores = bool(t.value)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None and not getattr(self, "_borrowed", False):
            _lib.cgtp_linear_destroy(h)

    def instruction(self, j: int):
        i, o, w = ctypes.c_int(), ctypes.c_int(), ctypes.c_int64()
        _check(lib().cgtp_linear_instruction(self._h, j, ctypes.byref(i), ctypes.byref(o),
                                             ctypes.byref(w)))
        return i.value, o.value, w.value

    def workspace_bytes(self, n: int):
        f, b = ctypes.c_size_t(), ctypes.c_size_t()
        _check(lib().cgtp_linear_workspace(self._h, n, ctypes.byref(f), ctypes.byref(b)))
        return f.value, b.value

    def _ws(self, nbytes, device):
        return torch.empty(max(1, (nbytes + 15) // 16) * 16, dtype=torch.uint8, device=device)

    def forward(self, x, W, out=None, workspace=None, cuda_cores: bool = False):
        n = x.shape[0]
        _need(x, "x", self.dtype, (n, self.dim_in))
        _need(W, "W", self.dtype, (self.weight_numel,))
        if out is None:
            out = torch.empty(n, self.dim_out, dtype=self.dtype, device=x.device)
        _need(out, "out", self.dtype, (n, self.dim_out))
        fb, _ = self.workspace_bytes(n)
        if workspace is None and fb > 0:
            workspace = self._ws(fb, x.device)
        nb = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check(lib().cgtp_linear_forward(self._h, n, _ptr(x), _ptr(W), _ptr(out), _ptr(workspace),
                                         nb, 1 if cuda_cores else 0, _stream()))
        return out

    def backward(self, x, W, grad_out, need=(True, True), workspace=None, cuda_cores: bool = False):
        """(grad_x, grad_W); an entry is None where ``need`` is False."""
        n = x.shape[0]
        _need(x, "x", self.dtype, (n, self.dim_in))
        _need(W, "W", self.dtype, (self.weight_numel,))
        _need(grad_out, "grad_out", self.dtype, (n, self.dim_out))
        gx = torch.empty_like(x) if need[0] else None
        gW = torch.empty_like(W) if need[1] else None
        _, bb = self.workspace_bytes(n)
        if workspace is None:
            workspace = self._ws(bb, x.device)
        nb = workspace.numel() * workspace.element_size()
        _check(lib().cgtp_linear_backward(self._h, n, _ptr(x), _ptr(W), _ptr(grad_out), _ptr(gx),
                                          _ptr(gW), _ptr(workspace), nb, 1 if cuda_cores else 0,
                                          _stream()))
        return gx, gW


def linear_device_status() -> int:
    c = ctypes.c_int()
    _check(lib().cgtp_linear_device_status(ctypes.byref(c)))
    return c.value


class UVWProduct:
    """'uvw' tensor product (``cgtp_uvw``): one [mul_in, mul_out] matrix per
    path, shared by all rows,
        out[b, k, m3, w] = sum_paths->k sum_u sum_{m1,m2} C[m1,m2,m3]
                           x[b, i1, m1, u] y[b, i2, m2] W_p[u, w],
    for every parity-allowed path (in1-major, then in2, then out); W holds the
    paths' matrices in order.  The library runs it as the 'uvu' product into
    one block per path (``mid``) followed by the channel mixing on the tensor
    cores; ``plan`` and ``linear`` are those two parts (borrowed)."""

    def __init__(self, irreps_in1: str, irreps_in2: str, irreps_out: str, dtype=torch.float32):
        L = lib()
        self.dtype = dtype
        h = ctypes.c_void_p()
        _check(L.cgtp_uvw_create(ctypes.byref(h), irreps_in1.encode(), irreps_in2.encode(),
                                 irreps_out.encode(), _dt(dtype)))
        self._h = h
        v = [ctypes.c_int64() for _ in range(5)]
        n = ctypes.c_int()
        _check(L.cgtp_uvw_info(h, *[ctypes.byref(t) for t in v], ctypes.byref(n)))
        (self.dim_in1, self.dim_in2, self.dim_out, self.dim_mid,
         self.weight_numel) = (t.value for t in v)
        self.n_paths = n.value
        # irreps of the per-path blocks: in1's multiplicity, each path's l3 and
        # the parity of its target irrep
        mul = int(irreps_in1.replace(" ", "").split("+")[0].split("x")[0])
        par = [t.strip()[-1] for t in irreps_out.split("+")]
        self.mid = "+".join(f"{mul}x{q[2]}{par[q[5]]}"
                            for q in (self.path(p) for p in range(self.n_paths)))
        ph, lh = ctypes.c_void_p(), ctypes.c_void_p()
        _check(L.cgtp_uvw_parts(h, ctypes.byref(ph), ctypes.byref(lh)))
        self.plan = _Borrowed(Plan, ph, self)
        self.linear = _Borrowed(Linear, lh, self)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.cgtp_uvw_destroy(h)
            self._h = None

    def path(self, p: int):
        """(l1, l2, l3, i_in1, i_in2, i_out, weight offset) of path p."""
        vals = [ctypes.c_int() for _ in range(6)]
        off = ctypes.c_int64()
        _check(lib().cgtp_uvw_path(self._h, p, *[ctypes.byref(t) for t in vals],
                                   ctypes.byref(off)))
        return tuple(t.value for t in vals) + (off.value,)

    def workspace_bytes(self, rows: int):
        f, b = ctypes.c_size_t(), ctypes.c_size_t()
        _check(lib().cgtp_uvw_workspace(self._h, rows, ctypes.byref(f), ctypes.byref(b)))
        return f.value, b.value

    def _ws(self, rows, bwd, device, workspace):
        if workspace is not None:
            return workspace, workspace.numel() * workspace.element_size()
        nb = self.workspace_bytes(rows)[1 if bwd else 0]
        t = torch.empty(max(256, nb), dtype=torch.uint8, device=device)
        return t, t.numel()

    def forward(self, x, y, W, out=None, mid=None, workspace=None):
        """out [B, dim_out]; ``mid`` (optional) receives the per-path blocks."""
        B = x.shape[0]
        _need(x, "x", self.dtype, (B, self.dim_in1))
        _need(y, "y", self.dtype, (B, self.dim_in2))
        _need(W, "W", self.dtype, (self.weight_numel,))
        if out is None:
            out = torch.empty(B, self.dim_out, dtype=self.dtype, device=x.device)
        _need(out, "out", self.dtype, (B, self.dim_out))
        if mid is not None:
            _need(mid, "mid", self.dtype, (B, self.dim_mid))
        ws, nb = self._ws(B, False, x.device, workspace)
        _check(lib().cgtp_uvw_forward(self._h, B, _ptr(x), _ptr(y), _ptr(W), _ptr(out),
                                      _ptr(mid), _ptr(ws), nb, _stream()))
        return out

    def backward(self, x, y, W, grad_out, mid=None, need=(True, True, True), workspace=None):
        """(grad_x, grad_y, grad_W) for dL/dout = grad_out; ``mid`` = the
        forward's per-path blocks (recomputed when None)."""
        B = x.shape[0]
        _need(grad_out, "grad_out", self.dtype, (B, self.dim_out))
        gx = torch.empty_like(x) if need[0] else None
        gy = torch.empty_like(y) if need[1] else None
        gW = torch.empty_like(W) if need[2] else None
        ws, nb = self._ws(B, True, x.device, workspace)
        _check(lib().cgtp_uvw_backward(self._h, B, _ptr(x), _ptr(y), _ptr(W), _ptr(grad_out),
                                       _ptr(mid), _ptr(gx), _ptr(gy), _ptr(gW), _ptr(ws), nb,
                                       _stream()))
        return gx, gy, gW

    def conv_forward(self, g: "Graph", x, y, W, scale: float = 1.0, out=None, mid=None,
                     workspace=None):
        """The fused convolution with 'uvw' paths: receiver sums of the per-path
        blocks (``mid`` [N, dim_mid]), then the mixing per node."""
        if out is None:
            out = torch.empty(g.N, self.dim_out, dtype=self.dtype, device=x.device)
        ws, nb = self._ws(g.N, False, x.device, workspace)
        _check(lib().cgtp_uvw_conv_forward(self._h, g.N, g.E, _ptr(g.rowptr), _ptr(g.sender),
                                           _ptr(x), _ptr(y), _ptr(W), float(scale), _ptr(out),
                                           _ptr(mid), _ptr(ws), nb, _stream()))
        return out

    def conv_backward(self, g: "Graph", x, y, W, scale, grad_out, mid=None,
                      need=(True, True, True), workspace=None):
        gx = torch.empty_like(x) if need[0] else None
        gy = torch.empty_like(y) if need[1] else None
        gW = torch.empty_like(W) if need[2] else None
        ws, nb = self._ws(g.N, True, x.device, workspace)
        _check(lib().cgtp_uvw_conv_backward(
            self._h, g.N, g.E, _ptr(g.rowptr), _ptr(g.sender), _ptr(g.s_rowptr), _ptr(g.s_perm),
            _ptr(g.s_recv), _ptr(x), _ptr(y), _ptr(W), float(scale), _ptr(grad_out), _ptr(mid),
            _ptr(gx), _ptr(gy), _ptr(gW), _ptr(ws), nb, _stream()))
        return gx, gy, gW


def _Borrowed(cls, handle, owner):
    """A Plan / Linear view of a handle owned by ``owner`` (never destroyed here)."""
    obj = cls.__new__(cls)
    obj._owner = owner
    if cls is Plan:
        L = lib()
        d1, d2, do, wn = (ctypes.c_int64() for _ in range(4))
        npth = ctypes.c_int()
        _check(L.cgtp_plan_info(handle, ctypes.byref(d1), ctypes.byref(d2), ctypes.byref(do),
                                ctypes.byref(wn), ctypes.byref(npth)))
        obj.dtype = obj.wdtype = owner.dtype
        obj.dim_in1, obj.dim_in2, obj.dim_out = d1.value, d2.value, do.value
        obj.weight_numel, obj.n_paths = wn.value, npth.value
        obj.shared_weights = True
    else:
        L = lib()
        a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        k = ctypes.c_int()
        _check(L.cgtp_linear_info(handle, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c),
                                  ctypes.byref(k)))
        obj.dtype = owner.dtype
        obj.dim_in, obj.dim_out, obj.weight_numel, obj.n_instr = a.value, b.value, c.value, k.value
        t = ctypes.c_int()
        _check(L.cgtp_linear_path(handle, ctypes.byref(t)))
        obj.tensor_cores = bool(t.value)
    obj._h = handle
    obj._borrowed = True
    return obj
