// The 'uvw' tensor product behind the C ABI: one [mul_in, mul_out] matrix per
// path, shared by every row.
//
// NVIDIA's SE(3)-Transformer blog ("TFN fusion") turns the per-degree channel
// contractions of a TFN layer into dense products: the pairwise degree
// convolutions that feed one output degree are summed, and the channel mixing
// runs as a matrix product.  Here that is two library operations:
//   1. the 'uvu' CG product with a shared weight row of ones, into one output
//      block per path (the "mid" row: path p's block has mul_in channels of
//      its l3 and parity), alone or fused with the graph convolution;
//   2. the per-irrep channel mixing from the mid blocks to irreps_out,
//      instruction p joining path p's block to the irrep of its l3 and parity
//      (cgtp_linear, tcgen05 for fp32).
// By linearity the convolution sums the blocks per receiver first and mixes
// once per node.  The path rule (triangle and parity, in1-major, then in2,
// then out) lives here, in the host planner, with the plan's own.
#include <cuda_runtime.h>

#include <array>
#include <cstdlib>
#include <memory>
#include <string>
#include <vector>

#include "cgtp.h"
#include "internal.hpp"

struct cgtp_uvw_s {
    cgtp_plan plan = nullptr;     // 'uvu' into the mid blocks, shared unit weights
    cgtp_linear lin = nullptr;    // mid blocks -> irreps_out
    cgtp_dtype dtype = CGTP_F32;
    int64_t dim1 = 0, dim2 = 0, dimo = 0, dimmid = 0, wtp = 0, wnumel = 0;
    std::vector<std::array<int, 6>> paths;  // l1, l2, l3, i_in1, i_in2, i_out
    std::vector<int64_t> woff;              // offset of W_p in the weight vector
    cgtp::LinTpDesc tp;                     // the paths as the mixing kernel's row source
    bool tp_ok = false;                     // tp describes every path
};

namespace cgtp {

static cgtp_status ufail(cgtp_status s, const std::string& m) {
    set_error_message(m);
    return s;
}

static size_t up256(size_t b) { return (b + 255) / 256 * 256; }

// Workspace layout: [unit weight row][mid rows][grad mid rows (backward)][mixing workspace].
struct UvwLayout {
    size_t ones = 0, mid = 0, gmid = 0, lin = 0, total = 0;
};

static UvwLayout uvw_layout(const cgtp_uvw_s& u, int64_t rows, bool bwd, bool need_mid) {
    const size_t es = u.dtype == CGTP_F64 ? 8 : 4;
    UvwLayout L;
    size_t fb = 0, bb = 0;
    cgtp_linear_workspace(u.lin, rows, &fb, &bb);
    size_t off = up256((size_t)u.wtp * es);
    L.mid = off;
    if (need_mid) off += up256((size_t)rows * u.dimmid * es);
    L.gmid = off;
    if (bwd) off += up256((size_t)rows * u.dimmid * es);
    L.lin = off;
    off += up256(bwd ? bb : fb);
    L.total = off;
    return L;
}

static unsigned char* at(void* ws, size_t off) { return static_cast<unsigned char*>(ws) + off; }

static cgtp_status uvw_ws_check(const cgtp_uvw_s& u, int64_t rows, bool bwd, const void* mid,
                                void* ws, size_t ws_bytes, UvwLayout& L) {
    L = uvw_layout(u, rows, bwd, mid == nullptr);
    if (!ws || ((uintptr_t)ws % 256) != 0 || ws_bytes < L.total)
        return ufail(CGTP_E_ARG, "the 'uvw' product needs a 256-byte aligned workspace of "
                                 "cgtp_uvw_workspace() bytes (" + std::to_string(L.total) + ")");
    return CGTP_OK;
}

}  // namespace cgtp

using namespace cgtp;

#define UGUARD_BEGIN try {
#define UGUARD_END                                                   \
    }                                                                \
    catch (const std::bad_alloc&) {                                  \
        return ufail(CGTP_E_NOMEM, "host allocation failed");        \
    }                                                                \
    catch (...) {                                                    \
        return ufail(CGTP_E_ARG, "unexpected internal exception");   \
    }

extern "C" {

cgtp_status cgtp_uvw_create(cgtp_uvw* out, const char* irreps_in1, const char* irreps_in2,
                            const char* irreps_out, cgtp_dtype dtype) {
    UGUARD_BEGIN
    if (!out) return ufail(CGTP_E_ARG, "NULL output handle");
    *out = nullptr;
    if (dtype != CGTP_F32 && dtype != CGTP_F64) return ufail(CGTP_E_ARG, "bad dtype");
    if (!irreps_in1 || !irreps_in2 || !irreps_out) return ufail(CGTP_E_ARG, "NULL irreps");
    std::vector<Irrep> a, b, c;
    std::string err;
    if (!parse_irreps(irreps_in1, a, err) || !parse_irreps(irreps_in2, b, err) ||
        !parse_irreps(irreps_out, c, err))
        return ufail(CGTP_E_IRREPS, err);
    if (a.empty() || b.empty() || c.empty()) return ufail(CGTP_E_IRREPS, "empty irreps");
    const int mul = a[0].mul;
    for (auto& r : a)
        if (r.mul != mul) return ufail(CGTP_E_IRREPS, "'uvw' needs one multiplicity in irreps_in1");
    for (auto& r : b)
        if (r.mul != 1) return ufail(CGTP_E_IRREPS, "irreps_in2 must have multiplicity 1");
    // paths: triangle and parity rule, in1-major, then in2, then out
    std::unique_ptr<cgtp_uvw_s> u(new cgtp_uvw_s);
    u->dtype = dtype;
    std::vector<cgtp_instr> tp;
    std::vector<cgtp_linear_instr> li;
    std::string mid;
    for (int i1 = 0; i1 < (int)a.size(); ++i1)
        for (int i2 = 0; i2 < (int)b.size(); ++i2)
            for (int k = 0; k < (int)c.size(); ++k) {
                const int l1 = a[i1].l, l2 = b[i2].l, l3 = c[k].l;
                if (l3 < std::abs(l1 - l2) || l3 > l1 + l2 || c[k].parity != a[i1].parity * b[i2].parity)
                    continue;
                const int blk = (int)u->paths.size();
                cgtp_instr I{i1, i2, blk, {'u', 'v', 'u', 0}};
                tp.push_back(I);
                li.push_back(cgtp_linear_instr{blk, k});
                if (!mid.empty()) mid += "+";
                mid += std::to_string(mul) + "x" + std::to_string(l3) + (c[k].parity > 0 ? "e" : "o");
                u->paths.push_back({l1, l2, l3, i1, i2, k});
            }
    if (u->paths.empty()) return ufail(CGTP_E_PATH, "no parity-allowed path");
    cgtp_status st = cgtp_plan_create(&u->plan, irreps_in1, irreps_in2, mid.c_str(), tp.data(),
                                      (int)tp.size(), dtype, CGTP_W_SHARED, 0);
    if (st != CGTP_OK) return st;
    st = cgtp_linear_create(&u->lin, mid.c_str(), irreps_out, li.data(), (int)li.size(), dtype);
    if (st != CGTP_OK) {
        cgtp_plan_destroy(u->plan);
        return st;
    }
    int np = 0, nl = 0;
    int64_t dmid2 = 0;
    cgtp_plan_info(u->plan, &u->dim1, &u->dim2, &u->dimmid, &u->wtp, &np);
    cgtp_linear_info(u->lin, &dmid2, &u->dimo, &u->wnumel, &nl);
    for (int j = 0; j < nl; ++j) {
        int ii = 0, io = 0;
        int64_t off = 0;
        cgtp_linear_instruction(u->lin, j, &ii, &io, &off);
        u->woff.push_back(off);
    }
    // the per-path blocks as a row source of the mixing kernel (fused forward):
    // path p's T entries [d3][d1] at t_off of a T row, each with its CG terms
    {
        LinTpDesc& T = u->tp;
        std::vector<int> x1off(a.size()), yoff(b.size());
        int acc = 0;
        for (size_t i = 0; i < a.size(); ++i) x1off[i] = acc, acc += a[i].mul * (2 * a[i].l + 1);
        acc = 0;
        for (size_t i = 0; i < b.size(); ++i) yoff[i] = acc, acc += 2 * b[i].l + 1;
        bool ok = (int)u->paths.size() <= kTpMaxPaths && acc <= 255;
        for (int p = 0; ok && p < (int)u->paths.size(); ++p) {
            const auto& q = u->paths[p];
            const int d1 = 2 * q[0] + 1, d2 = 2 * q[1] + 1, d3 = 2 * q[2] + 1;
            if (T.tdim + d1 * d3 > kTpMaxT) {
                ok = false;
                break;
            }
            std::vector<double> cg((size_t)d1 * d2 * d3);
            cgtp_plan_coefficients(u->plan, p, cg.data());
            T.path[p] = LinTpPath{x1off[q[3]], mul, T.tdim, d1, d3};
            for (int m3 = 0; m3 < d3 && ok; ++m3)
                for (int m1 = 0; m1 < d1 && ok; ++m1) {
                    T.estart[T.tdim++] = (short)T.nterms;
                    for (int m2 = 0; m2 < d2; ++m2) {
                        const double c = cg[((size_t)m1 * d2 + m2) * d3 + m3];
                        if (c == 0.0) continue;
                        if (T.nterms >= kTpMaxTerms) {
                            ok = false;
                            break;
                        }
                        T.term_y[T.nterms] = (unsigned char)(yoff[q[4]] + m2);
                        T.term_c[T.nterms] = (float)c;
                        ++T.nterms;
                    }
                }
        }
        T.estart[T.tdim] = (short)T.nterms;
        T.npaths = (int)u->paths.size();
        u->tp_ok = ok && dtype == CGTP_F32;
    }
    *out = u.release();
    return CGTP_OK;
    UGUARD_END
}

cgtp_status cgtp_uvw_destroy(cgtp_uvw u) {
    if (!u) return CGTP_OK;
    cgtp_plan_destroy(u->plan);
    cgtp_linear_destroy(u->lin);
    delete u;
    return CGTP_OK;
}

cgtp_status cgtp_uvw_info(cgtp_uvw u, int64_t* dim_in1, int64_t* dim_in2, int64_t* dim_out,
                          int64_t* dim_mid, int64_t* weight_numel, int* n_paths) {
    if (!u) return ufail(CGTP_E_ARG, "NULL 'uvw' product");
    if (dim_in1) *dim_in1 = u->dim1;
    if (dim_in2) *dim_in2 = u->dim2;
    if (dim_out) *dim_out = u->dimo;
    if (dim_mid) *dim_mid = u->dimmid;
    if (weight_numel) *weight_numel = u->wnumel;
    if (n_paths) *n_paths = (int)u->paths.size();
    return CGTP_OK;
}

cgtp_status cgtp_uvw_path(cgtp_uvw u, int p, int* l1, int* l2, int* l3, int* i_in1, int* i_in2,
                          int* i_out, int64_t* weight_offset) {
    if (!u) return ufail(CGTP_E_ARG, "NULL 'uvw' product");
    if (p < 0 || p >= (int)u->paths.size()) return ufail(CGTP_E_ARG, "path index out of range");
    const auto& q = u->paths[p];
    int* dst[6] = {l1, l2, l3, i_in1, i_in2, i_out};
    for (int i = 0; i < 6; ++i)
        if (dst[i]) *dst[i] = q[i];
    if (weight_offset) *weight_offset = u->woff[p];
    return CGTP_OK;
}

cgtp_status cgtp_uvw_parts(cgtp_uvw u, cgtp_plan* plan, cgtp_linear* lin) {
    if (!u) return ufail(CGTP_E_ARG, "NULL 'uvw' product");
    if (plan) *plan = u->plan;
    if (lin) *lin = u->lin;
    return CGTP_OK;
}

cgtp_status cgtp_uvw_workspace(cgtp_uvw u, int64_t rows, size_t* fwd_bytes, size_t* bwd_bytes) {
    UGUARD_BEGIN
    if (!u) return ufail(CGTP_E_ARG, "NULL 'uvw' product");
    if (rows < 0) return ufail(CGTP_E_ARG, "negative row count");
    if (fwd_bytes) *fwd_bytes = uvw_layout(*u, rows, false, true).total;
    if (bwd_bytes) *bwd_bytes = uvw_layout(*u, rows, true, true).total;
    return CGTP_OK;
    UGUARD_END
}

// conv: N rows (receivers), graph arguments as cgtp_conv_forward; else B rows.
static cgtp_status uvw_fwd(cgtp_uvw u, bool conv, int64_t rows, int64_t E, const int32_t* rowptr,
                           const int32_t* sender, const void* x, const void* y, const void* W,
                           double scale, void* out, void* mid, void* ws, size_t ws_bytes,
                           cgtp_stream stream) {
    if (!u) return ufail(CGTP_E_ARG, "NULL 'uvw' product");
    if (rows < 0 || E < 0) return ufail(CGTP_E_ARG, "negative size");
    UvwLayout L;
    cgtp_status st = uvw_ws_check(*u, rows, false, mid, ws, ws_bytes, L);
    if (st != CGTP_OK) return st;
    if (!conv && !mid && u->tp_ok) {
        // fused: the mixing kernel computes the per-path blocks where it reads
        // them (no intermediate in HBM)
        if (!x || !y || !W || !out) return ufail(CGTP_E_ARG, "NULL tensor");
        bool used = false;
        // the T rows take the place of the blocks in the workspace (mid region)
        cudaError_t e = launch_linear_forward_tp(
            cgtp_linear_impl(u->lin), u->tp, rows, x, u->dim1, y, u->dim2, W, out, at(ws, L.lin),
            ws_bytes - L.lin, at(ws, L.mid), L.gmid - L.mid,
            reinterpret_cast<cudaStream_t>(stream), &used);
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return ufail(CGTP_E_CUDA, std::string("uvw fused forward: ") + cudaGetErrorString(e));
        }
        if (used) return CGTP_OK;
    }
    void* ones = at(ws, L.ones);
    void* m = mid ? mid : at(ws, L.mid);
    cudaError_t e = launch_fill_ones(u->dtype == CGTP_F64, ones, u->wtp,
                                     reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return ufail(CGTP_E_CUDA, std::string("uvw unit weights: ") + cudaGetErrorString(e));
    }
    st = conv ? cgtp_conv_forward(u->plan, rows, E, rowptr, sender, x, y, ones, scale, m, stream)
              : cgtp_forward(u->plan, rows, x, y, ones, m, stream);
    if (st != CGTP_OK) return st;
    return cgtp_linear_forward(u->lin, rows, m, W, out, at(ws, L.lin),
                               ws_bytes - L.lin, 0, stream);
}

static cgtp_status uvw_bwd(cgtp_uvw u, bool conv, int64_t rows, int64_t E, const int32_t* rowptr,
                           const int32_t* sender, const int32_t* s_rowptr, const int32_t* s_perm,
                           const int32_t* s_recv, const void* x, const void* y, const void* W,
                           double scale, const void* grad_out, const void* mid, void* grad_x,
                           void* grad_y, void* grad_W, void* ws, size_t ws_bytes,
                           cgtp_stream stream) {
    if (!u) return ufail(CGTP_E_ARG, "NULL 'uvw' product");
    if (rows < 0 || E < 0) return ufail(CGTP_E_ARG, "negative size");
    UvwLayout L;
    cgtp_status st = uvw_ws_check(*u, rows, true, mid, ws, ws_bytes, L);
    if (st != CGTP_OK) return st;
    void* ones = at(ws, L.ones);
    cudaError_t e = launch_fill_ones(u->dtype == CGTP_F64, ones, u->wtp,
                                     reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return ufail(CGTP_E_CUDA, std::string("uvw unit weights: ") + cudaGetErrorString(e));
    }
    const void* m = mid;
    if (!m && (grad_W || grad_x || grad_y)) {  // recompute the per-path blocks
        void* mw = at(ws, L.mid);
        st = conv ? cgtp_conv_forward(u->plan, rows, E, rowptr, sender, x, y, ones, scale, mw, stream)
                  : cgtp_forward(u->plan, rows, x, y, ones, mw, stream);
        if (st != CGTP_OK) return st;
        m = mw;
    }
    const bool need_gmid = grad_x || grad_y;
    void* gmid = need_gmid ? at(ws, L.gmid) : nullptr;
    st = cgtp_linear_backward(u->lin, rows, m, W, grad_out, gmid, grad_W, at(ws, L.lin),
                              ws_bytes - L.lin, 0, stream);
    if (st != CGTP_OK || !need_gmid) return st;
    return conv ? cgtp_conv_backward(u->plan, rows, E, rowptr, sender, s_rowptr, s_perm, s_recv, x,
                                     y, ones, scale, gmid, grad_x, grad_y, nullptr, stream)
                : cgtp_backward(u->plan, rows, x, y, ones, gmid, grad_x, grad_y, nullptr, stream);
}

cgtp_status cgtp_uvw_forward(cgtp_uvw u, int64_t B, const void* x, const void* y, const void* W,
                             void* out, void* mid, void* workspace, size_t workspace_bytes,
                             cgtp_stream stream) {
    UGUARD_BEGIN
    return uvw_fwd(u, false, B, 0, nullptr, nullptr, x, y, W, 1.0, out, mid, workspace,
                   workspace_bytes, stream);
    UGUARD_END
}

cgtp_status cgtp_uvw_backward(cgtp_uvw u, int64_t B, const void* x, const void* y, const void* W,
                              const void* grad_out, const void* mid, void* grad_x, void* grad_y,
                              void* grad_W, void* workspace, size_t workspace_bytes,
                              cgtp_stream stream) {
    UGUARD_BEGIN
    return uvw_bwd(u, false, B, 0, nullptr, nullptr, nullptr, nullptr, nullptr, x, y, W, 1.0,
                   grad_out, mid, grad_x, grad_y, grad_W, workspace, workspace_bytes, stream);
    UGUARD_END
}

cgtp_status cgtp_uvw_conv_forward(cgtp_uvw u, int64_t N, int64_t E, const int32_t* rowptr,
                                  const int32_t* sender, const void* x, const void* y,
                                  const void* W, double scale, void* out, void* mid,
                                  void* workspace, size_t workspace_bytes, cgtp_stream stream) {
    UGUARD_BEGIN
    return uvw_fwd(u, true, N, E, rowptr, sender, x, y, W, scale, out, mid, workspace,
                   workspace_bytes, stream);
    UGUARD_END
}

cgtp_status cgtp_uvw_conv_backward(cgtp_uvw u, int64_t N, int64_t E, const int32_t* rowptr,
                                   const int32_t* sender, const int32_t* s_rowptr,
                                   const int32_t* s_perm, const int32_t* s_recv, const void* x,
                                   const void* y, const void* W, double scale,
                                   const void* grad_out, const void* mid, void* grad_x,
                                   void* grad_y, void* grad_W, void* workspace,
                                   size_t workspace_bytes, cgtp_stream stream) {
    UGUARD_BEGIN
    return uvw_bwd(u, true, N, E, rowptr, sender, s_rowptr, s_perm, s_recv, x, y, W, scale,
                   grad_out, mid, grad_x, grad_y, grad_W, workspace, workspace_bytes, stream);
    UGUARD_END
}

}  // extern "C"
