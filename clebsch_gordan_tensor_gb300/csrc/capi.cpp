// extern "C" entry points of the CG tensor-product library (declared in cgtp.h).
//
// Every call validates its arguments on the host, then launches kernels on the
// caller's stream.  Nothing here allocates device memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <climits>
#include <cstring>
#include <new>
#include <string>

#include "cgtp.h"
#include "internal.hpp"

struct cgtp_plan_s {
    cgtp::Plan p;
};

struct cgtp_linear_s {
    cgtp::LinearImpl* L;
};

namespace cgtp {

static thread_local int t_cuda_err = 0;
static thread_local std::string t_msg;
static std::atomic<int64_t> g_launches{0};

void set_cuda_error(cudaError_t e) { t_cuda_err = (int)e; }
void set_error_message(const std::string& m) { t_msg = m; }
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static cgtp_status fail(cgtp_status s, const std::string& m) {
    t_msg = m;
    return s;
}

static cgtp_status cuda_fail(cudaError_t e, const char* what) {
    t_cuda_err = (int)e;
    t_msg = std::string(what) + ": " + cudaGetErrorString(e);
    return CGTP_E_CUDA;
}

static bool aligned(const void* p, size_t a) { return p == nullptr || ((uintptr_t)p % a) == 0; }

// Alignment the plan's kernels need for feature, weight and gradient rows.
static size_t row_align(const Plan& p) {
    return p.dtype == CGTP_F64 ? 8 : (p.cpt == 2 ? 8 : 4);
}

// Weight rows: bfloat16 pairs are read as one 32-bit word per lane.
static size_t w_align(const Plan& p) {
    return p.w16() ? (p.cpt == 2 ? 4 : 2) : row_align(p);
}

static cgtp_status check_w(const Plan& p, const void* w) {
    if (!aligned(w, w_align(p)))
        return fail(CGTP_E_ARG, "weight pointer not aligned to " + std::to_string(w_align(p)) + " bytes");
    return CGTP_OK;
}

static cgtp_status check_rows(const Plan& p, std::initializer_list<const void*> ptrs) {
    const size_t a = row_align(p);
    for (const void* q : ptrs)
        if (!aligned(q, a))
            return fail(CGTP_E_ARG, "tensor pointer not aligned to " + std::to_string(a) + " bytes");
    return CGTP_OK;
}

static cgtp_status launch_tp(Plan& p, const char* name, int64_t n_items, void** args,
                             cudaStream_t s, bool staged = false, size_t smem = 0,
                             int threads = 0, int64_t max_rows = 0, int64_t* rows_used = nullptr) {
    if (n_items <= 0) return CGTP_OK;
    std::shared_ptr<Module> m;
    std::string err;
    cgtp_status st = get_module(p, true, m, err);
    if (st != CGTP_OK) return fail(st, err);
    cudaKernel_t k = m->kernels[name];
    if (!k) return fail(CGTP_E_ARG, std::string("kernel not in module: ") + name);
    cudaError_t e;
    if (!staged) {
        int64_t blocks = (n_items + p.slots - 1) / p.slots;
        if (blocks > INT_MAX) blocks = INT_MAX;
        if (max_rows > 0) {
            // each CTA writes p.slots partial rows: the scratch must hold one CTA's
            if (max_rows < p.slots)
                return fail(CGTP_E_ARG, "scratch holds " + std::to_string(max_rows) +
                                            " partial weight rows, fewer than the " +
                                            std::to_string(p.slots) + " one CTA writes");
            blocks = std::min<int64_t>(blocks, max_rows / p.slots);
        }
        if (rows_used) *rows_used = blocks * p.slots;
        e = cudaLaunchKernel((const void*)k, dim3((unsigned)blocks), dim3(p.block), args, 0, s);
    } else {
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
        int per_sm = 0, sms = 0;
        {
            std::lock_guard<std::mutex> g(p.mu);
            if (!m->smem_set.count(dev)) {
                const size_t need = std::max(p.fwd_smem, p.bwd_smem);
                e = cudaKernelSetAttributeForDevice(m->kernels["cgtp_fwd_conv_tma"],
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    (int)need, dev);
                for (const char* kn : {"cgtp_fwd_single_tma", "cgtp_bwd_conv_tma",
                                       "cgtp_bwd_conv_nogy_tma", "cgtp_bwd_single_tma",
                                       "cgtp_bwd_single_nogy_tma"})
                    if (e == cudaSuccess)
                        e = cudaKernelSetAttributeForDevice(
                            m->kernels[kn], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)need,
                            dev);
                if (e != cudaSuccess) return cuda_fail(e, "set max dynamic shared memory");
                m->smem_set[dev] = 1;
            }
            auto key = std::make_pair(dev, std::string(name));
            auto it = m->ctas_per_sm.find(key);
            if (it == m->ctas_per_sm.end()) {
                int n = 0;
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, (const void*)k, threads,
                                                                  smem) != cudaSuccess || n < 1) {
                    cudaGetLastError();
                    n = std::max(1, (int)((220 * 1024) / (smem + 4096)));
                }
                m->ctas_per_sm[key] = n;
                per_sm = n;
            } else {
                per_sm = it->second;
            }
        }
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        int64_t grid = std::min<int64_t>(n_items, (int64_t)sms * per_sm);
        if (max_rows > 0) grid = std::max<int64_t>(1, std::min<int64_t>(grid, max_rows));
        if (rows_used) *rows_used = grid;
        e = cudaLaunchKernel((const void*)k, dim3((unsigned)grid), dim3(threads), args, smem, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, name);
    count_launch();
    {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) {
            std::lock_guard<std::mutex> g(p.mu);
            m->launched_on.insert(dev);
        }
    }
    return CGTP_OK;
}

static bool a16(std::initializer_list<const void*> ptrs) {
    for (const void* q : ptrs)
        if (q && ((uintptr_t)q % 16) != 0) return false;
    return true;
}

// One forward-shaped launch: out (=|+=) scale * sum TP(a, b, c).
static cgtp_status fwd_launch(Plan& p, bool conv, int64_t n_items, const int32_t* rowptr,
                              const int32_t* sender, const void* a, const void* b, const void* c,
                              double scale, void* out, int accumulate, cudaStream_t s) {
    long long n = n_items;
    long long ws = p.wmode == CGTP_W_SHARED ? 0 : p.wdim;
    float sf = (float)scale;
    double sd = scale;
    void* sp = p.dtype == CGTP_F64 ? (void*)&sd : (void*)&sf;
    const bool staged = p.staged && a16({a, b, c, out});
    if (conv) {
        void* args[] = {&n, &rowptr, &sender, &a, &b, &c, &ws, &out, sp, &accumulate};
        return launch_tp(p, staged ? "cgtp_fwd_conv_tma" : "cgtp_fwd_conv", n_items, args, s,
                         staged, p.fwd_smem, (int)p.fwd_groups.size() * p.lanes);
    }
    void* args[] = {&n, &a, &b, &c, &ws, &out, sp, &accumulate};
    return launch_tp(p, staged ? "cgtp_fwd_single_tma" : "cgtp_fwd_single", n_items, args, s,
                     staged, p.fwd_smem, (int)p.fwd_groups.size() * p.lanes);
}

// One backward-shaped launch over items (senders or samples).
static cgtp_status bwd_launch(Plan& p, bool conv, int64_t n_items, const int32_t* s_rowptr,
                              const int32_t* s_perm, const int32_t* s_recv, const void* x,
                              const void* y, const void* w, const void* g, double scale, void* gx,
                              void* gy, void* gw, int mgx, int mgy, int mgw, cudaStream_t s,
                              void* wsp = nullptr, int64_t ws_rows = 0,
                              int64_t* rows_out = nullptr) {
    if (!mgx && !mgy && !mgw) return CGTP_OK;
    long long n = n_items;
    long long ws = p.wmode == CGTP_W_SHARED ? 0 : p.wdim;
    float sf = (float)scale;
    double sd = scale;
    void* sp = p.dtype == CGTP_F64 ? (void*)&sd : (void*)&sf;
    const bool shared = p.wmode == CGTP_W_SHARED && mgw;
    void* part = shared ? wsp : nullptr;
    void* args[] = {&n, &s_rowptr, &s_perm, &s_recv, &x, &y, &w, &ws, &g, sp,
                    &gx, &gy, &gw, &mgx, &mgy, &mgw, &part};
    const bool staged = p.staged && a16({x, y, w, g});
    std::string name = conv ? (mgy ? "cgtp_bwd_conv" : "cgtp_bwd_conv_nogy")
                            : (mgy ? "cgtp_bwd_single" : "cgtp_bwd_single_nogy");
    if (staged) name += "_tma";
    int64_t rows = 0;
    cgtp_status st = launch_tp(p, name.c_str(), n_items, args, s, staged, p.bwd_smem,
                               p.bwd_threads(), shared ? ws_rows : 0, &rows);
    if (st != CGTP_OK || !shared) return st;
    if (rows_out) {  // the caller adds these partial rows up with others
        *rows_out = rows;
        return CGTP_OK;
    }
    // ordered sum of the per-CTA partial rows into grad_w
    cudaError_t e = launch_reduce_rows(p.dtype == CGTP_F64, wsp, rows, p.wdim, gw, s);
    if (e != cudaSuccess) return cuda_fail(e, "weight-gradient reduction");
    return CGTP_OK;
}

static size_t esize(const Plan& p) { return p.dtype == CGTP_F64 ? 8 : 4; }

static cgtp_status zero(void* ptr, int64_t bytes, cudaStream_t s) {
    if (!ptr || bytes <= 0) return CGTP_OK;
    cudaError_t e = launch_fill_zero(ptr, bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "fill_zero");
    return CGTP_OK;
}

// Shared body of the standalone and convolution double backward.
static cgtp_status double_backward(Plan& p, bool conv, int64_t n_x, int64_t n_e,
                                   int64_t n_out, const int32_t* rowptr, const int32_t* sender,
                                   const int32_t* s_rowptr, const int32_t* s_perm,
                                   const int32_t* s_recv, const void* x, const void* y,
                                   const void* w, double scale, const void* g, const void* ggx,
                                   const void* ggy, const void* ggw, void* dx, void* dy, void* dw,
                                   void* dg, cudaStream_t s, void* wsp = nullptr,
                                   size_t wsb = 0) {
    cgtp_status st;
    // shared weight row: both d_w terms leave per-CTA partial rows side by side
    // in the workspace, added up in one ordered reduction at the end
    const bool shw = p.wmode == CGTP_W_SHARED && dw;
    const int64_t es = esize(p);
    const size_t part_bytes = (size_t)kSharedWRows * (size_t)p.wdim * (size_t)es;
    if (shw && (!wsp || wsb < 2 * part_bytes || !aligned(wsp, 16)))
        return fail(CGTP_E_ARG, "d_w of a shared weight row needs a 16-byte aligned workspace of " +
                                    std::to_string(2 * part_bytes) +
                                    " bytes (twice cgtp_weight_grad_workspace): use the _ws entry");
    int64_t rows_total = 0;
    auto part_at = [&]() { return (void*)((char*)wsp + rows_total * p.wdim * es); };
    if (dg) {
        int acc = 0;
        const void* terms[3][3] = {{ggx, y, w}, {x, ggy, w}, {x, y, ggw}};
        const bool live[3] = {ggx != nullptr, ggy != nullptr, ggw != nullptr};
        for (int t = 0; t < 3; ++t) {
            if (!live[t]) continue;
            st = fwd_launch(p, conv, n_out, rowptr, sender, terms[t][0], terms[t][1], terms[t][2],
                            scale, dg, acc, s);
            if (st != CGTP_OK) return st;
            acc = 1;
        }
        if (!acc && (st = zero(dg, n_out * p.dimo * (int64_t)esize(p), s)) != CGTP_OK) return st;
    }
    int wx = 0, wy = 0, ww = 0;  // already written?
    auto mode = [](void* out, int& written) {
        if (!out) return 0;
        const int m = written ? 2 : 1;
        written = 1;
        return m;
    };
    if (ggy) {  // f_x(g; ggy, w) -> dx, f_w(g; x, ggy) -> dw
        const int mx = mode(dx, wx), mw = mode(dw, ww);
        int64_t rows = 0;
        st = bwd_launch(p, conv, n_x, s_rowptr, s_perm, s_recv, x, ggy, w, g, scale, dx, nullptr,
                        dw, mx, 0, mw, s, shw ? part_at() : nullptr, kSharedWRows,
                        shw ? &rows : nullptr);
        if (st != CGTP_OK) return st;
        rows_total += rows;
    }
    if (ggw) {  // f_x(g; y, ggw) -> dx, f_y(g; x, ggw) -> dy
        const int mx = mode(dx, wx), my = mode(dy, wy);
        st = bwd_launch(p, conv, n_x, s_rowptr, s_perm, s_recv, x, y, ggw, g, scale, dx, dy,
                        nullptr, mx, my, 0, s);
        if (st != CGTP_OK) return st;
    }
    if (ggx) {  // f_y(g; ggx, w) -> dy, f_w(g; ggx, y) -> dw
        const int my = mode(dy, wy), mw = mode(dw, ww);
        int64_t rows = 0;
        st = bwd_launch(p, conv, n_x, s_rowptr, s_perm, s_recv, ggx, y, w, g, scale, nullptr, dy,
                        dw, 0, my, mw, s, shw ? part_at() : nullptr, kSharedWRows,
                        shw ? &rows : nullptr);
        if (st != CGTP_OK) return st;
        rows_total += rows;
    }
    if (shw && rows_total > 0) {
        cudaError_t e = launch_reduce_rows(p.dtype == CGTP_F64, wsp, rows_total, p.wdim, dw, s);
        if (e != cudaSuccess) return cuda_fail(e, "weight-gradient reduction");
    }
    if (dx && !wx && (st = zero(dx, n_x * p.dimx * es, s)) != CGTP_OK) return st;
    if (dy && !wy && (st = zero(dy, n_e * p.dimy * es, s)) != CGTP_OK) return st;
    if (dw && (shw ? rows_total == 0 : !ww) &&
        (st = zero(dw, (shw ? 1 : n_e) * p.wdim * es, s)) != CGTP_OK)
        return st;
    return CGTP_OK;
}

}  // namespace cgtp

using namespace cgtp;

#define GUARD_BEGIN try {
#define GUARD_END                                                  \
    }                                                              \
    catch (const std::bad_alloc&) {                                \
        return fail(CGTP_E_NOMEM, "host allocation failed");       \
    }                                                              \
    catch (...) {                                                  \
        return fail(CGTP_E_ARG, "unexpected internal exception");  \
    }

static inline cudaStream_t S(cgtp_stream s) { return reinterpret_cast<cudaStream_t>(s); }

extern "C" {

cgtp_status cgtp_plan_create(cgtp_plan* out, const char* irreps_in1, const char* irreps_in2,
                             const char* irreps_out, const cgtp_instr* instr, int n_instr,
                             cgtp_dtype dtype, cgtp_wmode wmode, unsigned flags) {
    GUARD_BEGIN
    if (!out) return fail(CGTP_E_ARG, "out is NULL");
    *out = nullptr;
    if (dtype != CGTP_F32 && dtype != CGTP_F64) return fail(CGTP_E_ARG, "bad dtype");
    if (wmode != CGTP_W_PER_EDGE && wmode != CGTP_W_SHARED) return fail(CGTP_E_ARG, "bad wmode");
    const bool w_bf16 = (flags & CGTP_PLAN_WEIGHTS_BF16) != 0;
    const bool w_f16 = (flags & CGTP_PLAN_WEIGHTS_F16) != 0;
    if (w_bf16 && w_f16) return fail(CGTP_E_ARG, "both 16-bit weight formats requested");
    if ((w_bf16 || w_f16) && dtype != CGTP_F32)
        return fail(CGTP_E_UNSUPPORTED, "16-bit weights need an fp32 plan");
    auto* h = new cgtp_plan_s();
    h->p.dtype = dtype;
    h->p.wmode = wmode;
    h->p.flags = flags;
    h->p.w_bf16 = w_bf16;
    h->p.w_f16 = w_f16;
    std::string err;
    cgtp_status st = build_plan(h->p, irreps_in1, irreps_in2, irreps_out, instr, n_instr, err);
    if (st != CGTP_OK) {
        delete h;
        return fail(st, err);
    }
    *out = h;
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_plan_destroy(cgtp_plan plan) {
    GUARD_BEGIN
    delete plan;
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_plan_info(cgtp_plan plan, int64_t* dim_in1, int64_t* dim_in2, int64_t* dim_out,
                           int64_t* weight_numel, int* n_paths) {
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    const Plan& p = plan->p;
    if (dim_in1) *dim_in1 = p.dimx;
    if (dim_in2) *dim_in2 = p.dimy;
    if (dim_out) *dim_out = p.dimo;
    if (weight_numel) *weight_numel = p.wdim;
    if (n_paths) *n_paths = (int)p.paths.size();
    return CGTP_OK;
}

cgtp_status cgtp_plan_path(cgtp_plan plan, int q, int* l1, int* l2, int* l3, int* i1, int* i2,
                           int* i3) {
    if (!plan || q < 0 || q >= (int)plan->p.paths.size()) return fail(CGTP_E_ARG, "bad path");
    const Path& P = plan->p.paths[q];
    if (l1) *l1 = P.l1;
    if (l2) *l2 = P.l2;
    if (l3) *l3 = P.l3;
    if (i1) *i1 = P.i1;
    if (i2) *i2 = P.i2;
    if (i3) *i3 = P.i3;
    return CGTP_OK;
}

cgtp_status cgtp_plan_coefficients(cgtp_plan plan, int q, double* out) {
    if (!plan || !out || q < 0 || q >= (int)plan->p.paths.size())
        return fail(CGTP_E_ARG, "bad path or NULL out");
    const auto& c = plan->p.paths[q].cg;
    memcpy(out, c.data(), c.size() * sizeof(double));
    return CGTP_OK;
}

cgtp_status cgtp_plan_compile(cgtp_plan plan, char* log, size_t cap) {
    GUARD_BEGIN
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    std::shared_ptr<Module> m;
    std::string err;
    cgtp_status st = get_module(plan->p, false, m, err);
    if (st != CGTP_OK) return fail(st, err);
    if (log && cap) {
        strncpy(log, m->log.c_str(), cap - 1);
        log[cap - 1] = 0;
    }
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_plan_source(cgtp_plan plan, char* buf, size_t cap, size_t* needed) {
    GUARD_BEGIN
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    const std::string src = plan->p.kernel_source();
    if (needed) *needed = src.size() + 1;
    if (buf && cap) {
        strncpy(buf, src.c_str(), cap - 1);
        buf[cap - 1] = 0;
    }
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_plan_device_status(cgtp_plan plan, int* code) {
    GUARD_BEGIN
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    if (code) *code = 0;
    std::shared_ptr<Module> m;
    {
        std::lock_guard<std::mutex> g(plan->p.mu);
        auto it = plan->p.modules.find("tp");
        if (it == plan->p.modules.end() || !it->second->lib || !it->second->err_flag) return CGTP_OK;
        m = it->second;
    }
    int v = 0;
    cudaError_t e = cudaMemcpy(&v, m->err_flag, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device error flag");
    if (code) *code = v;
    if (v) {
        const int zero = 0;
        cudaMemcpy(m->err_flag, &zero, sizeof(int), cudaMemcpyHostToDevice);
        return fail(CGTP_E_DEVICE, "a kernel timed out waiting for a bulk copy (code " +
                                       std::to_string(v) + ")");
    }
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_weight_grad_workspace(cgtp_plan plan, size_t* bytes) {
    if (!plan || !bytes) return fail(CGTP_E_ARG, "NULL argument");
    const Plan& p = plan->p;
    *bytes = p.wmode == CGTP_W_SHARED
                 ? (size_t)kSharedWRows * (size_t)p.wdim * (p.dtype == CGTP_F64 ? 8 : 4)
                 : 0;
    return CGTP_OK;
}

static cgtp_status check_ws(const Plan& p, const void* grad_w, const void* ws, size_t bytes) {
    if (p.wmode != CGTP_W_SHARED || !grad_w) return CGTP_OK;
    const size_t need = (size_t)kSharedWRows * (size_t)p.wdim * (p.dtype == CGTP_F64 ? 8 : 4);
    if (!ws || bytes < need)
        return fail(CGTP_E_ARG, "shared-weight gradient needs a workspace of " +
                                    std::to_string(need) + " bytes (cgtp_weight_grad_workspace)");
    if (!aligned(ws, 16)) return fail(CGTP_E_ARG, "workspace not 16-byte aligned");
    return CGTP_OK;
}

cgtp_status cgtp_forward(cgtp_plan plan, int64_t B, const void* x, const void* y, const void* w,
                         void* out, cgtp_stream stream) {
    GUARD_BEGIN
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    if (B < 0) return fail(CGTP_E_ARG, "B < 0");
    if (B == 0) return CGTP_OK;
    if (!x || !y || !w || !out) return fail(CGTP_E_ARG, "NULL tensor");
    Plan& p = plan->p;
    cgtp_status st = check_rows(p, {x, out});
    if (st != CGTP_OK) return st;
    if ((st = check_w(p, w)) != CGTP_OK) return st;
    return fwd_launch(p, false, B, nullptr, nullptr, x, y, w, 1.0, out, 0, S(stream));
    GUARD_END
}

cgtp_status cgtp_backward(cgtp_plan plan, int64_t B, const void* x, const void* y, const void* w,
                          const void* grad_out, void* grad_x, void* grad_y, void* grad_w,
                          cgtp_stream stream) {
    GUARD_BEGIN
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    if (B < 0) return fail(CGTP_E_ARG, "B < 0");
    if (B == 0) return CGTP_OK;
    if (!x || !y || !w || !grad_out) return fail(CGTP_E_ARG, "NULL input tensor");
    Plan& p = plan->p;
    if (p.wmode == CGTP_W_SHARED && grad_w)
        return fail(CGTP_E_ARG, "shared-weight gradient needs a workspace: use cgtp_backward_ws");
    cgtp_status st = check_rows(p, {x, grad_out, grad_x, grad_w});
    if (st != CGTP_OK) return st;
    if ((st = check_w(p, w)) != CGTP_OK) return st;
    return bwd_launch(p, false, B, nullptr, nullptr, nullptr, x, y, w, grad_out, 1.0, grad_x,
                      grad_y, grad_w, grad_x ? 1 : 0, grad_y ? 1 : 0, grad_w ? 1 : 0, S(stream));
    GUARD_END
}

cgtp_status cgtp_backward_ws(cgtp_plan plan, int64_t B, const void* x, const void* y,
                             const void* w, const void* grad_out, void* grad_x, void* grad_y,
                             void* grad_w, void* workspace, size_t workspace_bytes,
                             cgtp_stream stream) {
    GUARD_BEGIN
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    if (B < 0) return fail(CGTP_E_ARG, "B < 0");
    Plan& p = plan->p;
    cgtp_status st = check_ws(p, grad_w, workspace, workspace_bytes);
    if (st != CGTP_OK) return st;
    if (B == 0) {
        if (p.wmode == CGTP_W_SHARED && grad_w) return zero(grad_w, p.wdim * (int64_t)esize(p), S(stream));
        return CGTP_OK;
    }
    if (!x || !y || !w || !grad_out) return fail(CGTP_E_ARG, "NULL input tensor");
    if ((st = check_rows(p, {x, grad_out, grad_x, grad_w})) != CGTP_OK) return st;
    if ((st = check_w(p, w)) != CGTP_OK) return st;
    return bwd_launch(p, false, B, nullptr, nullptr, nullptr, x, y, w, grad_out, 1.0, grad_x,
                      grad_y, grad_w, grad_x ? 1 : 0, grad_y ? 1 : 0, grad_w ? 1 : 0, S(stream),
                      workspace, kSharedWRows);
    GUARD_END
}

cgtp_status cgtp_double_backward(cgtp_plan plan, int64_t B, const void* x, const void* y,
                                 const void* w, const void* grad_out, const void* gg_x,
                                 const void* gg_y, const void* gg_w, void* d_x, void* d_y,
                                 void* d_w, void* d_grad_out, cgtp_stream stream) {
    return cgtp_double_backward_ws(plan, B, x, y, w, grad_out, gg_x, gg_y, gg_w, d_x, d_y, d_w,
                                   d_grad_out, nullptr, 0, stream);
}

cgtp_status cgtp_double_backward_ws(cgtp_plan plan, int64_t B, const void* x, const void* y,
                                    const void* w, const void* grad_out, const void* gg_x,
                                    const void* gg_y, const void* gg_w, void* d_x, void* d_y,
                                    void* d_w, void* d_grad_out, void* workspace,
                                    size_t workspace_bytes, cgtp_stream stream) {
    GUARD_BEGIN
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    if (B < 0) return fail(CGTP_E_ARG, "B < 0");
    if (B == 0) {  // no rows: a shared weight row's d_w is zero
        Plan& p0 = plan->p;
        if (p0.wmode == CGTP_W_SHARED && d_w) return zero(d_w, p0.wdim * (int64_t)esize(p0), S(stream));
        return CGTP_OK;
    }
    if (!x || !y || !w || !grad_out) return fail(CGTP_E_ARG, "NULL input tensor");
    Plan& p = plan->p;
    if (p.w16()) return fail(CGTP_E_UNSUPPORTED, "double backward of a 16-bit-weight plan");
    cgtp_status st = check_rows(p, {x, grad_out, gg_x, gg_w, d_x, d_w, d_grad_out});
    if (st != CGTP_OK) return st;
    if ((st = check_w(p, w)) != CGTP_OK) return st;
    return double_backward(p, false, B, B, B, nullptr, nullptr, nullptr, nullptr, nullptr, x, y,
                           w, 1.0, grad_out, gg_x, gg_y, gg_w, d_x, d_y, d_w, d_grad_out,
                           S(stream), workspace, workspace_bytes);
    GUARD_END
}

static cgtp_status check_graph(int64_t N, int64_t E, const void* a, const void* b) {
    if (N < 0 || E < 0) return fail(CGTP_E_GRAPH, "negative graph size");
    if (N >= INT_MAX || E >= INT_MAX) return fail(CGTP_E_GRAPH, "graph too large for int32 CSR");
    if (N > 0 && !a) return fail(CGTP_E_GRAPH, "NULL CSR row pointer");
    if (E > 0 && !b) return fail(CGTP_E_GRAPH, "NULL CSR index array");
    return CGTP_OK;
}

cgtp_status cgtp_conv_forward(cgtp_plan plan, int64_t N, int64_t E, const int32_t* rowptr,
                              const int32_t* sender, const void* x, const void* y, const void* w,
                              double scale, void* out, cgtp_stream stream) {
    GUARD_BEGIN
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    cgtp_status st = check_graph(N, E, rowptr, sender);
    if (st != CGTP_OK) return st;
    if (N == 0) return CGTP_OK;
    if (!out || (E > 0 && (!x || !y || !w))) return fail(CGTP_E_ARG, "NULL tensor");
    Plan& p = plan->p;
    if ((st = check_rows(p, {x, out})) != CGTP_OK) return st;
    if ((st = check_w(p, w)) != CGTP_OK) return st;
    return fwd_launch(p, true, N, rowptr, sender, x, y, w, scale, out, 0, S(stream));
    GUARD_END
}

cgtp_status cgtp_conv_backward(cgtp_plan plan, int64_t N, int64_t E, const int32_t* rowptr,
                               const int32_t* sender, const int32_t* s_rowptr,
                               const int32_t* s_perm, const int32_t* s_recv, const void* x,
                               const void* y, const void* w, double scale, const void* grad_out,
                               void* grad_x, void* grad_y, void* grad_w, cgtp_stream stream) {
    GUARD_BEGIN
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    cgtp_status st = check_graph(N, E, s_rowptr, s_perm);
    if (st != CGTP_OK) return st;
    if (E > 0 && !s_recv) return fail(CGTP_E_GRAPH, "NULL s_recv");
    (void)rowptr;
    (void)sender;
    if (N == 0) return CGTP_OK;
    Plan& p = plan->p;
    if (p.wmode == CGTP_W_SHARED && grad_w)
        return fail(CGTP_E_ARG, "shared-weight gradient needs a workspace: use cgtp_conv_backward_ws");
    if (!x || !grad_out || (E > 0 && (!y || !w))) return fail(CGTP_E_ARG, "NULL input tensor");
    if ((st = check_rows(p, {x, grad_out, grad_x, grad_w})) != CGTP_OK) return st;
    if ((st = check_w(p, w)) != CGTP_OK) return st;
    return bwd_launch(p, true, N, s_rowptr, s_perm, s_recv, x, y, w, grad_out, scale, grad_x,
                      grad_y, grad_w, grad_x ? 1 : 0, grad_y ? 1 : 0, grad_w ? 1 : 0, S(stream));
    GUARD_END
}

cgtp_status cgtp_conv_backward_ws(cgtp_plan plan, int64_t N, int64_t E, const int32_t* rowptr,
                                  const int32_t* sender, const int32_t* s_rowptr,
                                  const int32_t* s_perm, const int32_t* s_recv, const void* x,
                                  const void* y, const void* w, double scale,
                                  const void* grad_out, void* grad_x, void* grad_y, void* grad_w,
                                  void* workspace, size_t workspace_bytes, cgtp_stream stream) {
    GUARD_BEGIN
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    cgtp_status st = check_graph(N, E, s_rowptr, s_perm);
    if (st != CGTP_OK) return st;
    if (E > 0 && !s_recv) return fail(CGTP_E_GRAPH, "NULL s_recv");
    (void)rowptr;
    (void)sender;
    Plan& p = plan->p;
    if ((st = check_ws(p, grad_w, workspace, workspace_bytes)) != CGTP_OK) return st;
    if (N == 0) {
        if (p.wmode == CGTP_W_SHARED && grad_w) return zero(grad_w, p.wdim * (int64_t)esize(p), S(stream));
        return CGTP_OK;
    }
    if (!x || !grad_out || (E > 0 && (!y || !w))) return fail(CGTP_E_ARG, "NULL input tensor");
    if ((st = check_rows(p, {x, grad_out, grad_x, grad_w})) != CGTP_OK) return st;
    if ((st = check_w(p, w)) != CGTP_OK) return st;
    return bwd_launch(p, true, N, s_rowptr, s_perm, s_recv, x, y, w, grad_out, scale, grad_x,
                      grad_y, grad_w, grad_x ? 1 : 0, grad_y ? 1 : 0, grad_w ? 1 : 0, S(stream),
                      workspace, kSharedWRows);
    GUARD_END
}

cgtp_status cgtp_conv_double_backward(cgtp_plan plan, int64_t N, int64_t E, const int32_t* rowptr,
                                      const int32_t* sender, const int32_t* s_rowptr,
                                      const int32_t* s_perm, const int32_t* s_recv, const void* x,
                                      const void* y, const void* w, double scale,
                                      const void* grad_out, const void* gg_x, const void* gg_y,
                                      const void* gg_w, void* d_x, void* d_y, void* d_w,
                                      void* d_grad_out, cgtp_stream stream) {
    return cgtp_conv_double_backward_ws(plan, N, E, rowptr, sender, s_rowptr, s_perm, s_recv, x,
                                        y, w, scale, grad_out, gg_x, gg_y, gg_w, d_x, d_y, d_w,
                                        d_grad_out, nullptr, 0, stream);
}

cgtp_status cgtp_conv_double_backward_ws(cgtp_plan plan, int64_t N, int64_t E,
                                         const int32_t* rowptr, const int32_t* sender,
                                         const int32_t* s_rowptr, const int32_t* s_perm,
                                         const int32_t* s_recv, const void* x, const void* y,
                                         const void* w, double scale, const void* grad_out,
                                         const void* gg_x, const void* gg_y, const void* gg_w,
                                         void* d_x, void* d_y, void* d_w, void* d_grad_out,
                                         void* workspace, size_t workspace_bytes,
                                         cgtp_stream stream) {
    GUARD_BEGIN
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    cgtp_status st = check_graph(N, E, rowptr, sender);
    if (st != CGTP_OK) return st;
    if ((st = check_graph(N, E, s_rowptr, s_perm)) != CGTP_OK) return st;
    if (E > 0 && !s_recv) return fail(CGTP_E_GRAPH, "NULL s_recv");
    if (N == 0) return CGTP_OK;
    if (!x || !grad_out || (E > 0 && (!y || !w))) return fail(CGTP_E_ARG, "NULL input tensor");
    Plan& p = plan->p;
    if (p.w16()) return fail(CGTP_E_UNSUPPORTED, "double backward of a 16-bit-weight plan");
    if ((st = check_rows(p, {x, grad_out, gg_x, gg_w, d_x, d_w, d_grad_out})) != CGTP_OK)
        return st;
    if ((st = check_w(p, w)) != CGTP_OK) return st;
    return double_backward(p, true, N, E, N, rowptr, sender, s_rowptr, s_perm, s_recv, x, y, w,
                           scale, grad_out, gg_x, gg_y, gg_w, d_x, d_y, d_w, d_grad_out,
                           S(stream), workspace, workspace_bytes);
    GUARD_END
}

static cgtp_status sh_check(int lmax, cgtp_dtype dt, int64_t E) {
    if (lmax < 0 || lmax > 6) return fail(CGTP_E_UNSUPPORTED, "lmax must be 0..6");
    if (dt != CGTP_F32 && dt != CGTP_F64) return fail(CGTP_E_ARG, "bad dtype");
    if (E < 0) return fail(CGTP_E_ARG, "E < 0");
    return CGTP_OK;
}

cgtp_status cgtp_sh_forward(int lmax, cgtp_dtype dtype, int64_t E, const void* vec, void* y,
                            cgtp_stream stream) {
    GUARD_BEGIN
    cgtp_status st = sh_check(lmax, dtype, E);
    if (st != CGTP_OK || E == 0) return st;
    if (!vec || !y) return fail(CGTP_E_ARG, "NULL tensor");
    cudaError_t e = launch_sh_forward(lmax, dtype == CGTP_F64, E, vec, y, S(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sh_forward");
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_sh_backward(int lmax, cgtp_dtype dtype, int64_t E, const void* vec,
                             const void* grad_y, void* grad_vec, cgtp_stream stream) {
    GUARD_BEGIN
    cgtp_status st = sh_check(lmax, dtype, E);
    if (st != CGTP_OK || E == 0) return st;
    if (!vec || !grad_y || !grad_vec) return fail(CGTP_E_ARG, "NULL tensor");
    cudaError_t e = launch_sh_backward(lmax, dtype == CGTP_F64, E, vec, grad_y, grad_vec, S(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sh_backward");
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_sh_jvp(int lmax, cgtp_dtype dtype, int64_t E, const void* vec,
                        const void* tangent_vec, void* tangent_y, cgtp_stream stream) {
    GUARD_BEGIN
    cgtp_status st = sh_check(lmax, dtype, E);
    if (st != CGTP_OK || E == 0) return st;
    if (!vec || !tangent_vec || !tangent_y) return fail(CGTP_E_ARG, "NULL tensor");
    cudaError_t e = launch_sh_jvp(lmax, dtype == CGTP_F64, E, vec, tangent_vec, tangent_y, S(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sh_jvp");
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_sh_hvp(int lmax, cgtp_dtype dtype, int64_t E, const void* vec,
                        const void* grad_y, const void* tangent_vec, void* out,
                        cgtp_stream stream) {
    GUARD_BEGIN
    cgtp_status st = sh_check(lmax, dtype, E);
    if (st != CGTP_OK || E == 0) return st;
    if (!vec || !grad_y || !tangent_vec || !out) return fail(CGTP_E_ARG, "NULL tensor");
    cudaError_t e =
        launch_sh_hvp(lmax, dtype == CGTP_F64, E, vec, grad_y, tangent_vec, out, S(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sh_hvp");
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_linear_create(cgtp_linear* out, const char* irreps_in, const char* irreps_out,
                               const cgtp_linear_instr* instr, int n_instr, cgtp_dtype dtype) {
    GUARD_BEGIN
    if (!out) return fail(CGTP_E_ARG, "NULL output handle");
    *out = nullptr;
    if (dtype != CGTP_F32 && dtype != CGTP_F64) return fail(CGTP_E_ARG, "bad dtype");
    LinearImpl* L = nullptr;
    std::string err;
    cgtp_status st = linear_create(irreps_in, irreps_out, instr, n_instr, dtype, &L, err);
    if (st != CGTP_OK) return fail(st, err);
    *out = new cgtp_linear_s{L};
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_linear_destroy(cgtp_linear lin) {
    GUARD_BEGIN
    if (!lin) return CGTP_OK;
    linear_destroy(lin->L);
    delete lin;
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_linear_info(cgtp_linear lin, int64_t* dim_in, int64_t* dim_out,
                             int64_t* weight_numel, int* n_instr) {
    GUARD_BEGIN
    if (!lin) return fail(CGTP_E_ARG, "NULL linear layer");
    linear_info(lin->L, dim_in, dim_out, weight_numel, n_instr);
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_linear_instruction(cgtp_linear lin, int j, int* i_in, int* i_out,
                                    int64_t* weight_offset) {
    GUARD_BEGIN
    if (!lin) return fail(CGTP_E_ARG, "NULL linear layer");
    if (!linear_instruction(lin->L, j, i_in, i_out, weight_offset))
        return fail(CGTP_E_ARG, "instruction index out of range");
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_linear_workspace(cgtp_linear lin, int64_t n, size_t* fwd_bytes,
                                  size_t* bwd_bytes) {
    GUARD_BEGIN
    if (!lin) return fail(CGTP_E_ARG, "NULL linear layer");
    if (n < 0) return fail(CGTP_E_ARG, "negative row count");
    if (fwd_bytes) *fwd_bytes = linear_fwd_workspace(lin->L);
    if (bwd_bytes) *bwd_bytes = linear_bwd_workspace(lin->L, n);
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_linear_path(cgtp_linear lin, int* tensor_cores) {
    GUARD_BEGIN
    if (!lin || !tensor_cores) return fail(CGTP_E_ARG, "NULL argument");
    *tensor_cores = linear_tensor_cores(lin->L) ? 1 : 0;
    return CGTP_OK;
    GUARD_END
}

static cgtp_status linear_check(cgtp_linear lin, int64_t n,
                                std::initializer_list<const void*> ptrs) {
    if (!lin) return fail(CGTP_E_ARG, "NULL linear layer");
    if (n < 0) return fail(CGTP_E_ARG, "negative row count");
    int64_t di = 0, dout = 0;
    linear_info(lin->L, &di, &dout, nullptr, nullptr);
    if (n > ((int64_t)1 << 40) / std::max<int64_t>(1, std::max(di, dout)))
        return fail(CGTP_E_ARG, "row count too large");
    for (const void* q : ptrs)
        if (!aligned(q, 4)) return fail(CGTP_E_ARG, "tensor pointer not aligned to its element");
    return CGTP_OK;
}

cgtp_status cgtp_linear_forward(cgtp_linear lin, int64_t n, const void* x, const void* W,
                                void* out, void* workspace, size_t workspace_bytes,
                                unsigned flags, cgtp_stream stream) {
    GUARD_BEGIN
    cgtp_status st = linear_check(lin, n, {x, W, out});
    if (st != CGTP_OK) return st;
    if (n == 0) return CGTP_OK;
    if (!x || !W || !out) return fail(CGTP_E_ARG, "NULL tensor");
    if (workspace && !aligned(workspace, 16)) return fail(CGTP_E_ARG, "workspace not 16-byte aligned");
    cudaError_t e = launch_linear_forward(lin->L, n, x, W, out, workspace, workspace_bytes,
                                          !(flags & CGTP_LINEAR_CUDA_CORES), S(stream),
                                          (flags & CGTP_LINEAR_TEST_WAIT_TIMEOUT) != 0);
    if (e != cudaSuccess) return cuda_fail(e, "linear_forward");
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_linear_backward(cgtp_linear lin, int64_t n, const void* x, const void* W,
                                 const void* grad_out, void* grad_x, void* grad_W,
                                 void* workspace, size_t workspace_bytes, unsigned flags,
                                 cgtp_stream stream) {
    GUARD_BEGIN
    cgtp_status st = linear_check(lin, n, {x, W, grad_out, grad_x, grad_W});
    if (st != CGTP_OK) return st;
    if (!grad_x && !grad_W) return CGTP_OK;
    if (n == 0) {  // no rows: grad_W is zero
        if (!grad_W) return CGTP_OK;
        cudaError_t e = launch_linear_backward(lin->L, 0, nullptr, nullptr, nullptr, nullptr,
                                               grad_W, nullptr, 0, false, S(stream));
        if (e != cudaSuccess) return cuda_fail(e, "linear_backward");
        return CGTP_OK;
    }
    if (!grad_out || (grad_x && !W) || (grad_W && !x)) return fail(CGTP_E_ARG, "NULL tensor");
    if (grad_W && (!workspace || workspace_bytes < linear_bwd_workspace(lin->L, n) ||
                   !aligned(workspace, 16)))
        return fail(CGTP_E_ARG, "grad_W needs a 16-byte aligned workspace of "
                                "cgtp_linear_workspace() bwd bytes");
    if (workspace && !aligned(workspace, 16)) return fail(CGTP_E_ARG, "workspace not 16-byte aligned");
    cudaError_t e = launch_linear_backward(lin->L, n, x, W, grad_out, grad_x, grad_W, workspace,
                                           workspace_bytes, !(flags & CGTP_LINEAR_CUDA_CORES),
                                           S(stream));
    if (e != cudaSuccess) return cuda_fail(e, "linear_backward");
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_linear_device_status(int* code) {
    GUARD_BEGIN
    if (!code) return fail(CGTP_E_ARG, "NULL output");
    cudaError_t e = linear_device_status(code);
    if (e != cudaSuccess) return cuda_fail(e, "linear_device_status");
    return CGTP_OK;
    GUARD_END
}

static cgtp_status radial_check(cgtp_dtype dt, int64_t E, int nb, double cutoff, int hidden,
                                int64_t n_out) {
    if (dt != CGTP_F32 && dt != CGTP_F64) return fail(CGTP_E_ARG, "bad dtype");
    if (E < 0) return fail(CGTP_E_ARG, "E < 0");
    if (nb < 1 || nb > 32) return fail(CGTP_E_ARG, "n_basis must be in 1..32");
    if (hidden < 1 || hidden > 256) return fail(CGTP_E_ARG, "hidden must be in 1..256");
    if (n_out < 1) return fail(CGTP_E_ARG, "n_out must be >= 1");
    if (!(cutoff > 0.0) || !std::isfinite(cutoff)) return fail(CGTP_E_ARG, "cutoff must be > 0");
    return CGTP_OK;
}

cgtp_status cgtp_radial_workspace(cgtp_dtype dtype, int n_basis, int hidden, int64_t n_out,
                                  size_t* bytes) {
    GUARD_BEGIN
    cgtp_status st = radial_check(dtype, 0, n_basis, 1.0, hidden, n_out);
    if (st != CGTP_OK) return st;
    if (!bytes) return fail(CGTP_E_ARG, "NULL output");
    *bytes = radial_workspace_bytes(dtype == CGTP_F64, n_basis, hidden, n_out);
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_radial_forward(cgtp_dtype dtype, int64_t E, int n_basis, double cutoff,
                                int hidden, int64_t n_out, const void* vec, const void* W1,
                                const void* W2, void* w, void* h, void* workspace,
                                size_t workspace_bytes, unsigned flags, cgtp_stream stream) {
    GUARD_BEGIN
    cgtp_status st = radial_check(dtype, E, n_basis, cutoff, hidden, n_out);
    if (st != CGTP_OK || E == 0) return st;
    if (!vec || !W1 || !W2 || !w) return fail(CGTP_E_ARG, "NULL tensor");
    const size_t es = dtype == CGTP_F64 ? 8 : 4;
    const bool out_bf16 = (flags & CGTP_RADIAL_OUT_BF16) != 0;
    const bool out_f16 = (flags & CGTP_RADIAL_OUT_F16) != 0;
    if (out_bf16 && out_f16) return fail(CGTP_E_ARG, "both 16-bit output formats requested");
    if ((out_bf16 || out_f16) && dtype != CGTP_F32)
        return fail(CGTP_E_UNSUPPORTED, "16-bit output needs fp32 inputs");
    for (const void* q : {vec, W1, W2, (const void*)h})
        if (!aligned(q, es)) return fail(CGTP_E_ARG, "tensor pointer not aligned to its element");
    if (!aligned(w, out_bf16 || out_f16 ? 2 : es))
        return fail(CGTP_E_ARG, "w not aligned to its element");
    const bool f64 = dtype == CGTP_F64;
    const size_t need = radial_workspace_bytes(f64, n_basis, hidden, n_out);
    const bool tc = !(flags & CGTP_RADIAL_CUDA_CORES) && need > 0 && workspace &&
                    workspace_bytes >= need && aligned(workspace, 16) &&
                    radial_tc_eligible(f64, n_basis, hidden, n_out, vec, W2, w, h);
    cudaError_t e = launch_radial_forward(f64, tc, out_bf16 ? 1 : out_f16 ? 2 : 0, E, n_basis,
                                          cutoff, hidden, n_out,
                                          vec, W1, W2, w, h, workspace, workspace_bytes,
                                          S(stream), (flags & CGTP_RADIAL_TEST_WAIT_TIMEOUT) != 0);
    if (e != cudaSuccess) return cuda_fail(e, "radial_forward");
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_radial_backward_workspace(cgtp_dtype dtype, int64_t E, int n_basis, int hidden,
                                           int64_t n_out, size_t* bytes) {
    GUARD_BEGIN
    cgtp_status st = radial_check(dtype, E, n_basis, 1.0, hidden, n_out);
    if (st != CGTP_OK) return st;
    if (!bytes) return fail(CGTP_E_ARG, "NULL output");
    *bytes = radial_backward_workspace_bytes(dtype == CGTP_F64, E, n_basis, hidden, n_out);
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_radial_backward(cgtp_dtype dtype, int64_t E, int n_basis, double cutoff,
                                 int hidden, int64_t n_out, const void* vec, const void* W1,
                                 const void* W2, const void* grad_w, void* grad_vec,
                                 void* grad_W1, void* grad_W2, void* workspace,
                                 size_t workspace_bytes, unsigned flags, cgtp_stream stream) {
    GUARD_BEGIN
    cgtp_status st = radial_check(dtype, E, n_basis, cutoff, hidden, n_out);
    if (st != CGTP_OK) return st;
    const bool f64 = dtype == CGTP_F64;
    const size_t es = f64 ? 8 : 4;
    if (!grad_vec && !grad_W1 && !grad_W2) return CGTP_OK;
    for (const void* q : {vec, W1, W2, grad_w, (const void*)grad_vec, (const void*)grad_W1,
                          (const void*)grad_W2, (const void*)workspace})
        if (!aligned(q, es)) return fail(CGTP_E_ARG, "tensor pointer not aligned to its element");
    if (E == 0) {  // empty sums
        if (grad_W1 && (st = zero(grad_W1, (int64_t)n_basis * hidden * es, S(stream))) != CGTP_OK)
            return st;
        if (grad_W2 && (st = zero(grad_W2, (int64_t)hidden * n_out * es, S(stream))) != CGTP_OK)
            return st;
        return CGTP_OK;
    }
    if (!vec || !W1 || !W2 || !grad_w) return fail(CGTP_E_ARG, "NULL input tensor");
    const size_t need = radial_backward_workspace_bytes(f64, E, n_basis, hidden, n_out);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16))
        return fail(CGTP_E_ARG, "workspace of " + std::to_string(workspace_bytes) +
                                    " bytes is smaller than the " + std::to_string(need) +
                                    " bytes cgtp_radial_backward_workspace reports");
    const bool tc = !(flags & CGTP_RADIAL_CUDA_CORES) &&
                    radial_tc_eligible(f64, n_basis, hidden, n_out, vec, W2, grad_w, nullptr);
    cudaError_t e = launch_radial_backward(f64, tc, E, n_basis, cutoff, hidden, n_out, vec, W1,
                                           W2, grad_w, grad_vec, grad_W1, grad_W2, workspace,
                                           S(stream));
    if (e != cudaSuccess) return cuda_fail(e, "radial_backward");
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_radial_path(cgtp_dtype dtype, int n_basis, int hidden, int64_t n_out,
                             int* tensor_cores) {
    GUARD_BEGIN
    cgtp_status st = radial_check(dtype, 0, n_basis, 1.0, hidden, n_out);
    if (st != CGTP_OK) return st;
    if (!tensor_cores) return fail(CGTP_E_ARG, "NULL output");
    *tensor_cores = radial_tc_eligible(dtype == CGTP_F64, n_basis, hidden, n_out, nullptr,
                                       nullptr, nullptr, nullptr) ? 1 : 0;
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_radial_device_status(int* code) {
    GUARD_BEGIN
    if (!code) return fail(CGTP_E_ARG, "NULL output");
    cudaError_t e = radial_device_status(code);
    if (e != cudaSuccess) return cuda_fail(e, "radial_device_status");
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_edge_forces(cgtp_dtype dtype, int64_t N, int64_t E, const int32_t* rowptr,
                             const int32_t* s_rowptr, const int32_t* s_perm, const void* dEdr,
                             void* forces, cgtp_stream stream) {
    GUARD_BEGIN
    if (dtype != CGTP_F32 && dtype != CGTP_F64) return fail(CGTP_E_ARG, "bad dtype");
    cgtp_status st = check_graph(N, E, rowptr, s_perm);
    if (st != CGTP_OK) return st;
    if (N > 0 && !s_rowptr) return fail(CGTP_E_GRAPH, "NULL s_rowptr");
    if (N == 0) return CGTP_OK;
    if (!forces || (E > 0 && !dEdr)) return fail(CGTP_E_ARG, "NULL tensor");
    cudaError_t e = launch_edge_forces(dtype == CGTP_F64, N, rowptr, s_rowptr, s_perm, dEdr,
                                       forces, S(stream));
    if (e != cudaSuccess) return cuda_fail(e, "edge_forces");
    return CGTP_OK;
    GUARD_END
}

cgtp_status cgtp_edge_forces_adjoint(cgtp_dtype dtype, int64_t N, int64_t E,
                                     const int32_t* rowptr, const int32_t* sender,
                                     const void* grad_forces, void* grad_dEdr,
                                     cgtp_stream stream) {
    GUARD_BEGIN
    if (dtype != CGTP_F32 && dtype != CGTP_F64) return fail(CGTP_E_ARG, "bad dtype");
    cgtp_status st = check_graph(N, E, rowptr, sender);
    if (st != CGTP_OK) return st;
    if (N == 0 || E == 0) return CGTP_OK;
    if (!grad_forces || !grad_dEdr) return fail(CGTP_E_ARG, "NULL tensor");
    cudaError_t e = launch_edge_forces_adjoint(dtype == CGTP_F64, N, rowptr, sender, grad_forces,
                                               grad_dEdr, S(stream));
    if (e != cudaSuccess) return cuda_fail(e, "edge_forces_adjoint");
    return CGTP_OK;
    GUARD_END
}

const char* cgtp_status_str(cgtp_status s) {
    switch (s) {
        case CGTP_OK: return "ok";
        case CGTP_E_ARG: return "invalid argument";
        case CGTP_E_IRREPS: return "irreps string does not parse";
        case CGTP_E_PATH: return "instruction is not an allowed path";
        case CGTP_E_UNSUPPORTED: return "unsupported";
        case CGTP_E_GRAPH: return "inconsistent graph";
        case CGTP_E_NOMEM: return "out of host memory";
        case CGTP_E_CUDA: return "CUDA error";
        case CGTP_E_COMPILE: return "kernel compilation failed";
        case CGTP_E_DEVICE: return "device-side error flag";
    }
    return "unknown status";
}

cgtp_status cgtp_last_cuda_error(int* cuda_err) {
    if (!cuda_err) return CGTP_E_ARG;
    *cuda_err = t_cuda_err;
    return CGTP_OK;
}

const char* cgtp_last_error_message(void) { return t_msg.c_str(); }

int64_t cgtp_launch_count(void) { return g_launches.load(); }

}  // extern "C"

namespace cgtp {

// Gradient of the fused convolution with the shared-weight partial rows
// written to `scratch` (at most scratch_bytes / row bytes of them); used by the
// entry point whose scratch is a fixed device array.
cgtp_status conv_backward_into_scratch(cgtp_plan plan, int64_t N, int64_t E,
                                       const int32_t* s_rowptr, const int32_t* s_perm,
                                       const int32_t* s_recv, const void* x, const void* y,
                                       const void* w, double scale, const void* grad_out,
                                       void* grad_x, void* grad_y, void* grad_w, void* scratch,
                                       size_t scratch_bytes, cudaStream_t s) {
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    cgtp_status st = check_graph(N, E, s_rowptr, s_perm);
    if (st != CGTP_OK) return st;
    if (E > 0 && !s_recv) return fail(CGTP_E_GRAPH, "NULL s_recv");
    Plan& p = plan->p;
    const int64_t row = p.wdim * (int64_t)esize(p);
    const bool shared = p.wmode == CGTP_W_SHARED && grad_w;
    const int64_t rows = shared ? (int64_t)(scratch_bytes / (size_t)row) : 0;
    if (shared && rows < 1)
        return fail(CGTP_E_ARG, "weight row of " + std::to_string(row) +
                                    " bytes exceeds the fixed scratch of " +
                                    std::to_string(scratch_bytes) + " bytes");
    if (N == 0) return shared ? zero(grad_w, row, s) : CGTP_OK;
    if (!x || !grad_out || (E > 0 && (!y || !w))) return fail(CGTP_E_ARG, "NULL input tensor");
    if ((st = check_rows(p, {x, grad_out, grad_x, grad_w})) != CGTP_OK) return st;
    if ((st = check_w(p, w)) != CGTP_OK) return st;
    return bwd_launch(p, true, N, s_rowptr, s_perm, s_recv, x, y, w, grad_out, scale, grad_x,
                      grad_y, grad_w, grad_x ? 1 : 0, grad_y ? 1 : 0, grad_w ? 1 : 0, s, scratch,
                      std::min<int64_t>(rows, kSharedWRows));
}

bool plan_module_loaded(cgtp_plan plan, int dev) {
    if (!plan) return false;
    std::lock_guard<std::mutex> g(plan->p.mu);
    auto it = plan->p.modules.find("tp");
    if (it == plan->p.modules.end() || it->second->lib == nullptr) return false;
    const std::set<int>& on = it->second->launched_on;
    return dev < 0 ? !on.empty() : on.count(dev) != 0;
}

int64_t plan_weight_row_bytes(cgtp_plan plan) {
    return plan ? plan->p.wdim * (int64_t)esize(plan->p) : 0;
}

bool plan_shared_weights(cgtp_plan plan) { return plan && plan->p.wmode == CGTP_W_SHARED; }

LinearImpl* cgtp_linear_impl(cgtp_linear lin) { return lin ? lin->L : nullptr; }

cgtp_status plan_preload_kernels(cgtp_plan plan, int dev) {
    if (!plan) return fail(CGTP_E_ARG, "plan is NULL");
    std::lock_guard<std::mutex> g(plan->p.mu);
    auto it = plan->p.modules.find("tp");
    if (it == plan->p.modules.end() || it->second->lib == nullptr)
        return fail(CGTP_E_ARG, "the plan's kernels are not loaded");
    Module& m = *it->second;
    if (m.preloaded_on.count(dev)) return CGTP_OK;
    cudaError_t e = cudaSuccess;
    for (auto& kv : m.kernels) {
        if (!kv.second) continue;
        cudaFuncAttributes a;
        if ((e = cudaFuncGetAttributes(&a, (const void*)kv.second)) != cudaSuccess)
            return cuda_fail(e, ("load kernel " + kv.first).c_str());
    }
    if ((e = preload_reduce_kernels()) != cudaSuccess) return cuda_fail(e, "load reduction kernels");
    m.preloaded_on.insert(dev);
    return CGTP_OK;
}

}  // namespace cgtp
