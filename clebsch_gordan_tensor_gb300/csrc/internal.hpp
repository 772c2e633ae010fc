// Internal declarations shared by the C-ABI, the JIT and the fixed kernels.
#pragma once

#include <cuda_runtime.h>

#include <map>
#include <memory>
#include <set>
#include <string>
#include <vector>

#include "plan.hpp"

namespace cgtp {

struct Module {
    std::vector<char> cubin;
    std::string log;  // NVRTC / ptxas log (register and spill report)
    cudaLibrary_t lib = nullptr;
    std::map<std::string, cudaKernel_t> kernels;
    void* err_flag = nullptr;           // device address of cgtp_device_error (staged)
    std::map<int, int> smem_set;        // device -> dynamic smem attribute already set
    std::map<std::pair<int, std::string>, int> ctas_per_sm;
    std::set<int> launched_on;          // devices a kernel of the module has run on
    std::set<int> preloaded_on;         // devices all its kernels were loaded on
    ~Module();
};

cgtp_status get_module(Plan& p, bool load, std::shared_ptr<Module>& out, std::string& err);

// Thread-local error state of the C ABI.
void set_cuda_error(cudaError_t e);
void set_error_message(const std::string& m);
void count_launch();

// Fixed kernels (sh.cu, graph.cu).  They return a cudaError_t of the launch.
cudaError_t launch_sh_forward(int lmax, bool f64, int64_t E, const void* vec, void* y,
                              cudaStream_t s);
cudaError_t launch_sh_backward(int lmax, bool f64, int64_t E, const void* vec, const void* gy,
                               void* gvec, cudaStream_t s);
cudaError_t launch_sh_jvp(int lmax, bool f64, int64_t E, const void* vec, const void* tvec,
                          void* ty, cudaStream_t s);
cudaError_t launch_sh_hvp(int lmax, bool f64, int64_t E, const void* vec, const void* gy,
                          const void* tvec, void* out, cudaStream_t s);
cudaError_t launch_edge_forces(bool f64, int64_t N, const int32_t* rowptr,
                               const int32_t* s_rowptr, const int32_t* s_perm, const void* dEdr,
                               void* F, cudaStream_t s);
cudaError_t launch_edge_forces_adjoint(bool f64, int64_t N, const int32_t* rowptr,
                                       const int32_t* sender, const void* gF, void* q,
                                       cudaStream_t s);
cudaError_t launch_fill_zero(void* p, int64_t bytes, cudaStream_t s);
cudaError_t launch_reduce_rows(bool f64, const void* partial, int64_t rows, int64_t cols,
                               void* out, cudaStream_t s);
cudaError_t preload_reduce_kernels();
// p[0..n) = 1 (fp32 or fp64).
cudaError_t launch_fill_ones(bool f64, void* p, int64_t n, cudaStream_t s);

// Radial network (radial.cu).
bool radial_tc_eligible(bool f64, int nb, int hidden, int64_t n_out, const void* vec,
                        const void* W2, const void* w, const void* h);
size_t radial_workspace_bytes(bool f64, int nb, int hidden, int64_t n_out);
cudaError_t launch_radial_forward(bool f64, bool tensor_cores, int out16, int64_t E, int nb,
                                  double rc, int hidden, int64_t n_out, const void* vec,
                                  const void* W1, const void* W2, void* w, void* h, void* ws,
                                  size_t ws_bytes, cudaStream_t s, bool test_fail = false);
cudaError_t radial_device_status(int* code);
size_t radial_backward_workspace_bytes(bool f64, int64_t E, int nb, int hidden, int64_t n_out);
cudaError_t launch_radial_backward(bool f64, bool tensor_cores, int64_t E, int nb, double rc,
                                   int hidden, int64_t n_out, const void* vec, const void* W1,
                                   const void* W2, const void* gw, void* gvec, void* gW1,
                                   void* gW2, void* ws, cudaStream_t s);

// Per-irrep channel mixing (linear.cu).
struct LinearImpl;

// Tensor-product source of a mixing layer's input rows (the fused 'uvw'
// forward): input irrep p of the layer is path p's block of the 'uvu' product
// with unit weights,
//   a[n, p, m3, u] = sum_m1 T[n, p, m3, m1] x1[n, x1_off + m1 mul1 + u],
//   T[n, p, m3, m1] = sum_m2 C_p[m1, m2, m3] y[n, m2],
// so the layer's input rows are computed where they are consumed.  T is
// channel-independent and small (one row of tdim values per sample, path p's
// [d3][d1] block at t_off); entry e of a T row sums the CG terms
// [estart[e], estart[e + 1]).  Passed by value as a kernel parameter.
constexpr int kTpMaxPaths = 64, kTpMaxT = 1024, kTpMaxTerms = 2048;
struct LinTpPath {
    int x1_off, mul1, t_off, d1, d3;
};
struct LinTpDesc {
    int npaths = 0, nterms = 0, tdim = 0;
    LinTpPath path[kTpMaxPaths];
    short estart[kTpMaxT + 1];
    unsigned char term_y[kTpMaxTerms];  // y element of the term
    float term_c[kTpMaxTerms];
};
// The fused forward: T for every sample into tbuf (n * tdim floats), then out =
// the layer applied to the rows described by tp (x1 [n, x1_stride], y [n,
// y_stride]).  *used = false when it is not eligible (nothing is launched).
cudaError_t launch_linear_forward_tp(const LinearImpl* L, const LinTpDesc& tp, int64_t n,
                                     const void* x1, int64_t x1_stride, const void* y,
                                     int64_t y_stride, const void* W, void* out, void* ws,
                                     size_t ws_bytes, void* tbuf, size_t tbuf_bytes,
                                     cudaStream_t s, bool* used);
cgtp_status linear_create(const char* irreps_in, const char* irreps_out,
                          const cgtp_linear_instr* instr, int n_instr, cgtp_dtype dt,
                          LinearImpl** res, std::string& err);
void linear_destroy(LinearImpl* L);
LinearImpl* cgtp_linear_impl(cgtp_linear lin);
void linear_info(const LinearImpl* L, int64_t* dim_in, int64_t* dim_out, int64_t* nw, int* ninstr);
bool linear_instruction(const LinearImpl* L, int j, int* i_in, int* i_out, int64_t* w_off);
bool linear_tensor_cores(const LinearImpl* L);
size_t linear_fwd_workspace(const LinearImpl* L);
size_t linear_bwd_workspace(const LinearImpl* L, int64_t n);
bool linear_uses_tc(const LinearImpl* L, int64_t n, const void* a, const void* out, const void* ws,
                    size_t ws_bytes, bool fwd);
cudaError_t launch_linear_forward(const LinearImpl* L, int64_t n, const void* x, const void* W,
                                  void* out, void* ws, size_t ws_bytes, bool allow_tc,
                                  cudaStream_t s, bool test_fail = false);
cudaError_t launch_linear_backward(const LinearImpl* L, int64_t n, const void* x, const void* W,
                                   const void* g, void* gx, void* gW, void* ws, size_t ws_bytes,
                                   bool allow_tc, cudaStream_t s);
cudaError_t linear_device_status(int* code);
bool radial_w2_tc_eligible(int hidden, int64_t n_out);
// The driver's cuTensorMapEncodeTiled (PFN_cuTensorMapEncodeTiled_v12000), or
// null where the driver does not provide it.
void* tensor_map_encoder();
cudaError_t launch_radial_w2_tc(int64_t E, int hidden, int64_t n_out, const float* h,
                                const float* gw, float* partial, int64_t S, cudaStream_t s);

// Partial weight-gradient rows a shared-weight backward may write (grid cap).
constexpr int64_t kSharedWRows = 2048;

cgtp_status conv_backward_into_scratch(cgtp_plan plan, int64_t N, int64_t E,
                                       const int32_t* s_rowptr, const int32_t* s_perm,
                                       const int32_t* s_recv, const void* x, const void* y,
                                       const void* w, double scale, const void* grad_out,
                                       void* grad_x, void* grad_y, void* grad_w, void* scratch,
                                       size_t scratch_bytes, cudaStream_t s);
// True once a kernel of the plan's module has run on device dev (dev < 0: on
// any device); loading the module into a device's context allocates.
bool plan_module_loaded(cgtp_plan plan, int dev);
// Bytes of one weight row of the plan (0 for a NULL plan).
int64_t plan_weight_row_bytes(cgtp_plan plan);
bool plan_shared_weights(cgtp_plan plan);
// Loads every kernel of the plan's module, and the fixed reduction kernels, into
// the current device's context (a no-op once done for that device).
cgtp_status plan_preload_kernels(cgtp_plan plan, int dev);

}  // namespace cgtp
