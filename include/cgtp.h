/*
 * cgtp.h -- C ABI of the GB300 (sm_103a) Clebsch-Gordan tensor-product library.
 *
 * The operation (from "An Efficient Sparse Kernel Generator for O(3)-Equivariant
 * Deep Networks", arXiv 2501.13986, abstract): the CG tensor product contracts
 * two dense irrep feature vectors x (irreps_in1) and y (irreps_in2) with the
 * fixed, highly structured sparse Clebsch-Gordan tensor into a dense output
 * (irreps_out); it is fused with the graph convolution around it; the library
 * also provides its gradient and the higher partial derivatives used for
 * interatomic forces.  The per-edge weights are the "radial profile" of the
 * TFN layer (NVIDIA SE(3)-Transformer blog, "Fused key and value computation");
 * a layer is the sum over degree pairs of the pairwise convolutions (same blog,
 * "TFN fusion", Fig. 5); a degree-l block has 2l+1 components.
 *
 * Conventions (the pages are silent; these are the library's):
 *  - Irreps strings: "16x0e+16x1o" (mul x l parity, parity e/o).
 *  - Paths are 'uvu': out[u] += w[path][u] * sum C[m1,m2,m3] x[u,m1] y[m2]; in2
 *    irreps have mul 1 and every in1 / out irrep has the same mul.  With
 *    instr == NULL every parity-allowed (|l1-l2| <= l3 <= l1+l2, p3 = p1 p2)
 *    triple is a path, listed with in1 outermost, then in2, then out.
 *  - CG coefficients are real-basis, unitary (sum_{m1,m2} C C' = delta), with
 *    the first nonzero entry of each path positive.  Real spherical harmonics
 *    are component-normalised (sum_m Y_lm^2 = 2l+1), m = -l..l, so that
 *    Y_1 = sqrt(3) (y, z, x).
 *  - Feature rows hold irrep blocks in irreps order; inside a block the element
 *    (m, u) sits at (m + l) * mul + u (channel fastest).  Weight rows hold one
 *    block of mul per path, in path order (weight_numel = n_paths * mul).
 *  - Graphs: rowptr[N+1] / sender[E] is a CSR over receivers (edges sorted by
 *    receiver).  The sender-grouped view (for gradients) is s_rowptr[N+1],
 *    s_perm[E] (edge ids grouped by sender, ascending within a sender) and
 *    s_recv[E] (receiver of edge s_perm[j]).  Edge vectors are
 *    pos[receiver] - pos[sender].
 *
 * Memory and errors:
 *  - Every tensor pointer is caller-owned DEVICE memory, contiguous, row-major,
 *    of the plan's dtype (int32 for graph arrays), 8-byte aligned at least.
 *    The library never allocates device memory in these calls.
 *  - Outputs are overwritten, never accumulated.  NULL outputs are skipped.
 *  - Calls are asynchronous on `stream` (NULL = legacy default stream).
 *    Argument errors return synchronously without launching.  A CUDA launch
 *    error returns CGTP_E_CUDA (cgtp_last_cuda_error gives the code).
 *  - No C++ exception crosses this interface.  Plans are immutable after
 *    creation and may be shared between threads.
 *  - The first GPU call of a plan compiles its kernels with NVRTC for sm_103a
 *    (tens of milliseconds to seconds); later calls reuse them.
 */
#ifndef CGTP_H
#define CGTP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cgtp_stream; /* == cudaStream_t */
typedef struct cgtp_plan_s* cgtp_plan;

typedef enum {
    CGTP_OK = 0,
    CGTP_E_ARG = 1,         /* bad pointer, size, or NULL where required */
    CGTP_E_IRREPS = 2,      /* irreps string does not parse */
    CGTP_E_PATH = 3,        /* an instruction is not an allowed path */
    CGTP_E_UNSUPPORTED = 4, /* valid request the library does not implement */
    CGTP_E_GRAPH = 5,       /* inconsistent graph sizes */
    CGTP_E_NOMEM = 6,       /* host allocation failed */
    CGTP_E_CUDA = 7,        /* CUDA runtime error */
    CGTP_E_COMPILE = 8,     /* NVRTC compilation or module load failed */
    CGTP_E_DEVICE = 9       /* a kernel reported an error flag */
} cgtp_status;

typedef enum { CGTP_F32 = 0, CGTP_F64 = 1 } cgtp_dtype;
typedef enum { CGTP_W_PER_EDGE = 0, CGTP_W_SHARED = 1 } cgtp_wmode;

/* One tensor-product path: irrep indices into in1, in2, out; mode "uvu". */
typedef struct {
    int i_in1, i_in2, i_out;
    char mode[4];
} cgtp_instr;

/* ------------------------------------------------------------- planning -- */

/* Parse the irreps, list or check the paths, compute the real-basis CG
 * coefficients (complex CG by the angular-momentum lowering recursion, taken to
 * the real basis) and lay out the per-path work.  Host only; no GPU needed.
 * irreps_in2 must have mul 1 per irrep (spherical harmonics); in1 and out must
 * share one mul.  l <= 6.
 * flags: 0 for automatic tuning, else overrides of the staged kernels' launch
 * shape: bits 0-3 forward warp groups (1-4), bits 4-7 backward warp groups,
 * bits 8-11 forward TMA ring depth (2-15), bits 12-15 backward ring depth,
 * bit 16: forward lanes load their weights directly (prefetched one edge ahead
 * in registers) instead of through the ring; bit 17: backward lanes take their
 * weights through the ring instead of loading them directly (direct loads are
 * the default for fp32 plans with two channels per lane, the ring for the
 * others); bit 18: directly loaded backward weights use one register
 * buffer (reloaded path by path) instead of two; bit 19: the backward puts
 * the grad_y contraction on a second warp of each CTA (one-warp path groups);
 * bits 20-23: the backward's register budget must allow that many resident
 * CTAs per SM; bit 27: the backward's T entries are stored as splatted pairs;
 * bit 28: the backward's two weight buffers alternate instead of the next
 * edge's being copied over.
 * CGTP_PLAN_WEIGHTS_BF16 (bit 24): the weights (w, per edge or shared) are
 * stored as bfloat16 and widened exactly to fp32 on load; all arithmetic,
 * every other tensor and grad_w stay fp32.  This halves the dominant weight
 * stream ("BF16/FP16 ... with FP32 accumulation", "Speeding Up MACE",
 * abstract).  fp32 plans only (else CGTP_E_UNSUPPORTED); the double backward
 * of such a plan returns CGTP_E_UNSUPPORTED. */
#define CGTP_PLAN_WEIGHTS_BF16 (1u << 24)
/* CGTP_PLAN_WEIGHTS_F16 (bit 25): as CGTP_PLAN_WEIGHTS_BF16 with the weights
 * stored as IEEE binary16 (11 significant bits, range +-65504; values below
 * 2^-14 are subnormal), widened exactly to fp32 on load.  Not combined with
 * CGTP_PLAN_WEIGHTS_BF16 (CGTP_E_ARG); the same restrictions otherwise. */
#define CGTP_PLAN_WEIGHTS_F16 (1u << 25)
/* CGTP_PLAN_TEST_WAIT_TIMEOUT (bit 26), for tests of the failure path only: in
 * the staged kernels the first bounded wait of every CTA gives up at once, as
 * if its bulk copy had not arrived within the limit.  The kernel then records
 * a code in the plan's device error flag, waits (bounded) for the copies it
 * has in flight and returns without finishing its outputs;
 * cgtp_plan_device_status returns CGTP_E_DEVICE with that code once and clears
 * the flag.  Never set it outside a test. */
#define CGTP_PLAN_TEST_WAIT_TIMEOUT (1u << 26)
cgtp_status cgtp_plan_create(cgtp_plan* out, const char* irreps_in1, const char* irreps_in2,
                             const char* irreps_out, const cgtp_instr* instr, int n_instr,
                             cgtp_dtype dtype, cgtp_wmode wmode, unsigned flags);
cgtp_status cgtp_plan_destroy(cgtp_plan plan);

/* Row widths (elements) of x, y, out; weight elements per row; path count. */
cgtp_status cgtp_plan_info(cgtp_plan plan, int64_t* dim_in1, int64_t* dim_in2, int64_t* dim_out,
                           int64_t* weight_numel, int* n_paths);

/* Path p: l1, l2, l3 and the irrep indices it couples. */
cgtp_status cgtp_plan_path(cgtp_plan plan, int p, int* l1, int* l2, int* l3, int* i_in1,
                           int* i_in2, int* i_out);

/* Dense real CG tensor of path p, out[((m1+l1)*(2l2+1) + m2+l2)*(2l3+1) + m3+l3]
 * (host memory, caller-owned, (2l1+1)(2l2+1)(2l3+1) doubles). */
cgtp_status cgtp_plan_coefficients(cgtp_plan plan, int p, double* out);

/* Compile the plan's kernels for sm_103a with NVRTC now (host only, no GPU
 * needed) instead of at the first GPU call.  If log != NULL, copies up to cap-1
 * bytes of the compiler log (ptxas register / spill report) into it. */
cgtp_status cgtp_plan_compile(cgtp_plan plan, char* log, size_t cap);

/* The CUDA source generated for the plan (constants, CG tables and unrolled
 * contraction streams).  *needed = bytes including the terminator. */
cgtp_status cgtp_plan_source(cgtp_plan plan, char* buf, size_t cap, size_t* needed);

/* Device-side error flag of the plan's kernels: CGTP_E_DEVICE (and *code != 0)
 * if a staged kernel gave up on a bounded wait for one of its bulk copies since
 * the last call; the flag is then cleared.  Synchronises with the device. */
cgtp_status cgtp_plan_device_status(cgtp_plan plan, int* code);

/* ------------------------------------------- standalone tensor product -- */

/* out[b] = sum_paths w[b,p,u] sum C x[b,l1,m1,u] y[b,l2,m2]   (b < B)
 * x [B, dim_in1], y [B, dim_in2], w [B, weight_numel] (or [weight_numel] for a
 * CGTP_W_SHARED plan), out [B, dim_out]. */
cgtp_status cgtp_forward(cgtp_plan plan, int64_t B, const void* x, const void* y, const void* w,
                         void* out, cgtp_stream stream);

/* Gradient for grad_out = dL/dout [B, dim_out]:
 *   grad_x[b,l1,m1,u] = sum C y[m2] w[p,u] g[l3,m3,u]
 *   grad_y[b,l2,m2]   = sum C x[m1,u] w[p,u] g[m3,u]   (summed over channels)
 *   grad_w[b,p,u]     = sum C x[m1,u] y[m2] g[m3,u]
 * Any output may be NULL.  For a CGTP_W_SHARED plan grad_w sums over the
 * samples and needs scratch memory: use cgtp_backward_ws (CGTP_E_ARG here). */
cgtp_status cgtp_backward(cgtp_plan plan, int64_t B, const void* x, const void* y, const void* w,
                          const void* grad_out, void* grad_x, void* grad_y, void* grad_w,
                          cgtp_stream stream);

/* Bytes of device scratch the weight gradient of a CGTP_W_SHARED plan needs
 * (0 for per-edge plans): one partial row of weight_numel per CTA, at most
 * 2048 rows.  The partial rows are summed in order, so results do not depend
 * on scheduling. */
cgtp_status cgtp_weight_grad_workspace(cgtp_plan plan, size_t* bytes);

/* cgtp_backward with caller-owned device scratch `workspace` (16-byte aligned,
 * at least cgtp_weight_grad_workspace bytes; contents need no initialisation
 * and are overwritten).  Required when grad_w != NULL on a CGTP_W_SHARED plan;
 * grad_w [weight_numel] = sum over samples. */
cgtp_status cgtp_backward_ws(cgtp_plan plan, int64_t B, const void* x, const void* y,
                             const void* w, const void* grad_out, void* grad_x, void* grad_y,
                             void* grad_w, void* workspace, size_t workspace_bytes,
                             cgtp_stream stream);

/* Higher partial derivatives ("a novel identity for the higher partial
 * derivatives", abstract of arXiv 2501.13986; the identity is not printed).
 * The library uses the trilinearity of f(x, y, w): with cotangents gg_x, gg_y,
 * gg_w (NULL = zero) of grad_x, grad_y, grad_w,
 *   d_grad_out = f(gg_x, y, w) + f(x, gg_y, w) + f(x, y, gg_w)
 *   d_x = f_x(g; gg_y, w) + f_x(g; y, gg_w)
 *   d_y = f_y(g; gg_x, w) + f_y(g; x, gg_w)
 *   d_w = f_w(g; gg_x, y) + f_w(g; x, gg_y)
 * Outputs may be NULL (skipped). */
cgtp_status cgtp_double_backward(cgtp_plan plan, int64_t B, const void* x, const void* y,
                                 const void* w, const void* grad_out, const void* gg_x,
                                 const void* gg_y, const void* gg_w, void* d_x, void* d_y,
                                 void* d_w, void* d_grad_out, cgtp_stream stream);
/* cgtp_double_backward with caller scratch: required (16-byte aligned, at
 * least twice cgtp_weight_grad_workspace() bytes, contents need not be set)
 * when d_w is requested from a CGTP_W_SHARED plan, whose d_w sums both terms
 * over all rows through per-CTA partial rows added in fixed order
 * (deterministic).  Calls sharing a workspace must not overlap in time. */
cgtp_status cgtp_double_backward_ws(cgtp_plan plan, int64_t B, const void* x, const void* y,
                                    const void* w, const void* grad_out, const void* gg_x,
                                    const void* gg_y, const void* gg_w, void* d_x, void* d_y,
                                    void* d_w, void* d_grad_out, void* workspace,
                                    size_t workspace_bytes, cgtp_stream stream);

/* -------------------------------------------- fused graph convolution -- */

/* out[n] = scale * sum_{e=rowptr[n]}^{rowptr[n+1]-1} TP(x[sender[e]], y[e], w[e])
 * ("fusing the CG tensor product with a subsequent graph convolution", abstract
 * of arXiv 2501.13986).  Every receiver row is written (zero if no edges).
 * x [N, dim_in1], y [E, dim_in2], w [E, weight_numel], out [N, dim_out]. */
cgtp_status cgtp_conv_forward(cgtp_plan plan, int64_t N, int64_t E, const int32_t* rowptr,
                              const int32_t* sender, const void* x, const void* y, const void* w,
                              double scale, void* out, cgtp_stream stream);

/* Gradient of cgtp_conv_forward for grad_out [N, dim_out]:
 *   grad_x[s] = scale * sum_{edges e with sender s} f_x(g[recv e]; y[e], w[e])
 *   grad_y[e] = scale * f_y(g[recv e]; x[sender e], w[e])
 *   grad_w[e] = scale * f_w(g[recv e]; x[sender e], y[e])
 * Uses the sender-grouped view (s_rowptr, s_perm, s_recv); no atomics.
 * For a CGTP_W_SHARED plan grad_w needs scratch: use cgtp_conv_backward_ws. */
cgtp_status cgtp_conv_backward(cgtp_plan plan, int64_t N, int64_t E, const int32_t* rowptr,
                               const int32_t* sender, const int32_t* s_rowptr,
                               const int32_t* s_perm, const int32_t* s_recv, const void* x,
                               const void* y, const void* w, double scale, const void* grad_out,
                               void* grad_x, void* grad_y, void* grad_w, cgtp_stream stream);

/* cgtp_conv_backward with caller-owned scratch (see cgtp_backward_ws); for a
 * CGTP_W_SHARED plan grad_w [weight_numel] sums over all edges. */
cgtp_status cgtp_conv_backward_ws(cgtp_plan plan, int64_t N, int64_t E, const int32_t* rowptr,
                                  const int32_t* sender, const int32_t* s_rowptr,
                                  const int32_t* s_perm, const int32_t* s_recv, const void* x,
                                  const void* y, const void* w, double scale,
                                  const void* grad_out, void* grad_x, void* grad_y, void* grad_w,
                                  void* workspace, size_t workspace_bytes, cgtp_stream stream);

/* cgtp_conv_backward_ws without a workspace argument, for callers that cannot
 * allocate device memory when they need the gradient (a framework whose own
 * pool owns all device memory, a plugin under a fixed memory budget, a loop
 * that cannot take the implicit synchronisation of cudaMalloc / cudaFree).
 * The pages have no counterpart: this entry point only changes where the
 * scratch lives.  The scratch is a fixed 8 MiB device array inside the library
 * (every GPU that loads the library holds it until exit).  A CGTP_W_SHARED plan
 * asking for grad_w sums it from partial rows in that array: its weight row may
 * take at most 64 KiB (8 MiB / 128, room for the partial rows of one CTA of any
 * kernel), else CGTP_E_ARG; at most min(2048, 8 MiB / row bytes) partial rows
 * are used.  The plan's kernels must already have run on the current device
 * through another entry point (that first load allocates), else CGTP_E_ARG.
 * Set-up: the first call on a device looks up the array's device address and
 * loads the rest of the plan's kernels and the reduction kernels into the
 * device's context, which can allocate device memory for their code; make that
 * first call before any stream capture and where allocation is acceptable.
 * Later calls on that device allocate and free nothing.  Every call shares the
 * one array and overwrites all of the rows it reads, so nothing in it needs
 * clearing; calls whose kernels overlap on the GPU (two streams, two threads)
 * race on it. */
cgtp_status cgtp_conv_backward_noalloc(cgtp_plan plan, int64_t N, int64_t E,
                                       const int32_t* rowptr, const int32_t* sender,
                                       const int32_t* s_rowptr, const int32_t* s_perm,
                                       const int32_t* s_recv, const void* x, const void* y,
                                       const void* w, double scale, const void* grad_out,
                                       void* grad_x, void* grad_y, void* grad_w,
                                       cgtp_stream stream);

/* The identity of cgtp_double_backward applied to the fused convolution.
 * CGTP_W_SHARED plans: d_w needs the workspace of cgtp_conv_double_backward_ws
 * (without one, a non-NULL d_w returns CGTP_E_ARG). */
cgtp_status cgtp_conv_double_backward(cgtp_plan plan, int64_t N, int64_t E, const int32_t* rowptr,
                                      const int32_t* sender, const int32_t* s_rowptr,
                                      const int32_t* s_perm, const int32_t* s_recv, const void* x,
                                      const void* y, const void* w, double scale,
                                      const void* grad_out, const void* gg_x, const void* gg_y,
                                      const void* gg_w, void* d_x, void* d_y, void* d_w,
                                      void* d_grad_out, cgtp_stream stream);
/* cgtp_conv_double_backward with caller scratch, as cgtp_double_backward_ws. */
cgtp_status cgtp_conv_double_backward_ws(cgtp_plan plan, int64_t N, int64_t E,
                                         const int32_t* rowptr, const int32_t* sender,
                                         const int32_t* s_rowptr, const int32_t* s_perm,
                                         const int32_t* s_recv, const void* x, const void* y,
                                         const void* w, double scale, const void* grad_out,
                                         const void* gg_x, const void* gg_y, const void* gg_w,
                                         void* d_x, void* d_y, void* d_w, void* d_grad_out,
                                         void* workspace, size_t workspace_bytes,
                                         cgtp_stream stream);

/* --------------------------------------------- spherical harmonics ------ */
/* The per-edge basis "depends on spherical harmonics" of the relative position
 * (NVIDIA SE(3)-Transformer blog, "Basis precomputation").  Component
 * normalisation, vectors normalised first, 0 <= lmax <= 6; y [E, (lmax+1)^2]. */
cgtp_status cgtp_sh_forward(int lmax, cgtp_dtype dtype, int64_t E, const void* vec, void* y,
                            cgtp_stream stream);
/* grad_vec[e] = J(vec[e])^T grad_y[e], J = dY/dvec. */
cgtp_status cgtp_sh_backward(int lmax, cgtp_dtype dtype, int64_t E, const void* vec,
                             const void* grad_y, void* grad_vec, cgtp_stream stream);
/* tangent_y[e] = J(vec[e]) tangent_vec[e] (the derivative of cgtp_sh_backward with
 * respect to grad_y, used by the force-loss chain). */
cgtp_status cgtp_sh_jvp(int lmax, cgtp_dtype dtype, int64_t E, const void* vec,
                        const void* tangent_vec, void* tangent_y, cgtp_stream stream);

/* out[e] = H_e tangent_vec[e], H_e the Hessian in r of grad_y[e] . Y(r) at
 * r = vec[e]: the derivative of cgtp_sh_backward along tangent_vec with grad_y
 * held fixed.  With grad_y = dE/dY and tangent_vec = cgtp_edge_forces_adjoint
 * of a force cotangent gF, out is dL/dr for L = sum gF . forces, and
 * cgtp_edge_forces(out) = -dL/dpos (the position part of the "higher partial
 * derivatives required to predict interatomic forces", abstract of arXiv
 * 2501.13986; the gradient of dE/dY in Y is zero for a product linear in Y).
 * vec, tangent_vec, out [E, 3]; grad_y [E, (lmax+1)^2]; 0 <= lmax <= 6. */
cgtp_status cgtp_sh_hvp(int lmax, cgtp_dtype dtype, int64_t E, const void* vec,
                        const void* grad_y, const void* tangent_vec, void* out,
                        cgtp_stream stream);

/* ---------------------------------------------------------- forces ------ */
/* Interatomic forces from per-edge energy gradients ("higher partial
 * derivatives required to predict interatomic forces", abstract of arXiv
 * 2501.13986), edge vector r_e = pos[recv] - pos[send]:
 *   forces[i] = -sum_{e: recv e = i} dEdr[e] + sum_{e: send e = i} dEdr[e]
 * dEdr [E, 3], forces [N, 3]; receiver CSR and sender-grouped view. */
cgtp_status cgtp_edge_forces(cgtp_dtype dtype, int64_t N, int64_t E, const int32_t* rowptr,
                             const int32_t* s_rowptr, const int32_t* s_perm, const void* dEdr,
                             void* forces, cgtp_stream stream);
/* Adjoint of cgtp_edge_forces: grad_dEdr[e] = grad_forces[sender e] - grad_forces[recv e]. */
cgtp_status cgtp_edge_forces_adjoint(cgtp_dtype dtype, int64_t N, int64_t E,
                                     const int32_t* rowptr, const int32_t* sender,
                                     const void* grad_forces, void* grad_dEdr, cgtp_stream stream);

/* ------------------------------------------- channel mixing (linear) ---- */
/* Per-irrep channel mixing, the dense 'uvw' contraction of a TFN layer: the
 * pairwise degree convolutions are summed per output degree and the fused
 * layers concatenate degrees so that the channel contractions become dense
 * products whose sizes are multiples of 16, for the tensor cores (NVIDIA
 * SE(3)-Transformer blog, "TFN fusion").  For each instruction j joining
 * input irrep i_in and output irrep i_out of the same l and parity, with the
 * matrix W_j [mul_in][mul_out] (row-major; instructions stored one after
 * another):
 *   out[n, i_out, m, w] += sum_u x[n, i_in, m, u] W_j[u, w]     (m = -l..l)
 * Outputs no instruction reaches are zero.  No normalisation is applied.
 * Rows use the library's layout: irrep blocks in order, [2l+1][mul] inside.
 * A 'uvw' tensor product with one matrix per path (shared by all rows) is the
 * 'uvu' product into one output irrep per path with a shared weight row of
 * ones, followed by this layer with instruction p joining path p's output to
 * the path's target irrep. */
typedef struct cgtp_linear_s* cgtp_linear;
typedef struct {
    int i_in, i_out;
} cgtp_linear_instr;
/* instr NULL: every (i_in, i_out) pair with equal l and parity, input-major.
 * Host only; the handle is immutable and may be shared between threads. */
cgtp_status cgtp_linear_create(cgtp_linear* out, const char* irreps_in, const char* irreps_out,
                               const cgtp_linear_instr* instr, int n_instr, cgtp_dtype dtype);
cgtp_status cgtp_linear_destroy(cgtp_linear lin);
cgtp_status cgtp_linear_info(cgtp_linear lin, int64_t* dim_in, int64_t* dim_out,
                             int64_t* weight_numel, int* n_instr);
/* Instruction j: its irreps and the offset of W_j in the weight vector. */
cgtp_status cgtp_linear_instruction(cgtp_linear lin, int j, int* i_in, int* i_out,
                                    int64_t* weight_offset);
/* Workspace bytes: fwd for cgtp_linear_forward (0: none is used), bwd for
 * cgtp_linear_backward with n rows. */
cgtp_status cgtp_linear_workspace(cgtp_linear lin, int64_t n, size_t* fwd_bytes,
                                  size_t* bwd_bytes);
/* Host query: *tensor_cores = 1 if fp32 and every multiplicity is a multiple
 * of 32 and at most 256 (the tcgen05 path, given a workspace and 16-byte
 * aligned tensors). */
cgtp_status cgtp_linear_path(cgtp_linear lin, int* tensor_cores);
/* flags & CGTP_LINEAR_CUDA_CORES: use the CUDA-core kernels. */
#define CGTP_LINEAR_CUDA_CORES 1u
/* CGTP_LINEAR_TEST_WAIT_TIMEOUT, for tests of the failure path only: in the
 * tensor-core forward the MMA issuer's first bounded wait gives up at once;
 * every role leaves its loop, the loader waits for the copies it started, the
 * tensor memory is freed and cgtp_linear_device_status reports 1; out is left
 * incomplete. */
#define CGTP_LINEAR_TEST_WAIT_TIMEOUT 2u
/* out [n, dim_out] = the layer applied to x [n, dim_in] with weights W
 * [weight_numel]; device, caller-owned, `dtype`, out overwritten.  On the
 * tensor-core path (see cgtp_linear_path; needs a 16-byte aligned workspace of
 * at least fwd_bytes, whose contents need not be set) each product runs as
 * TF32 hi*hi + hi*lo + lo*hi on tcgen05 with fp32 accumulation; calls sharing
 * a workspace must not overlap in time.  Otherwise, and for fp64, the CUDA
 * cores.  Asynchronous on `stream`; allocates nothing. */
cgtp_status cgtp_linear_forward(cgtp_linear lin, int64_t n, const void* x, const void* W,
                                void* out, void* workspace, size_t workspace_bytes,
                                unsigned flags, cgtp_stream stream);
/* Gradients for the cotangent grad_out [n, dim_out]: grad_x [n, dim_in]
 * (= grad_out through the transposed matrices, the tensor-core path as in the
 * forward) and grad_W [weight_numel] (= sum over rows of x^T grad_out per
 * instruction, on the tensor cores for tensor-core layers whose output
 * multiplicities are at most 128, else on the CUDA cores; partial sums over
 * fixed row ranges in the workspace, added in fixed order: deterministic);
 * either may be NULL (not computed).  The workspace (at least
 * bwd_bytes, 16-byte aligned) is required when grad_W is requested. */
cgtp_status cgtp_linear_backward(cgtp_linear lin, int64_t n, const void* x, const void* W,
                                 const void* grad_out, void* grad_x, void* grad_W,
                                 void* workspace, size_t workspace_bytes, unsigned flags,
                                 cgtp_stream stream);
/* Device status of the tensor-core kernel: *code = 1 if a bounded wait timed
 * out since the last query (the results of that call are invalid), then
 * cleared.  Synchronous. */
cgtp_status cgtp_linear_device_status(int* code);

/* ------------------------------------------------- 'uvw' product ------ */
/* The 'uvw' tensor product: one matrix W_p [mul_in][mul_out] per path, shared
 * by every row (NVIDIA SE(3)-Transformer blog, "TFN fusion": the pairwise
 * degree convolutions feeding one output degree are summed and the channel
 * contractions become dense products):
 *   out[b, k, m3, w] = sum over paths p -> k of sum_u sum_{m1,m2}
 *                      C_p[m1,m2,m3] x[b, i1(p), m1, u] y[b, i2(p), m2] W_p[u, w]
 * Paths: every (i_in1, i_in2, i_out) with |l1 - l2| <= l3 <= l1 + l2 and
 * p3 = p1 p2, listed in1-major, then in2, then out; W holds their matrices in
 * that order (cgtp_uvw_path gives each offset).  in1 has one multiplicity
 * (mul_in), in2 multiplicity 1 (spherical harmonics).  It runs as the 'uvu'
 * product into one block per path (the "mid" row, dim_mid wide) with unit
 * weights, then the channel mixing of cgtp_linear (tcgen05 for fp32); the
 * convolution sums the blocks per receiver first and mixes once per node.
 * Every call takes a caller-owned device workspace (256-byte aligned, at least
 * cgtp_uvw_workspace() bytes for its row count: B samples or N nodes; contents
 * need not be set; calls sharing one must not overlap in time).  Host only to
 * create; the handle is immutable and may be shared between threads. */
typedef struct cgtp_uvw_s* cgtp_uvw;
cgtp_status cgtp_uvw_create(cgtp_uvw* out, const char* irreps_in1, const char* irreps_in2,
                            const char* irreps_out, cgtp_dtype dtype);
cgtp_status cgtp_uvw_destroy(cgtp_uvw u);
cgtp_status cgtp_uvw_info(cgtp_uvw u, int64_t* dim_in1, int64_t* dim_in2, int64_t* dim_out,
                          int64_t* dim_mid, int64_t* weight_numel, int* n_paths);
/* Path p: l1, l2, l3, its irrep indices and the offset of W_p in W. */
cgtp_status cgtp_uvw_path(cgtp_uvw u, int p, int* l1, int* l2, int* l3, int* i_in1, int* i_in2,
                          int* i_out, int64_t* weight_offset);
/* The product's two parts (borrowed handles, valid while u lives). */
cgtp_status cgtp_uvw_parts(cgtp_uvw u, cgtp_plan* plan, cgtp_linear* lin);
/* Workspace bytes for `rows` rows: forward and backward (the backward's figure
 * covers recomputing the mid blocks when the caller does not pass them). */
cgtp_status cgtp_uvw_workspace(cgtp_uvw u, int64_t rows, size_t* fwd_bytes, size_t* bwd_bytes);
/* out [B, dim_out] from x [B, dim_in1], y [B, dim_in2], W [weight_numel];
 * mid [B, dim_mid] (optional, device) receives the per-path blocks for a later
 * backward.  Asynchronous on `stream`; allocates nothing. */
cgtp_status cgtp_uvw_forward(cgtp_uvw u, int64_t B, const void* x, const void* y, const void* W,
                             void* out, void* mid, void* workspace, size_t workspace_bytes,
                             cgtp_stream stream);
/* grad_x, grad_y, grad_W (each optional) for the cotangent grad_out; mid: the
 * forward's blocks, or NULL to recompute them in the workspace.  grad_W sums
 * over rows in fixed order (deterministic). */
cgtp_status cgtp_uvw_backward(cgtp_uvw u, int64_t B, const void* x, const void* y, const void* W,
                              const void* grad_out, const void* mid, void* grad_x, void* grad_y,
                              void* grad_W, void* workspace, size_t workspace_bytes,
                              cgtp_stream stream);
/* The fused graph convolution with 'uvw' paths: out[n] = scale * mixing of the
 * sum over n's edges of the per-path blocks (graph arguments as
 * cgtp_conv_forward / cgtp_conv_backward; mid is [N, dim_mid]). */
cgtp_status cgtp_uvw_conv_forward(cgtp_uvw u, int64_t N, int64_t E, const int32_t* rowptr,
                                  const int32_t* sender, const void* x, const void* y,
                                  const void* W, double scale, void* out, void* mid,
                                  void* workspace, size_t workspace_bytes, cgtp_stream stream);
cgtp_status cgtp_uvw_conv_backward(cgtp_uvw u, int64_t N, int64_t E, const int32_t* rowptr,
                                   const int32_t* sender, const int32_t* s_rowptr,
                                   const int32_t* s_perm, const int32_t* s_recv, const void* x,
                                   const void* y, const void* W, double scale,
                                   const void* grad_out, const void* mid, void* grad_x,
                                   void* grad_y, void* grad_W, void* workspace,
                                   size_t workspace_bytes, cgtp_stream stream);

/* --------------------------------------------------- radial network ---- */
/* Per-edge tensor-product weights from the radial network: the radial profile
 * of a TFN layer is a fully connected network of the edge length (NVIDIA
 * SE(3)-Transformer blog, "Fused key and value computation").  For edge e with
 * r = |vec[e]|:
 *   b_n  = sqrt(2/cutoff) sin(n pi r / cutoff) / r,  n = 1..n_basis
 *          (at r = 0 its limit sqrt(2/cutoff) n pi / cutoff)
 *   h[e] = silu(b W1),  silu(a) = a / (1 + exp(-a))
 *   w[e] = h[e] W2
 * vec [E,3], W1 [n_basis, hidden], W2 [hidden, n_out], w [E, n_out] and the
 * optional h [E, hidden] (NULL: not stored) are row-major device arrays of
 * `dtype`, owned by the caller; w and h are overwritten.  Limits:
 * 1 <= n_basis <= 32, 1 <= hidden <= 256, n_out >= 1, cutoff > 0; else
 * CGTP_E_ARG.  The last layer runs on the tensor cores (TF32 in three split
 * products, fp32 accuracy) for fp32 with n_basis <= 16, hidden % 8 == 0,
 * hidden <= 64, n_out % 128 == 0, 16-byte aligned vec / W2 / w / h and a
 * workspace of at least cgtp_radial_workspace() bytes (device, caller-owned,
 * 16-byte aligned, contents need not be set; the call packs W2's TF32 parts
 * into it, so calls sharing a workspace must not overlap in time).  Other
 * shapes, fp64, no workspace, or flags & CGTP_RADIAL_CUDA_CORES run it on the
 * CUDA cores.  Asynchronous on `stream`; allocates nothing. */
#define CGTP_RADIAL_CUDA_CORES 1u
/* flags & CGTP_RADIAL_OUT_BF16: w is written as bfloat16 (rounded to nearest
 * even; fp32 inputs only, else CGTP_E_UNSUPPORTED) for plans created with
 * CGTP_PLAN_WEIGHTS_BF16; h stays fp32. */
#define CGTP_RADIAL_OUT_BF16 2u
/* flags & CGTP_RADIAL_OUT_F16: w is written as IEEE binary16 (rounded to
 * nearest even), for plans created with CGTP_PLAN_WEIGHTS_F16; fp32 inputs
 * only; not combined with CGTP_RADIAL_OUT_BF16 (CGTP_E_ARG). */
#define CGTP_RADIAL_OUT_F16 4u
/* CGTP_RADIAL_TEST_WAIT_TIMEOUT, for tests of the failure path only: in the
 * tensor-core forward the MMA issuer's first bounded wait gives up at once;
 * every role then leaves its loop (their own waits are bounded), the kernel
 * waits a grace period for copies in flight, frees its tensor memory and sets
 * the flag cgtp_radial_device_status reports; w is left incomplete. */
#define CGTP_RADIAL_TEST_WAIT_TIMEOUT 8u
cgtp_status cgtp_radial_forward(cgtp_dtype dtype, int64_t E, int n_basis, double cutoff,
                                int hidden, int64_t n_out, const void* vec, const void* W1,
                                const void* W2, void* w, void* h, void* workspace,
                                size_t workspace_bytes, unsigned flags, cgtp_stream stream);
/* Workspace bytes cgtp_radial_forward uses for these sizes (0: it uses none). */
cgtp_status cgtp_radial_workspace(cgtp_dtype dtype, int n_basis, int hidden, int64_t n_out,
                                  size_t* bytes);
/* Vector-Jacobian product of cgtp_radial_forward's w for the cotangent grad_w
 * [E, n_out]: grad_vec [E,3] (edge vectors; zero for r = 0, where the basis is
 * flat), grad_W1 [n_basis, hidden], grad_W2 [hidden, n_out], each optional
 * (NULL: not computed), all `dtype`, device, caller-owned, overwritten.  Chain
 * rule: gh = grad_w W2^T, gpre = gh silu'(b W1), grad_W2 = h^T grad_w,
 * grad_W1 = b^T gpre, grad_vec = (gpre W1^T . db/dr) vec / r.  The sums over
 * edges are per-CTA partial rows in `workspace` (device, caller-owned, 16-byte
 * aligned, at least cgtp_radial_backward_workspace() bytes; contents need not
 * be set) added in fixed order, so results are deterministic.  Same size
 * limits as the forward.  gh = grad_w W2^T runs on the tensor cores (TF32
 * split products, fp32 accuracy) when the forward's tensor-core conditions
 * hold and flags lacks CGTP_RADIAL_CUDA_CORES.  grad_W2 = h^T grad_w runs on
 * the tensor cores too (the same split products, partial sums over 256-row
 * segments added in fp32) for fp32 with hidden a multiple of 32 up to 128,
 * n_out a multiple of 128 up to 16384, at most 16 basis functions, a 16-byte
 * aligned grad_w and no CGTP_RADIAL_CUDA_CORES; otherwise on the CUDA cores.
 * Asynchronous on `stream`; allocates nothing. */
cgtp_status cgtp_radial_backward(cgtp_dtype dtype, int64_t E, int n_basis, double cutoff,
                                 int hidden, int64_t n_out, const void* vec, const void* W1,
                                 const void* W2, const void* grad_w, void* grad_vec,
                                 void* grad_W1, void* grad_W2, void* workspace,
                                 size_t workspace_bytes, unsigned flags, cgtp_stream stream);
/* Workspace bytes cgtp_radial_backward needs for these sizes. */
cgtp_status cgtp_radial_backward_workspace(cgtp_dtype dtype, int64_t E, int n_basis, int hidden,
                                           int64_t n_out, size_t* bytes);
/* Host query: *tensor_cores = 1 if cgtp_radial_forward with these sizes (and
 * 16-byte aligned pointers, a large enough workspace, flags 0) takes the
 * tensor-core path, else 0. */
cgtp_status cgtp_radial_path(cgtp_dtype dtype, int n_basis, int hidden, int64_t n_out,
                             int* tensor_cores);
/* Reads and clears the radial kernels' device error flag (synchronous): 0, or
 * 1 when a bounded wait of the tensor-core kernel timed out (its output is then
 * incomplete). */
cgtp_status cgtp_radial_device_status(int* code);

/* ------------------------------------------------------------ misc ------ */
const char* cgtp_status_str(cgtp_status s);
/* CUDA error code behind the calling thread's last CGTP_E_CUDA / CGTP_E_COMPILE. */
cgtp_status cgtp_last_cuda_error(int* cuda_err);
/* Text of the calling thread's last error (NVRTC log, argument detail). */
const char* cgtp_last_error_message(void);
/* Number of kernel launches this process has issued through the library. */
int64_t cgtp_launch_count(void);

/* Measurement support (the pages have no counterpart): the roofline of the
 * CUDA-core kernels takes the FMA-pipe throughput of the device as its peak,
 * and this probe measures it instead of deriving it from unit counts.  Launches
 * `blocks` CTAs of `threads` threads (a multiple of 32, at most 1024); each
 * thread runs 8 independent chains of `iters` dependent fused multiply-adds in
 * `dtype` (packed = 1: fp32 pairs, one fma.rn.f32x2 per step) and stores one
 * 8-byte word to sink[blockIdx * threads + threadIdx] (device, caller-owned,
 * 8-byte aligned, blocks * threads words).  *flops (optional, host) receives the
 * floating-point operations the launch performs (2 per FMA).  Asynchronous on
 * `stream`: time it with events on that stream.  CGTP_E_ARG on bad sizes. */
cgtp_status cgtp_fma_probe(cgtp_dtype dtype, int packed, int64_t blocks, int threads,
                           int64_t iters, void* sink, int64_t* flops, cgtp_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* CGTP_H */
