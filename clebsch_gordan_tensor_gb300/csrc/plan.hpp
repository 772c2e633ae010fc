// Internal plan representation of the CG tensor-product library.
//
// A plan is the "static analysis at model compile-time" of "An Efficient Sparse
// Kernel Generator for O(3)-Equivariant Deep Networks" (abstract): it fixes the
// irreps, the paths and their real CG coefficients, and lays the per-edge work
// out so that every operand of one channel group lives in registers and the
// contraction is one long unrolled stream of fused multiply-adds.
#pragma once

#include <cstdint>
#include <map>
#include <memory>
#include <mutex>
#include <sstream>
#include <string>
#include <vector>

#include "cgtp.h"

namespace cgtp {

struct Irrep {
    int mul, l, parity;  // parity +1 (e) / -1 (o)
};

struct Path {
    int i1, i2, i3;  // irrep indices
    int l1, l2, l3;
    int r1;  // first x row (units of mul) of the in1 block
    int o2;  // first element of the in2 block inside a y row
    int r3;  // first out row (units of mul) of the out block
    std::vector<double> cg;  // dense [(2l1+1)][(2l2+1)][(2l3+1)]
};

// One entry of the per-edge matrix T_p[m1, m3] = sum_m2 C_p[m1, m2, m3] y[o2 + m2].
struct TEntry {
    int path, m1, m3;                           // m indices 0..2l
    std::vector<std::pair<int, double>> terms;  // (y element, coefficient)
};

// A loaded, compiled kernel module (one per plan and module kind).
struct Module;

struct Plan {
    std::string s1, s2, so;
    std::vector<Irrep> in1, in2, out;
    std::vector<Path> paths;
    std::vector<TEntry> T;  // grouped by path, in path order
    int mul = 0;
    int nx = 0, no = 0;     // rows per channel of x and out
    int ny = 0;             // y row width
    int64_t dimx = 0, dimy = 0, dimo = 0, wdim = 0;
    int maxterms = 1;
    cgtp_dtype dtype = CGTP_F32;
    cgtp_wmode wmode = CGTP_W_PER_EDGE;
    bool w_bf16 = false;  // weights stored as bfloat16 (fp32 arithmetic)
    bool w_f16 = false;   // weights stored as IEEE binary16 (fp32 arithmetic)
    bool w16() const { return w_bf16 || w_f16; }
    unsigned flags = 0;

    // launch geometry (fixed at plan creation)
    int cpt = 1;    // channels per thread
    int nch = 0;    // channel groups = mul / cpt
    int lanes = 0;  // threads per work slot (power of two <= 32, or multiple of 32)
    int slots = 0;  // slots per CTA
    int block = 0;  // threads per CTA
    // staged (TMA) kernels: one slot of `lanes` threads per CTA
    bool staged = false;
    int stages_f = 3, stages_b = 3;  // TMA ring depths (forward, backward)
    bool w_direct_f = false, w_direct_b = false;  // weights bypass the ring
    size_t fwd_smem = 0, bwd_smem = 0;  // dynamic shared memory per CTA
    int minb_b = 1;  // backward: resident CTAs per SM the register budget must allow
    // backward: a second warp per CTA computes grad_y while the first computes
    // grad_x and grad_w (one path group of one warp)
    bool gy_warp = false;
    bool test_wait0 = false;  // test only: the first wait of each CTA gives up at once
    int bwd_threads() const { return ((int)bwd_groups.size() + (gy_warp ? 1 : 0)) * lanes; }
    // warp groups of the staged kernels: each group of `lanes` threads runs the
    // generated stream of a subset of paths (longest-processing-time split)
    std::vector<std::vector<int>> fwd_groups, bwd_groups;

    std::mutex mu;
    std::map<std::string, std::shared_ptr<Module>> modules;

    std::string kernel_source() const;  // full NVRTC source of the TP module
    void gen_groups(std::ostringstream& g, const std::vector<int>& k0, bool f64) const;
};

// plan.cpp
cgtp_status build_plan(Plan& p, const char* s1, const char* s2, const char* so,
                       const cgtp_instr* instr, int n_instr, std::string& err);
// "16x0e+16x1o" -> irreps; false (with a message) on a syntax error.
bool parse_irreps(const char* s, std::vector<Irrep>& out, std::string& err);
// Real-basis CG tensor (dense, layout as Path::cg); false if the triangle fails.
bool real_cg(int l1, int l2, int l3, std::vector<double>& out);

}  // namespace cgtp
