// Host planner of the CG tensor-product library: irreps, paths, real CG
// coefficients, and the per-plan CUDA source handed to NVRTC.
//
// "static analysis at model compile-time ... break the tensor product into a
// series of smaller kernels with operands that fit entirely into registers ...
// emit long arithmetic instruction streams" ("An Efficient Sparse Kernel
// Generator for O(3)-Equivariant Deep Networks", abstract).  Here the analysis
// produces, per plan, one fully unrolled stream per direction in which every
// CG coefficient is an immediate and every operand index is a constant.
#include <algorithm>
#include <cmath>
#include <complex>
#include <cstdio>
#include <cstring>
#include <sstream>

#include "plan.hpp"

namespace cgtp {

extern const char* kTpKernelsSource;  // tp_kernels.cuh, embedded at build time

static constexpr int kMaxL = 6;

// ------------------------------------------------------------------ irreps

bool parse_irreps(const char* s, std::vector<Irrep>& out, std::string& err) {
    out.clear();
    if (!s) {
        err = "irreps string is NULL";
        return false;
    }
    std::string str(s);
    size_t pos = 0;
    while (pos <= str.size()) {
        size_t plus = str.find('+', pos);
        std::string tok = str.substr(pos, plus == std::string::npos ? std::string::npos : plus - pos);
        tok.erase(std::remove_if(tok.begin(), tok.end(), [](char c) { return c == ' '; }), tok.end());
        int mul = 1, l = -1;
        char par = 0;
        size_t xp = tok.find('x');
        std::string body = tok;
        if (xp != std::string::npos) {
            if (xp == 0 || sscanf(tok.substr(0, xp).c_str(), "%d", &mul) != 1 || mul <= 0) {
                err = "bad multiplicity in irrep '" + tok + "'";
                return false;
            }
            for (size_t i = 0; i < xp; ++i)
                if (tok[i] < '0' || tok[i] > '9') {
                    err = "bad multiplicity in irrep '" + tok + "'";
                    return false;
                }
            body = tok.substr(xp + 1);
        }
        if (body.size() < 2) {
            err = "bad irrep '" + tok + "'";
            return false;
        }
        par = body.back();
        std::string ls = body.substr(0, body.size() - 1);
        for (char c : ls)
            if (c < '0' || c > '9') {
                err = "bad degree in irrep '" + tok + "'";
                return false;
            }
        l = atoi(ls.c_str());
        if ((par != 'e' && par != 'o') || l < 0) {
            err = "bad irrep '" + tok + "'";
            return false;
        }
        if (l > kMaxL) {
            err = "degree above 6 in '" + tok + "'";
            return false;
        }
        out.push_back({mul, l, par == 'e' ? 1 : -1});
        if (plus == std::string::npos) break;
        pos = plus + 1;
    }
    return !out.empty();
}

// ------------------------------------------------- Clebsch-Gordan (planner)
//
// Complex CG by the angular-momentum ladder: the top state |J, J> of the
// coupled pair is the unit vector annihilated by J+ = J1+ + J2+ with positive
// <j1 j1; j2 J-j1 | J J> (Condon-Shortley), and each lower |J, M-1> is
// J- |J, M> / sqrt(J(J+1) - M(M-1)).

static double ladder(int j, int m, int dm) {  // <j m+dm | J(dm) | j m>
    return std::sqrt(double(j * (j + 1) - m * (m + dm)));
}

// tab[(m1 + j1) * (2J+1) + (M + J)] = <j1 m1 j2 M-m1 | J M>
static void complex_cg_ladder(int j1, int j2, int J, std::vector<double>& tab) {
    const int d1 = 2 * j1 + 1, dJ = 2 * J + 1;
    tab.assign((size_t)d1 * dJ, 0.0);
    auto at = [&](int m1, int M) -> double& { return tab[(size_t)(m1 + j1) * dJ + (M + J)]; };
    // top state
    const int lo = std::max(-j1, J - j2);
    std::vector<double> a(d1, 0.0);
    a[lo + j1] = 1.0;
    for (int k = lo + 1; k <= j1; ++k)  // coefficient of |k, J+1-k> in J+|J J> vanishes
        a[k + j1] = -a[k - 1 + j1] * ladder(j1, k - 1, +1) / ladder(j2, J - k, +1);
    double nrm = 0;
    for (double v : a) nrm += v * v;
    nrm = std::sqrt(nrm);
    const double sgn = a[2 * j1] >= 0 ? 1.0 : -1.0;
    for (int m1 = -j1; m1 <= j1; ++m1) at(m1, J) = sgn * a[m1 + j1] / nrm;
    // lower
    for (int M = J; M > -J; --M) {
        const double cJ = ladder(J, M, -1);
        for (int m1 = -j1; m1 <= j1; ++m1) {
            const int m2 = M - 1 - m1;
            if (m2 < -j2 || m2 > j2) continue;
            double v = 0;
            if (m1 + 1 <= j1 && std::abs(M - m1 - 1) <= j2) v += at(m1 + 1, M) * ladder(j1, m1 + 1, -1);
            if (std::abs(M - m1) <= j2) v += at(m1, M) * ladder(j2, M - m1, -1);
            at(m1, M - 1) = v / cJ;
        }
    }
}

// The real spherical-harmonic basis vector of real index m as a combination of
// complex ones: up to two (complex m, weight) terms.
//   m > 0: (|-m> + (-1)^m |m>) / sqrt2,  m = 0: |0>,  m < 0: i (|m> - (-1)^m |-m>) / sqrt2
struct CTerm {
    int mc;
    std::complex<double> c;
};
static int real_basis(int m, CTerm out[2]) {
    const double r = 1.0 / std::sqrt(2.0);
    const double s = (std::abs(m) % 2) ? -1.0 : 1.0;
    if (m == 0) {
        out[0] = {0, 1.0};
        return 1;
    }
    if (m > 0) {
        out[0] = {-m, r};
        out[1] = {m, s * r};
        return 2;
    }
    out[0] = {m, std::complex<double>(0, r)};
    out[1] = {-m, std::complex<double>(0, -s * r)};
    return 2;
}

bool real_cg(int l1, int l2, int l3, std::vector<double>& out) {
    const int d1 = 2 * l1 + 1, d2 = 2 * l2 + 1, d3 = 2 * l3 + 1;
    out.assign((size_t)d1 * d2 * d3, 0.0);
    if (l3 < std::abs(l1 - l2) || l3 > l1 + l2) return false;
    std::vector<double> tab;
    complex_cg_ladder(l1, l2, l3, tab);
    const int dJ = 2 * l3 + 1;
    std::vector<std::complex<double>> z((size_t)d1 * d2 * d3);
    double mre = 0, mim = 0;
    for (int a = -l1; a <= l1; ++a) {
        CTerm A[2];
        const int na = real_basis(a, A);
        for (int b = -l2; b <= l2; ++b) {
            CTerm B[2];
            const int nb = real_basis(b, B);
            for (int c = -l3; c <= l3; ++c) {
                CTerm Cc[2];
                const int nc = real_basis(c, Cc);
                std::complex<double> acc = 0;
                for (int i = 0; i < na; ++i)
                    for (int j = 0; j < nb; ++j)
                        for (int k = 0; k < nc; ++k) {
                            if (A[i].mc + B[j].mc != Cc[k].mc) continue;
                            const double cg = tab[(size_t)(A[i].mc + l1) * dJ + (Cc[k].mc + l3)];
                            acc += Cc[k].c * cg * std::conj(A[i].c) * std::conj(B[j].c);
                        }
                const size_t idx = ((size_t)(a + l1) * d2 + (b + l2)) * d3 + (c + l3);
                z[idx] = acc;
                mre = std::max(mre, std::abs(acc.real()));
                mim = std::max(mim, std::abs(acc.imag()));
            }
        }
    }
    const bool im = mim > mre;
    double sign = 0;
    for (size_t i = 0; i < z.size(); ++i) {
        double v = im ? z[i].imag() : z[i].real();
        if (std::abs(v) < 1e-14) v = 0;
        if (sign == 0 && v != 0) sign = v > 0 ? 1 : -1;
        out[i] = v;
    }
    for (double& v : out) v *= sign;
    return true;
}

// ---------------------------------------------------------------- planning

static int next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

cgtp_status build_plan(Plan& p, const char* s1, const char* s2, const char* so,
                       const cgtp_instr* instr, int n_instr, std::string& err) {
    if (!parse_irreps(s1, p.in1, err) || !parse_irreps(s2, p.in2, err) ||
        !parse_irreps(so, p.out, err))
        return CGTP_E_IRREPS;
    p.s1 = s1;
    p.s2 = s2;
    p.so = so;
    for (auto& ir : p.in2)
        if (ir.mul != 1) {
            err = "irreps_in2 must have multiplicity 1 per irrep";
            return CGTP_E_UNSUPPORTED;
        }
    p.mul = p.in1[0].mul;
    for (auto& ir : p.in1)
        if (ir.mul != p.mul) {
            err = "all irreps_in1 entries must share one multiplicity";
            return CGTP_E_UNSUPPORTED;
        }
    for (auto& ir : p.out)
        if (ir.mul != p.mul) {
            err = "irreps_out must share the multiplicity of irreps_in1";
            return CGTP_E_UNSUPPORTED;
        }
    std::vector<int> r1(p.in1.size()), o2(p.in2.size()), r3(p.out.size());
    int acc = 0;
    for (size_t i = 0; i < p.in1.size(); ++i) r1[i] = acc, acc += 2 * p.in1[i].l + 1;
    p.nx = acc;
    acc = 0;
    for (size_t i = 0; i < p.in2.size(); ++i) o2[i] = acc, acc += 2 * p.in2[i].l + 1;
    p.ny = acc;
    acc = 0;
    for (size_t i = 0; i < p.out.size(); ++i) r3[i] = acc, acc += 2 * p.out[i].l + 1;
    p.no = acc;

    auto allowed = [&](int a, int b, int c) {
        const Irrep &A = p.in1[a], &B = p.in2[b], &C = p.out[c];
        return C.l >= std::abs(A.l - B.l) && C.l <= A.l + B.l && C.parity == A.parity * B.parity;
    };
    auto add = [&](int a, int b, int c) {
        Path q{a, b, c, p.in1[a].l, p.in2[b].l, p.out[c].l, r1[a], o2[b], r3[c], {}};
        real_cg(q.l1, q.l2, q.l3, q.cg);
        p.paths.push_back(std::move(q));
    };
    if (instr == nullptr) {
        for (int a = 0; a < (int)p.in1.size(); ++a)
            for (int b = 0; b < (int)p.in2.size(); ++b)
                for (int c = 0; c < (int)p.out.size(); ++c)
                    if (allowed(a, b, c)) add(a, b, c);
    } else {
        if (n_instr < 0) {
            err = "negative instruction count";
            return CGTP_E_ARG;
        }
        for (int k = 0; k < n_instr; ++k) {
            const cgtp_instr& I = instr[k];
            if (I.i_in1 < 0 || I.i_in1 >= (int)p.in1.size() || I.i_in2 < 0 ||
                I.i_in2 >= (int)p.in2.size() || I.i_out < 0 || I.i_out >= (int)p.out.size()) {
                err = "instruction " + std::to_string(k) + " indexes outside the irreps";
                return CGTP_E_PATH;
            }
            if (strncmp(I.mode, "uvu", 3) != 0) {
                err = "instruction " + std::to_string(k) + ": only mode 'uvu' is supported";
                return CGTP_E_UNSUPPORTED;
            }
            if (!allowed(I.i_in1, I.i_in2, I.i_out)) {
                err = "instruction " + std::to_string(k) + " violates the triangle or parity rule";
                return CGTP_E_PATH;
            }
            add(I.i_in1, I.i_in2, I.i_out);
        }
    }
    p.dimx = (int64_t)p.nx * p.mul;
    p.dimy = p.ny;
    p.dimo = (int64_t)p.no * p.mul;
    p.wdim = (int64_t)p.paths.size() * p.mul;

    // T entries
    p.maxterms = 1;
    for (int q = 0; q < (int)p.paths.size(); ++q) {
        const Path& P = p.paths[q];
        const int d1 = 2 * P.l1 + 1, d2 = 2 * P.l2 + 1, d3 = 2 * P.l3 + 1;
        for (int a = 0; a < d1; ++a)
            for (int c = 0; c < d3; ++c) {
                TEntry t{q, a, c, {}};
                for (int b = 0; b < d2; ++b) {
                    const double v = P.cg[((size_t)a * d2 + b) * d3 + c];
                    if (v != 0.0) t.terms.push_back({P.o2 + b, v});
                }
                if (!t.terms.empty()) {
                    p.maxterms = std::max(p.maxterms, (int)t.terms.size());
                    p.T.push_back(std::move(t));
                }
            }
    }

    if (p.maxterms > 4 || p.ny > 255) {
        err = "CG term table exceeds the packed per-thread layout (more than 4 terms or y wider than 255)";
        return CGTP_E_UNSUPPORTED;
    }

    // launch geometry
    // fp32: two channels per lane (packed f32x2) when that still fills whole
    // warps; otherwise one.  fp64: one channel per lane.
    if (p.dtype == CGTP_F32 && p.mul % 64 == 0)
        p.cpt = 2;
    else if (p.dtype == CGTP_F32 && p.mul % 32 != 0 && p.mul % 2 == 0)
        p.cpt = 2;
    else
        p.cpt = 1;
    p.nch = p.mul / p.cpt;
    p.lanes = p.nch <= 32 ? next_pow2(p.nch) : ((p.nch + 31) / 32) * 32;
    if (p.lanes > 1024) {
        err = "multiplicity too large (more than 1024 channel groups)";
        return CGTP_E_UNSUPPORTED;
    }
    p.slots = std::max(1, 128 / p.lanes);
    if (p.lanes > 32) p.slots = std::min(p.slots, 15);
    const int nt = (int)p.T.size();
    const size_t vr = p.cpt == 2 ? 8 : (p.dtype == CGTP_F64 ? 8 : 4);
    auto smem = [&](int slots) {
        const size_t ntp = std::max(4, (nt + 3) / 4 * 4);
        const size_t nyp = next_pow2(std::max(1, p.ny));
        const size_t real = p.dtype == CGTP_F64 ? 8 : 4;
        return slots * (ntp * vr + nyp * real + (p.lanes > 32 ? (p.lanes / 32) * nyp * real : 0));
    };
    while (p.slots > 1 && smem(p.slots) > 40 * 1024) --p.slots;
    if (smem(p.slots) > 40 * 1024) {
        err = "too many CG entries for the shared-memory staging of one work slot";
        return CGTP_E_UNSUPPORTED;
    }
    p.block = p.slots * p.lanes;

    // staged kernels: whole warps of full channel groups, 16-byte rows
    const size_t es = p.dtype == CGTP_F64 ? 8 : 4;
    const size_t WB = (size_t)p.wdim * (p.w16() ? 2 : es), XB = (size_t)p.dimx * es,
                 GB = (size_t)p.dimo * es,
                 YB = (size_t)p.ny * es;
    const bool rows16 = WB % 16 == 0 && XB % 16 == 0 && GB % 16 == 0 && YB % 16 == 0;
    if (p.nch == p.lanes && p.lanes % 32 == 0 && rows16 && !p.paths.empty()) {
        // per-path costs in FMA-pipe cycles per channel group
        std::vector<double> cf(p.paths.size(), 0.0), cb(p.paths.size(), 0.0);
        std::vector<int> nTp(p.paths.size(), 0), nnzp(p.paths.size(), 0);
        for (auto& t : p.T) {
            nTp[t.path] += 1;
            nnzp[t.path] += (int)t.terms.size();
        }
        for (size_t q = 0; q < p.paths.size(); ++q) {
            const int d1 = 2 * p.paths[q].l1 + 1, d3 = 2 * p.paths[q].l3 + 1;
            cf[q] = nTp[q] + std::min(d1, d3);
            cb[q] = 2.0 * (nTp[q] + 3 * d1) + 2.0 * nTp[q] + nnzp[q];
        }
        // flags (0 = automatic): bits 0-3 forward warp groups, 4-7 backward
        // warp groups, 8-11 forward ring depth, 12-15 backward ring depth
        const int ovr_gf = (int)(p.flags & 15u), ovr_gb = (int)((p.flags >> 4) & 15u);
        const int ovr_sf = (int)((p.flags >> 8) & 15u), ovr_sb = (int)((p.flags >> 12) & 15u);
        auto lpt = [&](const std::vector<double>& c, int G) {
            std::vector<int> order(c.size());
            for (size_t i = 0; i < order.size(); ++i) order[i] = (int)i;
            std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return c[a] > c[b]; });
            std::vector<std::vector<int>> grp(G);
            std::vector<double> load(G, 0.0);
            for (int q : order) {
                int j = (int)(std::min_element(load.begin(), load.end()) - load.begin());
                grp[j].push_back(q);
                load[j] += c[q];
            }
            for (auto& v : grp) std::sort(v.begin(), v.end());
            return grp;
        };
        p.fwd_groups = lpt(cf, std::min(4, ovr_gf ? ovr_gf : 1));
        p.bwd_groups = lpt(cb, p.wmode == CGTP_W_SHARED ? 1 : std::min(4, ovr_gb ? ovr_gb : 1));
        // Ring depth and groups: on the 10k-atom convolution the fastest shape
        // was one warp group per CTA with a 2-deep ring (more resident CTAs beat
        // deeper prefetch); flags override both.
        const size_t stat = (size_t)std::max(4, (nt + 3) / 4 * 4) * es + 2048;
        // Weights loaded by the lanes (prefetched one edge ahead in registers)
        // instead of through the ring: default for the backward of plans with
        // two channels per lane (a lane's weight pair is one 8-byte load per
        // path, and the ring then carries only the gathered gradient row), not
        // for one channel per lane (a 4-byte load per path: the ring's one
        // bulk copy of the row measured 9% faster on the 32-channel TFN
        // layer) nor for the forward (its registers limit residency first).
        // Flag bit 16 turns it on for the forward (single warp group only),
        // bit 17 off for the backward.
        p.w_direct_f = ((p.flags >> 16) & 1u) && p.fwd_groups.size() == 1;
        p.w_direct_b = !((p.flags >> 17) & 1u) && p.cpt == 2 &&
                       p.dtype == CGTP_F32;  // fp64 pairs would double the prefetch registers
        // bits 20-23: resident backward CTAs per SM that the register budget
        // must allow (__launch_bounds__ minimum; 0 = no bound)
        p.minb_b = std::max(1, (int)((p.flags >> 20) & 15u));
        // bit 19: grad_y on a warp of its own (one-warp path group, direct weights)
        p.gy_warp = ((p.flags >> 19) & 1u) && p.bwd_groups.size() == 1 && p.lanes == 32;
        p.test_wait0 = (p.flags & CGTP_PLAN_TEST_WAIT_TIMEOUT) != 0;
        const size_t fst = (p.w_direct_f ? 0 : WB) + XB + YB;
        const size_t bst = (p.w_direct_b ? 0 : WB) + GB + YB + 16;
        const size_t budget = 216 * 1024;
        const size_t fbuf = p.fwd_groups.size() > 1 ? GB : 0;
        const size_t bbuf = 2 * XB + (p.bwd_groups.size() > 1 ? XB : 0);
        auto depth = [&](size_t stage, size_t extra, int ctas) {
            const long long room = (long long)(budget / ctas) - (long long)(extra + stat);
            return (int)std::max<long long>(0, std::min<long long>(15, room / (long long)stage));
        };
        int sf = std::min(2, depth(fst, fbuf, 1)), sb = std::min(2, depth(bst, bbuf, 1));
        if (ovr_sf) sf = std::max(2, std::min(ovr_sf, depth(fst, fbuf, 1)));
        if (ovr_sb) sb = std::max(2, std::min(ovr_sb, depth(bst, bbuf, 1)));
        if (sf >= 2 && sb >= 2) {
            p.staged = true;
            p.stages_f = sf;
            p.stages_b = sb;
            p.fwd_smem = sf * fst + fbuf;
            p.bwd_smem = sb * bst + bbuf;
        }
    }
    return CGTP_OK;
}

// -------------------------------------------------------------- code gen

static std::string lit(double v, bool f64) {
    char buf[64];
    if (f64)
        snprintf(buf, sizeof buf, "%.17g", v);
    else
        snprintf(buf, sizeof buf, "%.9gf", (double)(float)v);
    std::string s(buf);
    if (s.find_first_of(".eEn") == std::string::npos) {  // integral: make it a float literal
        if (f64)
            s += ".0";
        else
            s.insert(s.size() - 1, ".0");
    }
    return s;
}

// Emits T(k) loads: with two fp32 channels per lane, T entries are stored as
// duplicated pairs and fetched two at a time with one 128-bit shared load.
struct TLoader {
    int cpt;
    std::vector<bool> loaded;
    std::ostringstream* os;
    bool dup = false;  // entries stored as splatted pairs (two per 128-bit load)
    // T entries are stored as scalars; with two fp32 channels per lane four of
    // them come in one 128-bit shared load and each is splatted into a pair.
    std::string get(int k) {
        if (cpt != 2) return "Ts[" + std::to_string(k) + "]";
        if (dup) {
            const int q = k / 2;
            if (!loaded[q]) {
                *os << "    const ulonglong2 tp" << q << " = Tp[" << q << "];\n";
                loaded[q] = true;
            }
            return "tp" + std::to_string(q) + (k % 2 ? ".y" : ".x");
        }
        const int q = k / 4;
        if (!loaded[q]) {
            *os << "    const float4 tq" << q << " = Tq[" << q << "];\n";
            loaded[q] = true;
        }
        static const char* comp[4] = {".x", ".y", ".z", ".w"};
        return "vsplat(tq" + std::to_string(q) + comp[k % 4] + ")";
    }
};

// Per-group streams of the staged kernels.  Group g of the forward owns the
// paths fwd_groups[g]; its accumulators cover only the output rows those paths
// touch and its x registers only the rows they read.  The backward groups keep
// x rows and partial grad_x for their paths' input rows.
void Plan::gen_groups(std::ostringstream& g, const std::vector<int>& k0, bool f64) const {
    const int ntp = std::max(4, ((int)T.size() + 3) / 4 * 4);
    auto emit_tloader = [&](TLoader& L) { std::fill(L.loaded.begin(), L.loaded.end(), false); };
    // ---------------------------------------------------------------- forward
    g << "template <int GRP> struct FwdG;\n";
    for (size_t gi = 0; gi < fwd_groups.size(); ++gi) {
        const auto& P_ = fwd_groups[gi];
        std::vector<int> rows, xrows;
        for (int q : P_) {
            const Path& P = paths[q];
            for (int c = 0; c < 2 * P.l3 + 1; ++c) rows.push_back(P.r3 + c);
            for (int a = 0; a < 2 * P.l1 + 1; ++a) xrows.push_back(P.r1 + a);
        }
        std::sort(rows.begin(), rows.end());
        rows.erase(std::unique(rows.begin(), rows.end()), rows.end());
        std::sort(xrows.begin(), xrows.end());
        xrows.erase(std::unique(xrows.begin(), xrows.end()), xrows.end());
        std::map<int, int> ri, xi;
        for (size_t i = 0; i < rows.size(); ++i) ri[rows[i]] = (int)i;
        for (size_t i = 0; i < xrows.size(); ++i) xi[xrows[i]] = (int)i;
        g << "template <> struct FwdG<" << gi << "> {\n  static constexpr int NR = "
          << std::max<size_t>(1, rows.size()) << ", NXR = " << std::max<size_t>(1, xrows.size())
          << ";\n";
        g << "  __device__ static __forceinline__ void loadx(VR (&xr)[NXR], const REAL* xs, int ch) {\n";
        for (size_t i = 0; i < xrows.size(); ++i)
            g << "    xr[" << i << "] = lds_v(xs + " << xrows[i] << " * MUL, ch);\n";
        g << "  }\n";
        g << "  template <class FW>\n  __device__ static __forceinline__ void edge(VR (&acc)[NR], "
             "const REAL* __restrict__ Ts, const VR (&xr)[NXR], FW&& W) {\n";
        if (cpt == 2) g << "    const float4* __restrict__ Tq = reinterpret_cast<const float4*>(Ts);\n";
        TLoader L{cpt, std::vector<bool>(ntp / 4 + 1, false), &g};
        for (int q : P_) {
            const Path& P = paths[q];
            const int d1 = 2 * P.l1 + 1, d3 = 2 * P.l3 + 1;
            g << "    { // path " << q << ": " << P.l1 << " x " << P.l2 << " -> " << P.l3 << "\n";
            g << "    const VR w = W(" << q << ");\n";
            emit_tloader(L);
            if (d1 <= d3) {
                for (int a = 0; a < d1; ++a)
                    g << "    const VR z" << a << " = vmul(w, xr[" << xi[P.r1 + a] << "]);\n";
                for (int k = k0[q]; k < k0[q + 1]; ++k) {
                    const std::string t = L.get(k);
                    const int o = ri[P.r3 + T[k].m3];
                    g << "    acc[" << o << "] = vfma(" << t << ", z" << T[k].m1 << ", acc[" << o << "]);\n";
                }
            } else {
                std::vector<bool> started(d3, false);
                for (int k = k0[q]; k < k0[q + 1]; ++k) {
                    const std::string t = L.get(k);
                    const int c = T[k].m3;
                    const std::string xv = "xr[" + std::to_string(xi[P.r1 + T[k].m1]) + "]";
                    if (!started[c]) {
                        g << "    VR t" << c << " = vmul(" << t << ", " << xv << ");\n";
                        started[c] = true;
                    } else {
                        g << "    t" << c << " = vfma(" << t << ", " << xv << ", t" << c << ");\n";
                    }
                }
                for (int c = 0; c < d3; ++c)
                    if (started[c])
                        g << "    acc[" << ri[P.r3 + c] << "] = vfma(w, t" << c << ", acc["
                          << ri[P.r3 + c] << "]);\n";
            }
            g << "    }\n";
        }
        g << "  }\n";
        // combine: group 0 writes every row (zeros where it has none), others add
        g << "  __device__ static __forceinline__ void first(REAL* buf, const VR (&acc)[NR], int ch) {\n";
        for (int r = 0; r < no; ++r) {
            if (ri.count(r))
                g << "    stv(buf + " << r << " * MUL, ch, acc[" << ri[r] << "]);\n";
            else
                g << "    stv(buf + " << r << " * MUL, ch, vzero());\n";
        }
        g << "  }\n  __device__ static __forceinline__ void store(REAL* orow, const VR (&acc)[NR], int ch, "
             "VR sc, int accumulate) {\n";
        for (int r = 0; r < no; ++r) {
            const std::string v = ri.count(r) ? "vmul(acc[" + std::to_string(ri[r]) + "], sc)" : "vzero()";
            g << "    { VR v = " << v << "; if (accumulate) v = vadd(v, ldv_plain(orow + " << r
              << " * MUL, ch)); stv(orow + " << r << " * MUL, ch, v); }\n";
        }
        g << "  }\n  __device__ static __forceinline__ void add(REAL* buf, const VR (&acc)[NR], int ch) {\n";
        for (size_t i = 0; i < rows.size(); ++i)
            g << "    stv(buf + " << rows[i] << " * MUL, ch, vadd(lds_v(buf + " << rows[i]
              << " * MUL, ch), acc[" << i << "]));\n";
        g << "  }\n};\n\n";
    }
    // --------------------------------------------------------------- backward
    const int nyp_ = next_pow2(std::max(1, ny));
    g << "template <int GRP> struct BwdG;\n";
    for (size_t gi = 0; gi < bwd_groups.size(); ++gi) {
        // paths ordered by output block so one block's grad-output pairs are
        // live at a time (they are read from shared memory per path)
        std::vector<int> P_ = bwd_groups[gi];
        std::stable_sort(P_.begin(), P_.end(), [&](int a, int b) {
            return std::make_pair(paths[a].i3, paths[a].i1) < std::make_pair(paths[b].i3, paths[b].i1);
        });
        std::vector<int> xrows;
        for (int q : P_)
            for (int a = 0; a < 2 * paths[q].l1 + 1; ++a) xrows.push_back(paths[q].r1 + a);
        std::sort(xrows.begin(), xrows.end());
        xrows.erase(std::unique(xrows.begin(), xrows.end()), xrows.end());
        std::map<int, int> xi;
        for (size_t i = 0; i < xrows.size(); ++i) xi[xrows[i]] = (int)i;
        // wi[q]: slot of path q in the group's weight registers (direct loads)
        std::map<int, int> wi;
        for (size_t i = 0; i < P_.size(); ++i) wi[P_[i]] = (int)i;
        // grad_y partials of path q: per T entry the two-channel dot of (w x) and
        // g (or x and (w g), whichever needs fewer products), spread over its CG
        // terms into the lane's per-y-element sums
        // flag bit 29: odd paths add into a second set of partials (gyl[NYP +
        // i]), halving the dependent chains; bit 30: a path's dots are all
        // formed before their CG terms are spread
        const bool gy_split = (flags >> 29) & 1u, dots_first = (flags >> 30) & 1u;
        auto emit_gy = [&](int q, int slot) {
            const Path& P = paths[q];
            const int d1 = 2 * P.l1 + 1, d3 = 2 * P.l3 + 1;
            const bool zx = d1 <= d3;
            const int gofs = gy_split && (slot & 1) ? nyp_ : 0;
            if (zx) {
                for (int a = 0; a < d1; ++a)
                    g << "      const VR z" << a << " = vmul(w, xr[" << xi[P.r1 + a] << "]);\n";
            } else {
                for (int c = 0; c < d3; ++c)
                    g << "      const VR z" << c << " = vmul(w, G(" << P.r3 + c << "));\n";
            }
            auto dot = [&](const TEntry& t) {
                const std::string lhs =
                    zx ? "z" + std::to_string(t.m1) : "xr[" + std::to_string(xi[P.r1 + t.m1]) + "]";
                const std::string rhs =
                    zx ? "G(" + std::to_string(P.r3 + t.m3) + ")" : "z" + std::to_string(t.m3);
                return "vdot(" + lhs + ", " + rhs + ")";
            };
            auto spread = [&](const TEntry& t, const std::string& d, const char* ind) {
                for (auto& term : t.terms)
                    g << ind << "gyl[" << term.first + gofs << "] = fma(" << lit(term.second, f64)
                      << ", " << d << ", gyl[" << term.first + gofs << "]);\n";
            };
            if (dots_first) {
                for (int k = k0[q]; k < k0[q + 1]; ++k)
                    g << "      const REAL d" << k - k0[q] << " = " << dot(T[k]) << ";\n";
                for (int k = k0[q]; k < k0[q + 1]; ++k)
                    spread(T[k], "d" + std::to_string(k - k0[q]), "      ");
            } else {
                for (int k = k0[q]; k < k0[q + 1]; ++k) {
                    g << "      { const REAL d = " << dot(T[k]) << ";\n";
                    spread(T[k], "d", "        ");
                    g << "      }\n";
                }
            }
        };
        g << "template <> struct BwdG<" << gi << "> {\n  static constexpr int NXR = "
          << std::max<size_t>(1, xrows.size()) << ", NPW = " << std::max<size_t>(1, P_.size())
          << ";\n";
        // calls f(slot, path) for every path of the group
        g << "  template <class F> __device__ static __forceinline__ void each_w(F&& f) {\n";
        for (size_t i = 0; i < P_.size(); ++i) g << "    f(" << i << ", " << P_[i] << ");\n";
        g << "  }\n";
        g << "  __device__ static __forceinline__ void loadx(VR (&xr)[NXR], const REAL* xs, int ch) {\n";
        for (size_t i = 0; i < xrows.size(); ++i)
            g << "    xr[" << i << "] = lds_v(xs + " << xrows[i] << " * MUL, ch);\n";
        g << "  }\n";
        // FIX: grad_x and grad_w are both written (mode 1), so the stream has no
        // run-time branch and the whole edge is one block for the scheduler
        g << "  template <bool GY, bool FIX, class FG, class FW>\n  __device__ static __forceinline__ void edge("
             "VR (&gxa)[NXR], REAL (&gyl)[NYP * GYS], const REAL* __restrict__ Ts, const VR (&xr)[NXR],\n"
             "      FG&& G, FW&& W, REAL* __restrict__ gwrow, VR (&gwa)[NP], int ch, VR sc, bool dogx,\n"
             "      int mgw) {\n";
        // flag bit 27 (T_DUP_B) stores the backward's T entries as splatted pairs
        // (two per 128-bit load, no splat in the stream); scalar entries (four
        // per load) are the default.
        const bool tdup = cpt == 2 && ((flags >> 27) & 1u);
        if (cpt == 2) g << "    const float4* __restrict__ Tq = reinterpret_cast<const float4*>(Ts);\n";
        if (tdup) g << "    const ulonglong2* __restrict__ Tp = reinterpret_cast<const ulonglong2*>(Ts);\n";
        TLoader L{cpt, std::vector<bool>(ntp / 2 + 1, false), &g, tdup};
        for (int q : P_) {
            const Path& P = paths[q];
            const int d1 = 2 * P.l1 + 1, d3 = 2 * P.l3 + 1;
            g << "    { // path " << q << ": " << P.l1 << " x " << P.l2 << " -> " << P.l3 << "\n";
            g << "    const VR w = W(" << wi[q] << ", " << q << ");\n";
            emit_tloader(L);
            // h[m1] = sum_m3 T[m1,m3] g[m3]; entries ordered m3-major to interleave chains
            std::vector<int> ks;
            for (int k = k0[q]; k < k0[q + 1]; ++k) ks.push_back(k);
            std::stable_sort(ks.begin(), ks.end(), [&](int a, int b) { return T[a].m3 < T[b].m3; });
            // scalar entries: load all T of the path first (four per 128-bit
            // load); splatted pairs are loaded where first used (two per load,
            // twice the registers otherwise)
            if (!tdup)
                for (int k = k0[q]; k < k0[q + 1]; ++k) L.get(k);
            std::vector<bool> hs(d1, false);
            for (int k : ks) {
                const std::string t = L.get(k);
                const int a = T[k].m1;
                const std::string gv = "G(" + std::to_string(P.r3 + T[k].m3) + ")";
                if (!hs[a]) {
                    g << "    VR h" << a << " = vmul(" << t << ", " << gv << ");\n";
                    hs[a] = true;
                } else {
                    g << "    h" << a << " = vfma(" << t << ", " << gv << ", h" << a << ");\n";
                }
            }
            g << "    if (FIX || dogx) {\n";
            for (int a = 0; a < d1; ++a)
                if (hs[a])
                    g << "      gxa[" << xi[P.r1 + a] << "] = vfma(w, h" << a << ", gxa["
                      << xi[P.r1 + a] << "]);\n";
            g << "    }\n    if (FIX || mgw) {\n      VR s = vzero();\n";
            for (int a = 0; a < d1; ++a)
                if (hs[a]) g << "      s = vfma(xr[" << xi[P.r1 + a] << "], h" << a << ", s);\n";
            g << "      GWOUT_M(" << q << ", s, FIX ? 1 : mgw);\n    }\n";
            g << "    if (GY) {\n";
            emit_gy(q, wi[q]);
            g << "    }\n    }\n";
        }
        g << "  }\n";
        // grad_y alone (the CG coefficients are immediates: no T, no y), for
        // the CTA's grad-y warp
        g << "  template <class FG, class FW>\n  __device__ static __forceinline__ void edge_gy("
             "REAL (&gyl)[NYP * GYS], const VR (&xr)[NXR], FG&& G, FW&& W) {\n";
        for (int q : P_) {
            const Path& P = paths[q];
            g << "    { // path " << q << ": " << P.l1 << " x " << P.l2 << " -> " << P.l3 << "\n";
            g << "    const VR w = W(" << wi[q] << ", " << q << ");\n";
            emit_gy(q, wi[q]);
            g << "    }\n";
        }
        g << "  }\n";
        g << "  __device__ static __forceinline__ void first(REAL* buf, const VR (&gxa)[NXR], int ch) {\n";
        for (int r = 0; r < nx; ++r) {
            if (xi.count(r))
                g << "    stv(buf + " << r << " * MUL, ch, gxa[" << xi[r] << "]);\n";
            else
                g << "    stv(buf + " << r << " * MUL, ch, vzero());\n";
        }
        g << "  }\n  __device__ static __forceinline__ void store(REAL* orow, const VR (&gxa)[NXR], int ch, "
             "VR sc, int mode) {\n";
        for (int r = 0; r < nx; ++r) {
            const std::string v = xi.count(r) ? "vmul(gxa[" + std::to_string(xi[r]) + "], sc)" : "vzero()";
            g << "    { VR v = " << v << "; if (mode == 2) v = vadd(v, ldv_plain(orow + " << r
              << " * MUL, ch)); stv(orow + " << r << " * MUL, ch, v); }\n";
        }
        g << "  }\n  __device__ static __forceinline__ void add(REAL* buf, const VR (&gxa)[NXR], int ch) {\n";
        for (size_t i = 0; i < xrows.size(); ++i)
            g << "    stv(buf + " << xrows[i] << " * MUL, ch, vadd(lds_v(buf + " << xrows[i]
              << " * MUL, ch), gxa[" << i << "]));\n";
        g << "  }\n};\n\n";
    }
}

std::string Plan::kernel_source() const {
    const bool f64 = dtype == CGTP_F64;
    const int nt = (int)T.size();
    const int ntp = std::max(4, (nt + 3) / 4 * 4);
    const int nyp = next_pow2(std::max(1, ny));
    std::ostringstream os;
    os << "// generated for " << s1 << " (x) " << s2 << " -> " << so << ", " << paths.size()
       << " uvu paths, " << (f64 ? "fp64" : "fp32") << "\n";
    os << "#define REAL " << (f64 ? "double" : "float") << "\n";
    os << "#define IS_F64 " << (f64 ? 1 : 0) << "\n";
    os << "#define CPT " << cpt << "\n#define MUL " << mul << "\n#define NCH " << nch
       << "\n#define LANES " << lanes << "\n#define SLOTS " << slots << "\n#define BLOCK " << block
       << "\n#define NX " << nx << "\n#define NY " << ny << "\n#define NYP " << nyp
       << "\n#define NO " << no << "\n#define NP " << paths.size() << "\n#define NT " << nt
       << "\n#define NTP " << ntp << "\n#define MAXTERMS " << maxterms << "\n#define YPF "
       << (ny + lanes - 1) / lanes << "\n";
    os << "#define STAGED " << (staged ? 1 : 0) << "\n#define STAGES_F " << stages_f
       << "\n#define STAGES_B " << stages_b << "\n#define W_DIRECT_F " << (w_direct_f ? 1 : 0)
       << "\n#define W_DIRECT_B " << (w_direct_b ? 1 : 0) << "\n#define W_STORE " << (w_bf16 ? 1 : w_f16 ? 2 : 0)
       << "\n#define T_DUP_B " << ((cpt == 2 && ((flags >> 27) & 1u)) ? 1 : 0) << "\n#define W_BUF2 " << (((flags >> 18) & 1u) ? 0 : 1)
       << "\n#define SHARED_W " << (wmode == CGTP_W_SHARED ? 1 : 0)
       << "\n#define MINB_B " << minb_b << "\n#define GYW " << (gy_warp ? 1 : 0)
       << "\n#define TEST_WAIT0 " << (test_wait0 ? 1 : 0)
       << "\n#define W_ALT " << (((flags >> 28) & 1u) ? 1 : 0)
       << "\n#define GYS " << (((flags >> 29) & 1u) ? 2 : 1)
       << "\n#define GF " << std::max<size_t>(1, fwd_groups.size()) << "\n#define GB "
       << std::max<size_t>(1, bwd_groups.size()) << "\n";
    // T tables
    os << "__device__ const short T_IDX[" << std::max(1, nt * maxterms) << "] = {";
    for (int k = 0; k < nt; ++k)
        for (int q = 0; q < maxterms; ++q)
            os << (q < (int)T[k].terms.size() ? T[k].terms[q].first : 0) << ",";
    if (nt == 0) os << "0";
    os << "};\n";
    os << "__device__ const REAL T_CO[" << std::max(1, nt * maxterms) << "] = {";
    for (int k = 0; k < nt; ++k)
        for (int q = 0; q < maxterms; ++q)
            os << (q < (int)T[k].terms.size() ? lit(T[k].terms[q].second, f64) : (f64 ? "0.0" : "0.0f"))
               << ",";
    if (nt == 0) os << "0";
    os << "};\n";

    std::string tmpl(kTpKernelsSource);
    const std::string marker = "// @@GENERATED@@";
    const size_t cut = tmpl.find(marker);
    std::string head = tmpl.substr(0, cut), tail = tmpl.substr(cut);

    // T entries are grouped by path: k0[q] .. k0[q+1]-1 belong to path q
    std::vector<int> k0(paths.size() + 1, nt);
    {
        int k = 0;
        for (int q = 0; q < (int)paths.size(); ++q) {
            while (k < nt && T[k].path < q) ++k;
            k0[q] = k;
        }
    }

    std::ostringstream g;
    // ---- forward stream
    g << "template <class FX, class FW>\n__device__ __forceinline__ void gen_fwd(VR (&acc)[NO],\n"
         "    const REAL* __restrict__ Ts, FX&& X, FW&& W) {\n";
    if (cpt == 2) g << "    const float4* __restrict__ Tq = reinterpret_cast<const float4*>(Ts);\n";
    {
        TLoader L{cpt, std::vector<bool>(ntp / 4 + 1, false), &g};
        for (int q = 0; q < (int)paths.size(); ++q) {
            const Path& P = paths[q];
            const int d1 = 2 * P.l1 + 1, d3 = 2 * P.l3 + 1;
            g << "  { // path " << q << ": " << P.l1 << " x " << P.l2 << " -> " << P.l3 << "\n";
            g << "    const VR w = W(" << q << ");\n";
            std::fill(L.loaded.begin(), L.loaded.end(), false);  // loads are block-scoped
            if (d1 <= d3) {
                for (int a = 0; a < d1; ++a)
                    g << "    const VR z" << a << " = vmul(w, X(" << P.r1 + a << "));\n";
                for (int k = k0[q]; k < k0[q + 1]; ++k) {
                    const std::string t = L.get(k);
                    const int o = P.r3 + T[k].m3;
                    g << "    acc[" << o << "] = vfma(" << t << ", z" << T[k].m1 << ", acc[" << o << "]);\n";
                }
            } else {
                std::vector<bool> started(d3, false);
                for (int k = k0[q]; k < k0[q + 1]; ++k) {
                    const std::string t = L.get(k);
                    const int c = T[k].m3;
                    const std::string xv = "X(" + std::to_string(P.r1 + T[k].m1) + ")";
                    if (!started[c]) {
                        g << "    VR t" << c << " = vmul(" << t << ", " << xv << ");\n";
                        started[c] = true;
                    } else {
                        g << "    t" << c << " = vfma(" << t << ", " << xv << ", t" << c << ");\n";
                    }
                }
                for (int c = 0; c < d3; ++c)
                    if (started[c])
                        g << "    acc[" << P.r3 + c << "] = vfma(w, t" << c << ", acc[" << P.r3 + c
                          << "]);\n";
            }
            g << "  }\n";
        }
    }
    g << "}\n\n";

    // ---- backward stream
    g << "template <bool GY, class FX, class FG, class FW>\n__device__ __forceinline__ void gen_bwd(\n"
         "    VR (&gxa)[NX], REAL (&gyl)[NYP], const REAL* __restrict__ Ts, FX&& X, FG&& G, FW&& W,\n"
         "    REAL* __restrict__ gwrow, VR (&gwa)[NP], int ch, VR sc, bool dogx, int mgw) {\n";
    if (cpt == 2) g << "    const float4* __restrict__ Tq = reinterpret_cast<const float4*>(Ts);\n";
    {
        TLoader L{cpt, std::vector<bool>(ntp / 4 + 1, false), &g};
        for (int q = 0; q < (int)paths.size(); ++q) {
            const Path& P = paths[q];
            const int d1 = 2 * P.l1 + 1, d3 = 2 * P.l3 + 1;
            g << "  { // path " << q << ": " << P.l1 << " x " << P.l2 << " -> " << P.l3 << "\n";
            g << "    const VR w = W(" << q << ");\n";
            std::fill(L.loaded.begin(), L.loaded.end(), false);  // loads are block-scoped
            // h[m1] = sum_m3 T[m1,m3] g[m3]
            std::vector<bool> hs(d1, false);
            for (int k = k0[q]; k < k0[q + 1]; ++k) {
                const std::string t = L.get(k);
                const int a = T[k].m1;
                const std::string gv = "G(" + std::to_string(P.r3 + T[k].m3) + ")";
                if (!hs[a]) {
                    g << "    VR h" << a << " = vmul(" << t << ", " << gv << ");\n";
                    hs[a] = true;
                } else {
                    g << "    h" << a << " = vfma(" << t << ", " << gv << ", h" << a << ");\n";
                }
            }
            g << "    if (dogx) {\n";
            for (int a = 0; a < d1; ++a)
                if (hs[a])
                    g << "      gxa[" << P.r1 + a << "] = vfma(w, h" << a << ", gxa[" << P.r1 + a
                      << "]);\n";
            g << "    }\n    if (mgw) {\n      VR s = vzero();\n";
            for (int a = 0; a < d1; ++a)
                if (hs[a]) g << "      s = vfma(X(" << P.r1 + a << "), h" << a << ", s);\n";
            g << "      GWOUT(" << q << ", s);\n    }\n";
            // gy partials
            g << "    if (GY) {\n";
            const bool zx = d1 <= d3;
            if (zx) {
                for (int a = 0; a < d1; ++a)
                    g << "      const VR z" << a << " = vmul(w, X(" << P.r1 + a << "));\n";
            } else {
                for (int c = 0; c < d3; ++c)
                    g << "      const VR z" << c << " = vmul(w, G(" << P.r3 + c << "));\n";
            }
            for (int k = k0[q]; k < k0[q + 1]; ++k) {
                const TEntry& t = T[k];
                const std::string lhs =
                    zx ? "z" + std::to_string(t.m1) : "X(" + std::to_string(P.r1 + t.m1) + ")";
                const std::string rhs =
                    zx ? "G(" + std::to_string(P.r3 + t.m3) + ")" : "z" + std::to_string(t.m3);
                g << "      { const REAL d = vdot(" << lhs << ", " << rhs << ");\n";
                for (auto& term : t.terms)
                    g << "        gyl[" << term.first << "] = fma(" << lit(term.second, f64)
                      << ", d, gyl[" << term.first << "]);\n";
                g << "      }\n";
            }
            g << "    }\n  }\n";
        }
    }
    g << "}\n\n";

    if (staged) gen_groups(g, k0, f64);
    return os.str() + head + g.str() + tail;
}

}  // namespace cgtp
