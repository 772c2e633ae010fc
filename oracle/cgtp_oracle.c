/*
 * Oracle for the Clebsch-Gordan tensor product -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct fp64 CPU restatement of what the GPU path
 * computes.  Only tests/, the smoke check and the benchmark's CPU-baseline leg
 * may load this file's library; the product path never does.  It shares no
 * code, header, table or constant generator with the CUDA library.
 *
 * Sources (web pages on the subject):
 *  - "An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks"
 *    (arXiv 2501.13986), abstract: the CG tensor product contracts two dense
 *    feature vectors with a highly structured sparse tensor into a dense output;
 *    it is fused with a subsequent graph convolution; gradient kernels and
 *    higher partial derivatives for interatomic forces.
 *  - NVIDIA SE(3)-Transformer blog, section "TFN fusion": a degree-d feature has
 *    dimension 2d+1; a layer is a sum of pairwise degree convolutions whose
 *    contributions to one output degree are summed.  Section "basis
 *    precomputation": per-edge bases depend on spherical harmonics of the
 *    relative position.
 *
 * The pages print no formula.  Each function below writes out the textbook
 * definition that their statement of the problem implies:
 *  - complex CG by Racah's closed form (exact integer factorials, l <= 6);
 *  - real basis by the standard complex->real spherical-harmonic map;
 *  - real spherical harmonics from associated Legendre functions (no
 *    Condon-Shortley phase in the real functions), "component" normalised;
 *  - the tensor product as the plain sum over paths, channels and nonzero CG
 *    entries; the convolution as the plain sum over a receiver's edges, in
 *    edge order.
 *
 * Layouts (stated, since the pages are silent): feature rows hold irrep blocks
 * in irreps order; inside a block the index is m_index * mul + u (m_index =
 * m + l, channel u fastest).  Spherical-harmonic rows hold blocks l = 0..lmax of
 * width 2l+1.  Weight rows hold one block of mul per path, in path order.
 */
#include <complex.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_LMAX 6

/* ---------------------------------------------------------------- CG ---- */

static uint64_t fact(int n) {
    uint64_t r = 1;
    for (int i = 2; i <= n; ++i) r *= (uint64_t)i;
    return r;
}

/* <l1 m1 l2 m2 | l3 m3> (Condon-Shortley), Racah's closed form:
 *   delta(m3, m1+m2) * sqrt((2 l3+1) (l3+l1-l2)! (l3-l1+l2)! (l1+l2-l3)! / (l1+l2+l3+1)!)
 *   * sqrt((l3+m3)! (l3-m3)! (l1-m1)! (l1+m1)! (l2-m2)! (l2+m2)!)
 *   * sum_k (-1)^k / [k! (l1+l2-l3-k)! (l1-m1-k)! (l2+m2-k)! (l3-l2+m1+k)! (l3-l1-m2+k)!]
 * Factorials are exact 64-bit integers (19! is the largest needed for l <= 6).
 */
static long double cg_complex(int l1, int m1, int l2, int m2, int l3, int m3) {
    if (m3 != m1 + m2) return 0.0L;
    if (l3 < abs(l1 - l2) || l3 > l1 + l2) return 0.0L;
    if (abs(m1) > l1 || abs(m2) > l2 || abs(m3) > l3) return 0.0L;
    long double pre = (long double)(2 * l3 + 1) * (long double)fact(l3 + l1 - l2) *
                      (long double)fact(l3 - l1 + l2) * (long double)fact(l1 + l2 - l3) /
                      (long double)fact(l1 + l2 + l3 + 1);
    long double mterm = (long double)fact(l3 + m3) * (long double)fact(l3 - m3) *
                        (long double)fact(l1 - m1) * (long double)fact(l1 + m1) *
                        (long double)fact(l2 - m2) * (long double)fact(l2 + m2);
    long double s = 0.0L;
    for (int k = 0; k <= l1 + l2 + l3; ++k) {
        int a = l1 + l2 - l3 - k, b = l1 - m1 - k, c = l2 + m2 - k;
        int d = l3 - l2 + m1 + k, e = l3 - l1 - m2 + k;
        if (a < 0 || b < 0 || c < 0 || d < 0 || e < 0) continue;
        long double den = (long double)fact(k) * (long double)fact(a) * (long double)fact(b) *
                          (long double)fact(c) * (long double)fact(d) * (long double)fact(e);
        s += ((k & 1) ? -1.0L : 1.0L) / den;
    }
    return sqrtl(pre) * sqrtl(mterm) * s;
}

/* Exported for the pin against a library CG table. */
double oracle_cg_complex(int l1, int m1, int l2, int m2, int l3, int m3) {
    return (double)cg_complex(l1, m1, l2, m2, l3, m3);
}

/* Row r (real m = r - l) of the map from complex to real spherical harmonics:
 *   real m<0 : (i/sqrt2) (Y^m - (-1)^m Y^-m)
 *   real m=0 : Y^0
 *   real m>0 : (1/sqrt2) (Y^-m + (-1)^m Y^m)
 * A[r][k] with complex index k = mc + l.
 */
static void real_from_complex(int l, long double complex *A /* (2l+1)^2 */) {
    int d = 2 * l + 1;
    long double s2 = 1.0L / sqrtl(2.0L);
    for (int i = 0; i < d * d; ++i) A[i] = 0;
    for (int m = -l; m <= l; ++m) {
        int r = m + l;
        long double sgn = (abs(m) & 1) ? -1.0L : 1.0L;
        if (m < 0) {
            A[r * d + (m + l)] += I * s2;
            A[r * d + (-m + l)] += -I * s2 * sgn;
        } else if (m == 0) {
            A[r * d + l] = 1.0L;
        } else {
            A[r * d + (-m + l)] += s2;
            A[r * d + (m + l)] += s2 * sgn;
        }
    }
}

/* Real-basis CG tensor of the path l1 x l2 -> l3:
 *   C_real[m1,m2,m3] = sum A3[m3,M] C[M; k1,k2] conj(A1[m1,k1]) conj(A2[m2,k2])
 * (the coupling z = C (x (x) y) taken into the real basis, x = A^dagger x_real).
 * The result is purely real or purely imaginary; the nonzero part is kept.
 * Sign convention: the first nonzero entry in (m1, m2, m3) order is positive.
 * Output layout: out[(i1 * d2 + i2) * d3 + i3], i = m + l.
 * Returns 0 if the triangle rule fails (out zeroed), 1 otherwise, -1 on bad l.
 */
int oracle_cg_real(int l1, int l2, int l3, double *out) {
    if (l1 < 0 || l2 < 0 || l3 < 0 || l1 > ORACLE_LMAX || l2 > ORACLE_LMAX || l3 > ORACLE_LMAX)
        return -1;
    int d1 = 2 * l1 + 1, d2 = 2 * l2 + 1, d3 = 2 * l3 + 1;
    memset(out, 0, sizeof(double) * d1 * d2 * d3);
    if (l3 < abs(l1 - l2) || l3 > l1 + l2) return 0;
    long double complex A1[13 * 13], A2[13 * 13], A3[13 * 13];
    real_from_complex(l1, A1);
    real_from_complex(l2, A2);
    real_from_complex(l3, A3);
    long double complex *Cr = malloc(sizeof(long double complex) * d1 * d2 * d3);
    long double maxre = 0, maxim = 0;
    for (int a = 0; a < d1; ++a)
        for (int b = 0; b < d2; ++b)
            for (int c = 0; c < d3; ++c) {
                long double complex acc = 0;
                for (int k1 = 0; k1 < d1; ++k1)
                    for (int k2 = 0; k2 < d2; ++k2) {
                        int M = (k1 - l1) + (k2 - l2);
                        if (M < -l3 || M > l3) continue;
                        long double cg = cg_complex(l1, k1 - l1, l2, k2 - l2, l3, M);
                        if (cg == 0.0L) continue;
                        acc += A3[c * d3 + (M + l3)] * cg * conjl(A1[a * d1 + k1]) *
                               conjl(A2[b * d2 + k2]);
                    }
                Cr[(a * d2 + b) * d3 + c] = acc;
                if (fabsl(creall(acc)) > maxre) maxre = fabsl(creall(acc));
                if (fabsl(cimagl(acc)) > maxim) maxim = fabsl(cimagl(acc));
            }
    int use_im = maxim > maxre;
    long double sign = 0;
    for (int i = 0; i < d1 * d2 * d3; ++i) {
        long double v = use_im ? cimagl(Cr[i]) : creall(Cr[i]);
        if (fabsl(v) < 1e-15L) v = 0;
        if (sign == 0 && v != 0) sign = v > 0 ? 1.0L : -1.0L;
        out[i] = (double)v;
    }
    for (int i = 0; i < d1 * d2 * d3; ++i) out[i] = (double)(sign * out[i]);
    free(Cr);
    return 1;
}

/* --------------------------------------------------- spherical harmonics -- */

/* Q_lm(z) = d^m/dz^m P_l(z), P_l the Legendre polynomial written out as
 *   P_l(z) = 2^-l sum_k (-1)^k C(l,k) C(2l-2k, l) z^(l-2k).
 * The associated Legendre function without the Condon-Shortley phase is
 * (1 - z^2)^(m/2) Q_lm(z).
 */
static double legendre_deriv(int l, int m, double z) {
    double s = 0;
    for (int k = 0; 2 * k <= l; ++k) {
        int p = l - 2 * k; /* power of z */
        if (p < m) continue;
        double coef = (double)(fact(l) / (fact(k) * fact(l - k))) *
                      (double)(fact(2 * l - 2 * k) / (fact(l) * fact(l - 2 * k))) *
                      ((k & 1) ? -1.0 : 1.0);
        /* d^m/dz^m z^p = p!/(p-m)! z^(p-m) */
        coef *= (double)(fact(p) / fact(p - m));
        s += coef * pow(z, p - m);
    }
    return s / pow(2.0, l);
}

/* Component-normalised real spherical harmonic of the unit vector (x,y,z):
 *   Y_l0 = sqrt(2l+1) P_l(z)
 *   Y_lm = sqrt(2 (2l+1) (l-|m|)!/(l+|m|)!) P_l^|m|(z) cos(m phi)      m > 0
 *   Y_lm = sqrt(2 (2l+1) (l-|m|)!/(l+|m|)!) P_l^|m|(z) sin(|m| phi)    m < 0
 * with P_l^m(z) = (1-z^2)^(m/2) Q_lm(z) and the factor (1-z^2)^(m/2) e^{i m phi}
 * = (x + i y)^m for a unit vector.  Sum over m of Y_lm^2 is 2l+1.
 */
static double sh_norm(int l, int am) {
    double n = (double)(2 * l + 1) * (double)fact(l - am) / (double)fact(l + am);
    if (am != 0) n *= 2.0;
    return sqrt(n);
}

static void xy_power(int m, double x, double y, double *re, double *im) {
    double complex w = 1.0;
    for (int i = 0; i < m; ++i) w *= (x + I * y);
    *re = creal(w);
    *im = cimag(w);
}

static void sh_unit(int lmax, double x, double y, double z, double *out) {
    for (int l = 0; l <= lmax; ++l) {
        for (int m = -l; m <= l; ++m) {
            int am = abs(m);
            double re, im;
            xy_power(am, x, y, &re, &im);
            double ang = (m >= 0) ? re : im;
            out[l * l + (m + l)] = sh_norm(l, am) * legendre_deriv(l, am, z) * ang;
        }
    }
}

/* Gradient of the component-normalised real SH (as polynomials in a unit
 * vector u) with respect to u: d/du of Q_lm(z) * Re/Im((x+iy)^m), using
 *   d/dz Q_lm = Q_l,m+1,  d/dx (x+iy)^m = m (x+iy)^(m-1),  d/dy = i m (x+iy)^(m-1).
 */
static void sh_unit_grad(int lmax, double x, double y, double z, double *gx, double *gy,
                         double *gz) {
    for (int l = 0; l <= lmax; ++l) {
        for (int m = -l; m <= l; ++m) {
            int am = abs(m), i = l * l + (m + l);
            double N = sh_norm(l, am);
            double Q = legendre_deriv(l, am, z);
            double dQ = (am + 1 <= l) ? legendre_deriv(l, am + 1, z) : 0.0;
            double re, im, re1 = 0, im1 = 0;
            xy_power(am, x, y, &re, &im);
            if (am > 0) xy_power(am - 1, x, y, &re1, &im1);
            double ang = (m >= 0) ? re : im;
            /* d(x+iy)^m/dx = m (re1 + i im1) ; d/dy = m (i re1 - im1) */
            double dang_dx = (m >= 0) ? am * re1 : am * im1;
            double dang_dy = (m >= 0) ? -am * im1 : am * re1;
            gx[i] = N * Q * dang_dx;
            gy[i] = N * Q * dang_dy;
            gz[i] = N * dQ * ang;
        }
    }
}

/* Y[n, (lmax+1)^2] of vec[n, 3]; vectors are normalised first. */
int oracle_sh(int lmax, int64_t n, const double *vec, double *y) {
    if (lmax < 0 || lmax > ORACLE_LMAX) return -1;
    int dim = (lmax + 1) * (lmax + 1);
    for (int64_t e = 0; e < n; ++e) {
        double x = vec[3 * e], yy = vec[3 * e + 1], z = vec[3 * e + 2];
        double r = sqrt(x * x + yy * yy + z * z);
        sh_unit(lmax, x / r, yy / r, z / r, y + e * dim);
    }
    return 0;
}

/* Chain rule through u = r/|r|:  dY/dr = (grad_u Y) (I - u u^T) / |r|. */
static void sh_jacobian(int lmax, const double *v, double *J /* dim x 3 */) {
    int dim = (lmax + 1) * (lmax + 1);
    double r = sqrt(v[0] * v[0] + v[1] * v[1] + v[2] * v[2]);
    double u[3] = {v[0] / r, v[1] / r, v[2] / r};
    double gx[64], gy[64], gz[64];
    sh_unit_grad(lmax, u[0], u[1], u[2], gx, gy, gz);
    for (int i = 0; i < dim; ++i) {
        double g[3] = {gx[i], gy[i], gz[i]};
        double gu = g[0] * u[0] + g[1] * u[1] + g[2] * u[2];
        for (int k = 0; k < 3; ++k) J[i * 3 + k] = (g[k] - gu * u[k]) / r;
    }
}

/* grad_vec[e] = J(vec[e])^T grad_y[e] */
int oracle_sh_vjp(int lmax, int64_t n, const double *vec, const double *grad_y,
                  double *grad_vec) {
    if (lmax < 0 || lmax > ORACLE_LMAX) return -1;
    int dim = (lmax + 1) * (lmax + 1);
    double J[64 * 3];
    for (int64_t e = 0; e < n; ++e) {
        sh_jacobian(lmax, vec + 3 * e, J);
        for (int k = 0; k < 3; ++k) {
            double s = 0;
            for (int i = 0; i < dim; ++i) s += J[i * 3 + k] * grad_y[e * dim + i];
            grad_vec[3 * e + k] = s;
        }
    }
    return 0;
}

/* tangent_y[e] = J(vec[e]) tangent_vec[e] */
int oracle_sh_jvp(int lmax, int64_t n, const double *vec, const double *tangent_vec,
                  double *tangent_y) {
    if (lmax < 0 || lmax > ORACLE_LMAX) return -1;
    int dim = (lmax + 1) * (lmax + 1);
    double J[64 * 3];
    for (int64_t e = 0; e < n; ++e) {
        sh_jacobian(lmax, vec + 3 * e, J);
        for (int i = 0; i < dim; ++i) {
            double s = 0;
            for (int k = 0; k < 3; ++k) s += J[i * 3 + k] * tangent_vec[3 * e + k];
            tangent_y[e * dim + i] = s;
        }
    }
    return 0;
}

/* Second derivatives of the same polynomials in u: d2/dz2 Q_lm = Q_l,m+2,
 * d2/dx2 (x+iy)^m = m(m-1)(x+iy)^(m-2), d2/dxdy = i m(m-1)(x+iy)^(m-2),
 * d2/dy2 = -m(m-1)(x+iy)^(m-2), d2/dxdz = dQ m (x+iy)^(m-1), d2/dydz =
 * dQ i m (x+iy)^(m-1).  h[i][k] for k = xx, xy, xz, yy, yz, zz; the real
 * part for m >= 0, the imaginary part for m < 0.
 */
static void sh_unit_hess(int lmax, double x, double y, double z, double (*h)[6]) {
    for (int l = 0; l <= lmax; ++l) {
        for (int m = -l; m <= l; ++m) {
            int am = abs(m), i = l * l + (m + l);
            double N = sh_norm(l, am);
            double Q = legendre_deriv(l, am, z);
            double dQ = (am + 1 <= l) ? legendre_deriv(l, am + 1, z) : 0.0;
            double d2Q = (am + 2 <= l) ? legendre_deriv(l, am + 2, z) : 0.0;
            double re, im, re1 = 0, im1 = 0, re2 = 0, im2 = 0;
            xy_power(am, x, y, &re, &im);
            if (am >= 1) xy_power(am - 1, x, y, &re1, &im1);
            if (am >= 2) xy_power(am - 2, x, y, &re2, &im2);
            double complex w0 = re + I * im;
            double complex w1 = (double)am * (re1 + I * im1);
            double complex w2 = (double)am * (double)(am - 1) * (re2 + I * im2);
            double complex d[6] = {Q * w2, Q * I * w2, dQ * w1, -Q * w2, dQ * I * w1, d2Q * w0};
            for (int k = 0; k < 6; ++k) h[i][k] = N * ((m >= 0) ? creal(d[k]) : cimag(d[k]));
        }
    }
}

/* Hessian-vector product of s(r) = grad_y . Y(r/|r|):
 *   out[e] = (d^2 s / dr^2) tangent_vec[e].
 * With f = grad_u (grad_y . P)(u), F its second derivatives in u, rho = |r|,
 * u = r/rho and Pi = I - u u^T (chain rule through u = r/|r|, differentiated
 * twice):
 *   d^2 s/dr_j dr_k = [ (Pi F Pi)_jk - f_j u_k - f_k u_j - (f.u) delta_jk
 *                       + 3 (f.u) u_j u_k ] / rho^2.
 * It is the derivative of oracle_sh_vjp along tangent_vec (grad_y held fixed).
 */
int oracle_sh_hvp(int lmax, int64_t n, const double *vec, const double *grad_y,
                  const double *tangent_vec, double *out) {
    if (lmax < 0 || lmax > ORACLE_LMAX) return -1;
    int dim = (lmax + 1) * (lmax + 1);
    double gx[64], gy[64], gz[64], h[64][6];
    static const int sym[3][3] = {{0, 1, 2}, {1, 3, 4}, {2, 4, 5}};
    for (int64_t e = 0; e < n; ++e) {
        const double *v = vec + 3 * e, *g = grad_y + e * dim, *t = tangent_vec + 3 * e;
        double rho = sqrt(v[0] * v[0] + v[1] * v[1] + v[2] * v[2]);
        double u[3] = {v[0] / rho, v[1] / rho, v[2] / rho};
        sh_unit_grad(lmax, u[0], u[1], u[2], gx, gy, gz);
        sh_unit_hess(lmax, u[0], u[1], u[2], h);
        double f[3] = {0, 0, 0}, F[3][3] = {{0}};
        for (int i = 0; i < dim; ++i) {
            f[0] += g[i] * gx[i];
            f[1] += g[i] * gy[i];
            f[2] += g[i] * gz[i];
            for (int a = 0; a < 3; ++a)
                for (int b = 0; b < 3; ++b) F[a][b] += g[i] * h[i][sym[a][b]];
        }
        double Pi[3][3], PFP[3][3];
        for (int a = 0; a < 3; ++a)
            for (int b = 0; b < 3; ++b) Pi[a][b] = (a == b ? 1.0 : 0.0) - u[a] * u[b];
        for (int a = 0; a < 3; ++a)
            for (int b = 0; b < 3; ++b) {
                double s = 0;
                for (int c = 0; c < 3; ++c)
                    for (int d = 0; d < 3; ++d) s += Pi[a][c] * F[c][d] * Pi[d][b];
                PFP[a][b] = s;
            }
        double fu = f[0] * u[0] + f[1] * u[1] + f[2] * u[2];
        for (int j = 0; j < 3; ++j) {
            double s = 0;
            for (int k = 0; k < 3; ++k) {
                double H = PFP[j][k] - f[j] * u[k] - f[k] * u[j] - (j == k ? fu : 0.0) +
                           3.0 * fu * u[j] * u[k];
                s += H * t[k];
            }
            out[3 * e + j] = s / (rho * rho);
        }
    }
    return 0;
}

/* ------------------------------------------------------ tensor product -- */

/* One 'uvu' path: out block (l3) channel u gets
 *   sum_{m1,m2} C[m1,m2,m3] x[l1 block][m1][u] y[l2 block][m2] w[path][u]. */
typedef struct {
    int l1, l2, l3, mul;
    int64_t off1, off2, off3, offw; /* element offsets inside a row */
} oracle_path;

typedef struct {
    int n;
    const oracle_path *p;
    double **cg; /* per path, dense d1*d2*d3 */
} paths_t;

static int paths_init(paths_t *P, int n, const oracle_path *p) {
    P->n = n;
    P->p = p;
    P->cg = calloc((size_t)(n > 0 ? n : 1), sizeof(double *));
    for (int i = 0; i < n; ++i) {
        int d = (2 * p[i].l1 + 1) * (2 * p[i].l2 + 1) * (2 * p[i].l3 + 1);
        P->cg[i] = malloc(sizeof(double) * d);
        if (oracle_cg_real(p[i].l1, p[i].l2, p[i].l3, P->cg[i]) != 1) return -1;
    }
    return 0;
}

static void paths_free(paths_t *P) {
    for (int i = 0; i < P->n; ++i) free(P->cg[i]);
    free(P->cg);
}

/* acc[out row] += alpha * TP(x row, y row, w row) */
static void tp_row(const paths_t *P, const double *x, const double *y, const double *w,
                   double alpha, double *acc) {
    for (int q = 0; q < P->n; ++q) {
        const oracle_path *p = &P->p[q];
        int d1 = 2 * p->l1 + 1, d2 = 2 * p->l2 + 1, d3 = 2 * p->l3 + 1;
        const double *C = P->cg[q];
        for (int u = 0; u < p->mul; ++u)
            for (int a = 0; a < d1; ++a)
                for (int b = 0; b < d2; ++b)
                    for (int c = 0; c < d3; ++c) {
                        double cv = C[(a * d2 + b) * d3 + c];
                        if (cv == 0.0) continue;
                        acc[p->off3 + c * p->mul + u] += alpha * cv * x[p->off1 + a * p->mul + u] *
                                                         y[p->off2 + b] * w[p->offw + u];
                    }
    }
}

/* Partial contractions of <g, TP(x, y, w)> (the gradient of the tensor product):
 *   gx[l1][m1][u] += alpha sum C y[m2] w[u] g[l3][m3][u]
 *   gy[l2][m2]    += alpha sum C x[m1][u] w[u] g[m3][u]     (summed over u)
 *   gw[p][u]      += alpha sum C x[m1][u] y[m2] g[m3][u]
 * Any of gx, gy, gw may be NULL. */
static void tp_row_grad(const paths_t *P, const double *x, const double *y, const double *w,
                        const double *g, double alpha, double *gx, double *gy, double *gw) {
    for (int q = 0; q < P->n; ++q) {
        const oracle_path *p = &P->p[q];
        int d1 = 2 * p->l1 + 1, d2 = 2 * p->l2 + 1, d3 = 2 * p->l3 + 1;
        const double *C = P->cg[q];
        for (int u = 0; u < p->mul; ++u)
            for (int a = 0; a < d1; ++a)
                for (int b = 0; b < d2; ++b)
                    for (int c = 0; c < d3; ++c) {
                        double cv = C[(a * d2 + b) * d3 + c];
                        if (cv == 0.0) continue;
                        double xv = x[p->off1 + a * p->mul + u], yv = y[p->off2 + b];
                        double wv = w[p->offw + u], gv = g[p->off3 + c * p->mul + u];
                        if (gx) gx[p->off1 + a * p->mul + u] += alpha * cv * yv * wv * gv;
                        if (gy) gy[p->off2 + b] += alpha * cv * xv * wv * gv;
                        if (gw) gw[p->offw + u] += alpha * cv * xv * yv * gv;
                    }
    }
}

/* Standalone tensor product over B rows: out[b] = TP(x[b], y[b], w[b]).
 * w_stride = 0 shares one weight row across all samples. */
int oracle_tp_forward(int n_paths, const oracle_path *paths, int64_t B, int64_t dx, int64_t dy,
                      int64_t dw, int64_t dout, int64_t w_stride, const double *x, const double *y,
                      const double *w, double *out) {
    paths_t P;
    if (paths_init(&P, n_paths, paths)) { paths_free(&P); return -1; }
    (void)dw;
    for (int64_t b = 0; b < B; ++b) {
        double *o = out + b * dout;
        for (int64_t i = 0; i < dout; ++i) o[i] = 0;
        tp_row(&P, x + b * dx, y + b * dy, w + b * w_stride, 1.0, o);
    }
    paths_free(&P);
    return 0;
}

/* Standalone gradient: given g = dL/dout, returns dL/dx, dL/dy, dL/dw (NULL = skip).
 * With w_stride = 0 (shared weights) dL/dw is summed over the rows in order. */
int oracle_tp_backward(int n_paths, const oracle_path *paths, int64_t B, int64_t dx, int64_t dy,
                       int64_t dw, int64_t dout, int64_t w_stride, const double *x, const double *y,
                       const double *w, const double *g, double *gx, double *gy, double *gw) {
    paths_t P;
    if (paths_init(&P, n_paths, paths)) { paths_free(&P); return -1; }
    if (gw && w_stride == 0)
        for (int64_t i = 0; i < dw; ++i) gw[i] = 0;
    for (int64_t b = 0; b < B; ++b) {
        if (gx) for (int64_t i = 0; i < dx; ++i) gx[b * dx + i] = 0;
        if (gy) for (int64_t i = 0; i < dy; ++i) gy[b * dy + i] = 0;
        if (gw && w_stride) for (int64_t i = 0; i < dw; ++i) gw[b * dw + i] = 0;
        tp_row_grad(&P, x + b * dx, y + b * dy, w + b * w_stride, g + b * dout, 1.0,
                    gx ? gx + b * dx : NULL, gy ? gy + b * dy : NULL,
                    gw ? gw + b * w_stride : NULL);
    }
    paths_free(&P);
    return 0;
}

/* Fused graph convolution:
 *   out[n] = scale * sum_{e = rowptr[n]}^{rowptr[n+1]-1} TP(x[sender[e]], y[e], w[e])
 * edges taken in order.  If sel != NULL only receivers sel[0..n_sel) are written. */
int oracle_conv_forward(int n_paths, const oracle_path *paths, int64_t N, int64_t E,
                        const int32_t *rowptr, const int32_t *sender, int64_t dx, int64_t dy,
                        int64_t dw, int64_t dout, int64_t w_stride, const double *x,
                        const double *y, const double *w, double scale, double *out,
                        int64_t n_sel, const int64_t *sel) {
    paths_t P;
    if (paths_init(&P, n_paths, paths)) { paths_free(&P); return -1; }
    (void)E; (void)dw;
    int64_t cnt = sel ? n_sel : N;
    double *acc = malloc(sizeof(double) * (dout > 0 ? dout : 1));
    for (int64_t k = 0; k < cnt; ++k) {
        int64_t n = sel ? sel[k] : k;
        for (int64_t i = 0; i < dout; ++i) acc[i] = 0;
        for (int64_t e = rowptr[n]; e < rowptr[n + 1]; ++e)
            tp_row(&P, x + (int64_t)sender[e] * dx, y + e * dy, w + e * w_stride, 1.0, acc);
        for (int64_t i = 0; i < dout; ++i) out[n * dout + i] = scale * acc[i];
    }
    free(acc);
    paths_free(&P);
    return 0;
}

/* Gradient of the fused convolution for g = dL/dout[N, dout]:
 *   gx[s]  = sum over edges e with sender[e] = s (in edge order) of
 *            f_x(scale g[recv(e)]; y[e], w[e])
 *   gy[e]  = f_y(scale g[recv(e)]; x[sender[e]], w[e])
 *   gw[e]  = f_w(scale g[recv(e)]; x[sender[e]], y[e])
 * With node_sel (byte mask over N) only gx rows with node_sel[s] != 0 are
 * computed; with edge_sel (byte mask over E) only those gy/gw rows. */
int oracle_conv_backward(int n_paths, const oracle_path *paths, int64_t N, int64_t E,
                         const int32_t *rowptr, const int32_t *sender, int64_t dx, int64_t dy,
                         int64_t dw, int64_t dout, int64_t w_stride, const double *x,
                         const double *y, const double *w, double scale, const double *g,
                         double *gx, double *gy, double *gw, const uint8_t *node_sel,
                         const uint8_t *edge_sel) {
    paths_t P;
    if (paths_init(&P, n_paths, paths)) { paths_free(&P); return -1; }
    (void)E;
    if (gx)
        for (int64_t s = 0; s < N; ++s)
            if (!node_sel || node_sel[s])
                for (int64_t i = 0; i < dx; ++i) gx[s * dx + i] = 0;
    if (gw && w_stride == 0)
        for (int64_t i = 0; i < dw; ++i) gw[i] = 0;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t e = rowptr[n]; e < rowptr[n + 1]; ++e) {
            int64_t s = sender[e];
            int want_x = gx && (!node_sel || node_sel[s]);
            int want_e = !edge_sel || edge_sel[e];
            if (want_e) {
                if (gy) for (int64_t i = 0; i < dy; ++i) gy[e * dy + i] = 0;
                if (gw && w_stride) for (int64_t i = 0; i < dw; ++i) gw[e * dw + i] = 0;
            }
            if (!want_x && !want_e) continue;
            tp_row_grad(&P, x + s * dx, y + e * dy, w + e * w_stride, g + n * dout, scale,
                        want_x ? gx + s * dx : NULL, (want_e && gy) ? gy + e * dy : NULL,
                        (want_e && gw) ? gw + e * w_stride : NULL);
        }
    }
    paths_free(&P);
    return 0;
}

/* Forces from per-edge energy gradients, edge vector r_e = pos[recv] - pos[send]:
 *   F_i = - sum_e dE/dr_e (delta(i, recv(e)) - delta(i, send(e))). */
int oracle_edge_forces(int64_t N, int64_t E, const int32_t *rowptr, const int32_t *sender,
                       const double *dEdr, double *F) {
    (void)E;
    for (int64_t i = 0; i < 3 * N; ++i) F[i] = 0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t e = rowptr[n]; e < rowptr[n + 1]; ++e)
            for (int k = 0; k < 3; ++k) {
                F[3 * n + k] -= dEdr[3 * e + k];
                F[3 * (int64_t)sender[e] + k] += dEdr[3 * e + k];
            }
    return 0;
}
