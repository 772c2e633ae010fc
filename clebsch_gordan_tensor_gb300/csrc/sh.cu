// Real spherical harmonics of edge vectors and their derivatives (sm_103a).
//
// The per-edge basis of a TFN layer "depends on spherical harmonics" of the
// relative position (NVIDIA SE(3)-Transformer blog, "Basis precomputation");
// forces need their derivatives ("higher partial derivatives required to
// predict interatomic forces", abstract of arXiv 2501.13986).
//
// Method (independent of any table): for the unit vector u = (x, y, z),
//   C_m + i S_m = (x + i y)^m                      (C_{m+1} = x C_m - y S_m, ...)
//   Q_l^m(z): Q_m^m = (2m-1)!!,  Q_{m+1}^m = (2m+1) z Q_m^m,
//             (l-m) Q_l^m = (2l-1) z Q_{l-1}^m - (l+m-1) Q_{l-2}^m
//   Y_l0 = N_l0 Q_l^0,  Y_lm = N_lm Q_l^m C_m (m>0),  Y_l,-m = N_lm Q_l^m S_m,
//   N_lm = sqrt((2l+1) (l-m)!/(l+m)! * (m>0 ? 2 : 1))     (component normalised)
// and the gradient on the sphere uses dQ_l^m/dz = Q_l^(m+1), dC_m/dx = m C_{m-1},
// dC_m/dy = -m S_{m-1}, dS_m/dx = m S_{m-1}, dS_m/dy = m C_{m-1}, projected by
// (I - u u^T) / |r|.  One thread per edge.
//
// Second derivatives (the gradient of a force loss in the positions) are taken
// in forward mode over the backward: the backward's arithmetic evaluated on
// dual numbers a + b eps (eps^2 = 0) at r + eps t gives, in its eps part, the
// derivative of J(r)^T g along t, i.e. the Hessian of g . Y(r) applied to t.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.hpp"

namespace cgtp {

// Dual number a + b eps with eps^2 = 0: b carries the directional derivative.
template <typename T>
struct Dual {
    T v, d;
    __device__ __forceinline__ Dual() {}
    __device__ __forceinline__ Dual(T a) : v(a), d((T)0) {}
    __device__ __forceinline__ Dual(T a, T b) : v(a), d(b) {}
    __device__ __forceinline__ Dual& operator+=(const Dual& o) {
        v += o.v;
        d += o.d;
        return *this;
    }
    __device__ __forceinline__ Dual& operator*=(const Dual& o) {
        d = d * o.v + v * o.d;
        v *= o.v;
        return *this;
    }
};
template <typename T>
__device__ __forceinline__ Dual<T> operator+(Dual<T> a, Dual<T> b) { return {a.v + b.v, a.d + b.d}; }
template <typename T>
__device__ __forceinline__ Dual<T> operator-(Dual<T> a, Dual<T> b) { return {a.v - b.v, a.d - b.d}; }
template <typename T>
__device__ __forceinline__ Dual<T> operator-(Dual<T> a) { return {-a.v, -a.d}; }
template <typename T>
__device__ __forceinline__ Dual<T> operator*(Dual<T> a, Dual<T> b) {
    return {a.v * b.v, a.d * b.v + a.v * b.d};
}
template <typename T>
__device__ __forceinline__ Dual<T> operator*(T a, Dual<T> b) { return {a * b.v, a * b.d}; }
template <typename T>
__device__ __forceinline__ Dual<T> operator/(Dual<T> a, Dual<T> b) {
    const T inv = (T)1 / b.v, q = a.v * inv;
    return {q, (a.d - q * b.d) * inv};
}
template <typename T>
__device__ __forceinline__ Dual<T> dual_sqrt(Dual<T> a) {
    const T s = sqrt(a.v);
    return {s, a.d / (s + s)};
}

template <typename T>
__device__ __forceinline__ T sh_norm(int l, int m) {
    double r = 1.0;  // (l-m)!/(l+m)!
    for (int k = l - m + 1; k <= l + m; ++k) r /= (double)k;
    return (T)sqrt((2.0 * l + 1.0) * r * (m > 0 ? 2.0 : 1.0));
}

// Y (and optionally grad_u Y) of the unit vector u.
template <int L, typename T, bool GRAD>
__device__ __forceinline__ void sh_unit(T x, T y, T z, T* Y, T* gx, T* gy, T* gz) {
    constexpr int D = L + 1;
    T C[D + 1], S[D + 1];
    C[0] = (T)1;
    S[0] = (T)0;
#pragma unroll
    for (int m = 0; m < D; ++m) {
        C[m + 1] = x * C[m] - y * S[m];
        S[m + 1] = x * S[m] + y * C[m];
    }
    T Q[D + 1][D + 1];  // Q[l][m], m <= l, Q[l][l+1] = 0
#pragma unroll
    for (int l = 0; l <= L; ++l)
#pragma unroll
        for (int m = 0; m <= L; ++m) Q[l][m] = (T)0;
#pragma unroll
    for (int m = 0; m <= L; ++m) {
        T dfact = (T)1;
#pragma unroll
        for (int k = 1; k <= 2 * m - 1; k += 2) dfact *= (T)k;
        Q[m][m] = dfact;
        if (m + 1 <= L) Q[m + 1][m] = (T)(2 * m + 1) * z * dfact;
#pragma unroll
        for (int l = m + 2; l <= L; ++l)
            Q[l][m] = ((T)(2 * l - 1) * z * Q[l - 1][m] - (T)(l + m - 1) * Q[l - 2][m]) / (T)(l - m);
    }
#pragma unroll
    for (int l = 0; l <= L; ++l) {
#pragma unroll
        for (int m = -l; m <= l; ++m) {
            const int am = m < 0 ? -m : m;
            const T N = sh_norm<T>(l, am);
            const int i = l * l + m + l;
            const T ang = m > 0 ? C[am] : (m < 0 ? S[am] : (T)1);
            Y[i] = N * Q[l][am] * ang;
            if (GRAD) {
                const T q = Q[l][am];
                const T dq = am + 1 <= l ? Q[l][am + 1] : (T)0;
                T dax = (T)0, day = (T)0;
                if (m > 0) {
                    dax = (T)am * C[am - 1];
                    day = -(T)am * S[am - 1];
                } else if (m < 0) {
                    dax = (T)am * S[am - 1];
                    day = (T)am * C[am - 1];
                }
                gx[i] = N * q * dax;
                gy[i] = N * q * day;
                gz[i] = N * dq * ang;
            }
        }
    }
}

template <int L, typename T>
__global__ void __launch_bounds__(128) sh_forward_kernel(int64_t E, const T* __restrict__ vec,
                                                          T* __restrict__ out) {
    constexpr int D2 = (L + 1) * (L + 1);
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E;
         e += (int64_t)gridDim.x * blockDim.x) {
        const T x = vec[3 * e], y = vec[3 * e + 1], z = vec[3 * e + 2];
        const T inv = (T)1 / sqrt(x * x + y * y + z * z);
        T Y[D2];
        sh_unit<L, T, false>(x * inv, y * inv, z * inv, Y, nullptr, nullptr, nullptr);
#pragma unroll
        for (int i = 0; i < D2; ++i) out[e * D2 + i] = Y[i];
    }
}

// BACKWARD: out[e, 0..3) = J^T in[e];  JVP: out[e, 0..D2) = J in[e, 0..3).
template <int L, typename T, bool BACKWARD>
__global__ void __launch_bounds__(128) sh_deriv_kernel(int64_t E, const T* __restrict__ vec,
                                                        const T* __restrict__ in,
                                                        T* __restrict__ out) {
    constexpr int D2 = (L + 1) * (L + 1);
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E;
         e += (int64_t)gridDim.x * blockDim.x) {
        const T x = vec[3 * e], y = vec[3 * e + 1], z = vec[3 * e + 2];
        const T inv = (T)1 / sqrt(x * x + y * y + z * z);
        const T ux = x * inv, uy = y * inv, uz = z * inv;
        T Y[D2], gx[D2], gy[D2], gz[D2];
        sh_unit<L, T, true>(ux, uy, uz, Y, gx, gy, gz);
        if (BACKWARD) {
            T ax = 0, ay = 0, az = 0;
#pragma unroll
            for (int i = 0; i < D2; ++i) {
                const T g = in[e * D2 + i];
                ax += g * gx[i];
                ay += g * gy[i];
                az += g * gz[i];
            }
            const T r = ax * ux + ay * uy + az * uz;
            out[3 * e] = (ax - r * ux) * inv;
            out[3 * e + 1] = (ay - r * uy) * inv;
            out[3 * e + 2] = (az - r * uz) * inv;
        } else {
            T tx = in[3 * e], ty = in[3 * e + 1], tz = in[3 * e + 2];
            const T r = tx * ux + ty * uy + tz * uz;
            tx = (tx - r * ux) * inv;
            ty = (ty - r * uy) * inv;
            tz = (tz - r * uz) * inv;
#pragma unroll
            for (int i = 0; i < D2; ++i) out[e * D2 + i] = gx[i] * tx + gy[i] * ty + gz[i] * tz;
        }
    }
}

// HVP: out[e] = d/deps [J(vec[e] + eps t[e])^T g[e]] = H_e t[e], H_e the
// Hessian of g[e] . Y(r) at r = vec[e].
template <int L, typename T>
__global__ void __launch_bounds__(128) sh_hvp_kernel(int64_t E, const T* __restrict__ vec,
                                                      const T* __restrict__ gin,
                                                      const T* __restrict__ tvec,
                                                      T* __restrict__ out) {
    using D = Dual<T>;
    constexpr int D2 = (L + 1) * (L + 1);
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E;
         e += (int64_t)gridDim.x * blockDim.x) {
        const D x(vec[3 * e], tvec[3 * e]), y(vec[3 * e + 1], tvec[3 * e + 1]),
            z(vec[3 * e + 2], tvec[3 * e + 2]);
        const D inv = D((T)1) / dual_sqrt(x * x + y * y + z * z);
        const D ux = x * inv, uy = y * inv, uz = z * inv;
        D Y[D2], gx[D2], gy[D2], gz[D2];
        sh_unit<L, D, true>(ux, uy, uz, Y, gx, gy, gz);
        D ax((T)0), ay((T)0), az((T)0);
#pragma unroll
        for (int i = 0; i < D2; ++i) {
            const T g = gin[e * D2 + i];
            ax += g * gx[i];
            ay += g * gy[i];
            az += g * gz[i];
        }
        const D r = ax * ux + ay * uy + az * uz;
        out[3 * e] = ((ax - r * ux) * inv).d;
        out[3 * e + 1] = ((ay - r * uy) * inv).d;
        out[3 * e + 2] = ((az - r * uz) * inv).d;
    }
}

static dim3 grid_for(int64_t E) {
    int64_t b = (E + 127) / 128;
    if (b > (1 << 20)) b = 1 << 20;
    return dim3((unsigned)b);
}

template <typename T>
static cudaError_t sh_fwd_t(int lmax, int64_t E, const T* v, T* y, cudaStream_t s) {
    const dim3 g = grid_for(E);
    switch (lmax) {
        case 0: sh_forward_kernel<0, T><<<g, 128, 0, s>>>(E, v, y); break;
        case 1: sh_forward_kernel<1, T><<<g, 128, 0, s>>>(E, v, y); break;
        case 2: sh_forward_kernel<2, T><<<g, 128, 0, s>>>(E, v, y); break;
        case 3: sh_forward_kernel<3, T><<<g, 128, 0, s>>>(E, v, y); break;
        case 4: sh_forward_kernel<4, T><<<g, 128, 0, s>>>(E, v, y); break;
        case 5: sh_forward_kernel<5, T><<<g, 128, 0, s>>>(E, v, y); break;
        case 6: sh_forward_kernel<6, T><<<g, 128, 0, s>>>(E, v, y); break;
        default: return cudaErrorInvalidValue;
    }
    count_launch();
    return cudaGetLastError();
}

template <typename T, bool B>
static cudaError_t sh_der_t(int lmax, int64_t E, const T* v, const T* in, T* out, cudaStream_t s) {
    const dim3 g = grid_for(E);
    switch (lmax) {
        case 0: sh_deriv_kernel<0, T, B><<<g, 128, 0, s>>>(E, v, in, out); break;
        case 1: sh_deriv_kernel<1, T, B><<<g, 128, 0, s>>>(E, v, in, out); break;
        case 2: sh_deriv_kernel<2, T, B><<<g, 128, 0, s>>>(E, v, in, out); break;
        case 3: sh_deriv_kernel<3, T, B><<<g, 128, 0, s>>>(E, v, in, out); break;
        case 4: sh_deriv_kernel<4, T, B><<<g, 128, 0, s>>>(E, v, in, out); break;
        case 5: sh_deriv_kernel<5, T, B><<<g, 128, 0, s>>>(E, v, in, out); break;
        case 6: sh_deriv_kernel<6, T, B><<<g, 128, 0, s>>>(E, v, in, out); break;
        default: return cudaErrorInvalidValue;
    }
    count_launch();
    return cudaGetLastError();
}

template <typename T>
static cudaError_t sh_hvp_t(int lmax, int64_t E, const T* v, const T* g, const T* t, T* out,
                            cudaStream_t s) {
    const dim3 gr = grid_for(E);
    switch (lmax) {
        case 0: sh_hvp_kernel<0, T><<<gr, 128, 0, s>>>(E, v, g, t, out); break;
        case 1: sh_hvp_kernel<1, T><<<gr, 128, 0, s>>>(E, v, g, t, out); break;
        case 2: sh_hvp_kernel<2, T><<<gr, 128, 0, s>>>(E, v, g, t, out); break;
        case 3: sh_hvp_kernel<3, T><<<gr, 128, 0, s>>>(E, v, g, t, out); break;
        case 4: sh_hvp_kernel<4, T><<<gr, 128, 0, s>>>(E, v, g, t, out); break;
        case 5: sh_hvp_kernel<5, T><<<gr, 128, 0, s>>>(E, v, g, t, out); break;
        case 6: sh_hvp_kernel<6, T><<<gr, 128, 0, s>>>(E, v, g, t, out); break;
        default: return cudaErrorInvalidValue;
    }
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_sh_forward(int lmax, bool f64, int64_t E, const void* vec, void* y,
                              cudaStream_t s) {
    if (f64) return sh_fwd_t<double>(lmax, E, (const double*)vec, (double*)y, s);
    return sh_fwd_t<float>(lmax, E, (const float*)vec, (float*)y, s);
}

cudaError_t launch_sh_backward(int lmax, bool f64, int64_t E, const void* vec, const void* gy,
                               void* gvec, cudaStream_t s) {
    if (f64)
        return sh_der_t<double, true>(lmax, E, (const double*)vec, (const double*)gy,
                                      (double*)gvec, s);
    return sh_der_t<float, true>(lmax, E, (const float*)vec, (const float*)gy, (float*)gvec, s);
}

cudaError_t launch_sh_jvp(int lmax, bool f64, int64_t E, const void* vec, const void* tvec,
                          void* ty, cudaStream_t s) {
    if (f64)
        return sh_der_t<double, false>(lmax, E, (const double*)vec, (const double*)tvec,
                                       (double*)ty, s);
    return sh_der_t<float, false>(lmax, E, (const float*)vec, (const float*)tvec, (float*)ty, s);
}

cudaError_t launch_sh_hvp(int lmax, bool f64, int64_t E, const void* vec, const void* gy,
                          const void* tvec, void* out, cudaStream_t s) {
    if (f64)
        return sh_hvp_t<double>(lmax, E, (const double*)vec, (const double*)gy,
                                (const double*)tvec, (double*)out, s);
    return sh_hvp_t<float>(lmax, E, (const float*)vec, (const float*)gy, (const float*)tvec,
                           (float*)out, s);
}

}  // namespace cgtp
