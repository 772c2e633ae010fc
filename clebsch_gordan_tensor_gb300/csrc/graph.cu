// Graph-side kernels: interatomic forces from per-edge energy gradients, the
// adjoint used by the force-loss chain, and a zero fill (sm_103a).
//
// Forces are the gradient of the energy with respect to positions ("higher
// partial derivatives required to predict interatomic forces", abstract of
// arXiv 2501.13986).  With r_e = pos[recv] - pos[send],
//   F_i = -sum_{recv e = i} dE/dr_e + sum_{send e = i} dE/dr_e.
// One thread per atom walks its receiver segment then its sender segment:
// deterministic, no atomics.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.hpp"

namespace cgtp {

template <typename T>
__global__ void __launch_bounds__(128)
edge_forces_kernel(int64_t N, const int32_t* __restrict__ rowptr,
                   const int32_t* __restrict__ s_rowptr, const int32_t* __restrict__ s_perm,
                   const T* __restrict__ d, T* __restrict__ F) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N;
         i += (int64_t)gridDim.x * blockDim.x) {
        T fx = 0, fy = 0, fz = 0;
        for (int64_t e = rowptr[i]; e < rowptr[i + 1]; ++e) {
            fx -= d[3 * e];
            fy -= d[3 * e + 1];
            fz -= d[3 * e + 2];
        }
        for (int64_t j = s_rowptr[i]; j < s_rowptr[i + 1]; ++j) {
            const int64_t e = s_perm[j];
            fx += d[3 * e];
            fy += d[3 * e + 1];
            fz += d[3 * e + 2];
        }
        F[3 * i] = fx;
        F[3 * i + 1] = fy;
        F[3 * i + 2] = fz;
    }
}

// q[e] = gF[sender e] - gF[recv e], one thread per receiver.
template <typename T>
__global__ void __launch_bounds__(128)
edge_forces_adjoint_kernel(int64_t N, const int32_t* __restrict__ rowptr,
                           const int32_t* __restrict__ sender, const T* __restrict__ gF,
                           T* __restrict__ q) {
    for (int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; n < N;
         n += (int64_t)gridDim.x * blockDim.x) {
        const T ax = gF[3 * n], ay = gF[3 * n + 1], az = gF[3 * n + 2];
        for (int64_t e = rowptr[n]; e < rowptr[n + 1]; ++e) {
            const int64_t s = sender[e];
            q[3 * e] = gF[3 * s] - ax;
            q[3 * e + 1] = gF[3 * s + 1] - ay;
            q[3 * e + 2] = gF[3 * s + 2] - az;
        }
    }
}

// out[c] = sum over r of partial[r][c], rows added in order (deterministic).
template <typename T>
__global__ void __launch_bounds__(256)
reduce_rows_kernel(const T* __restrict__ partial, int64_t rows, int64_t cols, T* __restrict__ out) {
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < cols;
         c += (int64_t)gridDim.x * blockDim.x) {
        T s = 0;
        for (int64_t r = 0; r < rows; ++r) s += partial[r * cols + c];
        out[c] = s;
    }
}

__global__ void fill_zero_kernel(uint32_t* __restrict__ p, int64_t words) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words;
         i += (int64_t)gridDim.x * blockDim.x)
        p[i] = 0u;
}

static dim3 grid_for(int64_t n) {
    int64_t b = (n + 127) / 128;
    if (b > (1 << 20)) b = 1 << 20;
    if (b < 1) b = 1;
    return dim3((unsigned)b);
}

cudaError_t launch_edge_forces(bool f64, int64_t N, const int32_t* rowptr,
                               const int32_t* s_rowptr, const int32_t* s_perm, const void* dEdr,
                               void* F, cudaStream_t s) {
    if (f64)
        edge_forces_kernel<double><<<grid_for(N), 128, 0, s>>>(N, rowptr, s_rowptr, s_perm,
                                                              (const double*)dEdr, (double*)F);
    else
        edge_forces_kernel<float><<<grid_for(N), 128, 0, s>>>(N, rowptr, s_rowptr, s_perm,
                                                             (const float*)dEdr, (float*)F);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_edge_forces_adjoint(bool f64, int64_t N, const int32_t* rowptr,
                                       const int32_t* sender, const void* gF, void* q,
                                       cudaStream_t s) {
    if (f64)
        edge_forces_adjoint_kernel<double><<<grid_for(N), 128, 0, s>>>(
            N, rowptr, sender, (const double*)gF, (double*)q);
    else
        edge_forces_adjoint_kernel<float><<<grid_for(N), 128, 0, s>>>(
            N, rowptr, sender, (const float*)gF, (float*)q);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_reduce_rows(bool f64, const void* partial, int64_t rows, int64_t cols,
                               void* out, cudaStream_t s) {
    const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>((cols + 255) / 256, 4096));
    if (f64)
        reduce_rows_kernel<double><<<blocks, 256, 0, s>>>((const double*)partial, rows, cols,
                                                          (double*)out);
    else
        reduce_rows_kernel<float><<<blocks, 256, 0, s>>>((const float*)partial, rows, cols,
                                                         (float*)out);
    count_launch();
    return cudaGetLastError();
}

template <typename T>
__global__ void fill_ones_kernel(T* __restrict__ p, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        p[i] = (T)1;
}

cudaError_t launch_fill_ones(bool f64, void* p, int64_t n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    if (f64)
        fill_ones_kernel<double><<<grid_for(n), 128, 0, s>>>((double*)p, n);
    else
        fill_ones_kernel<float><<<grid_for(n), 128, 0, s>>>((float*)p, n);
    count_launch();
    return cudaGetLastError();
}

// Loads the weight-gradient reduction and zero-fill kernels into the current
// device's context now (with lazy module loading they would otherwise load,
// and allocate, at their first launch).
cudaError_t preload_reduce_kernels() {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, reduce_rows_kernel<float>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, reduce_rows_kernel<double>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, fill_zero_kernel);
    return e;
}

// bytes must be a multiple of 4 (every tensor here is fp32 or fp64).
cudaError_t launch_fill_zero(void* p, int64_t bytes, cudaStream_t s) {
    const int64_t words = bytes / 4;
    fill_zero_kernel<<<grid_for(words), 128, 0, s>>>((uint32_t*)p, words);
    count_launch();
    return cudaGetLastError();
}

}  // namespace cgtp
