// Fused multiply-add throughput probe of the current device: the denominator
// of the CUDA-core roofline of the tensor-product kernels, measured instead of
// derived from unit counts and clocks.
//
// Every thread runs kChains independent dependent chains acc = acc * a + b for
// `iters` steps (a just below 1 and b tiny keep the values finite and normal),
// so the FMA pipe, not latency, sets the pace once enough warps are resident.
// The chains' final values are folded into one word per thread and stored, so
// no chain can be removed by the compiler.  The caller times the launch (CUDA
// events on the same stream) and counts 2 * kChains * iters floating-point
// operations per thread, twice that for packed f32x2.
#include <cuda_runtime.h>

#include <cstdint>

#include "cgtp.h"
#include "internal.hpp"

namespace cgtp {

constexpr int kChains = 8;

template <typename T>
__global__ void __launch_bounds__(1024) fma_probe_kernel(int64_t iters, T a, T b,
                                                         unsigned long long* sink) {
    T acc[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) acc[i] = (T)(threadIdx.x + i) * (T)1e-3;
    // the multiplicands in registers (the compiler cannot prove the offset is
    // zero), as the tensor-product kernels have them
    const T z = (T)(iters >> 62);
    const T ar = a + z, br = b + z;
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) acc[i] = fma(acc[i], ar, br);
    }
    T s = 0;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += acc[i];
    unsigned long long bits = 0;
    if constexpr (sizeof(T) == 8)
        bits = (unsigned long long)__double_as_longlong((double)s);
    else
        bits = (unsigned long long)__float_as_uint((float)s);
    sink[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = bits;
}

// Two fp32 chains per 64-bit register, one fma.rn.f32x2 per step.
__global__ void __launch_bounds__(1024) fma_probe_f32x2_kernel(int64_t iters, float a, float b,
                                                               unsigned long long* sink) {
    typedef unsigned long long u64;
    const float z = (float)(iters >> 62);
    const u64 ua = __float_as_uint(a + z), ub = __float_as_uint(b + z);
    const u64 pa = (ua << 32) | ua, pb = (ub << 32) | ub;
    u64 acc[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) {
        const u64 v = __float_as_uint((float)(threadIdx.x + i) * 1e-3f);
        acc[i] = (v << 32) | v;
    }
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i)
            asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(acc[i]) : "l"(acc[i]), "l"(pa), "l"(pb));
    }
    u64 s = 0;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s ^= acc[i];
    sink[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace cgtp

extern "C" cgtp_status cgtp_fma_probe(cgtp_dtype dtype, int packed, int64_t blocks, int threads,
                                      int64_t iters, void* sink, int64_t* flops,
                                      cgtp_stream stream) {
    using namespace cgtp;
    if ((dtype != CGTP_F32 && dtype != CGTP_F64) || (packed && dtype != CGTP_F32) ||
        blocks < 1 || blocks > (1ll << 31) - 1 || threads < 32 || threads > 1024 ||
        threads % 32 != 0 || iters < 1 || !sink || ((uintptr_t)sink % 8) != 0) {
        set_error_message("cgtp_fma_probe: bad arguments");
        return CGTP_E_ARG;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned long long* out = static_cast<unsigned long long*>(sink);
    const dim3 g((unsigned)blocks), b((unsigned)threads);
    if (dtype == CGTP_F64)
        fma_probe_kernel<double><<<g, b, 0, s>>>(iters, 0.9999999, 1e-9, out);
    else if (packed)
        fma_probe_f32x2_kernel<<<g, b, 0, s>>>(iters, 0.9999f, 1e-7f, out);
    else
        fma_probe_kernel<float><<<g, b, 0, s>>>(iters, 0.9999f, 1e-7f, out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_cuda_error(e);
        set_error_message(std::string("cgtp_fma_probe: ") + cudaGetErrorString(e));
        return CGTP_E_CUDA;
    }
    count_launch();
    if (flops) *flops = blocks * (int64_t)threads * iters * kChains * 2 * (packed ? 2 : 1);
    return CGTP_OK;
}
