// The radial network that produces the per-edge tensor-product weights
// (sm_103a).
//
// NVIDIA's SE(3)-Transformer blog, section "Fused key and value computation":
// the radial profile inside a TFN layer is a fully connected network of the
// edge length whose outputs weight the pairwise convolutions.  Here, for edge
// e with length r = |vec[e]|:
//   b_n   = sqrt(2/rc) sin(n pi r / rc) / r,  n = 1..n_basis  (r = 0: its limit)
//   h     = silu(b W1)            W1 [n_basis, hidden]
//   w[e]  = h W2                  W2 [hidden, n_out]
//
// Two kernels:
//   * radial_tc_kernel (fp32, hidden % 8 == 0 and <= 64, n_out % 128 == 0):
//     the last layer -- the only dense contraction, 2 hidden * n_out FLOP per
//     edge -- runs on the tensor cores.  A tile of 128 edges' hidden
//     activations (A, 128 x hidden) and a 128-column slice of W2 (B) sit in
//     shared memory as TF32 "hi" and "lo" parts (x = hi + lo, both TF32);
//     tcgen05.mma accumulates hi*hi + hi*lo + lo*hi into a 128 x 128 fp32
//     accumulator in tensor memory, which keeps fp32 accuracy (the dropped
//     lo*lo term is 2^-22 relative).  One thread issues the MMAs; completion
//     arrives on an mbarrier; four warps read the accumulator back with
//     tcgen05.ld and store the rows.
//   * radial_simt_kernel (fp32 / fp64, any shape): shared-memory tiles and
//     FMA micro-tiles on the CUDA cores.
// Both compute b and h the same way on the CUDA cores.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "internal.hpp"

namespace cgtp {

__device__ int cgtp_radial_error;  // nonzero: a bounded wait timed out

template <typename T>
__device__ __forceinline__ T silu_f(T a) {
    return a / ((T)1 + exp(-a));
}

// Basis function n (1-based) at length r: sqrt(2/rc) sin(k r) / r, k = n pi / rc.
template <typename T>
__device__ __forceinline__ T bessel_f(int n, T r, T rc, T pref) {
    const T k = (T)n * (T)3.14159265358979323846 / rc;
    return pref * (r > (T)0 ? sin(k * r) / r : k);
}

// ------------------------------------------------------------- CUDA cores

constexpr int kSimtEdges = 32;   // edges per tile
constexpr int kSimtCols = 128;   // output columns per pass
constexpr int kSimtThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kSimtThreads)
radial_simt_kernel(int64_t E, int nb, T rc, int hidden, int64_t n_out, const T* __restrict__ vec,
                   const T* __restrict__ W1, const T* __restrict__ W2, T* __restrict__ w,
                   T* __restrict__ h) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* bS = reinterpret_cast<T*>(smem_raw);  // [kSimtEdges][nb]
    T* hS = bS + kSimtEdges * nb;            // [kSimtEdges][hidden]
    const int tid = threadIdx.x;
    const T pref = sqrt((T)2 / rc);
    for (int64_t e0 = (int64_t)blockIdx.x * kSimtEdges; e0 < E;
         e0 += (int64_t)gridDim.x * kSimtEdges) {
        const int ne = E - e0 < kSimtEdges ? (int)(E - e0) : kSimtEdges;
        for (int i = tid; i < kSimtEdges * nb; i += kSimtThreads) {
            const int le = i / nb, n = i % nb;
            T b = (T)0;
            if (le < ne) {
                const T* v = vec + 3 * (e0 + le);
                b = bessel_f<T>(n + 1, sqrt(v[0] * v[0] + v[1] * v[1] + v[2] * v[2]), rc, pref);
            }
            bS[i] = b;
        }
        __syncthreads();
        for (int i = tid; i < kSimtEdges * hidden; i += kSimtThreads) {
            const int le = i / hidden, j = i % hidden;
            T a = (T)0;
            for (int n = 0; n < nb; ++n) a = fma(bS[le * nb + n], __ldg(W1 + n * hidden + j), a);
            const T s = le < ne ? silu_f<T>(a) : (T)0;
            hS[i] = s;
            if (h && le < ne) h[(e0 + le) * hidden + j] = s;
        }
        __syncthreads();
        const int eg = tid / 32, cgp = tid % 32;  // 8 groups of 4 edges x 32 groups of 4 columns
        for (int64_t c0 = 0; c0 < n_out; c0 += kSimtCols) {
            T acc[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[i][q] = (T)0;
            for (int k = 0; k < hidden; ++k) {
                T a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = hS[(eg * 4 + i) * hidden + k];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int64_t c = c0 + cgp * 4 + q;
                    b[q] = c < n_out ? __ldg(W2 + (int64_t)k * n_out + c) : (T)0;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[i][q] = fma(a[i], b[q], acc[i][q]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int le = eg * 4 + i;
                if (le >= ne) continue;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int64_t c = c0 + cgp * 4 + q;
                    if (c < n_out) w[(e0 + le) * n_out + c] = acc[i][q];
                }
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------ tensor cores

constexpr int kTcM = 128;         // edges per tile (MMA M, TMEM lanes)
constexpr int kTcN = 128;         // output columns per chunk (MMA N)
constexpr int kTcKMax = 64;       // hidden width held in one tile
constexpr int kTcThreads = 128;   // four warps: one TMEM lane quarter each
constexpr unsigned kTcTmemCols = 128;
// Operand bytes: A hi/lo [128 x K] and B hi/lo [128 x K], tf32.
constexpr unsigned kTcOperand = kTcM * kTcKMax * 4;  // 32 KB each
// The operand region is followed by padding so that a descriptor stride read
// the other way round would still stay inside this CTA's shared memory.
constexpr unsigned kTcSmem = 4 * kTcOperand + 64 * 1024;

__device__ __forceinline__ unsigned smem_addr(const void* p) {
    return (unsigned)__cvta_generic_to_shared(p);
}

// Canonical K-major layout without swizzle: 8-row x 16-byte core matrices;
// the 8-row groups of one 4-wide K slice are contiguous (128 B apart) and the
// K slices follow each other (LBO = rows / 8 * 128 B apart).
__device__ __forceinline__ unsigned kmajor_offset(int row, int k, int rows) {
    return (unsigned)((k >> 2) * (rows / 8) * 128 + (row >> 3) * 128 + (row & 7) * 16 + (k & 3) * 4);
}

// Shared-memory matrix descriptor (tcgen05): start >> 4 in bits 0-13, leading
// byte offset >> 4 in 16-29, stride byte offset >> 4 in 32-45, the fixed
// version value 1 in bits 46-47, no swizzle (bits 61-63 = 0).
__device__ __forceinline__ uint64_t smem_desc(unsigned addr, unsigned lbo, unsigned sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor, kind::tf32: D fp32 (bits 4-5 = 1), A and B TF32
// (bits 7-9 and 10-12 = 2), both K-major, N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
constexpr uint32_t kTcIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(kTcN >> 3) << 17) |
                              ((uint32_t)(kTcM >> 4) << 24);

__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

__device__ __forceinline__ void mma_tf32(unsigned tmem_d, uint64_t a, uint64_t b, unsigned acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(kTcIdesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tc_mbar_init(unsigned long long* b) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(b)) : "memory");
}

// Bounded wait for phase `parity` (about a second at most).
__device__ __forceinline__ bool tc_mbar_wait(unsigned long long* b, unsigned parity) {
    const unsigned a = smem_addr(b);
    for (unsigned it = 0; it < (1u << 24); ++it) {
        unsigned ok;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
            : "=r"(ok) : "r"(a), "r"(parity) : "memory");
        if (ok) return true;
        if (it > 1024) __nanosleep(64);
    }
    return false;
}

__device__ __forceinline__ void tmem_ld32(unsigned taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kTcThreads, 1)
radial_tc_kernel(int64_t E, int nb, float rc, int hidden, int64_t n_out,
                 const float* __restrict__ vec, const float* __restrict__ W1,
                 const float* __restrict__ W2, float* __restrict__ w, float* __restrict__ h) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) unsigned long long mma_done;
    __shared__ unsigned tmem_base;
    __shared__ float bS[kTcM][33];
    unsigned char* Ahi = smem;
    unsigned char* Alo = smem + kTcOperand;
    unsigned char* Bhi = smem + 2 * kTcOperand;
    unsigned char* Blo = smem + 3 * kTcOperand;
    const int tid = threadIdx.x, warp = tid >> 5;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base)),
                     "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        tc_mbar_init(&mma_done);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const unsigned tmem = tmem_base;
    const float pref = sqrtf(2.0f / rc);
    const unsigned lbo = (kTcM / 8) * 128;  // next 4-wide K slice (A and B both have 128 rows)
    unsigned phase = 0;
    bool ok = true;

    for (int64_t e0 = (int64_t)blockIdx.x * kTcM; e0 < E && ok; e0 += (int64_t)gridDim.x * kTcM) {
        // hidden activations of the tile: thread tid owns edge row tid
        const int64_t e = e0 + tid;
        const bool live = e < E;
        {
            float r = 0.0f;
            if (live) {
                const float* v = vec + 3 * e;
                r = sqrtf(v[0] * v[0] + v[1] * v[1] + v[2] * v[2]);
            }
            for (int n = 0; n < nb; ++n) bS[tid][n] = live ? bessel_f<float>(n + 1, r, rc, pref) : 0.0f;
        }
        for (int k4 = 0; k4 < hidden; k4 += 4) {
            float hv[4], hi[4], lo[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float a = 0.0f;
                for (int n = 0; n < nb; ++n) a = fmaf(bS[tid][n], __ldg(W1 + n * hidden + k4 + q), a);
                hv[q] = live ? silu_f<float>(a) : 0.0f;
                hi[q] = to_tf32(hv[q]);
                lo[q] = to_tf32(hv[q] - hi[q]);
            }
            if (h && live)
                *reinterpret_cast<float4*>(h + e * hidden + k4) = make_float4(hv[0], hv[1], hv[2], hv[3]);
            const unsigned off = kmajor_offset(tid, k4, kTcM);
            *reinterpret_cast<float4*>(Ahi + off) = make_float4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<float4*>(Alo + off) = make_float4(lo[0], lo[1], lo[2], lo[3]);
        }
        for (int64_t c0 = 0; c0 < n_out; c0 += kTcN) {
            // B = W2[:, c0 : c0 + 128] as 128 K-major rows (row = output column)
            for (int i = tid; i < kTcN * (hidden / 4); i += kTcThreads) {
                const int n = i % kTcN, k4 = (i / kTcN) * 4;
                float hi[4], lo[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float x = __ldg(W2 + (int64_t)(k4 + q) * n_out + c0 + n);
                    hi[q] = to_tf32(x);
                    lo[q] = to_tf32(x - hi[q]);
                }
                const unsigned off = kmajor_offset(n, k4, kTcN);
                *reinterpret_cast<float4*>(Bhi + off) = make_float4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<float4*>(Blo + off) = make_float4(lo[0], lo[1], lo[2], lo[3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncthreads();
            if (tid == 0) {
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                for (int k8 = 0; k8 < hidden; k8 += 8) {
                    const unsigned koff = (unsigned)(k8 >> 2) * lbo;
                    const uint64_t ah = smem_desc(smem_addr(Ahi) + koff, lbo, 128);
                    const uint64_t al = smem_desc(smem_addr(Alo) + koff, lbo, 128);
                    const uint64_t bh = smem_desc(smem_addr(Bhi) + koff, lbo, 128);
                    const uint64_t bl = smem_desc(smem_addr(Blo) + koff, lbo, 128);
                    mma_tf32(tmem, ah, bh, k8 > 0 ? 1u : 0u);
                    mma_tf32(tmem, ah, bl, 1u);
                    mma_tf32(tmem, al, bh, 1u);
                }
                asm volatile(
                    "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                        smem_addr(&mma_done))
                    : "memory");
            }
            // every thread waits; all agree on the outcome before any
            // warp-collective tcgen05.ld
            const bool got = tc_mbar_wait(&mma_done, phase);
            if (!__syncthreads_and(got)) {
                if (tid == 0) atomicExch(&cgtp_radial_error, 1);
                ok = false;
                break;
            }
            phase ^= 1u;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            // accumulator rows 32 warp .. +31 -> this thread's edge row
#pragma unroll 1
            for (int cc = 0; cc < kTcN; cc += 32) {
                float v[32];
                tmem_ld32(tmem + ((unsigned)(warp * 32) << 16) + (unsigned)cc, v);
                if (live) {
                    float4* dst = reinterpret_cast<float4*>(w + e * n_out + c0 + cc);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncthreads();
        }
    }
    // after a timed-out wait give the MMAs in flight a second bounded wait,
    // then release the accumulator (every thread agrees on the exit first)
    if (!ok) tc_mbar_wait(&mma_done, phase);
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTcTmemCols)
                     : "memory");
}

// ------------------------------------------------------------------ host

bool radial_tc_eligible(bool f64, int nb, int hidden, int64_t n_out, const void* vec,
                        const void* W2, const void* w, const void* h) {
    auto a16 = [](const void* p) { return p == nullptr || ((uintptr_t)p % 16) == 0; };
    return !f64 && nb <= 32 && hidden % 8 == 0 && hidden <= kTcKMax && n_out % kTcN == 0 &&
           a16(w) && a16(h) && a16(W2) && a16(vec);
}

cudaError_t launch_radial_forward(bool f64, bool tensor_cores, int64_t E, int nb, double rc,
                                  int hidden, int64_t n_out, const void* vec, const void* W1,
                                  const void* W2, void* w, void* h, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (tensor_cores) {
        e = cudaFuncSetAttribute(radial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kTcSmem);
        if (e != cudaSuccess) return e;
        const int64_t tiles = (E + kTcM - 1) / kTcM;
        const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(tiles, sms));
        radial_tc_kernel<<<grid, kTcThreads, kTcSmem, s>>>(
            E, nb, (float)rc, hidden, n_out, (const float*)vec, (const float*)W1,
            (const float*)W2, (float*)w, (float*)h);
        return cudaGetLastError();
    }
    const size_t es = f64 ? 8 : 4;
    const size_t smem = (size_t)kSimtEdges * (nb + hidden) * es;
    auto* k64 = radial_simt_kernel<double>;
    auto* k32 = radial_simt_kernel<float>;
    e = f64 ? cudaFuncSetAttribute(k64, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
            : cudaFuncSetAttribute(k32, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (E + kSimtEdges - 1) / kSimtEdges;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)sms * 8));
    if (f64)
        k64<<<grid, kSimtThreads, smem, s>>>(E, nb, rc, hidden, n_out, (const double*)vec,
                                             (const double*)W1, (const double*)W2, (double*)w,
                                             (double*)h);
    else
        k32<<<grid, kSimtThreads, smem, s>>>(E, nb, (float)rc, hidden, n_out, (const float*)vec,
                                             (const float*)W1, (const float*)W2, (float*)w,
                                             (float*)h);
    return cudaGetLastError();
}

cudaError_t radial_device_status(int* code) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, cgtp_radial_error, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(cgtp_radial_error, &zero, sizeof(int));
    return e;
}

}  // namespace cgtp
