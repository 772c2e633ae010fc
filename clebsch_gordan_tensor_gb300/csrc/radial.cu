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
//   * radial_tc_kernel (fp32, n_basis <= 16, hidden % 8 == 0 and <= 64,
//     n_out % 128 == 0):
//     the last layer -- the only dense contraction, 2 hidden * n_out FLOP per
//     edge -- runs on the tensor cores.  A tile of 128 edges' hidden
//     activations (A, 128 x hidden) and a 128-column slice of W2 (B) sit in
//     shared memory as TF32 "hi" and "lo" parts (x = hi + lo, both TF32);
//     tcgen05.mma accumulates hi*hi + hi*lo + lo*hi into a 128 x 128 fp32
//     accumulator in tensor memory, which keeps fp32 accuracy (the dropped
//     lo*lo term is 2^-22 relative).  Four producer warps build A and B
//     (double-buffered) and one of their threads issues the MMAs; completion
//     arrives on an mbarrier; four epilogue warps read the accumulators
//     (double-buffered in tensor memory) back with tcgen05.ld and store whole
//     row segments.
//   * radial_simt_kernel (fp32 / fp64, any shape): shared-memory tiles and
//     FMA micro-tiles on the CUDA cores.
// Both compute b and h the same way on the CUDA cores.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "internal.hpp"
#include "tcgen05.cuh"

namespace cgtp {

__device__ int cgtp_radial_error;  // nonzero: a bounded wait timed out

// Output element: the compute type, bfloat16 or IEEE binary16 (each rounded
// to nearest even).
template <typename TW, typename T>
__device__ __forceinline__ TW out_cast(T v) {
    if constexpr (std::is_same_v<TW, __nv_bfloat16>) return __float2bfloat16_rn((float)v);
    else if constexpr (std::is_same_v<TW, __half>) return __float2half_rn((float)v);
    else return (TW)v;
}

// Two 16-bit outputs in one word (a in the low half).
template <typename TW>
__device__ __forceinline__ unsigned out_pack2(float a, float b) {
    if constexpr (std::is_same_v<TW, __nv_bfloat16>) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const unsigned*>(&v);
    } else {
        const __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<const unsigned*>(&v);
    }
}

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

template <typename T, typename TW>
__global__ void __launch_bounds__(kSimtThreads)
radial_simt_kernel(int64_t E, int nb, T rc, int hidden, int64_t n_out, const T* __restrict__ vec,
                   const T* __restrict__ W1, const T* __restrict__ W2, TW* __restrict__ w,
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
                    if (c < n_out) w[(e0 + le) * n_out + c] = out_cast<TW>(acc[i][q]);
                }
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------ tensor cores

constexpr int kTcM = 128;          // edges per tile (MMA M, TMEM lanes)
constexpr int kTcN = 128;          // output columns per chunk (MMA N)
constexpr int kTcKMax = 64;        // hidden width held in one tile
constexpr int kTcNbMax = 16;       // basis functions held in registers
constexpr int kTcEpiWarps = 8;     // two per TMEM lane quarter, 64 columns each
constexpr int kTcProdWarps = 4;    // one edge row per thread
constexpr int kTcThreads = 32 * (kTcEpiWarps + kTcProdWarps + 1);  // + the MMA issuer warp
constexpr int kTcBSlots = 2;       // B ring depth
// tensor memory: two fp32 accumulators (columns [0, 256)), then A: the hi part
// of the tile's activations in [256, 256 + hidden), the lo part from 320
constexpr unsigned kTcTmemCols = 512;
constexpr unsigned kTcAhi = 2 * kTcN, kTcAlo = kTcAhi + kTcKMax;
constexpr unsigned kTcB = kTcN * kTcKMax * 4;   // one tf32 part of B (32 KB)
constexpr unsigned kTcStagePitch = 36;                // floats per staged row (conflict-free)
constexpr unsigned kTcStage = 32 * 32 * 4;  // one epilogue warp's 32 x 32 block (either layout)
// the B ring (hi/lo per slot), the epilogue staging blocks, + 1 KB to align
// the 128-byte-swizzled staging blocks on 1024 bytes
constexpr unsigned kTcSmem = 1024 + 2 * kTcBSlots * kTcB + kTcEpiWarps * kTcStage;

// Instruction descriptor, kind::tf32: D fp32 (bits 4-5 = 1), A and B TF32
// (bits 7-9 and 10-12 = 2), both K-major, N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
constexpr uint32_t kTcIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(kTcN >> 3) << 17) |
                              ((uint32_t)(kTcM >> 4) << 24);

__device__ __forceinline__ void mma_tf32(unsigned tmem_d, uint64_t a, uint64_t b, unsigned acc) {
    mma_tf32_n(tmem_d, a, b, kTcIdesc, acc);
}

// W2 packed once per call as the shared-memory image of B: per 128-column
// chunk c, the TF32 "hi" part then the "lo" part, each 128 rows (output
// columns) x hidden in the K-major core-matrix layout (128 * hidden * 4 bytes).
__global__ void radial_pack_kernel(int hidden, int64_t n_out, const float* __restrict__ W2,
                                   unsigned char* __restrict__ img) {
    const int64_t total = (int64_t)hidden * n_out;
    const size_t part = (size_t)kTcN * hidden * 4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int k = (int)(i / n_out);
        const int64_t col = i % n_out;
        const int64_t c = col / kTcN;
        const int n = (int)(col % kTcN);
        const float x = W2[i];
        const float hi = to_tf32(x), lo = to_tf32(x - hi);
        unsigned char* base = img + (size_t)c * 2 * part + kmajor_offset(n, k, kTcN);
        *reinterpret_cast<float*>(base) = hi;
        *reinterpret_cast<float*>(base + part) = lo;
    }
}

// Warp roles, all persistent over this CTA's tiles of 128 edges:
//   producers (warps 8-11): thread = edge row; the hidden activations of the
//     next tile are computed into registers while the current tile is being
//     multiplied, then written to A (TF32 hi/lo) once a_free says the last MMA
//     reading A has completed; arrival on a_full publishes A.
//   issuer (warp 12, one thread): streams the packed W2 chunks into a 2-slot
//     ring with bulk copies (b_full), issues each chunk's MMAs into
//     accumulator chunk % 2 and commits them to mma_done (and, after a tile's
//     last chunk, to a_free).  Each CTA walks the column chunks in an order
//     rotated by its index, so the SMs do not all read the same image at once.
//   epilogue (warps 0-7): per chunk, wait for mma_done, read a 32-row x
//     64-column block of the accumulator (warp % 4 picks the TMEM lane
//     quarter, warp / 4 the column half), arrive on acc_free, then transpose
//     16 x 32 pieces through shared memory and store whole 128-byte row
//     segments.
// Chunk k of this CTA uses phase k / 2 of barriers k % 2 (accumulators and
// ring); tile t uses phase t of a_full and a_free.  Each waiter is never more
// than one phase behind the barrier it waits on.  Every wait is bounded; a
// timeout sets `fail`, each role leaves its loop, and the CTA releases its
// tensor memory after a grace period.
//
// With a tensor map of w (fp32 output, wmap_on), each epilogue warp writes its
// 32 x 32 blocks into a staging block in the 128-byte-swizzled layout and one
// thread stores the block with a 2D tensor copy (rows past E are clipped by
// the map); otherwise the lanes store 128-byte row segments themselves.
template <typename TW>
__global__ void __launch_bounds__(kTcThreads, 1)
radial_tc_kernel(int64_t E, int nb, float rc, int hidden, int64_t n_out,
                 const float* __restrict__ vec, const float* __restrict__ W1,
                 const unsigned char* __restrict__ img, TW* __restrict__ w,
                 float* __restrict__ h, int test_fail_first,
                 const __grid_constant__ CUtensorMap wmap, int wmap_on) {
    extern __shared__ __align__(1024) unsigned char smem_tc[];
    unsigned char* smem = smem_tc + ((1024u - (smem_addr(smem_tc) & 1023u)) & 1023u);
    __shared__ __align__(8) unsigned long long mma_done[2], acc_free[2], b_full[kTcBSlots];
    __shared__ __align__(8) unsigned long long a_full, a_free;
    __shared__ __align__(16) float W1s[kTcNbMax * kTcKMax];
    __shared__ unsigned tmem_base;
    __shared__ int fail;
    unsigned char* ring = smem;  // slot s: hi at 2 s kTcB, lo at (2 s + 1) kTcB
    float* stage_all = reinterpret_cast<float*>(smem + 2 * kTcBSlots * kTcB);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base)),
                     "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            tc_mbar_init(&mma_done[i], 1);
            tc_mbar_init(&acc_free[i], 32 * kTcEpiWarps);
        }
        for (int i = 0; i < kTcBSlots; ++i) tc_mbar_init(&b_full[i], 1);
        tc_mbar_init(&a_full, 32 * kTcProdWarps);
        tc_mbar_init(&a_free, 1);
        fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = tid; i < nb * hidden; i += kTcThreads) W1s[i] = W1[i];
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const unsigned tmem = tmem_base;
    const int64_t nchunk = n_out / kTcN;
    const int64_t tiles = (E + kTcM - 1) / kTcM;
    const int64_t my_tiles =
        tiles > (int64_t)blockIdx.x ? (tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int64_t nk = my_tiles * nchunk;  // chunks this CTA multiplies
    const unsigned part = (unsigned)(kTcN * hidden * 4);

    if (warp >= kTcEpiWarps && warp < kTcEpiWarps + kTcProdWarps) {
        // ---------------------------------------------------------- producers
        const int p = tid - 32 * kTcEpiWarps;
        const float pref = sqrtf(2.0f / rc);
        float hv[kTcKMax] = {};
        auto hidden_row = [&](int64_t t) {  // activations of row p of this CTA's tile t
            const int64_t e = ((int64_t)blockIdx.x + t * gridDim.x) * kTcM + p;
            const bool live = e < E;
            float b[kTcNbMax];
            float r = 0.0f;
            if (live) {
                const float* v = vec + 3 * e;
                r = sqrtf(v[0] * v[0] + v[1] * v[1] + v[2] * v[2]);
            }
#pragma unroll
            for (int n = 0; n < kTcNbMax; ++n)
                b[n] = (live && n < nb) ? bessel_f<float>(n + 1, r, rc, pref) : 0.0f;
#pragma unroll
            for (int k4 = 0; k4 < kTcKMax; k4 += 4) {
                if (k4 >= hidden) break;
                float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
                for (int n = 0; n < kTcNbMax; ++n)
                    if (n < nb) {
                        const float4 wv = *reinterpret_cast<const float4*>(W1s + n * hidden + k4);
                        a0 = fmaf(b[n], wv.x, a0);
                        a1 = fmaf(b[n], wv.y, a1);
                        a2 = fmaf(b[n], wv.z, a2);
                        a3 = fmaf(b[n], wv.w, a3);
                    }
                hv[k4] = live ? silu_f<float>(a0) : 0.0f;
                hv[k4 + 1] = live ? silu_f<float>(a1) : 0.0f;
                hv[k4 + 2] = live ? silu_f<float>(a2) : 0.0f;
                hv[k4 + 3] = live ? silu_f<float>(a3) : 0.0f;
                if (h && live)
                    *reinterpret_cast<float4*>(h + e * hidden + k4) =
                        make_float4(hv[k4], hv[k4 + 1], hv[k4 + 2], hv[k4 + 3]);
            }
        };
        if (my_tiles > 0) hidden_row(0);
        for (int64_t t = 0; t < my_tiles; ++t) {
            // A is free once the previous tile's last MMA has completed
            if (t > 0 && !tc_mbar_wait(&a_free, (unsigned)((t - 1) & 1))) {
                atomicExch(&fail, 1);
                break;
            }
            // this thread's row of A: TMEM lane p (warp % 4 is its lane quarter)
            const unsigned ta = tmem + ((unsigned)(p & ~31) << 16);
#pragma unroll
            for (int k16 = 0; k16 < kTcKMax; k16 += 16) {
                if (k16 >= hidden) break;
                float hi[16], lo[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    hi[q] = to_tf32(hv[k16 + q]);
                    lo[q] = to_tf32(hv[k16 + q] - hi[q]);
                }
                tmem_st16(ta + kTcAhi + (unsigned)k16, hi);
                tmem_st16(ta + kTcAlo + (unsigned)k16, lo);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            tc_mbar_arrive(&a_full);
            if (t + 1 < my_tiles) hidden_row(t + 1);
            if (*(volatile int*)&fail) break;
        }
    } else if (warp == kTcEpiWarps + kTcProdWarps) {
        // ------------------------------------------------------------- issuer
        if (lane == 0 && nk > 0) {
            const unsigned lb = (kTcN / 8) * 128;  // K-slice stride of B
            auto issue_b = [&](int64_t k) {
                const int s = (int)(k % kTcBSlots);
                const int64_t col = (k % nchunk + blockIdx.x) % nchunk;
                const unsigned char* src = img + (size_t)col * 2 * part;
                unsigned char* dst = ring + (size_t)s * 2 * kTcB;
                tc_expect_tx(&b_full[s], 2 * part);
                tc_bulk_g2s(dst, src, part, &b_full[s]);
                tc_bulk_g2s(dst + kTcB, src + part, part, &b_full[s]);
            };
            for (int64_t k = 0; k < nk && k < kTcBSlots - 1; ++k) issue_b(k);
            int64_t k = 0;
            bool ok = true;
            for (int64_t t = 0; t < my_tiles && ok; ++t) {
                // test_fail_first (tests only): the first wait gives up at once
                if (!tc_mbar_wait(&a_full, (unsigned)(t & 1),
                                  test_fail_first && t == 0 ? 0u : 1u << 24)) {
                    ok = false;
                    break;
                }
                for (int64_t c = 0; c < nchunk; ++c, ++k) {
                    const int s = (int)(k & 1), rs = (int)(k % kTcBSlots);
                    // B landed and the accumulator is free (the epilogue has
                    // read chunk k - 2)
                    if (!tc_mbar_wait(&b_full[rs], (unsigned)((k / kTcBSlots) & 1)) ||
                        (k >= 2 && !tc_mbar_wait(&acc_free[s], (unsigned)(((k - 2) >> 1) & 1)))) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const unsigned d = tmem + (unsigned)(s * kTcN);
                    const unsigned bhi = smem_addr(ring + (size_t)rs * 2 * kTcB);
                    for (int k8 = 0; k8 < hidden; k8 += 8) {
                        const unsigned kb = (unsigned)(k8 >> 2) * lb;
                        const unsigned ah = tmem + kTcAhi + (unsigned)k8, al = tmem + kTcAlo + (unsigned)k8;
                        const uint64_t bh = smem_desc(bhi + kb, lb, 128);
                        const uint64_t bl = smem_desc(bhi + kTcB + kb, lb, 128);
                        mma_tf32_tmem_a(d, ah, bh, kTcIdesc, k8 > 0 ? 1u : 0u);
                        mma_tf32_tmem_a(d, ah, bl, kTcIdesc, 1u);
                        mma_tf32_tmem_a(d, al, bh, kTcIdesc, 1u);
                    }
                    tc_commit(&mma_done[s]);
                    if (c == nchunk - 1) tc_commit(&a_free);
                    // refill the ring slot of chunk k - 1 with chunk k + 1 once
                    // chunk k - 1 has been multiplied
                    if (k + kTcBSlots - 1 < nk) {
                        if (k >= 1 &&
                            !tc_mbar_wait(&mma_done[(k - 1) & 1], (unsigned)(((k - 1) >> 1) & 1))) {
                            ok = false;
                            break;
                        }
                        issue_b(k + kTcBSlots - 1);
                    }
                    if (*(volatile int*)&fail) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) atomicExch(&fail, 1);
        }
    } else {
        // ----------------------------------------------------------- epilogue
        float* stage = stage_all + warp * (kTcStage / 4);
        const int quarter = warp & 3, half = warp >> 2;
        int64_t k = 0;
        bool ok = true;
        for (int64_t t = 0; t < my_tiles && ok; ++t) {
            const int64_t e0 = ((int64_t)blockIdx.x + t * gridDim.x) * kTcM + quarter * 32;
            for (int64_t c = 0; c < nchunk; ++c, ++k) {
                const int s = (int)(k & 1);
                const int64_t col0 = ((c + blockIdx.x) % nchunk) * kTcN + half * 64;
                // warp-uniform outcome before the warp-collective tcgen05.ld
                bool got = tc_mbar_wait(&mma_done[s], (unsigned)((k >> 1) & 1));
                got = __all_sync(0xffffffffu, got && !*(volatile int*)&fail);
                if (!got) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const unsigned ta = tmem + ((unsigned)(quarter * 32) << 16) + (unsigned)(s * kTcN + half * 64);
                float v0[32], v1[32];
                tmem_ld32(ta, v0);
                tmem_ld32(ta + 32, v1);
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                tc_mbar_arrive(&acc_free[s]);
                if constexpr (sizeof(TW) == 4) {
                    if (wmap_on) {
                        unsigned char* sb = reinterpret_cast<unsigned char*>(stage);
#pragma unroll
                        for (int blk = 0; blk < 2; ++blk) {
                            const float* v = blk ? v1 : v0;
                            // the staging block's previous store has been read
                            if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                            __syncwarp();
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                *reinterpret_cast<float4*>(sb + sw128_offset(lane, 4 * q)) =
                                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                            __syncwarp();
                            if (lane == 0 && e0 < E) {  // blocks wholly past E store nothing
                                asm volatile(
                                    "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                                    ::"l"(reinterpret_cast<uint64_t>(&wmap)), "r"((int)(col0 + 32 * blk)),
                                    "r"((int)e0), "r"(smem_addr(sb))
                                    : "memory");
                                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                            }
                        }
                        continue;
                    }
                }
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    const float* v = blk ? v1 : v0;
#pragma unroll
                    for (int hp = 0; hp < 2; ++hp) {
                        // rows 16 hp .. 16 hp + 15 of the 32 x 32 block into shared
                        // memory, then out as four 128-byte row segments per instruction
                        if ((lane >> 4) == hp) {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                *reinterpret_cast<float4*>(stage + (lane & 15) * kTcStagePitch + 4 * q) =
                                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                        }
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int r = 4 * i + (lane >> 3);
                            const int64_t e = e0 + 16 * hp + r;
                            const float4 val = *reinterpret_cast<const float4*>(
                                stage + r * kTcStagePitch + (lane & 7) * 4);
                            if (e < E) {
                                TW* dst = w + e * n_out + col0 + blk * 32 + (lane & 7) * 4;
                                if constexpr (sizeof(TW) == 2) {
                                    *reinterpret_cast<uint2*>(dst) =
                                        make_uint2(out_pack2<TW>(val.x, val.y), out_pack2<TW>(val.z, val.w));
                                } else {
                                    *reinterpret_cast<float4*>(dst) = val;
                                }
                            }
                        }
                        __syncwarp();
                    }
                }
            }
        }
        // the tensor stores of this warp have completed
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        if (!ok) atomicExch(&fail, 1);
    }
    __syncthreads();
    if (fail) {
        if (tid == 0) atomicExch(&cgtp_radial_error, 1);
        // let copies and MMAs that may still be in flight finish before the
        // CTA's shared and tensor memory are released
        for (int i = 0; i < 1000; ++i) __nanosleep(1000);
    }
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTcTmemCols)
                     : "memory");
}

// ---------------------------------------------------------------- gradient
//
// Vector-Jacobian product of w = silu(b(r) W1) W2 for a cotangent gw:
//   gh   = gw W2^T,   gpre = gh * silu'(pre),   silu'(a) = s (1 + a (1 - s))
//   gW2  = h^T gw,    gW1 = b^T gpre,           gb = gpre W1^T
//   dr   = sum_n gb_n db_n/dr,  db_n/dr = sqrt(2/rc) (k cos(k r) / r - sin(k r) / r^2)
//   gvec = dr vec / r   (0 at r = 0, where the basis is flat)
// Sums over edges (gW1, gW2) are per-CTA partial rows in the caller's
// workspace, added in fixed order afterwards: deterministic, no atomics.

constexpr int kBwEdges = 32;   // edges per tile
constexpr int kBwCols = 32;    // grad_w / W2 columns staged per step (edge kernel)
constexpr int kBwThreads = 256;
constexpr int kBwGrid1 = 512;  // CTAs of the edge kernel (at most)
constexpr int kBwW2Cols = 256; // output columns per CTA of the W2 kernel
constexpr int kBwW2Rows = 64;  // hidden units per pass of the W2 kernel

static inline int64_t bw_tiles(int64_t E) { return (E + kBwEdges - 1) / kBwEdges; }
static inline int64_t bw_grid1(int64_t E) {
    return std::max<int64_t>(1, std::min<int64_t>(bw_tiles(E), kBwGrid1));
}
static inline int64_t bw_splits(int64_t E, int64_t n_out) {
    const int64_t nc = (n_out + kBwW2Cols - 1) / kBwW2Cols;
    return std::max<int64_t>(1, std::min<int64_t>(bw_tiles(E), std::max<int64_t>(1, kBwGrid1 / nc)));
}

// Basis values of a tile's edges into bS [kBwEdges][nb] and, per edge, r.
template <typename T>
__device__ __forceinline__ void bw_basis(int64_t e0, int ne, int nb, T rc, const T* __restrict__ vec,
                                         T* bS, T* rS) {
    const T pref = sqrt((T)2 / rc);
    for (int i = threadIdx.x; i < kBwEdges * nb; i += blockDim.x) {
        const int le = i / nb, n = i % nb;
        T b = (T)0;
        if (le < ne) {
            const T* v = vec + 3 * (e0 + le);
            const T r = sqrt(v[0] * v[0] + v[1] * v[1] + v[2] * v[2]);
            b = bessel_f<T>(n + 1, r, rc, pref);
            if (n == 0) rS[le] = r;
        }
        bS[i] = b;
    }
}

// Per edge tile: gh (K = n_out), gpre, gb, dr and gvec; gW1 partial row of
// this CTA accumulated in place (the CTA owns the row).
template <typename T>
__global__ void __launch_bounds__(kBwThreads)
radial_bwd_edge_kernel(int64_t E, int nb, T rc, int hidden, int64_t n_out, const T* __restrict__ vec,
                       const T* __restrict__ W1, const T* __restrict__ W2,
                       const T* __restrict__ gw, T* __restrict__ gvec, T* __restrict__ gW1part) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* bS = reinterpret_cast<T*>(smem_raw);         // [kBwEdges][nb]
    T* rS = bS + kBwEdges * nb;                      // [kBwEdges]
    T* preS = rS + kBwEdges;                         // [kBwEdges][hidden]: pre, then gpre
    T* gS = preS + kBwEdges * hidden;                // [kBwEdges][kBwCols + 1]
    T* w2S = gS + kBwEdges * (kBwCols + 1);          // [hidden][kBwCols + 1]
    T* gbS = w2S + hidden * (kBwCols + 1);           // [kBwEdges][nb]
    const int tid = threadIdx.x;
    T* part = gW1part ? gW1part + (int64_t)blockIdx.x * nb * hidden : nullptr;
    if (part)
        for (int i = tid; i < nb * hidden; i += kBwThreads) part[i] = (T)0;
    const T pref = sqrt((T)2 / rc);
    const int eg = tid / 32, hq = tid % 32;  // 4 edges x hidden units hq, hq + 32, ...
    const int nt = (hidden + 31) / 32;       // at most 8
    for (int64_t e0 = (int64_t)blockIdx.x * kBwEdges; e0 < E; e0 += (int64_t)gridDim.x * kBwEdges) {
        const int ne = E - e0 < kBwEdges ? (int)(E - e0) : kBwEdges;
        bw_basis<T>(e0, ne, nb, rc, vec, bS, rS);
        __syncthreads();
        for (int i = tid; i < kBwEdges * hidden; i += kBwThreads) {
            const int le = i / hidden, j = i % hidden;
            T a = (T)0;
            for (int n = 0; n < nb; ++n) a = fma(bS[le * nb + n], __ldg(W1 + n * hidden + j), a);
            preS[i] = a;
        }
        // gh = gw W2^T, columns staged kBwCols at a time
        T acc[4][8];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int t = 0; t < 8; ++t) acc[i][t] = (T)0;
        for (int64_t k0 = 0; k0 < n_out; k0 += kBwCols) {
            const int kc = n_out - k0 < kBwCols ? (int)(n_out - k0) : kBwCols;
            __syncthreads();
            for (int i = tid; i < kBwEdges * kBwCols; i += kBwThreads) {
                const int le = i / kBwCols, k = i % kBwCols;
                gS[le * (kBwCols + 1) + k] = (le < ne && k < kc) ? gw[(e0 + le) * n_out + k0 + k] : (T)0;
            }
            for (int i = tid; i < hidden * kBwCols; i += kBwThreads) {
                const int j = i / kBwCols, k = i % kBwCols;
                w2S[j * (kBwCols + 1) + k] = k < kc ? __ldg(W2 + (int64_t)j * n_out + k0 + k) : (T)0;
            }
            __syncthreads();
            for (int k = 0; k < kBwCols; ++k) {
                T a[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = gS[(eg * 4 + i) * (kBwCols + 1) + k];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    if (t >= nt) break;
                    const int j = hq + 32 * t;
                    const T bv = j < hidden ? w2S[j * (kBwCols + 1) + k] : (T)0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i][t] = fma(a[i], bv, acc[i][t]);
                }
            }
        }
        __syncthreads();
        // gpre = gh * silu'(pre), in place of pre
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int j = hq + 32 * t;
                if (t < nt && j < hidden) {
                    const int idx = (eg * 4 + i) * hidden + j;
                    const T pre = preS[idx];
                    const T sg = (T)1 / ((T)1 + exp(-pre));
                    preS[idx] = acc[i][t] * sg * ((T)1 + pre * ((T)1 - sg));
                }
            }
        __syncthreads();
        // gb = gpre W1^T, then dr and gvec per edge
        for (int i = tid; i < kBwEdges * nb; i += kBwThreads) {
            const int le = i / nb, n = i % nb;
            T v = (T)0;
            for (int j = 0; j < hidden; ++j) v = fma(preS[le * hidden + j], __ldg(W1 + n * hidden + j), v);
            gbS[i] = v;
        }
        __syncthreads();
        if (gvec && tid < ne) {
            const T r = rS[tid];
            T dr = (T)0;
            if (r > (T)0) {
                for (int n = 0; n < nb; ++n) {
                    const T k = (T)(n + 1) * (T)3.14159265358979323846 / rc;
                    dr = fma(gbS[tid * nb + n], pref * (k * cos(k * r) / r - sin(k * r) / (r * r)), dr);
                }
                dr /= r;
            }
            const T* v = vec + 3 * (e0 + tid);
            T* o = gvec + 3 * (e0 + tid);
            o[0] = dr * v[0];
            o[1] = dr * v[1];
            o[2] = dr * v[2];
        }
        // gW1 partial += b^T gpre (this CTA's row, entries owned by threads)
        if (part)
            for (int i = tid; i < nb * hidden; i += kBwThreads) {
                const int n = i / hidden, j = i % hidden;
                T v = part[i];
                for (int le = 0; le < ne; ++le) v = fma(bS[le * nb + n], preS[le * hidden + j], v);
                part[i] = v;
            }
        __syncthreads();
    }
}

// Four consecutive values from shared memory (one 128-bit load for fp32).
template <typename T>
__device__ __forceinline__ void ld4(const T* p, T (&v)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = p[q];
}
template <>
__device__ __forceinline__ void ld4<float>(const float* p, float (&v)[4]) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    v[0] = t.x;
    v[1] = t.y;
    v[2] = t.z;
    v[3] = t.w;
}

// gW2 partial rows: CTA (chunk c, split s) sums h^T gw over its edge range for
// output columns [256 c, 256 c + 256), hidden units in passes of 64.  Thread
// (ty, tx) = (tid / 32, tid % 32) owns hidden rows 8 ty .. 8 ty + 7 and columns
// 4 tx .. 4 tx + 3 and 128 + 4 tx .. 128 + 4 tx + 3: per edge two broadcast
// loads of h and two 128-bit loads of gw feed 64 FMAs.
template <typename T>
__global__ void __launch_bounds__(kBwThreads)
radial_bwd_w2_kernel(int64_t E, int nb, T rc, int hidden, int64_t n_out, int64_t splits,
                     const T* __restrict__ vec, const T* __restrict__ W1,
                     const T* __restrict__ gw, T* __restrict__ part) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* hS = reinterpret_cast<T*>(smem_raw);   // [kBwEdges][kBwW2Rows]
    T* gS = hS + kBwEdges * kBwW2Rows;        // [kBwEdges][kBwW2Cols]
    T* bS = gS + kBwEdges * kBwW2Cols;        // [kBwEdges][nb]
    T* rS = bS + kBwEdges * nb;               // [kBwEdges]
    const int tid = threadIdx.x;
    const int64_t c = blockIdx.x / splits, sp = blockIdx.x % splits;
    const int64_t col0 = c * kBwW2Cols;
    const int ncol = n_out - col0 < kBwW2Cols ? (int)(n_out - col0) : kBwW2Cols;
    const int64_t ea = E * sp / splits, eb = E * (sp + 1) / splits;
    const int ty = tid / 32, tx = tid % 32;
    T* out = part + sp * (int64_t)hidden * n_out;
    for (int j0 = 0; j0 < hidden; j0 += kBwW2Rows) {
        const int nj = hidden - j0 < kBwW2Rows ? hidden - j0 : kBwW2Rows;
        T acc[8][8];
#pragma unroll
        for (int t = 0; t < 8; ++t)
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[t][q] = (T)0;
        for (int64_t e0 = ea; e0 < eb; e0 += kBwEdges) {
            const int ne = eb - e0 < kBwEdges ? (int)(eb - e0) : kBwEdges;
            __syncthreads();
            bw_basis<T>(e0, ne, nb, rc, vec, bS, rS);
            for (int i = tid; i < kBwEdges * kBwW2Cols; i += kBwThreads) {
                const int le = i / kBwW2Cols, k = i % kBwW2Cols;
                gS[i] = (le < ne && k < ncol) ? gw[(e0 + le) * n_out + col0 + k] : (T)0;
            }
            __syncthreads();
            for (int i = tid; i < kBwEdges * kBwW2Rows; i += kBwThreads) {
                const int le = i / kBwW2Rows, j = i % kBwW2Rows;
                T a = (T)0;
                if (le < ne && j < nj) {
                    for (int n = 0; n < nb; ++n) a = fma(bS[le * nb + n], __ldg(W1 + n * hidden + j0 + j), a);
                    a = silu_f<T>(a);
                }
                hS[i] = a;
            }
            __syncthreads();
            for (int le = 0; le < ne; ++le) {
                T ha[4], hb[4], ga[4], gb[4];
                ld4(hS + le * kBwW2Rows + 8 * ty, ha);
                ld4(hS + le * kBwW2Rows + 8 * ty + 4, hb);
                ld4(gS + le * kBwW2Cols + 4 * tx, ga);
                ld4(gS + le * kBwW2Cols + 128 + 4 * tx, gb);
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const T hv = t < 4 ? ha[t] : hb[t - 4];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        acc[t][q] = fma(hv, q < 4 ? ga[q] : gb[q - 4], acc[t][q]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int j = 8 * ty + t;
            if (j >= nj) continue;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int k = (q < 4 ? 4 * tx + q : 128 + 4 * tx + q - 4);
                if (k < ncol) out[(int64_t)(j0 + j) * n_out + col0 + k] = acc[t][q];
            }
        }
    }
}

// ------------------------------------------------- gradient on tensor cores
//
// gh = gw W2^T as an MMA with M = 128 edges, K = n_out (streamed 32 columns
// at a time), and N = 2 hidden: B holds W2^T's TF32 hi part in rows
// [0, hidden) and its lo part in rows [hidden, 2 hidden), so the two MMAs
// A_hi B and A_lo B give hi.hi + lo.hi in columns [0, hidden) and hi.lo +
// lo.lo in [hidden, 2 hidden); gh is their sum (fp32 accuracy, full-rate
// N = 128 instructions for hidden = 64).  The epilogue finishes the chain per
// edge (pre, silu', gpre, gb, dr, gvec) and adds b^T gpre of the tile to the
// CTA's grad_W1 partial row in fixed edge order.

constexpr int kGhK = 32;                 // grad_w columns per chunk
constexpr int kGhThreads = 32 * 9;       // 4 producer, 4 epilogue, 1 issuer warps
constexpr unsigned kGhA = kTcM * kGhK * 4;          // one tf32 part of an A chunk (16 KB)
constexpr unsigned kGhB = 2 * kTcKMax * kGhK * 4;   // a B chunk at hidden = 64 (16 KB)
constexpr int kGhBSlots = 4;                        // ring depth
// ring slot: the chunk of grad_w as copied (128 rows x 32 columns, 128-byte
// swizzle; it is the MMA's hi part), then the chunk of the packed W2 image
constexpr unsigned kGhSlot = kGhA + kGhB;
constexpr int kGhGp = kTcKMax + 1;   // padded row pitch of the gpre / basis staging
constexpr int kGhBp = kTcNbMax + 1;
// + 1 KB to align the swizzled tiles on 1024 bytes
constexpr unsigned kGhSmem =
    1024 + 2 * kGhA + kGhBSlots * kGhSlot + kTcM * kGhGp * 4 + kTcM * kGhBp * 4;

__host__ __device__ constexpr uint32_t gh_idesc(int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);
}

// W2^T packed per 32-column chunk c: rows r < hidden hold hi(W2[r][32 c + k]),
// rows hidden + r hold lo(...), K-major core matrices, 2 hidden x 32 x 4 bytes.
__global__ void radial_pack_t_kernel(int hidden, int64_t n_out, const float* __restrict__ W2,
                                     unsigned char* __restrict__ img) {
    const int64_t total = (int64_t)hidden * n_out;
    const size_t chunk = (size_t)2 * hidden * kGhK * 4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(i / n_out);
        const int64_t col = i % n_out;
        const int64_t c = col / kGhK;
        const int k = (int)(col % kGhK);
        const float x = W2[i];
        const float hi = to_tf32(x), lo = to_tf32(x - hi);
        unsigned char* base = img + (size_t)c * chunk;
        *reinterpret_cast<float*>(base + kmajor_offset(j, k, 2 * hidden)) = hi;
        *reinterpret_cast<float*>(base + kmajor_offset(hidden + j, k, 2 * hidden)) = lo;
    }
}

// Warp roles, persistent over this CTA's tiles of 128 edges, 32 columns of
// grad_w per chunk:
//   issuer (warp 8, one thread): per chunk one tensor-map copy of the grad_w
//     tile (gmap: [E][n_out], box 32 columns x 128 rows, 128-byte swizzle) and
//     one bulk copy of the W2 image's chunk into ring slot k % 4 (b_full),
//     refilled once chunk k - 1 has been multiplied; the MMAs of chunk k
//     (A hi = the copied tile, A lo from the producers) into accumulator
//     t % 2 of tile t, committed to mma_done and, after a tile's last chunk,
//     to acc_full.
//   producers (warps 0-3, thread = edge row): per chunk, read the row from the
//     copied tile, write lo = round_tf32(x - x cut to 10 bits) in the same
//     layout into lo slot k % 2 once chunk k - 2 is done, arrive on a_full.
//     (The tensor core reads the copied fp32 values as TF32, which keeps
//     their top 10 mantissa bits: x = hi + lo with both parts TF32.)
//   epilogue (warps 4-7): as described above.
__global__ void __launch_bounds__(kGhThreads, 1)
radial_bwd_tc_kernel(int64_t E, int nb, float rc, int hidden, int64_t n_out,
                     const float* __restrict__ vec, const float* __restrict__ W1,
                     const unsigned char* __restrict__ img, const __grid_constant__ CUtensorMap gmap,
                     float* __restrict__ gvec, float* __restrict__ gW1part) {
    extern __shared__ __align__(1024) unsigned char smem_tc[];
    unsigned char* smem = smem_tc + ((1024u - (smem_addr(smem_tc) & 1023u)) & 1023u);
    __shared__ __align__(8) unsigned long long a_full[2], mma_done[2], b_full[kGhBSlots];
    __shared__ __align__(8) unsigned long long acc_full[2], acc_free[2];
    __shared__ __align__(16) float W1s[kTcNbMax * kTcKMax];
    __shared__ unsigned tmem_base;
    __shared__ int fail;
    unsigned char* Ring = smem;                               // slot s at s kGhSlot
    unsigned char* Lo = smem + kGhBSlots * kGhSlot;           // lo slot s at s kGhA
    // [128][kGhGp] and [128][kGhBp]: odd pitches keep a warp's row-per-thread
    // stores in distinct banks
    float* gpS = reinterpret_cast<float*>(Lo + 2 * kGhA);
    float* bS = gpS + kTcM * kGhGp;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NB = 2 * hidden;
    const uint32_t idesc = gh_idesc(NB);
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base)),
                     "r"(256u)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            tc_mbar_init(&a_full[i], 4);  // one arrival per producer warp
            tc_mbar_init(&mma_done[i], 1);
            tc_mbar_init(&acc_full[i], 1);
            tc_mbar_init(&acc_free[i], 128);
        }
        for (int i = 0; i < kGhBSlots; ++i) tc_mbar_init(&b_full[i], 1);
        fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = tid; i < nb * hidden; i += kGhThreads) W1s[i] = W1[i];
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const unsigned tmem = tmem_base;
    const int64_t nchunk = n_out / kGhK;
    const int64_t tiles = (E + kTcM - 1) / kTcM;
    const int64_t my_tiles =
        tiles > (int64_t)blockIdx.x ? (tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int64_t nk = my_tiles * nchunk;
    const unsigned bchunk = (unsigned)(NB * kGhK * 4);
    const unsigned bslice = (unsigned)(NB / 8) * 128;  // K-slice stride of the W2 image
    const float pref = sqrtf(2.0f / rc);
    float* part = gW1part + (int64_t)blockIdx.x * nb * hidden;

    if (warp < 4) {
        // ---------------------------------------------------------- producers
        const int p = tid;
        bool ok = true;
        for (int64_t kk = 0; kk < nk && ok; ++kk) {
            const int rs = (int)(kk % kGhBSlots), s = (int)(kk & 1);
            if (!tc_mbar_wait(&b_full[rs], (unsigned)((kk / kGhBSlots) & 1))) {
                ok = false;
                break;
            }
            const unsigned char* raw = Ring + (size_t)rs * kGhSlot;
            float4 v[kGhK / 4];
#pragma unroll
            for (int q4 = 0; q4 < kGhK / 4; ++q4)
                v[q4] = *reinterpret_cast<const float4*>(raw + sw128_offset(p, 4 * q4));
            if (kk >= 2 && !tc_mbar_wait(&mma_done[s], (unsigned)(((kk - 2) >> 1) & 1))) {
                ok = false;
                break;
            }
            unsigned char* lo = Lo + (size_t)s * kGhA;
            auto lo1 = [](float x) {
                return to_tf32(x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u));
            };
#pragma unroll
            for (int q4 = 0; q4 < kGhK / 4; ++q4)
                *reinterpret_cast<float4*>(lo + sw128_offset(p, 4 * q4)) =
                    make_float4(lo1(v[q4].x), lo1(v[q4].y), lo1(v[q4].z), lo1(v[q4].w));
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();  // the warp's stores are ordered before its one arrival
            if ((p & 31) == 0) tc_mbar_arrive(&a_full[s]);
            ok = !*(volatile int*)&fail;
        }
        if (!ok) atomicExch(&fail, 1);
    } else if (warp == 8) {
        // ------------------------------------------------------------- issuer
        if (lane == 0 && nk > 0) {
            // chunk k's B into ring slot k % kGhBSlots; CTAs walk the K chunks
            // in an order rotated by their index (the producers do the same)
            auto issue_b = [&](int64_t k) {
                const int s = (int)(k % kGhBSlots);
                const int64_t t = k / nchunk, col = (k % nchunk + blockIdx.x) % nchunk;
                const int e0 = (int)(((int64_t)blockIdx.x + t * gridDim.x) * kTcM);
                unsigned char* slot = Ring + (size_t)s * kGhSlot;
                // rows past E read as zeros and still count their bytes
                tc_expect_tx(&b_full[s], kGhA + bchunk);
                tma_tile_g2s(slot, &gmap, (int)col * kGhK, e0, &b_full[s]);
                tc_bulk_g2s(slot + kGhA, img + (size_t)col * bchunk, bchunk, &b_full[s]);
            };
            for (int64_t k = 0; k < nk && k < kGhBSlots - 1; ++k) issue_b(k);
            int64_t k = 0;
            bool ok = true;
            for (int64_t t = 0; t < my_tiles && ok; ++t) {
                const int as = (int)(t & 1);
                if (t >= 2 && !tc_mbar_wait(&acc_free[as], (unsigned)(((t - 2) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                const unsigned d = tmem + (unsigned)(as * 128);
                for (int64_t c = 0; c < nchunk; ++c, ++k) {
                    const int s = (int)(k & 1);
                    const int bs = (int)(k % kGhBSlots);
                    if (!tc_mbar_wait(&a_full[s], (unsigned)((k >> 1) & 1)) ||
                        !tc_mbar_wait(&b_full[bs], (unsigned)((k / kGhBSlots) & 1))) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const unsigned ahi = smem_addr(Ring + (size_t)bs * kGhSlot);
                    const unsigned alo = smem_addr(Lo + (size_t)s * kGhA);
                    const unsigned bb = ahi + kGhA;
                    for (int k8 = 0; k8 < kGhK; k8 += 8) {
                        const unsigned ka = (unsigned)k8 * 4, kb = (unsigned)(k8 >> 2) * bslice;
                        const uint64_t bd = smem_desc(bb + kb, bslice, 128);
                        mma_tf32_n(d, smem_desc_sw128(ahi + ka), bd, idesc, (c > 0 || k8 > 0) ? 1u : 0u);
                        mma_tf32_n(d, smem_desc_sw128(alo + ka), bd, idesc, 1u);
                    }
                    tc_commit(&mma_done[s]);
                    if (c == nchunk - 1) tc_commit(&acc_full[as]);
                    // chunk k + 3's B into the slot of chunk k - 1 once that is done
                    if (k + kGhBSlots - 1 < nk) {
                        if (k >= 1 && !tc_mbar_wait(&mma_done[s ^ 1], (unsigned)(((k - 1) >> 1) & 1))) {
                            ok = false;
                            break;
                        }
                        issue_b(k + kGhBSlots - 1);
                    }
                    if (*(volatile int*)&fail) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) atomicExch(&fail, 1);
        }
    } else {
        // ----------------------------------------------------------- epilogue
        const int q = tid - 128;  // edge row of the tile; TMEM lane quarter = warp % 4
        for (int64_t t = 0; t < my_tiles; ++t) {
            const int64_t e = ((int64_t)blockIdx.x + t * gridDim.x) * kTcM + q;
            const bool live = e < E;
            float r = 0.0f, vx = 0.0f, vy = 0.0f, vz = 0.0f;
            if (live) {
                vx = vec[3 * e]; vy = vec[3 * e + 1]; vz = vec[3 * e + 2];
                r = sqrtf(vx * vx + vy * vy + vz * vz);
            }
            float b[kTcNbMax];
#pragma unroll
            for (int n = 0; n < kTcNbMax; ++n) b[n] = (live && n < nb) ? bessel_f<float>(n + 1, r, rc, pref) : 0.0f;
            const int as = (int)(t & 1);
            // every epilogue thread waits (bounded) and the four warps agree on
            // the outcome at their named barrier before any of them leaves
            if (!tc_mbar_wait(&acc_full[as], (unsigned)((t >> 1) & 1))) atomicExch(&fail, 1);
            asm volatile("bar.sync 2, 128;" ::: "memory");
            if (*(volatile int*)&fail) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const unsigned ta = tmem + ((unsigned)((warp & 3) * 32) << 16) + (unsigned)(as * 128);
            float gb[kTcNbMax];
#pragma unroll
            for (int n = 0; n < kTcNbMax; ++n) gb[n] = 0.0f;
#pragma unroll 1
            for (int j0 = 0; j0 < hidden; j0 += 8) {  // hidden % 8 == 0
                float d0[8], d1[8];
                tmem_ld8(ta + (unsigned)j0, d0);
                tmem_ld8(ta + (unsigned)(hidden + j0), d1);
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int j = j0 + jj;
                    float pre = 0.0f;
#pragma unroll
                    for (int n = 0; n < kTcNbMax; ++n)
                        if (n < nb) pre = fmaf(b[n], W1s[n * hidden + j], pre);
                    const float sg = 1.0f / (1.0f + expf(-pre));
                    const float gp = live ? (d0[jj] + d1[jj]) * sg * (1.0f + pre * (1.0f - sg)) : 0.0f;
                    gpS[q * kGhGp + j] = gp;
#pragma unroll
                    for (int n = 0; n < kTcNbMax; ++n)
                        if (n < nb) gb[n] = fmaf(gp, W1s[n * hidden + j], gb[n]);
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            tc_mbar_arrive(&acc_free[as]);
#pragma unroll
            for (int n = 0; n < kTcNbMax; ++n)
                if (n < nb) bS[q * kGhBp + n] = b[n];
            if (gvec && live) {
                float dr = 0.0f;
                if (r > 0.0f) {
#pragma unroll
                    for (int n = 0; n < kTcNbMax; ++n)
                        if (n < nb) {
                            const float kk = (float)(n + 1) * 3.14159265358979323846f / rc;
                            dr = fmaf(gb[n], pref * (kk * cosf(kk * r) / r - sinf(kk * r) / (r * r)), dr);
                        }
                    dr /= r;
                }
                gvec[3 * e] = dr * vx;
                gvec[3 * e + 1] = dr * vy;
                gvec[3 * e + 2] = dr * vz;
            }
            // grad_W1 partial += b^T gpre over the tile's edges, fixed order
            asm volatile("bar.sync 2, 128;" ::: "memory");
            for (int i = q; i < nb * hidden; i += 128) {
                const int n = i / hidden, j = i % hidden;
                float v = t == 0 ? 0.0f : part[i];
                for (int le = 0; le < kTcM; ++le) v = fmaf(bS[le * kGhBp + n], gpS[le * kGhGp + j], v);
                part[i] = v;
            }
            asm volatile("bar.sync 2, 128;" ::: "memory");
        }
        if (my_tiles == 0)
            for (int i = q; i < nb * hidden; i += 128) part[i] = 0.0f;
    }
    __syncthreads();
    if (fail) {
        if (tid == 0) atomicExch(&cgtp_radial_error, 1);
        for (int i = 0; i < 1000; ++i) __nanosleep(1000);
    }
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256u)
                     : "memory");
}

static bool radial_bwd_tc_eligible(bool f64, int nb, int hidden, int64_t n_out) {
    return !f64 && nb <= kTcNbMax && hidden % 8 == 0 && hidden <= kTcKMax && n_out % kGhK == 0;
}

// Workspace: [packed W2^T image, tensor-core path only][grad_W1 partial rows]
// [grad_W2 partial rows]; every region starts 16-byte aligned.
static size_t bw_image_bytes(bool f64, int nb, int hidden, int64_t n_out) {
    return radial_bwd_tc_eligible(f64, nb, hidden, n_out) ? (size_t)n_out * 2 * hidden * 4 : 0;
}

// The hidden activations h [E, hidden] stored for the tensor-core grad_W2.
static size_t bw_h_bytes(bool f64, int64_t E, int hidden, int64_t n_out) {
    return !f64 && radial_w2_tc_eligible(hidden, n_out) ? ((size_t)E * hidden * 4 + 255) / 256 * 256
                                                         : 0;
}

size_t radial_backward_workspace_bytes(bool f64, int64_t E, int nb, int hidden, int64_t n_out) {
    const size_t es = f64 ? 8 : 4;
    const size_t p1 = ((size_t)bw_grid1(E) * nb * hidden * es + 15) / 16 * 16;
    const size_t p2 = ((size_t)bw_splits(E, n_out) * hidden * n_out * es + 255) / 256 * 256;
    return bw_image_bytes(f64, nb, hidden, n_out) + p1 + p2 + bw_h_bytes(f64, E, hidden, n_out);
}

// h[e] = silu(b(|vec[e]|) W1), one thread per edge (for the tensor-core grad_W2).
__global__ void __launch_bounds__(128) radial_h_kernel(int64_t E, int nb, float rc, int hidden,
                                                       const float* __restrict__ vec,
                                                       const float* __restrict__ W1,
                                                       float* __restrict__ h) {
    const float pref = sqrtf(2.0f / rc);
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E;
         e += (int64_t)gridDim.x * blockDim.x) {
        const float* v = vec + 3 * e;
        const float r = sqrtf(v[0] * v[0] + v[1] * v[1] + v[2] * v[2]);
        float b[kTcNbMax];
#pragma unroll
        for (int n = 0; n < kTcNbMax; ++n) b[n] = n < nb ? bessel_f<float>(n + 1, r, rc, pref) : 0.0f;
        for (int k4 = 0; k4 < hidden; k4 += 4) {
            float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int n = 0; n < kTcNbMax; ++n)
                if (n < nb) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) a[q] = fmaf(b[n], __ldg(W1 + n * hidden + k4 + q), a[q]);
                }
            *reinterpret_cast<float4*>(h + e * hidden + k4) =
                make_float4(silu_f<float>(a[0]), silu_f<float>(a[1]), silu_f<float>(a[2]),
                            silu_f<float>(a[3]));
        }
    }
}

// Tensor map of grad_w [E][n_out] (fp32) for the gh kernel: tiles of 32
// columns x 128 rows with 128-byte swizzle, rows past E read as zeros.
static bool gh_map(const float* gw, int64_t E, int64_t n_out, CUtensorMap* m) {
    const auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
    if (!encode || E < 1 || E > 0x7fffffff || n_out % kGhK != 0 || ((uintptr_t)gw & 15) != 0)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)n_out, (cuuint64_t)E};
    const cuuint64_t strides[1] = {(cuuint64_t)n_out * 4};
    const cuuint32_t box[2] = {(cuuint32_t)kGhK, (cuuint32_t)kTcM};
    const cuuint32_t es[2] = {1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(gw), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_radial_backward(bool f64, bool tensor_cores, int64_t E, int nb, double rc,
                                   int hidden, int64_t n_out, const void* vec, const void* W1,
                                   const void* W2, const void* gw, void* gvec, void* gW1,
                                   void* gW2, void* ws, cudaStream_t s) {
    const size_t es = f64 ? 8 : 4;
    const int64_t g1 = bw_grid1(E), sp = bw_splits(E, n_out);
    const int64_t nc = (n_out + kBwW2Cols - 1) / kBwW2Cols;
    unsigned char* img = (unsigned char*)ws;
    unsigned char* p1 = img + bw_image_bytes(f64, nb, hidden, n_out);
    unsigned char* p2 = p1 + ((size_t)g1 * nb * hidden * es + 15) / 16 * 16;
    CUtensorMap gmap{};
    const bool tc = tensor_cores && radial_bwd_tc_eligible(f64, nb, hidden, n_out) &&
                    (gvec || gW1) && gh_map((const float*)gw, E, n_out, &gmap);
    const size_t sm1 = es * ((size_t)kBwEdges * nb + kBwEdges + (size_t)kBwEdges * hidden +
                             (size_t)kBwEdges * (kBwCols + 1) + (size_t)hidden * (kBwCols + 1) +
                             (size_t)kBwEdges * nb);
    const size_t sm2 = es * ((size_t)kBwEdges * kBwW2Rows + (size_t)kBwEdges * kBwW2Cols +
                             (size_t)kBwEdges * nb + kBwEdges);
    cudaError_t e;
    if ((gvec || gW1) && tc) {
        int dev = 0, sms = 0;
        if ((e = cudaGetDevice(&dev))) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
        const int64_t total = (int64_t)hidden * n_out;
        const unsigned pg =
            (unsigned)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, (int64_t)sms * 8));
        radial_pack_t_kernel<<<pg, 256, 0, s>>>(hidden, n_out, (const float*)W2, img);
        count_launch();
        if ((e = cudaGetLastError())) return e;
        if ((e = cudaFuncSetAttribute(radial_bwd_tc_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGhSmem)))
            return e;
        const int64_t tiles = (E + kTcM - 1) / kTcM;
        const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(tiles, sms));
        radial_bwd_tc_kernel<<<(unsigned)grid, kGhThreads, kGhSmem, s>>>(
            E, nb, (float)rc, hidden, n_out, (const float*)vec, (const float*)W1, img, gmap,
            (float*)gvec, (float*)p1);
        count_launch();
        if ((e = cudaGetLastError())) return e;
        if (gW1 && (e = launch_reduce_rows(false, p1, grid, (int64_t)nb * hidden, gW1, s))) return e;
    } else if (gvec || gW1) {
        if (f64) {
            auto* k = radial_bwd_edge_kernel<double>;
            if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)))
                return e;
            k<<<(unsigned)g1, kBwThreads, sm1, s>>>(E, nb, rc, hidden, n_out, (const double*)vec,
                                                   (const double*)W1, (const double*)W2,
                                                   (const double*)gw, (double*)gvec,
                                                   gW1 ? (double*)p1 : nullptr);
            count_launch();
        } else {
            auto* k = radial_bwd_edge_kernel<float>;
            if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)))
                return e;
            k<<<(unsigned)g1, kBwThreads, sm1, s>>>(E, nb, (float)rc, hidden, n_out,
                                                   (const float*)vec, (const float*)W1,
                                                   (const float*)W2, (const float*)gw,
                                                   (float*)gvec, gW1 ? (float*)p1 : nullptr);
            count_launch();
        }
        if ((e = cudaGetLastError())) return e;
        if (gW1 && (e = launch_reduce_rows(f64, p1, g1, (int64_t)nb * hidden, gW1, s))) return e;
    }
    if (gW2 && !f64 && tensor_cores && radial_w2_tc_eligible(hidden, n_out) && nb <= kTcNbMax &&
        ((uintptr_t)gw & 15) == 0) {
        // h into the workspace, then h^T grad_w on the tensor cores
        float* hbuf = reinterpret_cast<float*>(
            p2 + ((size_t)sp * hidden * n_out * es + 255) / 256 * 256);
        const unsigned hg = (unsigned)std::max<int64_t>(1, std::min<int64_t>((E + 127) / 128, 65535));
        radial_h_kernel<<<hg, 128, 0, s>>>(E, nb, (float)rc, hidden, (const float*)vec,
                                           (const float*)W1, hbuf);
        count_launch();
        if ((e = cudaGetLastError())) return e;
        if ((e = launch_radial_w2_tc(E, hidden, n_out, hbuf, (const float*)gw, (float*)p2, sp, s)))
            return e;
        if ((e = launch_reduce_rows(false, p2, sp, (int64_t)hidden * n_out, gW2, s))) return e;
    } else if (gW2) {
        if (f64) {
            auto* k = radial_bwd_w2_kernel<double>;
            if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2)))
                return e;
            k<<<(unsigned)(nc * sp), kBwThreads, sm2, s>>>(E, nb, rc, hidden, n_out, sp,
                                                          (const double*)vec, (const double*)W1,
                                                          (const double*)gw, (double*)p2);
            count_launch();
        } else {
            auto* k = radial_bwd_w2_kernel<float>;
            if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2)))
                return e;
            k<<<(unsigned)(nc * sp), kBwThreads, sm2, s>>>(E, nb, (float)rc, hidden, n_out, sp,
                                                          (const float*)vec, (const float*)W1,
                                                          (const float*)gw, (float*)p2);
            count_launch();
        }
        if ((e = cudaGetLastError())) return e;
        if ((e = launch_reduce_rows(f64, p2, sp, (int64_t)hidden * n_out, gW2, s))) return e;
    }
    return cudaSuccess;
}

// ------------------------------------------------------------------ host

bool radial_tc_eligible(bool f64, int nb, int hidden, int64_t n_out, const void* vec,
                        const void* W2, const void* w, const void* h) {
    auto a16 = [](const void* p) { return p == nullptr || ((uintptr_t)p % 16) == 0; };
    return !f64 && nb <= kTcNbMax && hidden % 8 == 0 && hidden <= kTcKMax && n_out % kTcN == 0 &&
           a16(w) && a16(h) && a16(W2) && a16(vec);
}

size_t radial_workspace_bytes(bool f64, int nb, int hidden, int64_t n_out) {
    if (!radial_tc_eligible(f64, nb, hidden, n_out, nullptr, nullptr, nullptr, nullptr)) return 0;
    return (size_t)n_out * hidden * 8;  // TF32 hi and lo parts of W2, packed
}

// The fp32 launches for output element TW (float, bfloat16 or binary16).
template <typename TW>
static cudaError_t radial_forward_f32(bool tensor_cores, int sms, int64_t E, int nb, float rc,
                                      int hidden, int64_t n_out, const float* vec,
                                      const float* W1, const float* W2, TW* w, float* h,
                                      void* ws, cudaStream_t s, bool test_fail) {
    cudaError_t e;
    if (tensor_cores) {
        e = cudaFuncSetAttribute(radial_tc_kernel<TW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kTcSmem);
        if (e != cudaSuccess) return e;
        const int64_t total = (int64_t)hidden * n_out;
        const unsigned pg =
            (unsigned)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, (int64_t)sms * 8));
        radial_pack_kernel<<<pg, 256, 0, s>>>(hidden, n_out, W2, (unsigned char*)ws);
        count_launch();
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        const int64_t tiles = (E + kTcM - 1) / kTcM;
        const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(tiles, sms));
        // fp32 output: stores through a tensor map of w [E][n_out] (32 x 32
        // boxes, 128-byte swizzle, rows past E clipped)
        CUtensorMap wmap{};
        int wmap_on = 0;
        const auto encode =
            reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
        if (sizeof(TW) == 4 && encode && E >= 1 && E <= 0x7fffffff && ((uintptr_t)w & 15) == 0) {
            const cuuint64_t dims[2] = {(cuuint64_t)n_out, (cuuint64_t)E};
            const cuuint64_t strides[1] = {(cuuint64_t)n_out * 4};
            const cuuint32_t box[2] = {32, 32};
            const cuuint32_t es[2] = {1, 1};
            wmap_on = encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, (void*)w, dims, strides, box,
                             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_NONE,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        }
        radial_tc_kernel<TW><<<grid, kTcThreads, kTcSmem, s>>>(E, nb, rc, hidden, n_out, vec, W1,
                                                               (const unsigned char*)ws, w, h,
                                                               test_fail ? 1 : 0, wmap, wmap_on);
        count_launch();
        return cudaGetLastError();
    }
    const size_t smem = (size_t)kSimtEdges * (nb + hidden) * 4;
    const int64_t tiles = (E + kSimtEdges - 1) / kSimtEdges;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)sms * 8));
    auto* k = radial_simt_kernel<float, TW>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kSimtThreads, smem, s>>>(E, nb, rc, hidden, n_out, vec, W1, W2, w, h);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_radial_forward(bool f64, bool tensor_cores, int out16, int64_t E, int nb,
                                  double rc, int hidden, int64_t n_out, const void* vec,
                                  const void* W1, const void* W2, void* w, void* h, void* ws,
                                  size_t ws_bytes, cudaStream_t s, bool test_fail) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    (void)ws_bytes;
    if (f64) {
        const size_t smem = (size_t)kSimtEdges * (nb + hidden) * 8;
        const int64_t tiles = (E + kSimtEdges - 1) / kSimtEdges;
        const unsigned grid =
            (unsigned)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)sms * 8));
        auto* k = radial_simt_kernel<double, double>;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k<<<grid, kSimtThreads, smem, s>>>(E, nb, rc, hidden, n_out, (const double*)vec,
                                           (const double*)W1, (const double*)W2, (double*)w,
                                           (double*)h);
        count_launch();
        return cudaGetLastError();
    }
    const float* v = (const float*)vec;
    const float* a = (const float*)W1;
    const float* b = (const float*)W2;
    if (out16 == 1)
        return radial_forward_f32(tensor_cores, sms, E, nb, (float)rc, hidden, n_out, v, a, b,
                                  (__nv_bfloat16*)w, (float*)h, ws, s, test_fail);
    if (out16 == 2)
        return radial_forward_f32(tensor_cores, sms, E, nb, (float)rc, hidden, n_out, v, a, b,
                                  (__half*)w, (float*)h, ws, s, test_fail);
    return radial_forward_f32(tensor_cores, sms, E, nb, (float)rc, hidden, n_out, v, a, b,
                              (float*)w, (float*)h, ws, s, test_fail);
}

cudaError_t radial_device_status(int* code) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, cgtp_radial_error, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(cgtp_radial_error, &zero, sizeof(int));
    return e;
}

}  // namespace cgtp
