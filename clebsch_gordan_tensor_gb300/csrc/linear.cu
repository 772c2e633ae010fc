// Per-irrep channel mixing ("linear" layer, the dense 'uvw' contraction)
// (sm_103a).
//
// NVIDIA's SE(3)-Transformer blog, section "TFN fusion": the pairwise degree
// convolutions are summed per output degree, and the fused layers concatenate
// degrees so that the channel contractions become dense products with sizes
// that are multiples of 16, for the tensor cores.  For an instruction j that
// joins input irrep i and output irrep o (same l and parity) with a matrix
// W_j [mul_in, mul_out]:
//     out[n, o, m, w] += sum_u x[n, i, m, u] W_j[u, w]          (m = -l..l)
// Rows (n, m) of one output block form a GEMM with M = n * (2l+1) rows,
// K = the concatenated u ranges of every instruction into that block and
// N = mul_out.  The gradient in x is the same GEMM with W_j transposed, one
// block per input irrep; the gradient in W_j sums x^T g over the rows.
//
// Kernels:
//   * linear_tc_kernel (fp32; every mul a multiple of 32, mul_out <= 256,
//     16-byte aligned rows): 128-row tiles on tcgen05 with kind::tf32.  A (the
//     rows, as TF32 hi + lo parts) is written into tensor memory by producer
//     warps; B (the packed hi/lo image of W, one bulk copy per 32-wide K
//     chunk) streams through a shared-memory ring; one thread issues hi*hi +
//     hi*lo + lo*hi into fp32 accumulators in tensor memory (the dropped
//     lo*lo term is about 2^-21 relative); epilogue warps store the results.
//   * linear_simt_kernel (fp32 / fp64, any shape): shared-memory tiles and 4 x 4
//     FMA micro-tiles on the CUDA cores.
//   * linear_wgrad_tc_kernel (fp32 tensor-core layers, mul_out <= 128): the
//     gradient in W on tcgen05, K = the rows: X^T in tensor memory, G^T as a
//     stacked K-major image, per-unit partial sums over a fixed row range;
//     linear_wgrad_kernel does the same on the CUDA cores for other layers.
//     The partial rows are added in a fixed order (deterministic).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "internal.hpp"
#include "tcgen05.cuh"

namespace cgtp {

__device__ int cgtp_linear_error;  // nonzero: a bounded wait timed out

// ------------------------------------------------------------ descriptors

// One output block of a GEMM pass (an output irrep in the forward, an input
// irrep in the x-gradient): rows (n, m), m < d, written at
// out[n * out_stride + out_off + m * ncols + c] for c < ncols.
struct LinBlock {
    int out_off, ncols, d, chunk0, nchunk;
};
// One K chunk of a block: columns a_off + m * a_mul + k0 + k (k < kc) of the
// input rows, against B[k][c] = W[w_off + (k0 + k) * w_ks + c * w_ns]; the
// packed tensor-core image of the chunk starts at byte img_off.
struct LinChunk {
    int a_off, a_mul, k0, kc, w_off, w_ks, w_ns, img_off;
    int src;  // source irrep of the chunk (its path, for a tensor-product source)
};

constexpr int kLinMaxBlocks = 32;
constexpr int kLinMaxChunks = 384;
struct LinDesc {
    int nblocks, nchunks;
    int64_t in_stride, out_stride;
    LinBlock blk[kLinMaxBlocks];
    LinChunk ch[kLinMaxChunks];
    // unit order of the tensor-core kernel: groups of blocks that read the
    // same input rows (same d, same chunk sources), tile-major inside a group,
    // so that the blocks of a group read a row tile at the same time and all
    // but the first read come from L2 (the x-gradient of a layer whose output
    // irreps feed several instructions); group g holds grp_nb[g] blocks,
    // grp_b[grp_b0[g] ..], each of grp_nt[g] tiles, from unit grp_u0[g]
    int ngrp;
    int grp_nb[kLinMaxBlocks], grp_b0[kLinMaxBlocks], grp_b[kLinMaxBlocks];
    int64_t grp_nt[kLinMaxBlocks], grp_u0[kLinMaxBlocks + 1];  // per launch
};

// --------------------------------------------------------------- CUDA cores

constexpr int kLsT = 64;   // rows per tile
constexpr int kLsC = 64;   // columns per tile
constexpr int kLsK = 16;   // K per shared-memory step
constexpr int kLsThreads = 256;

// grid: x = row tile, y = column tile, z = block
template <typename T>
__global__ void __launch_bounds__(kLsThreads)
linear_simt_kernel(const __grid_constant__ LinDesc D, int64_t n, const T* __restrict__ x,
                   const T* __restrict__ W, T* __restrict__ out) {
    const LinBlock& B = D.blk[blockIdx.z];
    const int64_t rows = n * B.d;
    const int64_t r0 = (int64_t)blockIdx.x * kLsT;
    const int c0 = blockIdx.y * kLsC;
    if (r0 >= rows || c0 >= B.ncols) return;
    __shared__ T As[kLsK][kLsT + 1];
    __shared__ T Bs[kLsK][kLsC];
    const int tid = threadIdx.x, tr = tid / 16, tc = tid % 16;
    T acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = (T)0;
    for (int ci = 0; ci < B.nchunk; ++ci) {
        const LinChunk& C = D.ch[B.chunk0 + ci];
        for (int kk = 0; kk < C.kc; kk += kLsK) {
            __syncthreads();
            for (int i = tid; i < kLsK * kLsT; i += kLsThreads) {
                const int k = i % kLsK, r = i / kLsK;
                const int64_t R = r0 + r;
                T v = (T)0;
                if (R < rows && kk + k < C.kc) {
                    const int64_t item = R / B.d;
                    const int m = (int)(R % B.d);
                    v = x[item * D.in_stride + C.a_off + (int64_t)m * C.a_mul + C.k0 + kk + k];
                }
                As[k][r] = v;
            }
            for (int i = tid; i < kLsK * kLsC; i += kLsThreads) {
                const int c = i % kLsC, k = i / kLsC;
                T v = (T)0;
                if (c0 + c < B.ncols && kk + k < C.kc)
                    v = W[C.w_off + (int64_t)(C.k0 + kk + k) * C.w_ks + (int64_t)(c0 + c) * C.w_ns];
                Bs[k][c] = v;
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < kLsK; ++k) {
                T a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[k][tr * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = Bs[k][tc + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fma(a[i], b[j], acc[i][j]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t R = r0 + tr * 4 + i;
        if (R >= rows) continue;
        const int64_t item = R / B.d;
        const int m = (int)(R % B.d);
        T* o = out + item * D.out_stride + B.out_off + (int64_t)m * B.ncols;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = c0 + tc + 16 * j;
            if (c < B.ncols) o[c] = acc[i][j];
        }
    }
}

// Zero the output columns of blocks that no instruction reaches.
template <typename T>
__global__ void linear_zero_kernel(int64_t n, int64_t stride, int off, int width,
                                   T* __restrict__ out) {
    const int64_t total = n * width;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x)
        out[(i / width) * stride + off + i % width] = (T)0;
}

// ------------------------------------------------------------- W gradient

// Instruction j of the gradient: gW_j[u, w] = sum_{n, m} x[n, xo + m mi + u]
// g[n, go + m mo + w]; tile0 = first 32 x 32 tile of j in the flat tile list.
struct LinGrad {
    int xo, mi, go, mo, d, w_off, tile0;
    int mt0;  // first 128-row M tile of j in the tensor-core kernel's list
    int ldw;  // row stride of gW_j in the output (mo for the layer's own layout)
    int tr;   // 1: gW_j is stored transposed, element (u, w) at w_off + w ldw + u
};
constexpr int kLinMaxGrad = 128;
constexpr int kLinMaxMT = 2 * kLinMaxGrad;  // M tiles: multiplicities up to 256
constexpr int kLinMaxCls = 16;
struct LinGradDesc {
    int ninstr, ntiles, nmt;  // nmt: M tiles (128 input channels) over all instructions
    int64_t x_stride, g_stride, nw;
    LinGrad g[kLinMaxGrad];
    // order of the tensor-core kernel's units (wgrad_schedule): classes of M
    // tiles with equal rows per item, widest first; class c holds cls_n[c]
    // consecutive entries of qord (M tile indices)
    int ncls;
    int cls_n[kLinMaxCls];
    int qord[kLinMaxMT];
};

constexpr int kLgRows = 32;  // rows staged per step

// The tensor-core weight gradient's unit order: M tiles grouped into classes
// of equal rows per item (d), widest first; inside a class by g offset (the
// output irrep), then tile index.
static void wgrad_schedule(LinGradDesc& G) {
    std::vector<int> q(G.nmt), dq(G.nmt), go(G.nmt);
    for (int j = 0; j < G.ninstr; ++j) {
        const int end = j + 1 < G.ninstr ? G.g[j + 1].mt0 : G.nmt;
        for (int t = G.g[j].mt0; t < end; ++t) {
            dq[t] = G.g[j].d;
            go[t] = G.g[j].go;
        }
    }
    for (int t = 0; t < G.nmt; ++t) q[t] = t;
    std::stable_sort(q.begin(), q.end(), [&](int a, int b) {
        if (dq[a] != dq[b]) return dq[a] > dq[b];
        return go[a] < go[b];
    });
    G.ncls = 0;
    for (int i = 0; i < G.nmt; ++i) {
        G.qord[i] = q[i];
        // widths beyond the class table share the last class
        if (i == 0 || (dq[q[i]] != dq[q[i - 1]] && G.ncls < kLinMaxCls)) G.cls_n[G.ncls++] = 0;
        ++G.cls_n[G.ncls - 1];
    }
    if (G.ncls == 0) {
        G.ncls = 1;
        G.cls_n[0] = 0;
    }
}

// grid: x = tile (instruction, u tile, w tile), y = row split.  Split s covers
// items [s * per, (s + 1) * per) and writes its partial sums to
// partial[s * nw + ...]; every partial element is written.
template <typename T>
__global__ void __launch_bounds__(256)
linear_wgrad_kernel(const __grid_constant__ LinGradDesc D, int64_t n, int64_t per,
                    const T* __restrict__ x, const T* __restrict__ g, T* __restrict__ partial) {
    int j = 0;
    while (j + 1 < D.ninstr && D.g[j + 1].tile0 <= (int)blockIdx.x) ++j;
    const LinGrad& G = D.g[j];
    const int t = blockIdx.x - G.tile0;
    const int ntw = (G.mo + 31) / 32;
    const int u0 = (t / ntw) * 32, w0 = (t % ntw) * 32;
    const int tid = threadIdx.x, ty = tid >> 5, tx = tid & 31;
    __shared__ T Xs[kLgRows][33];
    __shared__ T Gs[kLgRows][33];
    T acc[4] = {(T)0, (T)0, (T)0, (T)0};
    const int64_t i0 = (int64_t)blockIdx.y * per;
    const int64_t i1 = min(n, i0 + per);
    const int64_t r0 = i0 * G.d, r1 = i1 > i0 ? i1 * G.d : r0;
    for (int64_t rb = r0; rb < r1; rb += kLgRows) {
        __syncthreads();
        for (int i = tid; i < kLgRows * 32; i += 256) {
            const int r = i >> 5, c = i & 31;
            const int64_t R = rb + r;
            T xv = (T)0, gv = (T)0;
            if (R < r1) {
                const int64_t item = R / G.d;
                const int m = (int)(R % G.d);
                if (u0 + c < G.mi) xv = x[item * D.x_stride + G.xo + (int64_t)m * G.mi + u0 + c];
                if (w0 + c < G.mo) gv = g[item * D.g_stride + G.go + (int64_t)m * G.mo + w0 + c];
            }
            Xs[r][c] = xv;
            Gs[r][c] = gv;
        }
        __syncthreads();
#pragma unroll 8
        for (int r = 0; r < kLgRows; ++r) {
            const T gv = Gs[r][tx];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = fma(Xs[r][ty * 4 + q], gv, acc[q]);
        }
    }
    T* P = partial + (int64_t)blockIdx.y * D.nw + G.w_off;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int u = u0 + ty * 4 + q, w = w0 + tx;
        if (u < G.mi && w < G.mo)
            P[G.tr ? (int64_t)w * G.ldw + u : (int64_t)u * G.ldw + w] = acc[q];
    }
}

// ------------------------------------------------------------ tensor cores

constexpr int kLtM = 128;                    // rows per tile (MMA M, TMEM lanes)
constexpr int kLtK = 32;                     // K per chunk
constexpr int kLtEpiWarps = 4;               // one per TMEM lane quarter
constexpr int kLtProdWarps = 8;              // two per lane quarter, 16 K columns each
constexpr int kLtThreads = 32 * (kLtEpiWarps + kLtProdWarps + 2);  // + MMA issuer, loader
constexpr unsigned kLtTmemCols = 512;        // accumulators in [0, 256), A stages in [256, 512)
constexpr unsigned kLtAcol = 256;            // first column of A stage 0 (hi 32, lo 32 per stage)

// Dynamic shared memory: RB B slots (hi + lo of up to nmax rows), the
// epilogue warps' staging blocks and the block / chunk tables.
constexpr unsigned kLtStagePitch = 36;  // floats per staged epilogue row (conflict-free)
// Epilogue staging per warp: 32 rows x (nmax + 4) floats holding a whole tile
// row block (stacked products), else one 32 x 32 block at a time.
__host__ __device__ constexpr unsigned lt_stage_pitch(int nmax, bool wide) {
    return wide ? (unsigned)nmax + 4 : kLtStagePitch;
}
__host__ __device__ constexpr unsigned lt_smem_bytes(int nmax, int RB, bool wide, bool tpa = false) {
    return (unsigned)RB * 2u * (unsigned)nmax * kLtK * 4 +
           kLtEpiWarps * 32 * lt_stage_pitch(nmax, wide) * 4 +
           (unsigned)((kLinMaxBlocks + 1) * sizeof(LinBlock) + kLinMaxChunks * sizeof(LinChunk)) +
           (tpa ? (unsigned)sizeof(LinTpDesc) : 0u);
}

// Kernel argument of the tensor-product source (empty without one).
template <bool TPA>
struct TpArg {};
template <>
struct TpArg<true> {
    LinTpDesc d;
    const float* x1;
    int64_t x1_stride;
    const float* t;  // T rows, tdim floats per sample
};

// Bounded wait that sleeps between polls (about a second at most): for the
// producer and epilogue warps, whose polling would otherwise compete with the
// MMA issuer for the shared-memory pipe.
__device__ __forceinline__ bool tc_mbar_wait_sleep(unsigned long long* b, unsigned parity) {
    const unsigned a = smem_addr(b);
    for (unsigned it = 0; it < (1u << 22); ++it) {
        unsigned ok;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
            : "=r"(ok) : "r"(a), "r"(parity) : "memory");
        if (ok) return true;
        __nanosleep(128);
    }
    return false;
}

// R / d for a row index and a block's 2l+1 (32-bit division when R fits).
__device__ __forceinline__ int64_t row_item(int64_t R, int d) {
    return R < 0x7fffffff ? (int64_t)((unsigned)R / (unsigned)d) : R / d;
}



// Packed B image of every chunk: rows = output columns c < ncols, K-major
// core matrices, the TF32 hi part then the lo part (ncols * 32 * 4 bytes each);
// stacked: one image of 2 ncols rows, hi in rows c, lo in rows ncols + c (the
// B operand of a single N = 2 ncols product A_hi [B_hi | B_lo]).
// grid: x = chunk.
__global__ void linear_pack_kernel(const __grid_constant__ LinDesc D, const float* __restrict__ W,
                                   unsigned char* __restrict__ img, bool stacked) {
    const int ci = blockIdx.x;
    int b = 0;
    while (b + 1 < D.nblocks && D.blk[b + 1].chunk0 <= ci) ++b;
    const int N = D.blk[b].ncols;
    const LinChunk& C = D.ch[ci];
    unsigned char* base = img + C.img_off;
    const unsigned part = (unsigned)N * kLtK * 4;
    for (int i = threadIdx.x; i < N * kLtK; i += blockDim.x) {
        const int c = i / kLtK, k = i % kLtK;
        const float v =
            k < C.kc ? W[C.w_off + (int64_t)(C.k0 + k) * C.w_ks + (int64_t)c * C.w_ns] : 0.0f;
        const float hi = to_tf32(v), lo = to_tf32(v - hi);
        if (stacked) {
            *reinterpret_cast<float*>(base + kmajor_offset(c, k, 2 * N)) = hi;
            *reinterpret_cast<float*>(base + kmajor_offset(N + c, k, 2 * N)) = lo;
        } else {
            const unsigned o = kmajor_offset(c, k, N);
            *reinterpret_cast<float*>(base + o) = hi;
            *reinterpret_cast<float*>(base + part + o) = lo;
        }
    }
}

// Work units are (block, 128-row tile) pairs, blocks in order; CTA c takes
// units c, c + grid, ...; every role walks the same sequence, taking a unit's
// chunks in an order rotated by c (the CTAs then read different B chunks at
// the same time).  Chunk k uses stage k % S: A columns in tensor memory and a
// B slot in shared memory.  Warp roles:
//   producers (warps 4-11; warp 4 + p serves TMEM lanes 32 (p % 4) .. + 31,
//     one row per lane, K columns 16 (p / 4) .. + 15 of each chunk): the rows
//     are loaded into registers three chunks ahead (four buffers taken in
//     rotation by name, so no copy waits for a load); once the MMAs of chunk
//     k - S have released the stage (empty) the warp writes chunk k's values
//     as they are (the tensor cores read them as the TF32 "hi" part, which
//     keeps the leading 10 fraction bits) and the "lo" parts, lo =
//     round_tf32(x - x cut to 10 fraction bits), with tcgen05.st and arrives
//     on full (one arrival per warp).
//   loader (warp 13, one thread): once the stage is empty, starts the bulk
//     copy of chunk k's B image into its slot, arriving on full with the
//     expected byte count.
//   MMA issuer (warp 12, lane 0 issuing): one wait per chunk (full: A written
//     and B landed), then the products (A from tensor memory, B from shared
//     memory) into accumulator t % NACC of unit t (after acc_free says the
//     epilogue has read unit t - NACC), committed to empty and, after a unit's
//     last chunk, to acc_full.  Each wait of this thread leaves the tensor
//     pipe without queued work for its latency, so it waits once per chunk.
//   epilogue (warps 0-3): per unit, wait acc_full, read the 32 rows of its lane
//     quarter, transpose 32 x 32 pieces through shared memory, store whole
//     128-byte row segments and arrive on acc_free.
// Chunk k uses phase (k / S) % 2 of full / empty; unit t uses phase
// (t / NACC) % 2 of acc_full / acc_free.  Every wait is bounded; after a
// timeout the remaining waits return at once, each role leaves its loop, and
// the loader drains the copies it started.
//
// TPD > 0 (the fused 'uvw' forward): the producers compute their rows from
// the tensor-product source instead of loading them.  For row (n, m3) and a
// chunk of path p's block: sum over m1 < d1 (at most TPD) of the T entry
// T[n, p, m3, m1] (precomputed per sample by lin_tp_t_kernel) times the 16
// channels of x1[n, m1].  The path table is copied to shared memory with the
// others.
template <int S, int NACC, bool STACK, int TPD>
__global__ void __launch_bounds__(kLtThreads, 1)  // 128 registers: 4 of the 14 warps share a sub-partition
linear_tc_kernel(const __grid_constant__ LinDesc D, int64_t n, int nmax,
                 const float* __restrict__ x, const unsigned char* __restrict__ img,
                 float* __restrict__ out, const __grid_constant__ TpArg<(TPD > 0)> tp,
                 int test_fail_first) {
    constexpr bool TPA = TPD > 0;
    constexpr int RA = S;
    constexpr int RB = S;
    constexpr unsigned accw = 256 / NACC;  // columns per accumulator
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) unsigned long long full[S], empty[S];
    __shared__ __align__(8) unsigned long long acc_full[2], acc_free[2];
    __shared__ unsigned tmem_base;
    __shared__ int fail;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned char* Bbase = smem;  // slot j: j * bslot
    const unsigned bslot = 2u * (unsigned)nmax * kLtK * 4;
    float* stage_all = reinterpret_cast<float*>(Bbase + (size_t)RB * bslot);
    // the block and chunk tables, copied to shared memory (indexed lookups in
    // the parameter space would go through the small constant cache)
    const unsigned pitch = lt_stage_pitch(nmax, STACK);
    LinBlock* sblk = reinterpret_cast<LinBlock*>(stage_all + kLtEpiWarps * 32 * pitch);
    LinChunk* sch = reinterpret_cast<LinChunk*>(sblk + kLinMaxBlocks + 1);
    for (int i = tid; i < D.nblocks; i += kLtThreads) sblk[i] = D.blk[i];
    for (int i = tid; i < D.nchunks; i += kLtThreads) sch[i] = D.ch[i];
    LinTpDesc* stp = reinterpret_cast<LinTpDesc*>(sch + kLinMaxChunks);
    if constexpr (TPA) {
        const int* src = reinterpret_cast<const int*>(&tp.d);
        int* dst = reinterpret_cast<int*>(stp);
        for (int i = tid; i < (int)(sizeof(LinTpDesc) / 4); i += kLtThreads) dst[i] = src[i];
    }
    const int nblocks = D.nblocks;
    const int64_t in_stride = D.in_stride, out_stride = D.out_stride;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base)),
                     "r"(kLtTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            tc_mbar_init(&full[i], kLtProdWarps + 1);  // producer warps + the loader
            tc_mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc_mbar_init(&acc_full[i], 1);
            tc_mbar_init(&acc_free[i], 32 * kLtEpiWarps);
        }
        fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const unsigned tmem = tmem_base;

    const bool issuer = warp == kLtEpiWarps + kLtProdWarps;
    const bool loader = warp == kLtEpiWarps + kLtProdWarps + 1;
    // after a timeout elsewhere the remaining waits return at once (the issuer
    // reads the flag once per unit instead, and its next wait runs out)
    auto wait = [&](unsigned long long* bar, unsigned parity) -> bool {
        if (!issuer && *(volatile int*)&fail) return false;
        if (issuer || loader ? tc_mbar_wait(bar, parity) : tc_mbar_wait_sleep(bar, parity))
            return true;
        atomicExch(&fail, 1);
        return false;
    };
    // position in this CTA's chunk sequence, with the current block's fields
    // held in registers (the issuer reads no table per chunk)
    struct Pos {
        int64_t u, t;
        int b, ci, nch, ncols, chunk0, rot;
        bool valid;
    };
    // unit u -> group g (units [grp_u0[g], grp_u0[g + 1])), tile-major inside
    // The fused forward (single-block groups) runs window by window instead: a
    // window of 128 items holds d tiles of a block whose rows have d
    // components, uw = sum_b d units in block order, so all blocks of a window
    // read its x1 rows close together in time (L2 keeps them); units past a
    // block's last tile (in the last window) are skipped by every role alike.
    int uw = 0;
    if constexpr (TPA)
        for (int g = 0; g < D.ngrp; ++g) uw += sblk[D.grp_b[g]].d;
    const int64_t nwin = (n + kLtM - 1) / kLtM;
    auto locate = [&](Pos& p) {
        const int ng = D.ngrp;
        if constexpr (TPA) {
            for (;;) {
                p.valid = p.u < nwin * uw;
                if (!p.valid) return;
                int64_t w;
                int r;
                if (p.u < (int64_t)0xffffffff) {
                    w = (unsigned)p.u / (unsigned)uw;
                    r = (int)((unsigned)p.u - (unsigned)w * (unsigned)uw);
                } else {
                    w = p.u / uw;
                    r = (int)(p.u - w * uw);
                }
                int g = 0, acc = 0;
                while (g + 1 < ng && r >= acc + sblk[D.grp_b[g]].d) acc += sblk[D.grp_b[g++]].d;
                p.b = D.grp_b[g];
                p.t = w * sblk[p.b].d + (r - acc);
                if (p.t < D.grp_nt[g]) break;
                p.u += gridDim.x;
            }
        } else {
        p.valid = p.u < D.grp_u0[ng];
        if (!p.valid) return;
        int g = 0;
        while (g + 1 < ng && p.u >= D.grp_u0[g + 1]) ++g;
        const int64_t ul = p.u - D.grp_u0[g];
        const int nb = D.grp_nb[g];
        int r = 0;
        if (nb == 1) {
            p.t = ul;
        } else if (ul < (int64_t)0xffffffff) {
            const unsigned q = (unsigned)ul / (unsigned)nb;
            p.t = q;
            r = (int)((unsigned)ul - q * (unsigned)nb);
        } else {
            p.t = ul / nb;
            r = (int)(ul - p.t * nb);
        }
        p.b = D.grp_b[D.grp_b0[g] + r];
        }
        const LinBlock& B = sblk[p.b];
        p.nch = B.nchunk;
        p.ncols = B.ncols;
        p.chunk0 = B.chunk0;
        // the chunks of a unit are taken in an order rotated by the CTA index,
        // so that the CTAs do not all read the same B chunk at once
        p.rot = (int)(blockIdx.x % (unsigned)B.nchunk);
    };
    auto advance = [&](Pos& p) {
        if (p.ci + 1 < p.nch) {
            ++p.ci;
        } else {
            p.u += gridDim.x;
            p.ci = 0;
            locate(p);
        }
    };
    auto chunk_index = [&](const Pos& p) {
        const int c = p.ci + p.rot;
        return p.chunk0 + (c >= p.nch ? c - p.nch : c);
    };
    auto chunk_of = [&](const Pos& p) -> const LinChunk& { return sch[chunk_index(p)]; };
    Pos start{(int64_t)blockIdx.x, 0, 0, 0, 1, 0, 0, 0, false};
    locate(start);

    if (warp >= kLtEpiWarps && warp < kLtEpiWarps + kLtProdWarps) {
        // ---------------------------------------------------------- producers
        const int pw = warp - kLtEpiWarps, qa = pw & 3, h = pw >> 2;
        const int r = 32 * qa + lane;  // this lane's row of every tile
        int64_t rbase = 0;
        int rm = -1;
        int64_t row_u = -1;
        auto load = [&](const Pos& p, float4 (&v)[4]) {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (!p.valid) return;
            const LinBlock& B = sblk[p.b];
            const LinChunk& C = chunk_of(p);
            if (p.u != row_u) {
                row_u = p.u;
                const int64_t R = p.t * kLtM + r;
                rm = -1;
                if (R < n * B.d) {
                    const int64_t item = row_item(R, B.d);
                    rm = (int)(R - item * B.d);
                    rbase = TPA ? item : item * in_stride;
                }
            }
            if (rm < 0) return;
            const float* src = x + rbase + C.a_off + (int64_t)rm * C.a_mul + C.k0 + 16 * h;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (16 * h + 4 * j < C.kc) v[j] = *reinterpret_cast<const float4*>(src + 4 * j);
        };
        Pos pre = start, cur = start;
        bool stop = false;
        // write chunk k's values into its stage once the stage is empty
        auto put = [&](int64_t k, const float4 (&v)[4]) {
            const int s = (int)(k % RA);
            if (k >= S && !wait(&empty[s], (unsigned)(((k - S) / S) & 1))) {
                stop = true;
                return;
            }
            float hi[16], lo[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float in[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    hi[4 * j + q] = in[q];
                    lo[4 * j + q] =
                        to_tf32(in[q] - __uint_as_float(__float_as_uint(in[q]) & 0xFFFFE000u));
                }
            }
            const unsigned ta = tmem + ((unsigned)(32 * qa) << 16) + kLtAcol + 64u * s + 16u * h;
            tmem_st16(ta, hi);
            tmem_st16(ta + 32, lo);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) tc_mbar_arrive(&full[s]);  // one arrival per warp
            advance(cur);
            if (*(volatile int*)&fail) stop = true;
        };
        // chunk k: load chunk k + 3 into `nxt`, then write chunk k (in `v`)
        auto step = [&](int64_t k, float4 (&v)[4], float4 (&nxt)[4]) {
            load(pre, nxt);
            if (pre.valid) advance(pre);
            put(k, v);
        };
        if constexpr (TPA) {
            // rows computed from the tensor-product source: for the row's
            // (n, m3) and the chunk's path p, the T entries of m1 < d1 (at most
            // TPD) and the 16 channels of x1[n, m1], all loads independent,
            // then the sums; each chunk when its stage comes (the eight
            // producer warps build one chunk together)
            constexpr int G = TPD > 0 ? TPD : 1;
            auto load_tp = [&](const Pos& p, float4 (&v)[4]) {
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (!p.valid) return;
                const LinBlock& B = sblk[p.b];
                const LinChunk& C = chunk_of(p);
                if (p.u != row_u) {
                    row_u = p.u;
                    const int64_t R = p.t * kLtM + r;
                    rm = -1;
                    if (R < n * B.d) {
                        const int64_t item = row_item(R, B.d);
                        rm = (int)(R - item * B.d);
                        rbase = item;
                    }
                }
                if (rm < 0) return;
                const LinTpPath& P = stp->path[C.src];
                const float* xr = tp.x1 + rbase * tp.x1_stride + P.x1_off + C.k0 + 16 * h;
                const float* tr = tp.t + rbase * stp->tdim + P.t_off + rm * P.d1;
                float tv[G];
                float4 a[G][4];
#pragma unroll
                for (int g = 0; g < G; ++g)
                    if (g < P.d1) {
                        tv[g] = __ldg(tr + g);
                        const float4* xs = reinterpret_cast<const float4*>(xr + (int64_t)g * P.mul1);
#pragma unroll
                        for (int j = 0; j < 4; ++j) a[g][j] = __ldg(xs + j);
                    }
#pragma unroll
                for (int g = 0; g < G; ++g)
                    if (g < P.d1)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            v[j].x = fmaf(tv[g], a[g][j].x, v[j].x);
                            v[j].y = fmaf(tv[g], a[g][j].y, v[j].y);
                            v[j].z = fmaf(tv[g], a[g][j].z, v[j].z);
                            v[j].w = fmaf(tv[g], a[g][j].w, v[j].w);
                        }
            };
            for (int64_t k = 0; cur.valid && !stop; ++k) {
                float4 v[4];
                load_tp(cur, v);
                put(k, v);
            }
        } else {
            // four register buffers taken in rotation by name (a copy between
            // them would wait for the load just issued)
            float4 b0[4], b1[4], b2[4], b3[4];
            load(pre, b0);
            if (pre.valid) advance(pre);
            load(pre, b1);
            if (pre.valid) advance(pre);
            load(pre, b2);
            if (pre.valid) advance(pre);
            for (int64_t k = 0; cur.valid && !stop; k += 4) {
                step(k, b0, b3);
                if (!cur.valid || stop) break;
                step(k + 1, b1, b0);
                if (!cur.valid || stop) break;
                step(k + 2, b2, b1);
                if (!cur.valid || stop) break;
                step(k + 3, b3, b2);
            }
        }
    } else if (loader) {
        // ------------------------------------------------------------- loader
        if (lane == 0) {
            Pos bp = start;
            int img_b = -1, img0 = 0;  // block whose first-chunk image offset is cached
            int64_t k = 0;
            for (; bp.valid; ++k) {
                const int s = (int)(k % S);
                if (k >= S && !wait(&empty[s], (unsigned)(((k - S) / S) & 1))) break;
                const unsigned bytes = 2u * (unsigned)bp.ncols * kLtK * 4;
                if (bp.b != img_b) {  // a block's chunk images are consecutive, equal in size
                    img_b = bp.b;
                    img0 = sch[bp.chunk0].img_off;
                }
                const int c = chunk_index(bp) - bp.chunk0;
                tc_expect_tx(&full[s], bytes);
                tc_bulk_g2s(Bbase + (size_t)s * bslot, img + img0 + (size_t)c * bytes, bytes,
                            &full[s]);
                advance(bp);
                if ((k & 15) == 15 && *(volatile int*)&fail) {
                    ++k;
                    break;
                }
            }
            // drain: the copies of the last S chunks may still be in flight;
            // each completes its stage's phase once the producers arrived too,
            // so wait on the copies alone through a fresh phase check of the
            // transaction count (bounded)
            for (int64_t c = k > S ? k - S : 0; c < k; ++c)
                tc_mbar_wait(&full[c % S], (unsigned)((c / S) & 1));
        }
    } else if (issuer) {
        // ---------------------------------------------------------- MMA issuer
        // the whole warp walks the loop (converged); lane 0 issues
        const bool leader = lane == 0;
        Pos cur = start;
        int64_t k = 0, t = 0, last_commit = -1;
        while (cur.valid) {
            const int s = (int)(k % S);
            const int N = cur.ncols;
            const bool first = cur.ci == 0, last = cur.ci + 1 == cur.nch;
            const int acc = (int)(t % NACC);
            // test_fail_first (tests only): the first wait gives up at once
            bool ok = test_fail_first && k == 0
                          ? (tc_mbar_wait(&full[s], 0u, 0u) || (atomicExch(&fail, 1), false))
                          : wait(&full[s], (unsigned)((k / S) & 1));
            if (ok && first && t >= NACC)
                ok = wait(&acc_free[acc], (unsigned)(((t - NACC) / NACC) & 1));
            if (!__all_sync(0xffffffffu, ok)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t idesc = tf32_idesc(kLtM, N);
            const unsigned b0 = smem_addr(Bbase + (size_t)s * bslot);
            const unsigned d = tmem + (unsigned)acc * accw;
            const unsigned a0 = tmem + kLtAcol + 64u * s;
            if (leader) {
                if (STACK) {
                    // A_hi [B_hi | B_lo] (N = 2 ncols) into columns [0, 2 ncols),
                    // A_lo B_hi into [0, ncols); the epilogue adds the halves
                    const uint32_t idesc2 = tf32_idesc(kLtM, 2 * N);
                    const unsigned lb = (unsigned)(2 * N / 8) * 128;
#pragma unroll
                    for (int k8 = 0; k8 < kLtK; k8 += 8) {
                        const uint64_t bd = smem_desc(b0 + (unsigned)(k8 >> 2) * lb, lb, 128);
                        mma_tf32_tmem_a(d, a0 + k8, bd, idesc2, (first && k8 == 0) ? 0u : 1u);
                        mma_tf32_tmem_a(d, a0 + 32 + k8, bd, idesc, 1u);
                    }
                } else {
                    const unsigned lb = (unsigned)(N / 8) * 128;
                    const unsigned bpart = (unsigned)N * kLtK * 4;
#pragma unroll
                    for (int k8 = 0; k8 < kLtK; k8 += 8) {
                        const unsigned kk = (unsigned)(k8 >> 2) * lb;
                        const uint64_t bh = smem_desc(b0 + kk, lb, 128);
                        const uint64_t bl = smem_desc(b0 + bpart + kk, lb, 128);
                        mma_tf32_tmem_a(d, a0 + k8, bh, idesc, (first && k8 == 0) ? 0u : 1u);
                        mma_tf32_tmem_a(d, a0 + k8, bl, idesc, 1u);
                        mma_tf32_tmem_a(d, a0 + 32 + k8, bh, idesc, 1u);
                    }
                }
                tc_commit(&empty[s]);
                if (last) tc_commit(&acc_full[acc]);
            }
            __syncwarp();
            last_commit = k;
            if (last) ++t;
            advance(cur);
            ++k;
            if (last && __any_sync(0xffffffffu, *(volatile int*)&fail)) break;
        }
        if (leader && last_commit >= 0)  // the MMAs must finish before tensor memory is freed
            tc_mbar_wait(&empty[last_commit % S], (unsigned)((last_commit / S) & 1));
    } else {
        // ----------------------------------------------------------- epilogue
        const int q = warp;  // TMEM lane quarter
        Pos cur = start;
        float* stage = stage_all + q * (32 * pitch);
        for (int64_t t = 0; cur.valid; ++t) {
            const int acc = (int)(t % NACC);
            bool got = wait(&acc_full[acc], (unsigned)((t / NACC) & 1));
            got = __all_sync(0xffffffffu, got);
            if (!got) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const LinBlock& EB = sblk[cur.b];
            const int N = EB.ncols;
            const int64_t R = cur.t * kLtM + 32 * q + lane;
            const bool live = R < n * EB.d;
            float* o = out;  // this lane's row
            if (live) {
                const int64_t item = row_item(R, EB.d);
                const int m = (int)(R - item * EB.d);
                o = out + item * out_stride + EB.out_off + (int64_t)m * N;
            }
            if (STACK) {
                // the whole row block into shared memory (+ the A_hi B_lo half),
                // then the accumulator is free while the rows go out
                for (int c0 = 0; c0 < N; c0 += 32) {
                    float v[32], v2[32];
                    const unsigned ta =
                        tmem + ((unsigned)(32 * q) << 16) + (unsigned)acc * accw + (unsigned)c0;
                    tmem_ld32(ta, v);
                    tmem_ld32(ta + (unsigned)N, v2);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<float4*>(stage + lane * pitch + c0 + 4 * i) = make_float4(
                            v[4 * i] + v2[4 * i], v[4 * i + 1] + v2[4 * i + 1],
                            v[4 * i + 2] + v2[4 * i + 2], v[4 * i + 3] + v2[4 * i + 3]);
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                tc_mbar_arrive(&acc_free[acc]);
                __syncwarp();
                for (int rr = 0; rr < 32; ++rr) {  // one row per step, 16 bytes per lane
                    float* orow = reinterpret_cast<float*>(
                        __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(o), rr));
                    const bool rlive = __shfl_sync(0xffffffffu, live, rr);
                    for (int c = 4 * lane; c < N; c += 128)
                        if (rlive)
                            *reinterpret_cast<float4*>(orow + c) =
                                *reinterpret_cast<const float4*>(stage + rr * pitch + c);
                }
                __syncwarp();
            } else {
                for (int c0 = 0; c0 < N; c0 += 32) {
                    float v[32];
                    tmem_ld32(tmem + ((unsigned)(32 * q) << 16) + (unsigned)acc * accw + (unsigned)c0, v);
                    // transpose through shared memory: 8 lanes store one row's 128 bytes
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<float4*>(stage + lane * pitch + 4 * i) =
                            make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    __syncwarp();
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int rr = 4 * it + (lane >> 3), cq = lane & 7;
                        float* orow = reinterpret_cast<float*>(
                            __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(o), rr));
                        const bool rlive = __shfl_sync(0xffffffffu, live, rr);
                        const float4 w4 = *reinterpret_cast<const float4*>(stage + rr * pitch + 4 * cq);
                        if (rlive) *reinterpret_cast<float4*>(orow + c0 + 4 * cq) = w4;
                    }
                    __syncwarp();
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                tc_mbar_arrive(&acc_free[acc]);
            }
            cur.u += gridDim.x;
            cur.ci = 0;
            locate(cur);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (tid == 0 && fail) atomicExch(&cgtp_linear_error, 1);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kLtTmemCols)
                     : "memory");
}

// --------------------------------------------- W gradient on tensor cores
//
// gW_j = X_j^T G_j summed over the rows (n, m) of instruction j, as
// D[u, w] = sum_k A[u, k] B[w, k] with K = rows: A = X^T in tensor memory (lane
// = input channel u, columns = 32 rows of a chunk), B = G^T in shared memory
// (K-major, [hi | lo] stacked along N = 2 mul_out), the same three split
// products as the forward in two instructions per K step (A_hi [B_hi | B_lo]
// into 2 mul_out columns, A_lo B_hi added to the first mul_out).  Work units are
// (instruction, 128-channel M tile, row split s), split s holding the rows of
// items [s per, (s + 1) per); each unit writes its partial sums to
// partial[s nw + ...] (zeros for an empty split), added in fixed order
// afterwards.  Warp roles:
//   epilogue (warps 0-3): per segment, wait acc_full, read D (lane u), add it
//     to the unit's sums; after the last one store the partial row; arrive on
//     acc_free.
//   loader (warp 12): lane i starts the bulk copies of row i of chunk k (its
//     128 x columns of the M tile and its g row) into staging stage k % 3 once
//     the producers have released it (raw_empty), lane 0 announcing the bytes
//     on raw_full.
//   A producers (warps 4-7, lane quarter warp % 4): each thread reads its
//     channel u of the chunk's 32 staged rows, releases the staging stage,
//     writes hi = the values and lo = round_tf32(x - x cut to 10 bits) with
//     tcgen05.st once the MMA stage is empty, and arrives on full.
//   B producers (warps 8-11, output channel w = 32 (warp - 8) + lane): read w
//     of the 32 staged rows, release the staging stage, write four rows at a
//     time into the K-major image (hi rows w, lo rows mul_out + w), fence to
//     the async proxy, arrive on full.  (Warps 13-15 have no role.)
//   MMA issuer (warp 16): one wait per chunk, the products, commit to empty
//     (and acc_full after a unit's last chunk).
// Chunk k (counted over the CTA's units) uses MMA stage k % 2 and phase
// (k / 2) % 2 of full / empty, staging stage k % 3 and phase (k / 3) % 2 of
// raw_full / raw_empty.  Precision: the tensor core's fp32 accumulator loses low
// bits on every addition, so its error grows with the number of rows it sums.
// A unit's chunks are therefore cut into segments; each segment starts a
// fresh accumulator and the epilogue adds it, in plain fp32 arithmetic and
// segment order, into the unit's sums in shared memory.  With every mul_out <=
// 64 (accumulators of at most 128 columns) two buffers, columns [0, 128) and
// [128, 256), alternate so that the epilogue drains one while the MMA fills the
// other, with segments of kWgSeg / 2 chunks; wider outputs use one buffer and
// segments of kWgSeg chunks.  The t-th segment (counted over the CTA) uses
// buffer t % nacc and phase (t / nacc) % 2 of acc_full / acc_free.
// Waits are bounded as in the forward kernel.
constexpr int kWgStages = 2;    // MMA stages: A in tensor memory, B image in shared memory
constexpr int kWgRaw = 3;       // staging stages of the rows (bulk or tensor-map copies)
constexpr int kWgThreads = 32 * 17;
constexpr int kWgRows = 32;  // rows (K) per chunk
constexpr int kWgSeg = 16;   // chunks (512 rows) per segment of a single buffer
constexpr int kWgLoaderWarp = 12;
// one staging stage: 32 rows of x (128 columns of the M tile) and of g (up to
// 128 output channels)
constexpr size_t kWgRawBytes = 2 * (size_t)kWgRows * 128 * 4;
// dynamic shared memory: the MMA stages' B images, the epilogue's sums
// [128 w][128 u], then the staging ring
constexpr size_t kWgSmem = kWgStages * (size_t)(2 * 128 * kWgRows * 4) + 128 * 128 * 4 +
                           kWgRaw * kWgRawBytes;

// Tensor maps of the weight gradient (wgrad_maps), for layers whose
// instructions all take 128 input channels and the same number of output
// channels: x viewed as [n][x_stride / 128][128] and g as
// [n][g_stride / mo][mo]; map (d - 1) / 2 has the box [32 / d items][d][128 or
// mo], so that one copy per operand stages a chunk of whole items (the rows
// past 32 / d items, d of them each, are left out of the chunk).
constexpr int kWgMaxD = 8;  // item widths d = 1, 3, ..., 15
struct WgMaps {
    CUtensorMap x[kWgMaxD], g[kWgMaxD];
    int on;    // 1: the maps are set
    int gbox;  // g channels per staged row (= mo)
};

// 3D tile copy through a tensor map, coordinates innermost first.
__device__ __forceinline__ void tma_3d_g2s(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                           unsigned long long* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
        : "memory");
}

__global__ void __launch_bounds__(kWgThreads, 1)
linear_wgrad_tc_kernel(const __grid_constant__ LinGradDesc D, int64_t n, int64_t per, int S,
                       int nacc, const float* __restrict__ x, const float* __restrict__ g,
                       float* __restrict__ partial, const __grid_constant__ WgMaps M) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) unsigned long long full[kWgStages], empty[kWgStages];
    __shared__ __align__(8) unsigned long long raw_full[kWgRaw], raw_empty[kWgRaw];
    __shared__ __align__(8) unsigned long long acc_full[2], acc_free[2];
    __shared__ unsigned tmem_base;
    __shared__ int fail;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr unsigned bslot = 2u * 128 * kWgRows * 4;  // stacked image, mul_out <= 128
    unsigned char* const raw0 = smem + kWgStages * (size_t)bslot + 128 * 128 * 4;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base)),
                     "r"(kLtTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int i = 0; i < kWgStages; ++i) {
            tc_mbar_init(&full[i], 8);  // 4 A warps + 4 B warps
            tc_mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < kWgRaw; ++i) {
            tc_mbar_init(&raw_full[i], 1);   // the loader's arrival with the byte count
            tc_mbar_init(&raw_empty[i], 8);  // the producer warps
        }
        for (int i = 0; i < 2; ++i) {
            tc_mbar_init(&acc_full[i], 1);
            tc_mbar_init(&acc_free[i], 128);
        }
        fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const unsigned tmem = tmem_base;
    const bool issuer = warp == 16;
    const bool tight = issuer || warp == kWgLoaderWarp;  // these two poll without sleeping
    const int seg = nacc == 2 ? kWgSeg / 2 : kWgSeg;
    auto wait = [&](unsigned long long* bar, unsigned parity) -> bool {
        if (!issuer && *(volatile int*)&fail) return false;
        if (tight ? tc_mbar_wait(bar, parity) : tc_mbar_wait_sleep(bar, parity)) return true;
        atomicExch(&fail, 1);
        return false;
    };
    // unit u -> instruction j, M tile mt, split s and its rows [r0, r1).
    // Units run class by class (M tiles with the same rows per item, widest
    // first) and split-major inside a class: the CTAs running at one time hold
    // every M tile of a class for the same few row splits, so g rows that
    // instructions of one output irrep share (they have the same width) are
    // read from HBM once and served to the others from L2.  Round r of
    // gridDim.x units goes to the CTAs in ascending order when r is even and
    // descending when odd, which evens out the CTAs' rows.
    // With the maps a chunk is ipc = 32 / d whole items (rows past ipc * d
    // are zero); without them, 32 consecutive rows.
    struct Unit {
        int j, mt, nch, sp, ipc;
        int64_t r0, r1, i0, i1;
    };
    const int64_t units = (int64_t)D.nmt * S;
    auto unit_at = [&](int64_t r) -> int64_t {
        return r * gridDim.x + ((r & 1) ? (int64_t)(gridDim.x - 1 - blockIdx.x) : (int64_t)blockIdx.x);
    };
    auto unit_of = [&](int64_t u, Unit& U) {
        int c = 0, q0 = 0;
        while (c + 1 < D.ncls && u >= (int64_t)D.cls_n[c] * S) {
            u -= (int64_t)D.cls_n[c] * S;
            q0 += D.cls_n[c];
            ++c;
        }
        const int sp = (int)(u / D.cls_n[c]);
        const int q = D.qord[q0 + (int)(u % D.cls_n[c])];
        int j = 0;
        while (j + 1 < D.ninstr && D.g[j + 1].mt0 <= q) ++j;
        U.j = j;
        U.sp = sp;
        U.mt = q - D.g[j].mt0;
        const int64_t i0 = (int64_t)sp * per, i1 = i0 + per < n ? i0 + per : n;
        const int d = D.g[j].d;
        U.i0 = i0 < n ? i0 : 0;
        U.i1 = i0 < n ? i1 : 0;
        U.r0 = U.i0 * d;
        U.r1 = U.i1 * d;
        U.ipc = M.on ? kWgRows / d : 0;
        U.nch = U.ipc ? (int)((U.i1 - U.i0 + U.ipc - 1) / U.ipc)
                      : (int)((U.r1 - U.r0 + kWgRows - 1) / kWgRows);
    };
    // first row and number of live rows of chunk ci
    auto chunk_rows = [&](const Unit& U, int ci, int64_t& rb, int& valid) {
        if (U.ipc) {
            const int64_t it = U.i0 + (int64_t)ci * U.ipc;
            const int d = D.g[U.j].d;
            rb = it * d;
            valid = (int)min((int64_t)U.ipc, U.i1 - it) * d;
        } else {
            rb = U.r0 + (int64_t)ci * kWgRows;
            valid = (int)min((int64_t)kWgRows, U.r1 - rb);
        }
    };

    if (warp >= 4 && warp < 12) {
        // ---------------------------------------------------------- producers
        const bool isA = warp < 8;
        const int q = warp & 3;
        auto lo = [](float v) {
            return to_tf32(v - __uint_as_float(__float_as_uint(v) & 0xFFFFE000u));
        };
        int64_t k = 0;
        bool stop = false;
        for (int64_t r = 0, u; (u = unit_at(r)) < units && !stop; ++r) {
            Unit U;
            unit_of(u, U);
            if (U.nch == 0) continue;
            const LinGrad& G = D.g[U.j];
            // this thread's column of the staged rows: A -> input channel of the
            // M tile, B -> output channel
            const int col = isA ? 32 * q + lane : 32 * (warp - 8) + lane;
            const int lim = isA ? min(128, G.mi - U.mt * 128) : G.mo;
            for (int ci = 0; ci < U.nch; ++ci, ++k) {
                const int rs = (int)(k % kWgRaw);
                int64_t rb;
                int valid;
                chunk_rows(U, ci, rb, valid);
                if (!wait(&raw_full[rs], (unsigned)((k / kWgRaw) & 1))) {
                    stop = true;
                    break;
                }
                const float* src = reinterpret_cast<const float*>(raw0 + (size_t)rs * kWgRawBytes) +
                                   (isA ? 0 : kWgRows * 128);
                // staged row stride: 128 floats, except g rows copied through the
                // maps (gbox floats per row)
                const int pitch = (!isA && M.on) ? M.gbox : 128;
                float v[kWgRows];
#pragma unroll
                for (int i = 0; i < kWgRows; ++i)
                    v[i] = (i < valid && col < lim) ? src[i * pitch + col] : 0.0f;
                __syncwarp();
                if (lane == 0) tc_mbar_arrive(&raw_empty[rs]);
                const int st = (int)(k % kWgStages);
                if (k >= kWgStages &&
                    !wait(&empty[st], (unsigned)(((k - kWgStages) / kWgStages) & 1))) {
                    stop = true;
                    break;
                }
                if (isA) {
                    const unsigned ta = tmem + ((unsigned)(32 * q) << 16) + kLtAcol + 64u * st;
                    float hv[16], lv[16];
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            hv[i] = v[16 * half + i];
                            lv[i] = lo(v[16 * half + i]);
                        }
                        tmem_st16(ta + 16u * half, hv);
                        tmem_st16(ta + 32 + 16u * half, lv);
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                } else {
                    const int w = col;
                    const int mo = G.mo;
                    if (w < mo) {
                        unsigned char* bs = smem + (size_t)st * bslot;
#pragma unroll
                        for (int k4 = 0; k4 < kWgRows; k4 += 4) {
                            *reinterpret_cast<float4*>(bs + kmajor_offset(w, k4, 2 * mo)) =
                                make_float4(v[k4], v[k4 + 1], v[k4 + 2], v[k4 + 3]);
                            *reinterpret_cast<float4*>(bs + kmajor_offset(mo + w, k4, 2 * mo)) =
                                make_float4(lo(v[k4]), lo(v[k4 + 1]), lo(v[k4 + 2]), lo(v[k4 + 3]));
                        }
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                __syncwarp();
                if (lane == 0) tc_mbar_arrive(&full[st]);
                if (*(volatile int*)&fail) {
                    stop = true;
                    break;
                }
            }
        }
    } else if (warp == kWgLoaderWarp) {
        // ------------------------------------------------------------- loader
        int64_t k = 0;
        bool stop = false;
        for (int64_t r = 0, u; (u = unit_at(r)) < units && !stop; ++r) {
            Unit U;
            unit_of(u, U);
            if (U.nch == 0) continue;
            const LinGrad& G = D.g[U.j];
            const int cols = min(128, G.mi - U.mt * 128);
            const unsigned abytes = (unsigned)cols * 4, bbytes = (unsigned)G.mo * 4;
            for (int ci = 0; ci < U.nch; ++ci, ++k) {
                const int rs = (int)(k % kWgRaw);
                if (k >= kWgRaw && !wait(&raw_empty[rs], (unsigned)(((k - kWgRaw) / kWgRaw) & 1))) {
                    stop = true;
                    break;
                }
                int64_t rb;
                int valid;
                chunk_rows(U, ci, rb, valid);
                unsigned char* dst = raw0 + (size_t)rs * kWgRawBytes;
                if (U.ipc) {
                    // one copy per operand: items it .. it + ipc - 1, all d rows
                    // each (items past the unit are ignored by the producers,
                    // items past n read as zeros); the full boxes count
                    if (lane == 0) {
                        const int it = (int)(U.i0 + (int64_t)ci * U.ipc), di = (G.d - 1) / 2;
                        const unsigned rows = (unsigned)(U.ipc * G.d);
                        tc_expect_tx(&raw_full[rs], rows * (128u + (unsigned)M.gbox) * 4u);
                        tma_3d_g2s(dst, &M.x[di], 0, (G.xo + U.mt * 128) / 128, it, &raw_full[rs]);
                        tma_3d_g2s(dst + (size_t)kWgRows * 512, &M.g[di], 0, G.go / M.gbox, it,
                                   &raw_full[rs]);
                    }
                    __syncwarp();
                    if (__any_sync(0xffffffffu, *(volatile int*)&fail)) {
                        ++k;
                        stop = true;
                        break;
                    }
                    continue;
                }
                if (lane == 0) tc_expect_tx(&raw_full[rs], (unsigned)valid * (abytes + bbytes));
                __syncwarp();
                if (lane < valid) {
                    // rows m, m + 1, ... of one item are consecutive in memory; when a
                    // row slice is exactly one 512-byte staging row, the lane holding
                    // the first row of a run copies the whole run at once
                    const int64_t R = rb + lane;
                    const int64_t item = row_item(R, G.d);
                    const int m = (int)(R - item * G.d);
                    const int run = min(G.d - m, valid - lane);
                    const bool head = lane == 0 || m == 0;
                    const bool arun = abytes == 512 && G.mi == 128, brun = bbytes == 512;
                    if (!arun || head)
                        tc_bulk_g2s(dst + (size_t)lane * 512,
                                    x + G.xo + item * D.x_stride + (int64_t)m * G.mi + U.mt * 128,
                                    arun ? 512u * run : abytes, &raw_full[rs]);
                    if (!brun || head)
                        tc_bulk_g2s(dst + (size_t)(kWgRows + lane) * 512,
                                    g + G.go + item * D.g_stride + (int64_t)m * G.mo,
                                    brun ? 512u * run : bbytes, &raw_full[rs]);
                }
                if (__any_sync(0xffffffffu, *(volatile int*)&fail)) {
                    ++k;
                    stop = true;
                    break;
                }
            }
        }
        // after a timeout the copies of the last stages may still be in flight:
        // wait for them (bounded) before the CTA's shared memory is released
        if (stop)
            for (int64_t c = k > kWgRaw ? k - kWgRaw : 0; c < k; ++c)
                tc_mbar_wait(&raw_full[c % kWgRaw], (unsigned)((c / kWgRaw) & 1));
    } else if (issuer) {
        // ---------------------------------------------------------- MMA issuer
        const bool leader = lane == 0;
        int64_t k = 0, t = 0, last_commit = -1;
        for (int64_t r = 0, u; (u = unit_at(r)) < units; ++r) {
            Unit U;
            unit_of(u, U);
            if (U.nch == 0) continue;
            const int mo = D.g[U.j].mo;
            const uint32_t idesc = tf32_idesc(kLtM, mo), idesc2 = tf32_idesc(kLtM, 2 * mo);
            const unsigned lb = (unsigned)(2 * mo / 8) * 128;
            bool ok = true;
            for (int ci = 0; ci < U.nch && ok; ++ci, ++k) {
                const int st = (int)(k % kWgStages);
                const bool first = ci % seg == 0;
                const bool last = ci + 1 == U.nch || (ci + 1) % seg == 0;
                const int b = (int)(t % nacc);
                ok = wait(&full[st], (unsigned)((k / kWgStages) & 1));
                if (ok && first && t >= nacc)
                    ok = wait(&acc_free[b], (unsigned)(((t - nacc) / nacc) & 1));
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (leader) {
                    const unsigned b0 = smem_addr(smem + (size_t)st * bslot);
                    const unsigned a0 = tmem + kLtAcol + 64u * st;
                    const unsigned acc = tmem + 128u * b;
#pragma unroll
                    for (int k8 = 0; k8 < kWgRows; k8 += 8) {
                        const uint64_t bd = smem_desc(b0 + (unsigned)(k8 >> 2) * lb, lb, 128);
                        mma_tf32_tmem_a(acc, a0 + k8, bd, idesc2, (first && k8 == 0) ? 0u : 1u);
                        mma_tf32_tmem_a(acc, a0 + 32 + k8, bd, idesc, 1u);
                    }
                    tc_commit(&empty[st]);
                    if (last) tc_commit(&acc_full[b]);
                }
                __syncwarp();
                last_commit = k;
                if (last) ++t;
            }
            if (!ok) break;
            if (__any_sync(0xffffffffu, *(volatile int*)&fail)) break;
        }
        if (leader && last_commit >= 0)
            tc_mbar_wait(&empty[last_commit % kWgStages], (unsigned)((last_commit / kWgStages) & 1));
    } else if (warp < 4) {
        // ----------------------------------------------------------- epilogue
        int64_t t = 0;
        for (int64_t r = 0, u; (u = unit_at(r)) < units; ++r) {
            Unit U;
            unit_of(u, U);
            const LinGrad& G = D.g[U.j];
            const int sp = U.sp;
            const int urow = U.mt * 128 + 32 * warp + lane;  // input channel of this lane
            // element (urow, w) at prow[w * ws]: rows of the layer's layout, or
            // a column of a transposed output (lanes then store consecutive words)
            float* prow = partial + (int64_t)sp * D.nw + G.w_off +
                          (G.tr ? (int64_t)urow : (int64_t)urow * G.ldw);
            const int64_t ws = G.tr ? G.ldw : 1;
            const bool live = urow < G.mi;
            if (U.nch == 0) {  // empty split: its partial sums are zero
                if (live)
                    for (int w = 0; w < G.mo; ++w) prow[w * ws] = 0.0f;
                continue;
            }
            // this thread's running sums, column w at sums[128 w] (lanes contiguous)
            float* sums = reinterpret_cast<float*>(smem + kWgStages * (size_t)bslot) + 32 * warp + lane;
            const int nseg = (U.nch + seg - 1) / seg;
            bool got = true;
            for (int sg = 0; sg < nseg && got; ++sg, ++t) {
                const int b = (int)(t % nacc);
                got = wait(&acc_full[b], (unsigned)((t / nacc) & 1));
                got = __all_sync(0xffffffffu, got);
                if (!got) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const bool fin = sg + 1 == nseg;
                for (int c0 = 0; c0 < G.mo; c0 += 32) {
                    float v[32], v2[32];
                    const unsigned ta = tmem + ((unsigned)(32 * warp) << 16) + 128u * b + (unsigned)c0;
                    tmem_ld32(ta, v);
                    tmem_ld32(ta + (unsigned)G.mo, v2);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        v[i] += v2[i];
                        if (sg > 0) v[i] = sums[128 * (c0 + i)] + v[i];
                        if (!fin) sums[128 * (c0 + i)] = v[i];
                    }
                    if (!fin) continue;
                    if (live && !G.tr) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            *reinterpret_cast<float4*>(prow + c0 + 4 * i) =
                                make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    } else if (live) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) prow[(int64_t)(c0 + i) * ws] = v[i];
                    }
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                tc_mbar_arrive(&acc_free[b]);
            }
            if (!got) break;
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (tid == 0 && fail) atomicExch(&cgtp_linear_error, 1);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kLtTmemCols)
                     : "memory");
}

// ------------------------------------------------------------------- host

struct LinearImpl {
    std::vector<Irrep> in, out;
    std::vector<int> off_in, off_out;
    std::vector<std::pair<int, int>> instr;  // (input irrep, output irrep)
    std::vector<int64_t> w_off;
    int64_t dim_in = 0, dim_out = 0, nw = 0;
    cgtp_dtype dtype = CGTP_F32;
    LinDesc fwd{}, bwd{};  // forward (blocks = outputs) and x gradient (blocks = inputs)
    std::vector<std::pair<int, int>> fwd_zero, bwd_zero;  // unreached blocks: (offset, width)
    LinGradDesc grad{};
    bool tc = false;
    size_t fwd_img = 0, bwd_img = 0;
    int fwd_nmax = 0, bwd_nmax = 0;
};

static size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Blocks of one pass: for every target irrep reached by an instruction, its
// chunks (instruction order, 32 source channels each).  fwd: target = output.
// Groups of blocks that read the same input rows: equal d and the same
// chunk sequence (source offset, width, K range); the tensor-core kernel runs
// a group's units tile-major.
static void lin_groups(LinDesc& D) {
    auto same = [&](int a, int b) {
        const LinBlock &A = D.blk[a], &B = D.blk[b];
        if (A.d != B.d || A.nchunk != B.nchunk) return false;
        for (int i = 0; i < A.nchunk; ++i) {
            const LinChunk &x = D.ch[A.chunk0 + i], &y = D.ch[B.chunk0 + i];
            if (x.a_off != y.a_off || x.a_mul != y.a_mul || x.k0 != y.k0 || x.kc != y.kc) return false;
        }
        return true;
    };
    std::vector<std::vector<int>> grp;
    for (int b = 0; b < D.nblocks; ++b) {
        bool placed = false;
        for (auto& g : grp)
            if (same(g[0], b)) {
                g.push_back(b);
                placed = true;
                break;
            }
        if (!placed) grp.push_back({b});
    }
    D.ngrp = (int)grp.size();
    int k = 0;
    for (int g = 0; g < D.ngrp; ++g) {
        D.grp_nb[g] = (int)grp[g].size();
        D.grp_b0[g] = k;
        for (int b : grp[g]) D.grp_b[k++] = b;
    }
}

// Units of the tensor-core kernel for n rows of items: per group, its blocks
// times the 128-row tiles of one block (n d rows).
static int64_t lin_units(LinDesc& D, int64_t n) {
    D.grp_u0[0] = 0;
    for (int g = 0; g < D.ngrp; ++g) {
        D.grp_nt[g] = (n * D.blk[D.grp_b[D.grp_b0[g]]].d + kLtM - 1) / kLtM;
        D.grp_u0[g + 1] = D.grp_u0[g] + D.grp_nb[g] * D.grp_nt[g];
    }
    return D.grp_u0[D.ngrp];
}

static bool build_pass(LinearImpl& L, bool fwd, std::string& err) {
    LinDesc& D = fwd ? L.fwd : L.bwd;
    auto& zero = fwd ? L.fwd_zero : L.bwd_zero;
    const auto& tgt = fwd ? L.out : L.in;
    const auto& toff = fwd ? L.off_out : L.off_in;
    D.in_stride = fwd ? L.dim_in : L.dim_out;
    D.out_stride = fwd ? L.dim_out : L.dim_in;
    D.nblocks = D.nchunks = 0;
    size_t img = 0;
    int nmax = 0;
    for (int t = 0; t < (int)tgt.size(); ++t) {
        const int ncols = tgt[t].mul, d = 2 * tgt[t].l + 1;
        const int c0 = D.nchunks;
        for (int j = 0; j < (int)L.instr.size(); ++j) {
            const int src = fwd ? L.instr[j].first : L.instr[j].second;
            if ((fwd ? L.instr[j].second : L.instr[j].first) != t) continue;
            const int mi = L.in[L.instr[j].first].mul, mo = L.out[L.instr[j].second].mul;
            const int ksrc = fwd ? mi : mo;
            for (int k0 = 0; k0 < ksrc; k0 += kLtK) {
                if (D.nchunks >= kLinMaxChunks) {
                    err = "too many weight chunks for one linear layer";
                    return false;
                }
                LinChunk& C = D.ch[D.nchunks++];
                C.src = src;
                C.a_off = fwd ? L.off_in[src] : L.off_out[src];
                C.a_mul = ksrc;
                C.k0 = k0;
                C.kc = std::min(kLtK, ksrc - k0);
                C.w_off = (int)L.w_off[j];
                C.w_ks = fwd ? mo : 1;
                C.w_ns = fwd ? 1 : mo;
                C.img_off = (int)img;
                img += (size_t)2 * ncols * kLtK * 4;
            }
        }
        if (D.nchunks == c0) {
            zero.emplace_back(toff[t], ncols * d);
            continue;
        }
        if (D.nblocks >= kLinMaxBlocks) {
            err = "too many irreps for one linear layer";
            return false;
        }
        D.blk[D.nblocks++] = LinBlock{toff[t], ncols, d, c0, D.nchunks - c0};
        nmax = std::max(nmax, ncols);
    }
    (fwd ? L.fwd_img : L.bwd_img) = img;
    (fwd ? L.fwd_nmax : L.bwd_nmax) = nmax;
    lin_groups(D);
    return true;
}

cgtp_status linear_create(const char* sin, const char* sout, const cgtp_linear_instr* instr,
                          int n_instr, cgtp_dtype dt, LinearImpl** res, std::string& err) {
    auto L = std::make_unique<LinearImpl>();
    if (!parse_irreps(sin, L->in, err) || !parse_irreps(sout, L->out, err)) return CGTP_E_IRREPS;
    L->dtype = dt;
    for (auto* v : {&L->in, &L->out}) {
        int64_t off = 0;
        auto& offs = v == &L->in ? L->off_in : L->off_out;
        for (const Irrep& r : *v) {
            offs.push_back((int)off);
            off += (int64_t)r.mul * (2 * r.l + 1);
        }
        (v == &L->in ? L->dim_in : L->dim_out) = off;
    }
    if (L->dim_in >= (1 << 30) || L->dim_out >= (1 << 30)) {
        err = "irreps too wide";
        return CGTP_E_IRREPS;
    }
    if (instr == nullptr) {
        for (int i = 0; i < (int)L->in.size(); ++i)
            for (int o = 0; o < (int)L->out.size(); ++o)
                if (L->in[i].l == L->out[o].l && L->in[i].parity == L->out[o].parity)
                    L->instr.emplace_back(i, o);
    } else {
        if (n_instr < 0) {
            err = "negative instruction count";
            return CGTP_E_ARG;
        }
        for (int j = 0; j < n_instr; ++j) {
            const int i = instr[j].i_in, o = instr[j].i_out;
            if (i < 0 || i >= (int)L->in.size() || o < 0 || o >= (int)L->out.size()) {
                err = "instruction " + std::to_string(j) + " indexes outside the irreps";
                return CGTP_E_PATH;
            }
            if (L->in[i].l != L->out[o].l || L->in[i].parity != L->out[o].parity) {
                err = "instruction " + std::to_string(j) + " joins irreps of different l or parity";
                return CGTP_E_PATH;
            }
            L->instr.emplace_back(i, o);
        }
    }
    if ((int)L->instr.size() > kLinMaxGrad) {
        err = "too many instructions for one linear layer";
        return CGTP_E_UNSUPPORTED;
    }
    for (auto& [i, o] : L->instr) {
        L->w_off.push_back(L->nw);
        L->nw += (int64_t)L->in[i].mul * L->out[o].mul;
    }
    if (L->nw >= (1ll << 31)) {
        err = "weights too large";
        return CGTP_E_UNSUPPORTED;
    }
    if (!build_pass(*L, true, err) || !build_pass(*L, false, err)) return CGTP_E_UNSUPPORTED;
    // gradient in W
    LinGradDesc& G = L->grad;
    G.ninstr = (int)L->instr.size();
    G.x_stride = L->dim_in;
    G.g_stride = L->dim_out;
    G.nw = L->nw;
    int tiles = 0;
    for (int j = 0; j < G.ninstr; ++j) {
        const auto [i, o] = L->instr[j];
        G.g[j] = LinGrad{L->off_in[i], L->in[i].mul, L->off_out[o], L->out[o].mul,
                         2 * L->in[i].l + 1, (int)L->w_off[j], tiles, G.nmt, L->out[o].mul, 0};
        tiles += ((L->in[i].mul + 31) / 32) * ((L->out[o].mul + 31) / 32);
        G.nmt += (L->in[i].mul + 127) / 128;
    }
    G.ntiles = tiles;
    wgrad_schedule(G);
    bool tc = dt == CGTP_F32;
    for (const auto* v : {&L->in, &L->out})
        for (const Irrep& r : *v) tc = tc && r.mul % 32 == 0 && r.mul <= 256;
    L->tc = tc;
    *res = L.release();
    return CGTP_OK;
}

void linear_destroy(LinearImpl* L) { delete L; }

void linear_info(const LinearImpl* L, int64_t* dim_in, int64_t* dim_out, int64_t* nw, int* ni) {
    if (dim_in) *dim_in = L->dim_in;
    if (dim_out) *dim_out = L->dim_out;
    if (nw) *nw = L->nw;
    if (ni) *ni = (int)L->instr.size();
}

bool linear_instruction(const LinearImpl* L, int j, int* i_in, int* i_out, int64_t* w_off) {
    if (j < 0 || j >= (int)L->instr.size()) return false;
    if (i_in) *i_in = L->instr[j].first;
    if (i_out) *i_out = L->instr[j].second;
    if (w_off) *w_off = L->w_off[j];
    return true;
}

bool linear_tensor_cores(const LinearImpl* L) { return L->tc; }

// Row splits of the W gradient: partial sums per split, added in split order.
static int64_t wgrad_splits(int64_t n) { return std::max<int64_t>(1, std::min<int64_t>(64, (n + 63) / 64)); }

size_t linear_fwd_workspace(const LinearImpl* L) { return L->tc ? L->fwd_img : 0; }

size_t linear_bwd_workspace(const LinearImpl* L, int64_t n) {
    const size_t es = L->dtype == CGTP_F64 ? 8 : 4;
    return round_up(L->tc ? L->bwd_img : 0, 256) + (size_t)wgrad_splits(n) * L->nw * es;
}

static int sm_count() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        return 148;
    return v;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

template <typename T>
static cudaError_t zero_blocks(const std::vector<std::pair<int, int>>& z, int64_t n, int64_t stride,
                               T* out, cudaStream_t s) {
    for (auto [off, width] : z) {
        const int64_t total = n * width;
        if (total == 0) continue;
        const unsigned g = (unsigned)std::min<int64_t>((total + 255) / 256, 4096);
        linear_zero_kernel<T><<<g, 256, 0, s>>>(n, stride, off, width, out);
        count_launch();
    }
    return cudaGetLastError();
}

// One GEMM pass (forward or x gradient) into `out`.
static cudaError_t run_pass(const LinearImpl& L, const LinDesc& D, int nmax, size_t img_bytes,
                            bool test_fail,
                            int64_t n, const void* a, const void* W, void* out, void* img,
                            bool use_tc, cudaStream_t s) {
    if (D.nblocks == 0 || n == 0) return cudaSuccess;
    if (L.dtype == CGTP_F64) {
        int dmax = 1;
        for (int b = 0; b < D.nblocks; ++b) dmax = std::max(dmax, D.blk[b].d);
        const dim3 g((unsigned)((n * dmax + kLsT - 1) / kLsT), (unsigned)((nmax + kLsC - 1) / kLsC),
                     (unsigned)D.nblocks);
        linear_simt_kernel<double><<<g, kLsThreads, 0, s>>>(D, n, (const double*)a,
                                                            (const double*)W, (double*)out);
        count_launch();
        return cudaGetLastError();
    }
    if (!use_tc) {
        int dmax = 1;
        for (int b = 0; b < D.nblocks; ++b) dmax = std::max(dmax, D.blk[b].d);
        const dim3 g((unsigned)((n * dmax + kLsT - 1) / kLsT), (unsigned)((nmax + kLsC - 1) / kLsC),
                     (unsigned)D.nblocks);
        linear_simt_kernel<float><<<g, kLsThreads, 0, s>>>(D, n, (const float*)a, (const float*)W,
                                                           (float*)out);
        count_launch();
        return cudaGetLastError();
    }
    // up to 128 columns: A_hi [B_hi | B_lo] as one N = 2 ncols product (stacked
    // B image), one accumulator of 2 ncols columns; 256: three products.
    // Blocks of at most four K chunks (the x-gradient of a layer whose
    // instructions each take one 128-channel irrep): three products into two
    // alternating 128-column accumulators, so that one unit's epilogue and
    // the next unit's products overlap.
    int kmax = 0;
    for (int b = 0; b < D.nblocks; ++b) kmax = std::max(kmax, D.blk[b].nchunk);
    const bool twoacc = nmax <= 128 && kmax <= 4;
    const bool stack = nmax <= 128 && !twoacc;
    linear_pack_kernel<<<(unsigned)D.nchunks, 256, 0, s>>>(D, (const float*)W, (unsigned char*)img,
                                                          stack);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // per-launch copy with the tile ranges of the blocks for this n
    auto Dn = std::make_unique<LinDesc>(D);
    const int64_t units = lin_units(*Dn, n);
    const unsigned grid = (unsigned)std::min<int64_t>(units, sm_count());
    // stages (A in tensor memory, B in shared memory): 4 up to 128 columns, 3 at 256
    const size_t smem = std::max<size_t>(
        120 * 1024, stack    ? lt_smem_bytes(nmax, 4, true)
                    : twoacc ? lt_smem_bytes(nmax, 4, false)
                             : lt_smem_bytes(nmax, 3, false));
    auto* kern = stack    ? linear_tc_kernel<4, 1, true, 0>
                 : twoacc ? linear_tc_kernel<4, 2, false, 0>
                          : linear_tc_kernel<3, 1, false, 0>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    (void)img_bytes;
    kern<<<grid, kLtThreads, smem, s>>>(*Dn, n, nmax, (const float*)a, (const unsigned char*)img,
                                        (float*)out, TpArg<false>{}, test_fail ? 1 : 0);
    count_launch();
    return cudaGetLastError();
}

bool linear_uses_tc(const LinearImpl* L, int64_t n, const void* a, const void* out, const void* ws,
                    size_t ws_bytes, bool fwd) {
    (void)n;
    return L->tc && ws && ws_bytes >= (fwd ? L->fwd_img : L->bwd_img) && aligned16(a) &&
           aligned16(out) && aligned16(ws);
}

cudaError_t launch_linear_forward(const LinearImpl* L, int64_t n, const void* x, const void* W,
                                  void* out, void* ws, size_t ws_bytes, bool allow_tc,
                                  cudaStream_t s, bool test_fail) {
    cudaError_t e = L->dtype == CGTP_F64
                        ? zero_blocks(L->fwd_zero, n, L->dim_out, (double*)out, s)
                        : zero_blocks(L->fwd_zero, n, L->dim_out, (float*)out, s);
    if (e != cudaSuccess) return e;
    const bool tc = allow_tc && linear_uses_tc(L, n, x, out, ws, ws_bytes, true);
    return run_pass(*L, L->fwd, L->fwd_nmax, L->fwd_img, test_fail, n, x, W, out, ws, tc, s);
}

// T rows of the fused 'uvw' forward: t[n, e] = sum over entry e's CG terms of
// c * y[n, term_y] (channel-independent).  One CTA per sample at a time, the
// term table in shared memory.
__global__ void __launch_bounds__(256)
lin_tp_t_kernel(const __grid_constant__ LinTpDesc D, int64_t n, const float* __restrict__ y,
                int64_t y_stride, float* __restrict__ t) {
    __shared__ short es[kTpMaxT + 1];
    __shared__ unsigned char ty[kTpMaxTerms];
    __shared__ float tc[kTpMaxTerms];
    for (int i = threadIdx.x; i <= D.tdim; i += blockDim.x) es[i] = D.estart[i];
    for (int i = threadIdx.x; i < D.nterms; i += blockDim.x) {
        ty[i] = D.term_y[i];
        tc[i] = D.term_c[i];
    }
    __syncthreads();
    for (int64_t item = blockIdx.x; item < n; item += gridDim.x) {
        const float* yr = y + item * y_stride;
        for (int e = threadIdx.x; e < D.tdim; e += blockDim.x) {
            float a = 0.0f;
            for (int k = es[e]; k < es[e + 1]; ++k) a = fmaf(tc[k], __ldg(yr + ty[k]), a);
            t[item * D.tdim + e] = a;
        }
    }
}

cudaError_t launch_linear_forward_tp(const LinearImpl* L, const LinTpDesc& tp, int64_t n,
                                     const void* x1, int64_t x1_stride, const void* y,
                                     int64_t y_stride, const void* W, void* out, void* ws,
                                     size_t ws_bytes, void* tbuf, size_t tbuf_bytes,
                                     cudaStream_t s, bool* used) {
    *used = false;
    const LinDesc& D = L->fwd;
    const int nmax = L->fwd_nmax;
    // the stacked tensor-core shape (every output multiplicity <= 128), one
    // source path per input irrep, 16-byte aligned x1 rows and channel groups
    if (!L->tc || nmax > 128 || !ws || ws_bytes < L->fwd_img || !aligned16(ws) ||
        !aligned16(x1) || !aligned16(out) || (x1_stride % 4) != 0 || ((uintptr_t)y & 3) != 0 ||
        tp.npaths != (int)L->in.size() || tp.tdim <= 0 || tp.tdim > kTpMaxT ||
        tp.nterms > kTpMaxTerms || !tbuf || ((uintptr_t)tbuf & 3) != 0 ||
        tbuf_bytes < (size_t)n * tp.tdim * 4)
        return cudaSuccess;
    int groups = 1;  // m1 values of one row (d1), at most 7 here
    for (int p = 0; p < tp.npaths; ++p) {
        if (tp.path[p].x1_off % 4 != 0 || tp.path[p].mul1 % 4 != 0 ||
            tp.path[p].mul1 != L->in[p].mul || tp.path[p].d3 != 2 * L->in[p].l + 1)
            return cudaSuccess;
        groups = std::max(groups, tp.path[p].d1);
    }
    if (groups > 7) return cudaSuccess;
    for (int g = 0; g < D.ngrp; ++g)  // the fused kernel takes single-block groups
        if (D.grp_nb[g] != 1) return cudaSuccess;
    *used = true;
    cudaError_t e = zero_blocks(L->fwd_zero, n, L->dim_out, (float*)out, s);
    if (e != cudaSuccess || D.nblocks == 0 || n == 0) return e;
    const unsigned tg = (unsigned)std::max<int64_t>(1, std::min<int64_t>(n, 8 * sm_count()));
    lin_tp_t_kernel<<<tg, 256, 0, s>>>(tp, n, (const float*)y, y_stride, (float*)tbuf);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    linear_pack_kernel<<<(unsigned)D.nchunks, 256, 0, s>>>(D, (const float*)W, (unsigned char*)ws,
                                                          true);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    auto Dn = std::make_unique<LinDesc>(D);
    const int64_t units = lin_units(*Dn, n);
    const unsigned grid = (unsigned)std::min<int64_t>(units, sm_count());
    const size_t smem = std::max<size_t>(120 * 1024, lt_smem_bytes(nmax, 4, true, true));
    auto* kern = groups <= 3 ? linear_tc_kernel<4, 1, true, 3>
                             : groups <= 5 ? linear_tc_kernel<4, 1, true, 5>
                                           : linear_tc_kernel<4, 1, true, 7>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    auto arg = std::make_unique<TpArg<true>>();
    arg->d = tp;
    arg->x1 = (const float*)x1;
    arg->x1_stride = x1_stride;
    arg->t = (const float*)tbuf;
    kern<<<grid, kLtThreads, smem, s>>>(*Dn, n, nmax, nullptr, (const unsigned char*)ws,
                                        (float*)out, *arg, 0);
    count_launch();
    return cudaGetLastError();
}

void* tensor_map_encoder() {
    static void* encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = fn;
        else
            cudaGetLastError();
    });
    return encode;
}

// The weight gradient's tensor maps (WgMaps) for x [n][x_stride] and g
// [n][g_stride], fp32: set when every instruction takes 128 input channels at
// a 128-aligned offset, all take the same mo output channels (mo % 32 == 0) at
// mo-aligned offsets, d is odd and at most 15, and the data are 16-byte
// aligned.  M->on stays 0 otherwise (row-by-row copies).
static void wgrad_maps(const LinGradDesc& G, int64_t n, const void* x, const void* g, WgMaps* M) {
    M->on = 0;
    M->gbox = 128;
    const auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
    if (!encode || n < 1 || n > 0x7fffffff || G.ninstr < 1 || !aligned16(x) || !aligned16(g)) return;
    const int mo = G.g[0].mo;
    if (mo % 32 != 0 || mo > 128 || G.x_stride % 128 != 0 || G.g_stride % mo != 0) return;
    bool used[kWgMaxD] = {};
    for (int j = 0; j < G.ninstr; ++j) {
        const LinGrad& L = G.g[j];
        if (L.mi != 128 || L.xo % 128 != 0 || L.mo != mo || L.go % mo != 0 || L.d % 2 != 1 ||
            L.d > 2 * kWgMaxD - 1)
            return;
        used[(L.d - 1) / 2] = true;
    }
    auto enc = [&](CUtensorMap* m, const void* base, int width, int64_t stride, int d) {
        const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)(stride / width), (cuuint64_t)n};
        const cuuint64_t strides[2] = {(cuuint64_t)width * 4, (cuuint64_t)stride * 4};
        const cuuint32_t box[3] = {(cuuint32_t)width, (cuuint32_t)d, (cuuint32_t)(kWgRows / d)};
        const cuuint32_t es[3] = {1, 1, 1};
        return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                      box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    for (int i = 0; i < kWgMaxD; ++i)
        if (used[i] && !(enc(&M->x[i], x, 128, G.x_stride, 2 * i + 1) &&
                         enc(&M->g[i], g, mo, G.g_stride, 2 * i + 1)))
            return;
    M->gbox = mo;
    M->on = 1;
}

// Accumulator buffers of the tensor-core weight gradient: two when every
// stacked [hi | lo] accumulator (2 mul_out columns) fits in 128 columns.  (The
// three split products as N = mul_out instructions into one mul_out-column
// accumulator would allow two buffers at mul_out = 128 too; measured slower.)
static int wgrad_accumulators(const LinGradDesc& G) {
    for (int j = 0; j < G.ninstr; ++j)
        if (G.g[j].mo > 64) return 1;
    return 2;
}

// The tensor-core weight gradient: fp32 tensor-core layer with every output
// multiplicity at most 128 (the stacked [hi | lo] image), 16-byte aligned data.
static bool linear_wgrad_tc_ok(const LinearImpl* L, const void* x, const void* g, const void* part) {
    if (!L->tc) return false;
    for (int j = 0; j < L->grad.ninstr; ++j)
        if (L->grad.g[j].mo > 128) return false;
    return aligned16(x) && aligned16(g) && aligned16(part);
}

cudaError_t launch_linear_backward(const LinearImpl* L, int64_t n, const void* x, const void* W,
                                   const void* g, void* gx, void* gW, void* ws, size_t ws_bytes,
                                   bool allow_tc, cudaStream_t s) {
    const bool f64 = L->dtype == CGTP_F64;
    cudaError_t e = cudaSuccess;
    if (gx) {
        e = f64 ? zero_blocks(L->bwd_zero, n, L->dim_in, (double*)gx, s)
                : zero_blocks(L->bwd_zero, n, L->dim_in, (float*)gx, s);
        if (e != cudaSuccess) return e;
        const bool tc = allow_tc && linear_uses_tc(L, n, g, gx, ws, ws_bytes, false);
        e = run_pass(*L, L->bwd, L->bwd_nmax, L->bwd_img, false, n, g, W, gx, ws, tc, s);
        if (e != cudaSuccess) return e;
    }
    if (gW && L->nw > 0) {
        if (n == 0) return launch_fill_zero(gW, L->nw * (f64 ? 8 : 4), s);
        const int64_t S = wgrad_splits(n), per = (n + S - 1) / S;
        unsigned char* part = (unsigned char*)ws + round_up(L->tc ? L->bwd_img : 0, 256);
        const dim3 grid((unsigned)L->grad.ntiles, (unsigned)S);
        if (allow_tc && linear_wgrad_tc_ok(L, x, g, part)) {
            const int64_t units = (int64_t)L->grad.nmt * S;
            const unsigned gr = (unsigned)std::min<int64_t>(units, sm_count());
            e = cudaFuncSetAttribute(linear_wgrad_tc_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWgSmem);
            if (e != cudaSuccess) return e;
            // one copy per operand and chunk of whole items where the layer's
            // shape allows, else row-by-row copies merged per item
            auto M = std::make_unique<WgMaps>();
            wgrad_maps(L->grad, n, x, g, M.get());
            linear_wgrad_tc_kernel<<<gr, kWgThreads, kWgSmem, s>>>(
                L->grad, n, per, (int)S, wgrad_accumulators(L->grad), (const float*)x,
                (const float*)g, (float*)part, *M);
        } else if (f64)
            linear_wgrad_kernel<double><<<grid, 256, 0, s>>>(L->grad, n, per, (const double*)x,
                                                             (const double*)g, (double*)part);
        else
            linear_wgrad_kernel<float><<<grid, 256, 0, s>>>(L->grad, n, per, (const float*)x,
                                                            (const float*)g, (float*)part);
        count_launch();
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        e = launch_reduce_rows(f64, part, S, L->nw, gW, s);
    }
    return e;
}

cudaError_t linear_device_status(int* code) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, cgtp_linear_error, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(cgtp_linear_error, &zero, sizeof(int));
    return e;
}

// grad_W2 = h^T grad_w of the radial network (a sum over edges) on the tensor
// cores through the weight-gradient kernel: "x" = grad_w [E, n_out] in
// 128-column instructions (M = the output columns), "g" = h [E, hidden]
// (N = hidden), each instruction's [128 x hidden] block stored transposed into
// the row-major [hidden, n_out] partial rows.  fp32, hidden % 32 == 0 and
// <= 128, n_out % 128 == 0 and <= 128 * kLinMaxGrad, 16-byte aligned data.
bool radial_w2_tc_eligible(int hidden, int64_t n_out) {
    return hidden % 32 == 0 && hidden <= 128 && n_out % 128 == 0 && n_out / 128 <= kLinMaxGrad;
}

cudaError_t launch_radial_w2_tc(int64_t E, int hidden, int64_t n_out, const float* h,
                                const float* gw, float* partial, int64_t S, cudaStream_t s) {
    auto G = std::make_unique<LinGradDesc>();
    G->ninstr = (int)(n_out / 128);
    G->ntiles = 0;
    G->nmt = G->ninstr;
    G->x_stride = n_out;
    G->g_stride = hidden;
    G->nw = (int64_t)hidden * n_out;
    for (int j = 0; j < G->ninstr; ++j)
        G->g[j] = LinGrad{128 * j, 128, 0, hidden, 1, 128 * j, 0, j, (int)n_out, 1};
    wgrad_schedule(*G);
    const int64_t per = (E + S - 1) / S;
    const int64_t units = (int64_t)G->nmt * S;
    const unsigned gr = (unsigned)std::min<int64_t>(units, sm_count());
    cudaError_t e = cudaFuncSetAttribute(linear_wgrad_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWgSmem);
    if (e != cudaSuccess) return e;
    auto M = std::make_unique<WgMaps>();
    wgrad_maps(*G, E, gw, h, M.get());
    linear_wgrad_tc_kernel<<<gr, kWgThreads, kWgSmem, s>>>(*G, E, per, (int)S,
                                                           wgrad_accumulators(*G), gw, h, partial,
                                                           *M);
    count_launch();
    return cudaGetLastError();
}

}  // namespace cgtp
