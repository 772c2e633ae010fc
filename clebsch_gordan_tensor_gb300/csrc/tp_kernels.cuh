// Tensor-product kernels of the CG library, compiled at run time by NVRTC for
// sm_103a once per plan.  The plan generator prepends the constants, the CG
// tables and the fully unrolled per-path contraction streams (gen_fwd,
// gen_bwd); this file holds the parts that do not depend on the irreps.
//
// Method ("An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep
// Networks", abstract): the CG tensor product of x (irreps_in1) and y
// (irreps_in2) under per-edge weights, alone and fused with the graph
// convolution (gather x by sender, product per edge, sum into the receiver),
// plus its gradient.  Operands of one channel group are held in registers and
// the CG coefficients are immediates of one long FMA stream.
//
// Work decomposition.  A "slot" of LANES threads owns one item: a receiver
// (fused convolution forward), a sender (convolution gradient) or a sample
// (standalone product).  Lane `ch` of a slot owns channels [CPT*ch, CPT*ch+CPT)
// of every irrep block; with CPT == 2 (fp32) the pair is one 64-bit register
// and every FMA is a packed fma.rn.f32x2.  Per edge the slot first builds
//   T_p[m1, m3] = sum_m2 C_p[m1, m2, m3] y[e, o2 + m2]
// cooperatively in shared memory (it is the same for every channel), then
// each lane runs the generated stream
//   out[r3 + m3] += T_p[m1, m3] * (w[e, p, ch] * x[s, r1 + m1, ch]).
// Receiver sums run in edge order inside one slot: no atomics, deterministic.
//
// Provided by the generator: REAL, CPT, MUL, NCH, LANES, SLOTS, BLOCK, NX, NY,
// NYP, NO, NP, NT, NTP, MAXTERMS, YPF, IS_F64, T_IDX[], T_CO[], gen_fwd,
// gen_bwd.

typedef unsigned long long u64;

#define DIMX ((long long)NX * MUL)
#define DIMO ((long long)NO * MUL)
#define WDIM ((long long)NP * MUL)

#if CPT == 2
typedef u64 VR;  // two fp32 channels
__device__ __forceinline__ VR vfma(VR a, VR b, VR c) {
    VR d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ VR vmul(VR a, VR b) {
    VR d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ VR vadd(VR a, VR b) {
    VR d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ VR vzero() { return 0ull; }
__device__ __forceinline__ VR vsplat(float s) {
    const u64 u = __float_as_uint(s);
    return (u << 32) | u;
}
__device__ __forceinline__ float vlo(VR a) { return __uint_as_float((unsigned)a); }
__device__ __forceinline__ float vhi(VR a) { return __uint_as_float((unsigned)(a >> 32)); }
// sum over the two channels of a * b
__device__ __forceinline__ float vdot(VR a, VR b) { return fmaf(vlo(a), vlo(b), vhi(a) * vhi(b)); }
__device__ __forceinline__ VR ldv(const REAL* p, int ch) {
    return __ldg(reinterpret_cast<const u64*>(p) + ch);
}
__device__ __forceinline__ void stv(REAL* p, int ch, VR v) { reinterpret_cast<u64*>(p)[ch] = v; }
__device__ __forceinline__ VR ldv_plain(const REAL* p, int ch) {
    return reinterpret_cast<const u64*>(p)[ch];
}
#else
typedef REAL VR;  // one channel
__device__ __forceinline__ VR vfma(VR a, VR b, VR c) { return fma(a, b, c); }
__device__ __forceinline__ VR vmul(VR a, VR b) { return a * b; }
__device__ __forceinline__ VR vadd(VR a, VR b) { return a + b; }
__device__ __forceinline__ VR vzero() { return (REAL)0; }
__device__ __forceinline__ VR vsplat(REAL s) { return s; }
__device__ __forceinline__ REAL vdot(VR a, VR b) { return a * b; }
__device__ __forceinline__ VR ldv(const REAL* p, int ch) { return __ldg(p + ch); }
__device__ __forceinline__ void stv(REAL* p, int ch, VR v) { p[ch] = v; }
__device__ __forceinline__ VR ldv_plain(const REAL* p, int ch) { return p[ch]; }
#endif

#if NCH == LANES
#define CH_ACTIVE(ch) true
#else
#define CH_ACTIVE(ch) ((ch) < NCH)
#endif

__device__ __forceinline__ VR ldv_m(const REAL* p, int ch) {
    return CH_ACTIVE(ch) ? ldv(p, ch) : vzero();
}

// Weight storage (W_STORE): 0 = REAL; 1 = bfloat16, 2 = IEEE binary16, each
// widened exactly to fp32 on load (every value of either format is an fp32
// value); the arithmetic is the same in all three.  WRAW is what one lane
// loads for its channels (two 16-bit values in one 32-bit word when CPT == 2:
// channel 2ch in the low half).
#if W_STORE == 2
__device__ __forceinline__ float h2f(unsigned short h) {
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
    return f;
}
#endif
#if W_STORE != 0
typedef unsigned short WT;
#if CPT == 2
typedef unsigned WRAW;
__device__ __forceinline__ VR wcvt(WRAW u) {
#if W_STORE == 1
    return ((u64)(u & 0xffff0000u) << 32) | (u64)(u << 16);
#else
    return ((u64)__float_as_uint(h2f((unsigned short)(u >> 16))) << 32) |
           (u64)__float_as_uint(h2f((unsigned short)(u & 0xffffu)));
#endif
}
#else
typedef unsigned short WRAW;
#if W_STORE == 1
__device__ __forceinline__ VR wcvt(WRAW u) { return __uint_as_float((unsigned)u << 16); }
#else
__device__ __forceinline__ VR wcvt(WRAW u) { return h2f(u); }
#endif
#endif
#else
typedef REAL WT;
typedef VR WRAW;
__device__ __forceinline__ VR wcvt(WRAW u) { return u; }
#endif
__device__ __forceinline__ WRAW ldw_raw(const WT* p, int ch) {
    return __ldg(reinterpret_cast<const WRAW*>(p) + ch);
}
__device__ __forceinline__ VR ldw(const WT* p, int ch) { return wcvt(ldw_raw(p, ch)); }
__device__ __forceinline__ VR ldw_m(const WT* p, int ch) {
    return CH_ACTIVE(ch) ? ldw(p, ch) : vzero();
}
// from a shared-memory stage
__device__ __forceinline__ VR lds_w(const WT* p, int ch) {
    return wcvt(reinterpret_cast<const WRAW*>(p)[ch]);
}

// Weight of path p for this lane's channels, from global memory (direct
// kernels) or from the shared-memory stage (staged kernels).
__device__ __forceinline__ VR lds_v(const REAL* p, int ch) {
    return reinterpret_cast<const VR*>(p)[ch];
}

#if LANES <= 32
__device__ __forceinline__ unsigned slot_mask() {
    if (LANES == 32) return 0xffffffffu;
    const unsigned base = ((threadIdx.x & 31u) / LANES) * LANES;
    return (LANES == 32 ? 0xffffffffu : ((1u << LANES) - 1u)) << base;
}
__device__ __forceinline__ void slot_sync(int) { __syncwarp(slot_mask()); }
#else
// LANES / 32 warps per slot: named barrier 1 + slot.
__device__ __forceinline__ unsigned slot_mask() { return 0xffffffffu; }
__device__ __forceinline__ void slot_sync(int slot) {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + slot), "r"(LANES) : "memory");
}
#endif

// Per-edge T entries, lane-strided over the slot.  Ys holds the edge's y row.
__device__ __forceinline__ void build_T(REAL* __restrict__ Ts, const REAL* __restrict__ Ys, int lane) {
    for (int k = lane; k < NT; k += LANES) {
        REAL t = (REAL)0;
#pragma unroll
        for (int q = 0; q < MAXTERMS; ++q)
            t = fma(T_CO[k * MAXTERMS + q], Ys[T_IDX[k * MAXTERMS + q]], t);
        Ts[k] = t;
    }
}

// Recursive-halving sum of v[0..N) over the W lanes of this thread's segment
// (lanes differing in the bits below 2*OFF).  Afterwards the lane holds the
// totals of indices base .. base + N/W - 1 (at least one); `owner` is false on
// lanes that merely duplicate another lane's totals.
__device__ __forceinline__ REAL shfl_x(unsigned mask, REAL v, int off) {
    return __shfl_xor_sync(mask, v, off);
}
template <int OFF, int N>
__device__ __forceinline__ void seg_reduce(REAL* v, int lane, unsigned mask, int& base,
                                           bool& owner) {
    if constexpr (OFF >= 1) {
        const bool upper = (lane & OFF) != 0;
        if constexpr (N > 1) {
            constexpr int H = N / 2;
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const REAL send = upper ? v[i] : v[i + H];
                const REAL keep = upper ? v[i + H] : v[i];
                v[i] = keep + shfl_x(mask, send, OFF);
            }
            if (upper) base += H;
            seg_reduce<OFF / 2, H>(v, lane, mask, base, owner);
        } else {
            v[0] += shfl_x(mask, v[0], OFF);
            if (upper) owner = false;
            seg_reduce<OFF / 2, 1>(v, lane, mask, base, owner);
        }
    }
}

constexpr int WSEG = LANES < 32 ? LANES : 32;  // lanes of one slot inside one warp
constexpr int NRED = NYP / WSEG > 0 ? NYP / WSEG : 1;

// grad_w of one path: stored per edge, or (shared weights) added to the
// thread's running partial, which the kernel writes once per CTA / slot.
__device__ __forceinline__ void gw_store(REAL* gp, int ch, VR s, VR sc, int mgw) {
    s = vmul(s, sc);
    if (mgw == 2) s = vadd(s, ldv_plain(gp, ch));
    if (CH_ACTIVE(ch)) stv(gp, ch, s);
}
#if SHARED_W
#define GWOUT(q, s) (gwa[q] = vadd(gwa[q], (s)))
#define GWOUT_M(q, s, mode) (gwa[q] = vadd(gwa[q], (s)))
#else
#define GWOUT(q, s) gw_store(gwrow + (long long)(q) * MUL, ch, (s), sc, mgw)
#define GWOUT_M(q, s, mode) gw_store(gwrow + (long long)(q) * MUL, ch, (s), sc, (mode))
#endif
// Partial weight-gradient row of a CTA or slot (shared weights).
__device__ __forceinline__ void gw_partial(REAL* __restrict__ row, const VR (&gwa)[NP], int ch,
                                           VR sc) {
    if (!CH_ACTIVE(ch)) return;
#pragma unroll
    for (int q = 0; q < NP; ++q) stv(row + (long long)q * MUL, ch, vmul(gwa[q], sc));
}

// @@GENERATED@@ (per-plan contraction streams are inserted here)

// ------------------------------------------------------------------ forward

template <bool CONV>
__device__ __forceinline__ void fwd_body(long long n_items, const int* __restrict__ rowptr,
                                         const int* __restrict__ sender,
                                         const REAL* __restrict__ x, const REAL* __restrict__ y,
                                         const WT* __restrict__ w, long long w_stride,
                                         REAL* __restrict__ out, REAL scale, int accumulate) {
    __shared__ __align__(16) REAL Ts_all[SLOTS][NTP];
    __shared__ __align__(16) REAL Ys_all[SLOTS][NYP];
    const int slot = threadIdx.x / LANES, lane = threadIdx.x % LANES;
    REAL* Ts = Ts_all[slot];
    REAL* Ys = Ys_all[slot];
    const int ch = lane;
    for (long long item = (long long)blockIdx.x * SLOTS + slot; item < n_items;
         item += (long long)gridDim.x * SLOTS) {
        long long e0, e1;
        if (CONV) {
            e0 = rowptr[item];
            e1 = rowptr[item + 1];
        } else {
            e0 = item;
            e1 = item + 1;
        }
        VR acc[NO];
#pragma unroll
        for (int r = 0; r < NO; ++r) acc[r] = vzero();
        REAL ypf[YPF];
        int snext = 0;
        if (e0 < e1) {
#pragma unroll
            for (int j = 0; j < YPF; ++j) {
                const int k = lane + j * LANES;
                ypf[j] = k < NY ? __ldg(y + e0 * NY + k) : (REAL)0;
            }
            if (CONV) snext = __ldg(sender + e0);
        }
        for (long long e = e0; e < e1; ++e) {
#pragma unroll
            for (int j = 0; j < YPF; ++j) {
                const int k = lane + j * LANES;
                if (k < NY) Ys[k] = ypf[j];
            }
            const long long src = CONV ? (long long)snext : e;
            slot_sync(slot);
            if (e + 1 < e1) {
#pragma unroll
                for (int j = 0; j < YPF; ++j) {
                    const int k = lane + j * LANES;
                    ypf[j] = k < NY ? __ldg(y + (e + 1) * NY + k) : (REAL)0;
                }
                if (CONV) snext = __ldg(sender + e + 1);
            }
            build_T(Ts, Ys, lane);
            slot_sync(slot);
            VR xr[NX];
            const REAL* xrow = x + src * DIMX;
#pragma unroll
            for (int r = 0; r < NX; ++r) xr[r] = ldv_m(xrow + r * MUL, ch);
            const WT* wrow = w + e * w_stride;
            gen_fwd(acc, Ts, [&](int r) { return xr[r]; },
                    [&](int p) { return ldw_m(wrow + (long long)p * MUL, ch); });
            slot_sync(slot);
        }
        if (CH_ACTIVE(ch)) {
            REAL* orow = out + item * DIMO;
            const VR sc = vsplat(scale);
#pragma unroll
            for (int r = 0; r < NO; ++r) {
                VR v = vmul(acc[r], sc);
                if (accumulate) v = vadd(v, ldv_plain(orow + r * MUL, ch));
                stv(orow + r * MUL, ch, v);
            }
        }
    }
}

extern "C" __global__ void __launch_bounds__(BLOCK)
cgtp_fwd_conv(long long n_items, const int* __restrict__ rowptr, const int* __restrict__ sender,
              const REAL* __restrict__ x, const REAL* __restrict__ y, const WT* __restrict__ w,
              long long w_stride, REAL* __restrict__ out, REAL scale, int accumulate) {
    fwd_body<true>(n_items, rowptr, sender, x, y, w, w_stride, out, scale, accumulate);
}

extern "C" __global__ void __launch_bounds__(BLOCK)
cgtp_fwd_single(long long n_items, const REAL* __restrict__ x, const REAL* __restrict__ y,
                const WT* __restrict__ w, long long w_stride, REAL* __restrict__ out, REAL scale,
                int accumulate) {
    fwd_body<false>(n_items, nullptr, nullptr, x, y, w, w_stride, out, scale, accumulate);
}

// ----------------------------------------------------------------- backward
//
// Per item (sender s, or sample b) and each of its edges e with receiver n:
//   h_p[m1]   = sum_m3 T_p[m1, m3] g[n, r3 + m3]
//   gx[r1+m1] += w[e,p] * h_p[m1]                    (summed over the edges)
//   gw[e,p]    = sum_m1 x[r1+m1] * h_p[m1]
//   gy[e,o2+m2] = sum_{p,m1,m3,u} C_p[m1,m2,m3] w[e,p,u] x[r1+m1,u] g[n,r3+m3,u]
// gy is a sum over channels: per-lane partials, then a shuffle reduction.
// mode flags: 0 skip, 1 write, 2 add to the existing output.

template <bool CONV, bool GY>
__device__ __forceinline__ void bwd_body(long long n_items, const int* __restrict__ s_rowptr,
                                         const int* __restrict__ s_perm,
                                         const int* __restrict__ s_recv,
                                         const REAL* __restrict__ x, const REAL* __restrict__ y,
                                         const WT* __restrict__ w, long long w_stride,
                                         const REAL* __restrict__ g, REAL scale,
                                         REAL* __restrict__ gx, REAL* __restrict__ gy,
                                         REAL* __restrict__ gw, int mgx, int mgy, int mgw,
                                         REAL* __restrict__ wsp) {
    __shared__ __align__(16) REAL Ts_all[SLOTS][NTP];
    __shared__ __align__(16) REAL Ys_all[SLOTS][NYP];
#if LANES > 32
    __shared__ REAL Gy_all[SLOTS][LANES / 32][NYP];
#endif
    const int slot = threadIdx.x / LANES, lane = threadIdx.x % LANES;
    REAL* Ts = Ts_all[slot];
    REAL* Ys = Ys_all[slot];
    const int ch = lane;
    const VR sc = vsplat(scale);
    VR gwa[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) gwa[q] = vzero();
    for (long long item = (long long)blockIdx.x * SLOTS + slot; item < n_items;
         item += (long long)gridDim.x * SLOTS) {
        long long j0, j1;
        if (CONV) {
            j0 = s_rowptr[item];
            j1 = s_rowptr[item + 1];
        } else {
            j0 = item;
            j1 = item + 1;
        }
        VR xr[NX], gxa[NX];
        const REAL* xrow = x + item * DIMX;
#pragma unroll
        for (int r = 0; r < NX; ++r) {
            xr[r] = ldv_m(xrow + r * MUL, ch);
            gxa[r] = vzero();
        }
        REAL ypf[YPF];
        long long enext = j0, nnext = j0;
        if (j0 < j1) {
            if (CONV) {
                enext = __ldg(s_perm + j0);
                nnext = __ldg(s_recv + j0);
            }
#pragma unroll
            for (int j = 0; j < YPF; ++j) {
                const int k = lane + j * LANES;
                ypf[j] = k < NY ? __ldg(y + enext * NY + k) : (REAL)0;
            }
        }
        for (long long jj = j0; jj < j1; ++jj) {
            const long long e = enext, n = nnext;
#pragma unroll
            for (int j = 0; j < YPF; ++j) {
                const int k = lane + j * LANES;
                if (k < NY) Ys[k] = ypf[j];
            }
            slot_sync(slot);
            if (jj + 1 < j1) {
                if (CONV) {
                    enext = __ldg(s_perm + jj + 1);
                    nnext = __ldg(s_recv + jj + 1);
                } else {
                    enext = jj + 1;
                    nnext = jj + 1;
                }
#pragma unroll
                for (int j = 0; j < YPF; ++j) {
                    const int k = lane + j * LANES;
                    ypf[j] = k < NY ? __ldg(y + enext * NY + k) : (REAL)0;
                }
            }
            build_T(Ts, Ys, lane);
            slot_sync(slot);
            VR gr[NO];
            const REAL* grow = g + n * DIMO;
#pragma unroll
            for (int r = 0; r < NO; ++r) gr[r] = ldv_m(grow + r * MUL, ch);
            const WT* wrow = w + e * w_stride;
            REAL* gwrow = gw ? gw + e * WDIM : nullptr;
            REAL gyl[NYP];
#pragma unroll
            for (int i = 0; i < NYP; ++i) gyl[i] = (REAL)0;
            gen_bwd<GY>(gxa, gyl, Ts, [&](int r) { return xr[r]; }, [&](int r) { return gr[r]; },
                        [&](int p) { return ldw_m(wrow + (long long)p * MUL, ch); }, gwrow, gwa,
                        ch, sc, mgx != 0, mgw);
            if (GY && mgy) {
                int base = 0;
                bool owner = true;
                seg_reduce<WSEG / 2, NYP>(gyl, lane, slot_mask(), base, owner);
#if LANES > 32
                if (owner && (lane & 31) < WSEG)
                    for (int i = 0; i < NRED; ++i) Gy_all[slot][lane / 32][base + i] = gyl[i];
                slot_sync(slot);
                for (int k = lane; k < NY; k += LANES) {
                    REAL t = (REAL)0;
                    for (int q = 0; q < LANES / 32; ++q) t += Gy_all[slot][q][k];
                    t *= scale;
                    if (mgy == 2) t += gy[e * NY + k];
                    gy[e * NY + k] = t;
                }
#else
                if (owner) {
#pragma unroll
                    for (int i = 0; i < NRED; ++i) {
                        const int k = base + i;
                        if (k < NY) {
                            REAL t = gyl[i] * scale;
                            if (mgy == 2) t += gy[e * NY + k];
                            gy[e * NY + k] = t;
                        }
                    }
                }
#endif
            }
            slot_sync(slot);
        }
        if (mgx && CH_ACTIVE(ch)) {
            REAL* orow = gx + item * DIMX;
#pragma unroll
            for (int r = 0; r < NX; ++r) {
                VR v = vmul(gxa[r], sc);
                if (mgx == 2) v = vadd(v, ldv_plain(orow + r * MUL, ch));
                stv(orow + r * MUL, ch, v);
            }
        }
    }
    if (SHARED_W && mgw) gw_partial(wsp + ((long long)blockIdx.x * SLOTS + slot) * WDIM, gwa, ch, sc);
}

#define CGTP_BWD_ENTRY(NAME, CONV, GY)                                                          \
    extern "C" __global__ void __launch_bounds__(BLOCK) NAME(                                 \
        long long n_items, const int* __restrict__ s_rowptr, const int* __restrict__ s_perm,  \
        const int* __restrict__ s_recv, const REAL* __restrict__ x,                           \
        const REAL* __restrict__ y, const WT* __restrict__ w, long long w_stride,             \
        const REAL* __restrict__ g, REAL scale, REAL* __restrict__ gx, REAL* __restrict__ gy, \
        REAL* __restrict__ gw, int mgx, int mgy, int mgw, REAL* __restrict__ wsp) {           \
        bwd_body<CONV, GY>(n_items, s_rowptr, s_perm, s_recv, x, y, w, w_stride, g, scale,    \
                           gx, gy, gw, mgx, mgy, mgw, wsp);                                   \
    }

CGTP_BWD_ENTRY(cgtp_bwd_conv, true, true)
CGTP_BWD_ENTRY(cgtp_bwd_conv_nogy, true, false)
CGTP_BWD_ENTRY(cgtp_bwd_single, false, true)
CGTP_BWD_ENTRY(cgtp_bwd_single_nogy, false, false)

// ===================================================================== staged
//
// Staged kernels (generated when every lane has a full channel group, rows are
// 16-byte multiples and the plan fits): one slot per CTA, persistent grid, each
// CTA owns a contiguous item range balanced by edge count.  Thread 0 streams the
// per-edge rows (weights, the gathered x or g row, y) into an S-deep ring of
// shared-memory stages with cp.async.bulk (TMA, completion on an mbarrier),
// STAGES-1 edges ahead of the edge being computed, so HBM latency overlaps the
// FMA stream.  Every wait is bounded: on timeout the kernel records an error
// code in cgtp_device_error and stops.

#if STAGED

__device__ int cgtp_device_error;

__device__ __forceinline__ unsigned smem_u32(const void* p) {
    return (unsigned)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(unsigned long long* b, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* b, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)),
                 "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes,
                                         unsigned long long* b) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(b)) : "memory");
}
// Bounded wait for phase `parity` of barrier b: at most `polls` polls (the
// default, 2^24 polls sleeping 64 ns between late ones, is about a second).
// Returns false on timeout.
constexpr unsigned kWaitPolls = 1u << 24;
__device__ __forceinline__ bool mbar_wait(unsigned long long* b, unsigned parity,
                                          unsigned polls = kWaitPolls) {
    const unsigned a = smem_u32(b);
    for (unsigned it = 0; it < polls; ++it) {
        unsigned ok;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
            : "=r"(ok) : "r"(a), "r"(parity) : "memory");
        if (ok) return true;
        if (it > 1024) __nanosleep(64);
    }
    return false;
}

// TEST_WAIT0 (a test-only plan flag): the first wait of every CTA gives up at
// once, so the timeout path (error flag, drain of the copies in flight, early
// return) runs without any real stall.

// First index n in [0, N] with ptr[n] >= target (ptr non-decreasing), computed
// by one warp with 32-way probes.
__device__ __forceinline__ long long warp_lower_bound(const int* __restrict__ ptr, long long N,
                                                      long long target) {
    const int lane = threadIdx.x & 31;
    long long lo = 0, hi = N;  // answer in [lo, hi]
    while (hi - lo > 32) {
        const long long step = (hi - lo + 31) / 32;
        long long probe = lo + (long long)lane * step;
        if (probe > hi) probe = hi;
        const bool ge = __ldg(ptr + probe) >= target;
        const unsigned m = __ballot_sync(0xffffffffu, ge);
        const int f = m ? __ffs(m) - 1 : 32;  // first probe with ptr >= target
        const long long nhi = f < 32 ? lo + (long long)f * step : hi;
        const long long nlo = f > 0 ? lo + (long long)(f - 1) * step : lo;
        lo = nlo;
        hi = nhi < hi ? nhi : hi;
    }
    const long long probe = lo + lane;
    const bool ge = probe <= hi && __ldg(ptr + probe) >= target;
    const unsigned m = __ballot_sync(0xffffffffu, ge);
    return m ? lo + (__ffs(m) - 1) : hi;
}

// Item range of this CTA: items whose first edge lies in its share of edges.
__device__ __forceinline__ void cta_items(const int* __restrict__ ptr, long long n_items,
                                          long long& i0, long long& i1) {
    __shared__ long long sh_range[2];
    if (threadIdx.x < 32) {
        const long long total = ptr ? (long long)__ldg(ptr + n_items) : n_items;
        const long long c = blockIdx.x, nc = gridDim.x;
        const long long t0 = total * c / nc, t1 = total * (c + 1) / nc;
        long long a, b;
        if (ptr) {
            a = c == 0 ? 0 : warp_lower_bound(ptr, n_items, t0);
            b = c == nc - 1 ? n_items : warp_lower_bound(ptr, n_items, t1);
        } else {
            a = t0;
            b = t1;
        }
        if (threadIdx.x == 0) {
            sh_range[0] = a;
            sh_range[1] = b;
        }
    }
    __syncthreads();
    i0 = sh_range[0];
    i1 = sh_range[1];
}

__device__ __forceinline__ void cta_sync() { __syncthreads(); }
// Barrier that also agrees on a flag: true only if every thread's ok is true.
__device__ __forceinline__ bool cta_all(bool ok) { return __syncthreads_and(ok) != 0; }
// After a timed-out wait: record the error, give every barrier a short bounded
// wait so no copy is left writing into this CTA's shared memory, then return.
__device__ __noinline__ void fail_and_drain(int code, unsigned long long* bars, int n) {
    if (threadIdx.x == 0) atomicExch(&cgtp_device_error, code);
    for (int s = 0; s < n; ++s)
        for (unsigned ph = 0; ph < 2; ++ph) {
            const unsigned a = smem_u32(&bars[s]);
            for (int it = 0; it < 4096; ++it) {
                unsigned ok;
                asm volatile(
                    "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                    : "=r"(ok) : "r"(a), "r"(ph) : "memory");
                if (ok) break;
                __nanosleep(1000);
            }
        }
}

// The CG terms of the T entries a thread computes (entries tid, tid + NTHR,
// ...): coefficients and packed y indices, loaded once per CTA into registers
// so the per-edge T build reads only y from shared memory.
template <int NTHR>
struct TTerms {
    static constexpr int R = (NT + NTHR - 1) / NTHR;
    REAL c[R][MAXTERMS];
    unsigned idx[R];  // MAXTERMS indices of 8 bits each
    __device__ __forceinline__ void load() {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int k = threadIdx.x + r * NTHR;
            idx[r] = 0u;
#pragma unroll
            for (int q = 0; q < MAXTERMS; ++q) {
                c[r][q] = k < NT ? __ldg(&T_CO[k * MAXTERMS + q]) : (REAL)0;
                const unsigned i = k < NT ? (unsigned)__ldg(&T_IDX[k * MAXTERMS + q]) : 0u;
                idx[r] |= i << (8 * q);
            }
        }
    }
};

// T entries of one edge, computed by all NTHR threads of the CTA with the CG
// terms read from the (L1-resident) global tables.  With DUP the entries are
// stored as splatted register pairs (no unpacking in the stream).
template <int NTHR, bool DUP = false>
__device__ __forceinline__ void build_T_cta(REAL* __restrict__ Ts, const REAL* __restrict__ Ys) {
    constexpr int ROUNDS = (NT + NTHR - 1) / NTHR;
    REAL t[ROUNDS];
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        const int k = threadIdx.x + r * NTHR;
        t[r] = (REAL)0;
        if (k < NT) {
#pragma unroll
            for (int q = 0; q < MAXTERMS; ++q)
                t[r] = fma(__ldg(&T_CO[k * MAXTERMS + q]), Ys[__ldg(&T_IDX[k * MAXTERMS + q])], t[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        const int k = threadIdx.x + r * NTHR;
        if (k < NT) {
            if constexpr (DUP)
                reinterpret_cast<VR*>(Ts)[k] = vsplat(t[r]);
            else
                Ts[k] = t[r];
        }
    }
}

// The same with the CG terms held in registers (TTerms).
template <int NTHR, bool DUP = false>
__device__ __forceinline__ void build_T_cta(REAL* __restrict__ Ts, const REAL* __restrict__ Ys,
                                            const TTerms<NTHR>& tt) {
#pragma unroll
    for (int r = 0; r < TTerms<NTHR>::R; ++r) {
        const int k = threadIdx.x + r * NTHR;
        REAL t = (REAL)0;
#pragma unroll
        for (int q = 0; q < MAXTERMS; ++q) t = fma(tt.c[r][q], Ys[(tt.idx[r] >> (8 * q)) & 255u], t);
        if (k < NT) {
            if constexpr (DUP)
                reinterpret_cast<VR*>(Ts)[k] = vsplat(t);
            else
                Ts[k] = t;
        }
    }
}

// Stage layout: [W row][x or g row][y row][int header]; all offsets 16-aligned.
constexpr unsigned SZ = sizeof(REAL);
constexpr unsigned WB = (unsigned)(NP * MUL) * (unsigned)sizeof(WT);
constexpr unsigned XB = (unsigned)(NX * MUL) * SZ;
constexpr unsigned GB_ = (unsigned)(NO * MUL) * SZ;
constexpr unsigned YB = (unsigned)NY * SZ;
// With W_DIRECT_* the lanes load their weight pairs straight from global
// memory (prefetched one edge ahead in registers) and the ring carries only the
// gathered row and y.
constexpr unsigned WSF = W_DIRECT_F ? 0u : WB;  // weight bytes in a forward stage
constexpr unsigned WSB = W_DIRECT_B ? 0u : WB;  // weight bytes in a backward stage
constexpr unsigned FWD_STAGE = WSF + XB + YB;
constexpr unsigned BWD_STAGE = WSB + GB_ + YB + 16;
constexpr int NTF = GF * LANES;  // threads of a forward CTA
constexpr int NTB = (GB + GYW) * LANES;  // threads of a backward CTA (GYW: + a grad-y warp)

// A 32-entry window of an int array, held one entry per lane of warp 0, with
// the next window prefetched.  get(j) must be called by all lanes of warp 0
// with non-decreasing j.
struct IdxWindow {
    const int* __restrict__ a;
    long long end, base;
    int cur, nxt;
    __device__ __forceinline__ void init(const int* __restrict__ arr, long long b, long long e) {
        a = arr;
        end = e;
        base = b;
        const int lane = threadIdx.x & 31;
        cur = base + lane < end ? __ldg(a + base + lane) : 0;
        nxt = base + 32 + lane < end ? __ldg(a + base + 32 + lane) : 0;
    }
    __device__ __forceinline__ int get(long long j) {
        while (j >= base + 32) {
            base += 32;
            cur = nxt;
            const int lane = threadIdx.x & 31;
            nxt = base + 32 + lane < end ? __ldg(a + base + 32 + lane) : 0;
        }
        return __shfl_sync(0xffffffffu, cur, (int)(j - base));
    }
};

// ----------------------------------------------------------- staged forward

struct FwdArgs {
    long long n_items;
    const int* __restrict__ rowptr;
    const int* __restrict__ sender;
    const REAL* __restrict__ x;
    const REAL* __restrict__ y;
    const WT* __restrict__ w;
    long long w_stride;
    REAL* __restrict__ out;
    REAL scale;
    int accumulate;
};

struct FwdShared {
    unsigned char* stages;
    REAL* buf;
    unsigned long long* full;
    REAL* Ts;
    long long i0, i1, e_begin, e_end;
};

// Called by all of warp 0: stream edge j's rows into its stage.
template <bool CONV>
__device__ __forceinline__ void fwd_issue(const FwdArgs& A, const FwdShared& S, IdxWindow& win,
                                          long long j) {
    const long long src = CONV ? (long long)win.get(j) : j;
    if (threadIdx.x == 0) {
        unsigned char* st = S.stages + (size_t)((j - S.e_begin) % STAGES_F) * FWD_STAGE;
        unsigned long long* b = &S.full[(j - S.e_begin) % STAGES_F];
        mbar_expect_tx(b, FWD_STAGE);
        if (!W_DIRECT_F) bulk_g2s(st, A.w + j * A.w_stride, WB, b);
        bulk_g2s(st + WSF, A.x + src * DIMX, XB, b);
        bulk_g2s(st + WSF + XB, A.y + j * NY, YB, b);
    }
}

template <int GRP, bool CONV>
__device__ __forceinline__ void fwd_group(const FwdArgs& A, const FwdShared& S, IdxWindow& win) {
    using FG = FwdG<GRP>;
    const int tid = threadIdx.x, ch = tid % LANES;
    const VR sc = vsplat(A.scale);
    TTerms<NTF> tt;
    tt.load();
    VR acc[FG::NR];
#if W_DIRECT_F
    // wbuf[p] holds this edge's weight pair of path p; the stream reads it and
    // at once reloads the slot with the next edge's value (one edge of latency)
    VR wbuf[NP];
    if (S.e_begin < S.e_end)
#pragma unroll
        for (int p = 0; p < NP; ++p) wbuf[p] = ldw(A.w + S.e_begin * A.w_stride + p * MUL, ch);
#endif
    long long j = S.e_begin;
    long long nend = CONV ? (long long)__ldg(A.rowptr + S.i0 + 1) : S.i0 + 1;
    for (long long item = S.i0; item < S.i1; ++item) {
        const long long e1 = nend;
        if (item + 1 < S.i1) nend = CONV ? (long long)__ldg(A.rowptr + item + 2) : item + 2;
#pragma unroll
        for (int r = 0; r < FG::NR; ++r) acc[r] = vzero();
        for (; j < e1; ++j) {
            const long long k = j - S.e_begin;
            const unsigned char* st = S.stages + (size_t)(k % STAGES_F) * FWD_STAGE;
            const bool ok = mbar_wait(&S.full[k % STAGES_F], (unsigned)((k / STAGES_F) & 1),
                                      TEST_WAIT0 && k == 0 ? 0u : kWaitPolls);
            build_T_cta<NTF>(S.Ts, reinterpret_cast<const REAL*>(st + WSF + XB), tt);
            if (!cta_all(ok)) {
                fail_and_drain(1, S.full, STAGES_F);
                return;
            }
            VR xr[FG::NXR];
            FG::loadx(xr, reinterpret_cast<const REAL*>(st + WSF), ch);
#if W_DIRECT_F
            const WT* wnext = A.w + (j + 1 < S.e_end ? j + 1 : j) * A.w_stride;
            FG::edge(acc, S.Ts, xr, [&](int p) {
                const VR v = wbuf[p];
                wbuf[p] = ldw(wnext + p * MUL, ch);
                return v;
            });
#else
            const WT* ws = reinterpret_cast<const WT*>(st);
            FG::edge(acc, S.Ts, xr, [&](int p) { return lds_w(ws + p * MUL, ch); });
#endif
            cta_sync();
            if constexpr (GRP == 0)
                if (tid < 32 && j + STAGES_F < S.e_end) fwd_issue<CONV>(A, S, win, j + STAGES_F);
        }
        REAL* orow = A.out + item * DIMO;
        if constexpr (GF == 1) {
            FG::store(orow, acc, ch, sc, A.accumulate);
        } else {
            // partial sums of the groups, added in group order
            if constexpr (GRP == 0) FG::first(S.buf, acc, ch);
            cta_sync();
#pragma unroll
            for (int g = 1; g < GF; ++g) {
                if (g == GRP) FG::add(S.buf, acc, ch);
                cta_sync();
            }
            for (int i = tid; i < NO * NCH; i += NTF) {
                const int r = i / NCH, c = i % NCH;
                VR v = vmul(lds_v(S.buf + r * MUL, c), sc);
                if (A.accumulate) v = vadd(v, ldv_plain(orow + r * MUL, c));
                stv(orow + r * MUL, c, v);
            }
            cta_sync();
        }
    }
}

template <bool CONV>
__device__ __forceinline__ void fwd_staged(const FwdArgs& A) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) unsigned long long full[STAGES_F];
    __shared__ __align__(16) REAL Ts[NTP];
    FwdShared S;
    cta_items(CONV ? A.rowptr : nullptr, A.n_items, S.i0, S.i1);
    if (S.i0 >= S.i1) return;
    S.stages = smem;
    S.buf = reinterpret_cast<REAL*>(smem + (size_t)STAGES_F * FWD_STAGE);
    S.full = full;
    S.Ts = Ts;
    S.e_begin = CONV ? (long long)__ldg(A.rowptr + S.i0) : S.i0;
    S.e_end = CONV ? (long long)__ldg(A.rowptr + S.i1) : S.i1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES_F; ++s) mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    IdxWindow win;
    if (threadIdx.x < 32) {
        if (CONV) win.init(A.sender, S.e_begin, S.e_end);
        for (long long j = S.e_begin; j < S.e_begin + STAGES_F && j < S.e_end; ++j)
            fwd_issue<CONV>(A, S, win, j);
    }
    const int grp = threadIdx.x / LANES;
    if (grp == 0) fwd_group<0, CONV>(A, S, win);
#if GF > 1
    else if (grp == 1) fwd_group<1, CONV>(A, S, win);
#endif
#if GF > 2
    else if (grp == 2) fwd_group<2, CONV>(A, S, win);
#endif
#if GF > 3
    else if (grp == 3) fwd_group<3, CONV>(A, S, win);
#endif
}

extern "C" __global__ void __launch_bounds__(NTF)
cgtp_fwd_conv_tma(long long n_items, const int* __restrict__ rowptr,
                  const int* __restrict__ sender, const REAL* __restrict__ x,
                  const REAL* __restrict__ y, const WT* __restrict__ w, long long w_stride,
                  REAL* __restrict__ out, REAL scale, int accumulate) {
    fwd_staged<true>(FwdArgs{n_items, rowptr, sender, x, y, w, w_stride, out, scale, accumulate});
}

extern "C" __global__ void __launch_bounds__(NTF)
cgtp_fwd_single_tma(long long n_items, const REAL* __restrict__ x, const REAL* __restrict__ y,
                    const WT* __restrict__ w, long long w_stride, REAL* __restrict__ out,
                    REAL scale, int accumulate) {
    fwd_staged<false>(FwdArgs{n_items, nullptr, nullptr, x, y, w, w_stride, out, scale, accumulate});
}

// ---------------------------------------------------------- staged backward
//
// Items are senders (or samples).  Stages carry w[e], g[n] and y[e] of the
// item's edges (e = s_perm[j], n = s_recv[j]); the item's own x row comes
// through a second, double-buffered TMA slot.  grad_w is stored by the group
// owning the path; grad_y is reduced per warp, then across warps in warp order;
// grad_x partials are added in group order at the end of the item.

struct BwdArgs {
    long long n_items;
    const int* __restrict__ s_rowptr;
    const int* __restrict__ s_perm;
    const int* __restrict__ s_recv;
    const REAL* __restrict__ x;
    const REAL* __restrict__ y;
    const WT* __restrict__ w;
    long long w_stride;
    const REAL* __restrict__ g;
    REAL scale;
    REAL* __restrict__ gx;
    REAL* __restrict__ gy;
    REAL* __restrict__ gw;
    int mgx, mgy, mgw;
    REAL* __restrict__ wsp;  // partial weight-gradient rows (shared weights)
};

constexpr int NWB = NTB / 32;  // warps of a backward CTA

struct BwdShared {
    unsigned char* stages;
    unsigned char* xring;
    REAL* buf;
    unsigned long long* full;
    unsigned long long* xfull;
    REAL* Ts;
    REAL (*gyS)[NYP];
    long long i0, i1, j_begin, j_end;
};

template <bool CONV>
__device__ __forceinline__ void bwd_issue(const BwdArgs& A, const BwdShared& S, IdxWindow& we,
                                          IdxWindow& wn, long long j) {
    const long long e = CONV ? (long long)we.get(j) : j;
    const long long n = CONV ? (long long)wn.get(j) : j;
    if (threadIdx.x == 0) {
        unsigned char* st = S.stages + (size_t)((j - S.j_begin) % STAGES_B) * BWD_STAGE;
        unsigned long long* b = &S.full[(j - S.j_begin) % STAGES_B];
        *reinterpret_cast<int*>(st + WSB + GB_ + YB) = (int)e;
        mbar_expect_tx(b, WSB + GB_ + YB);
        if (!W_DIRECT_B) bulk_g2s(st, A.w + e * A.w_stride, WB, b);
        bulk_g2s(st + WSB, A.g + n * DIMO, GB_, b);
        bulk_g2s(st + WSB + GB_, A.y + e * NY, YB, b);
    }
}

__device__ __forceinline__ void bwd_issue_x(const BwdArgs& A, const BwdShared& S, long long item,
                                            int slot) {
    if (threadIdx.x == 0) {
        mbar_expect_tx(&S.xfull[slot], XB);
        bulk_g2s(S.xring + (size_t)slot * XB, A.x + item * DIMX, XB, &S.xfull[slot]);
    }
}

template <int GRP, bool CONV, bool GY, bool FIX>
__device__ __forceinline__ void bwd_group(const BwdArgs& A, const BwdShared& S, IdxWindow& we,
                                          IdxWindow& wn) {
    using BG = BwdG<GRP>;
    const int tid = threadIdx.x, ch = tid % LANES, lane = tid & 31;
    const VR sc = vsplat(A.scale);
    VR gwa[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) gwa[q] = vzero();
    long long j = S.j_begin;
    long long nend = CONV ? (long long)__ldg(A.s_rowptr + S.i0 + 1) : S.i0 + 1;
#if W_DIRECT_B
    // edge ids come from the stage headers (written before the barrier that
    // follows their issue); the first stage was issued before this loop
    // W_BUF2: the next edge's weights land in a second register array loaded
    // ahead of the stream (the arrays alternate from edge to edge); otherwise
    // the stream reads a path's weight and reloads that slot with the next
    // edge's value.
    // (slot i of a group's registers holds the weight pair of its path q)
    WRAW wbuf[BG::NPW];
#if W_BUF2
    WRAW wnext[BG::NPW];
#endif
    if (S.j_begin < S.j_end) {
        const long long e0 = *reinterpret_cast<const int*>(S.stages + WSB + GB_ + YB);
        BG::each_w([&](int i, int q) { wbuf[i] = ldw_raw(A.w + e0 * A.w_stride + q * MUL, ch); });
    }
#endif
    for (long long item = S.i0; item < S.i1; ++item) {
        const long long kk = item - S.i0;
        const long long e1 = nend;
        if (item + 1 < S.i1) nend = CONV ? (long long)__ldg(A.s_rowptr + item + 2) : item + 2;
        if (!cta_all(mbar_wait(&S.xfull[kk & 1], (unsigned)((kk >> 1) & 1),
                               TEST_WAIT0 && kk == 0 ? 0u : kWaitPolls))) {
            fail_and_drain(2, S.full, STAGES_B);
            fail_and_drain(2, S.xfull, 2);
            return;
        }
        VR xr[BG::NXR], gxa[BG::NXR];
        BG::loadx(xr, reinterpret_cast<const REAL*>(S.xring + (size_t)(kk & 1) * XB), ch);
#pragma unroll
        for (int r = 0; r < BG::NXR; ++r) gxa[r] = vzero();
        cta_sync();  // every thread holds its x before the slot is refilled
        if (item + 1 < S.i1) bwd_issue_x(A, S, item + 1, (int)((kk + 1) & 1));
        for (; j < e1; ++j) {
            const long long k = j - S.j_begin;
            const unsigned char* st = S.stages + (size_t)(k % STAGES_B) * BWD_STAGE;
            const bool ok = mbar_wait(&S.full[k % STAGES_B], (unsigned)((k / STAGES_B) & 1));
            const long long e = *reinterpret_cast<const int*>(st + WSB + GB_ + YB);
            build_T_cta<NTB, T_DUP_B && CPT == 2>(S.Ts, reinterpret_cast<const REAL*>(st + WSB + GB_));
            if (!cta_all(ok)) {
                fail_and_drain(3, S.full, STAGES_B);
                fail_and_drain(3, S.xfull, 2);
                return;
            }
            const REAL* gs = reinterpret_cast<const REAL*>(st + WSB);
            REAL gyl[NYP * GYS];  // GYS == 2: odd paths use the second half
#pragma unroll
            for (int i = 0; i < NYP * GYS; ++i) gyl[i] = (REAL)0;
            REAL* gwrow = A.gw ? A.gw + e * WDIM : nullptr;
#if W_DIRECT_B
            long long e1 = e;
            if (j + 1 < S.j_end) {
                const unsigned char* st1 = S.stages + (size_t)((k + 1) % STAGES_B) * BWD_STAGE;
                e1 = *reinterpret_cast<const int*>(st1 + WSB + GB_ + YB);
            }
            const WT* wrow1 = A.w + e1 * A.w_stride;
#if W_BUF2
            // W_ALT: the two register buffers take turns (this edge reads one
            // while the next edge's weights land in the other, no copy between
            // them); else the next edge's weights are copied over after use
            if (!W_ALT || (k & 1) == 0) {
                BG::each_w([&](int i, int q) { wnext[i] = ldw_raw(wrow1 + q * MUL, ch); });
                BG::template edge<GY, FIX>(gxa, gyl, S.Ts, xr,
                                           [&](int r) { return lds_v(gs + r * MUL, ch); },
                                           [&](int i, int) { return wcvt(wbuf[i]); }, gwrow, gwa,
                                           ch, sc, A.mgx != 0, A.mgw);
                if (!W_ALT) {
#pragma unroll
                    for (int i = 0; i < BG::NPW; ++i) wbuf[i] = wnext[i];
                }
            } else {
                BG::each_w([&](int i, int q) { wbuf[i] = ldw_raw(wrow1 + q * MUL, ch); });
                BG::template edge<GY, FIX>(gxa, gyl, S.Ts, xr,
                                           [&](int r) { return lds_v(gs + r * MUL, ch); },
                                           [&](int i, int) { return wcvt(wnext[i]); }, gwrow, gwa,
                                           ch, sc, A.mgx != 0, A.mgw);
            }
#else
            BG::template edge<GY, FIX>(gxa, gyl, S.Ts, xr,
                                  [&](int r) { return lds_v(gs + r * MUL, ch); },
                                  [&](int i, int q) {
                                      const VR v = wcvt(wbuf[i]);
                                      wbuf[i] = ldw_raw(wrow1 + q * MUL, ch);
                                      return v;
                                  },
                                  gwrow, gwa, ch, sc, A.mgx != 0, A.mgw);
#endif
#else
            const WT* ws = reinterpret_cast<const WT*>(st);
            BG::template edge<GY, FIX>(gxa, gyl, S.Ts, xr,
                                  [&](int r) { return lds_v(gs + r * MUL, ch); },
                                  [&](int, int q) { return lds_w(ws + q * MUL, ch); }, gwrow, gwa,
                                  ch, sc, A.mgx != 0, A.mgw);
#endif
            if (GY && A.mgy) {
                if (GYS == 2)
#pragma unroll
                    for (int i = 0; i < NYP; ++i) gyl[i] += gyl[NYP * (GYS - 1) + i];
                int base = 0;
                bool owner = true;
                seg_reduce<16, NYP>(gyl, lane, 0xffffffffu, base, owner);
                if (owner)
#pragma unroll
                    for (int i = 0; i < NRED; ++i) S.gyS[tid / 32][base + i] = gyl[i];
            }
            cta_sync();
            if (GY && A.mgy && tid < NY) {
                REAL t = (REAL)0;
#pragma unroll
                for (int q = 0; q < NWB; ++q) t += S.gyS[q][tid];
                t *= A.scale;
                if (A.mgy == 2) t += A.gy[e * NY + tid];
                A.gy[e * NY + tid] = t;
            }
            if constexpr (GRP == 0)
                if (tid < 32 && j + STAGES_B < S.j_end) bwd_issue<CONV>(A, S, we, wn, j + STAGES_B);
        }
        if (A.mgx) {
            REAL* orow = A.gx + item * DIMX;
            if constexpr (GB == 1) {
                BG::store(orow, gxa, ch, sc, A.mgx);
            } else {
                if constexpr (GRP == 0) BG::first(S.buf, gxa, ch);
                cta_sync();
#pragma unroll
                for (int g = 1; g < GB; ++g) {
                    if (g == GRP) BG::add(S.buf, gxa, ch);
                    cta_sync();
                }
                for (int i = tid; i < NX * NCH; i += NTB) {
                    const int r = i / NCH, c = i % NCH;
                    VR v = vmul(lds_v(S.buf + r * MUL, c), sc);
                    if (A.mgx == 2) v = vadd(v, ldv_plain(orow + r * MUL, c));
                    stv(orow + r * MUL, c, v);
                }
                cta_sync();
            }
        }
    }
    if (SHARED_W && A.mgw) gw_partial(A.wsp + (long long)blockIdx.x * WDIM, gwa, ch, sc);
}

#if GYW
// The grad-y warp: walks the same items and ring stages as group 0, passing
// the same CTA barriers in the same order, and computes only grad_y (the CG
// coefficients are immediates, so it reads x, the staged g row and the
// weights, not T).  Group 0 then runs without grad_y.
template <bool CONV, bool GY>
__device__ __forceinline__ void bwd_gy_role(const BwdArgs& A, const BwdShared& S) {
    using BG = BwdG<0>;
    const int tid = threadIdx.x, ch = tid % LANES, lane = tid & 31;
    const bool dogy = GY && A.mgy;
    long long j = S.j_begin;
    long long nend = CONV ? (long long)__ldg(A.s_rowptr + S.i0 + 1) : S.i0 + 1;
#if W_DIRECT_B
    WRAW wbuf[BG::NPW];
#if W_BUF2
    WRAW wnext[BG::NPW];
#endif
    if (dogy && S.j_begin < S.j_end) {
        const long long e0 = *reinterpret_cast<const int*>(S.stages + WSB + GB_ + YB);
        BG::each_w([&](int i, int q) { wbuf[i] = ldw_raw(A.w + e0 * A.w_stride + q * MUL, ch); });
    }
#endif
    for (long long item = S.i0; item < S.i1; ++item) {
        const long long kk = item - S.i0;
        const long long e1 = nend;
        if (item + 1 < S.i1) nend = CONV ? (long long)__ldg(A.s_rowptr + item + 2) : item + 2;
        if (!cta_all(mbar_wait(&S.xfull[kk & 1], (unsigned)((kk >> 1) & 1),
                               TEST_WAIT0 && kk == 0 ? 0u : kWaitPolls))) {
            fail_and_drain(2, S.full, STAGES_B);
            fail_and_drain(2, S.xfull, 2);
            return;
        }
        VR xr[BG::NXR];
        BG::loadx(xr, reinterpret_cast<const REAL*>(S.xring + (size_t)(kk & 1) * XB), ch);
        cta_sync();  // every thread holds its x before the slot is refilled
        for (; j < e1; ++j) {
            const long long k = j - S.j_begin;
            const unsigned char* st = S.stages + (size_t)(k % STAGES_B) * BWD_STAGE;
            const bool ok = mbar_wait(&S.full[k % STAGES_B], (unsigned)((k / STAGES_B) & 1));
            const long long e = *reinterpret_cast<const int*>(st + WSB + GB_ + YB);
            build_T_cta<NTB, T_DUP_B && CPT == 2>(S.Ts, reinterpret_cast<const REAL*>(st + WSB + GB_));
            if (!cta_all(ok)) {
                fail_and_drain(3, S.full, STAGES_B);
                fail_and_drain(3, S.xfull, 2);
                return;
            }
            if (dogy) {
                const REAL* gs = reinterpret_cast<const REAL*>(st + WSB);
                REAL gyl[NYP * GYS];
#pragma unroll
                for (int i = 0; i < NYP * GYS; ++i) gyl[i] = (REAL)0;
#if W_DIRECT_B
                long long en = e;
                if (j + 1 < S.j_end) {
                    const unsigned char* st1 = S.stages + (size_t)((k + 1) % STAGES_B) * BWD_STAGE;
                    en = *reinterpret_cast<const int*>(st1 + WSB + GB_ + YB);
                }
                const WT* wrow1 = A.w + en * A.w_stride;
#if W_BUF2
                if (!W_ALT || (k & 1) == 0) {
                    BG::each_w([&](int i, int q) { wnext[i] = ldw_raw(wrow1 + q * MUL, ch); });
                    BG::edge_gy(gyl, xr, [&](int r) { return lds_v(gs + r * MUL, ch); },
                                [&](int i, int) { return wcvt(wbuf[i]); });
                    if (!W_ALT) {
#pragma unroll
                        for (int i = 0; i < BG::NPW; ++i) wbuf[i] = wnext[i];
                    }
                } else {
                    BG::each_w([&](int i, int q) { wbuf[i] = ldw_raw(wrow1 + q * MUL, ch); });
                    BG::edge_gy(gyl, xr, [&](int r) { return lds_v(gs + r * MUL, ch); },
                                [&](int i, int) { return wcvt(wnext[i]); });
                }
#else
                BG::edge_gy(gyl, xr, [&](int r) { return lds_v(gs + r * MUL, ch); },
                            [&](int i, int q) {
                                const VR v = wcvt(wbuf[i]);
                                wbuf[i] = ldw_raw(wrow1 + q * MUL, ch);
                                return v;
                            });
#endif
#else
                const WT* ws = reinterpret_cast<const WT*>(st);
                BG::edge_gy(gyl, xr, [&](int r) { return lds_v(gs + r * MUL, ch); },
                            [&](int, int q) { return lds_w(ws + q * MUL, ch); });
#endif
                if (GYS == 2)
#pragma unroll
                    for (int i = 0; i < NYP; ++i) gyl[i] += gyl[NYP * (GYS - 1) + i];
                int base = 0;
                bool owner = true;
                seg_reduce<16, NYP>(gyl, lane, 0xffffffffu, base, owner);
                if (owner) {
#pragma unroll
                    for (int i = 0; i < NRED; ++i) {
                        const int c = base + i;
                        if (c < NY) {
                            REAL t = gyl[i] * A.scale;
                            if (A.mgy == 2) t += A.gy[e * NY + c];
                            A.gy[e * NY + c] = t;
                        }
                    }
                }
            }
            cta_sync();
        }
    }
}
#endif

template <bool CONV, bool GY>
__device__ __forceinline__ void bwd_staged(const BwdArgs& A) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) unsigned long long full[STAGES_B];
    __shared__ __align__(8) unsigned long long xfull[2];
    __shared__ __align__(16) REAL Ts[NTP * (T_DUP_B ? CPT : 1)];
    __shared__ REAL gyS[NWB][NYP];
    BwdShared S;
    cta_items(CONV ? A.s_rowptr : nullptr, A.n_items, S.i0, S.i1);
    if (S.i0 >= S.i1) {
        if (SHARED_W && A.mgw) {  // every CTA owns one partial row, even an empty one
            VR z[NP];
#pragma unroll
            for (int q = 0; q < NP; ++q) z[q] = vzero();
            if (threadIdx.x < LANES) gw_partial(A.wsp + (long long)blockIdx.x * WDIM, z, threadIdx.x, z[0]);
        }
        return;
    }
    S.stages = smem;
    S.xring = smem + (size_t)STAGES_B * BWD_STAGE;
    S.buf = reinterpret_cast<REAL*>(S.xring + 2 * (size_t)XB);
    S.full = full;
    S.xfull = xfull;
    S.Ts = Ts;
    S.gyS = gyS;
    S.j_begin = CONV ? (long long)__ldg(A.s_rowptr + S.i0) : S.i0;
    S.j_end = CONV ? (long long)__ldg(A.s_rowptr + S.i1) : S.i1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES_B; ++s) mbar_init(&full[s], 1);
        mbar_init(&xfull[0], 1);
        mbar_init(&xfull[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    IdxWindow we, wn;
    if (threadIdx.x < 32) {
        if (CONV) {
            we.init(A.s_perm, S.j_begin, S.j_end);
            wn.init(A.s_recv, S.j_begin, S.j_end);
        }
        for (long long j = S.j_begin; j < S.j_begin + STAGES_B && j < S.j_end; ++j)
            bwd_issue<CONV>(A, S, we, wn, j);
    }
    bwd_issue_x(A, S, S.i0, 0);
    __syncthreads();  // stage headers of the first edges are visible to all threads
    const int grp = threadIdx.x / LANES;
    // grad_x and grad_w both written: the branch-free stream
    const bool fix = A.mgx == 1 && A.mgw == 1;
#define CGTP_BWD_GROUP(G_, GY_)                                  \
    (fix ? bwd_group<G_, CONV, GY_, true>(A, S, we, wn)          \
         : bwd_group<G_, CONV, GY_, false>(A, S, we, wn))
#if GYW
    if (grp == 0)
        CGTP_BWD_GROUP(0, false);
    else
        bwd_gy_role<CONV, GY>(A, S);
#else
    if (grp == 0) CGTP_BWD_GROUP(0, GY);
#endif
#if GB > 1
    else if (grp == 1) CGTP_BWD_GROUP(1, GY);
#endif
#if GB > 2
    else if (grp == 2) CGTP_BWD_GROUP(2, GY);
#endif
#if GB > 3
    else if (grp == 3) CGTP_BWD_GROUP(3, GY);
#endif
#undef CGTP_BWD_GROUP
}

#define CGTP_BWD_TMA_ENTRY(NAME, CONV, GY)                                                      \
    extern "C" __global__ void __launch_bounds__(NTB, MINB_B) NAME(                           \
        long long n_items, const int* __restrict__ s_rowptr, const int* __restrict__ s_perm,  \
        const int* __restrict__ s_recv, const REAL* __restrict__ x,                           \
        const REAL* __restrict__ y, const WT* __restrict__ w, long long w_stride,             \
        const REAL* __restrict__ g, REAL scale, REAL* __restrict__ gx, REAL* __restrict__ gy, \
        REAL* __restrict__ gw, int mgx, int mgy, int mgw, REAL* __restrict__ wsp) {           \
        bwd_staged<CONV, GY>(BwdArgs{n_items, s_rowptr, s_perm, s_recv, x, y, w, w_stride, g, \
                                     scale, gx, gy, gw, mgx, mgy, mgw, wsp});                 \
    }

CGTP_BWD_TMA_ENTRY(cgtp_bwd_conv_tma, true, true)
CGTP_BWD_TMA_ENTRY(cgtp_bwd_conv_nogy_tma, true, false)
CGTP_BWD_TMA_ENTRY(cgtp_bwd_single_tma, false, true)
CGTP_BWD_TMA_ENTRY(cgtp_bwd_single_nogy_tma, false, false)

#endif  // STAGED
