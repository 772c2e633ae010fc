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

// Weight of path p for this lane's channels.
#define LDW(p) ldv_m(wrow + (long long)(p) * MUL, ch)

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
__device__ __forceinline__ void build_T(VR* __restrict__ Ts, const REAL* __restrict__ Ys, int lane) {
    for (int k = lane; k < NT; k += LANES) {
        REAL t = (REAL)0;
#pragma unroll
        for (int q = 0; q < MAXTERMS; ++q)
            t = fma(T_CO[k * MAXTERMS + q], Ys[T_IDX[k * MAXTERMS + q]], t);
        Ts[k] = vsplat(t);
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

// @@GENERATED@@ (per-plan contraction streams are inserted here)

// ------------------------------------------------------------------ forward

template <bool CONV>
__device__ __forceinline__ void fwd_body(long long n_items, const int* __restrict__ rowptr,
                                         const int* __restrict__ sender,
                                         const REAL* __restrict__ x, const REAL* __restrict__ y,
                                         const REAL* __restrict__ w, long long w_stride,
                                         REAL* __restrict__ out, REAL scale, int accumulate) {
    __shared__ __align__(16) VR Ts_all[SLOTS][NTP];
    __shared__ __align__(16) REAL Ys_all[SLOTS][NYP];
    const int slot = threadIdx.x / LANES, lane = threadIdx.x % LANES;
    VR* Ts = Ts_all[slot];
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
            const REAL* wrow = w + e * w_stride;
            gen_fwd(acc, Ts, xr, wrow, ch);
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
              const REAL* __restrict__ x, const REAL* __restrict__ y, const REAL* __restrict__ w,
              long long w_stride, REAL* __restrict__ out, REAL scale, int accumulate) {
    fwd_body<true>(n_items, rowptr, sender, x, y, w, w_stride, out, scale, accumulate);
}

extern "C" __global__ void __launch_bounds__(BLOCK)
cgtp_fwd_single(long long n_items, const REAL* __restrict__ x, const REAL* __restrict__ y,
                const REAL* __restrict__ w, long long w_stride, REAL* __restrict__ out, REAL scale,
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
                                         const REAL* __restrict__ w, long long w_stride,
                                         const REAL* __restrict__ g, REAL scale,
                                         REAL* __restrict__ gx, REAL* __restrict__ gy,
                                         REAL* __restrict__ gw, int mgx, int mgy, int mgw) {
    __shared__ __align__(16) VR Ts_all[SLOTS][NTP];
    __shared__ __align__(16) REAL Ys_all[SLOTS][NYP];
#if LANES > 32
    __shared__ REAL Gy_all[SLOTS][LANES / 32][NYP];
#endif
    const int slot = threadIdx.x / LANES, lane = threadIdx.x % LANES;
    VR* Ts = Ts_all[slot];
    REAL* Ys = Ys_all[slot];
    const int ch = lane;
    const VR sc = vsplat(scale);
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
            const REAL* wrow = w + e * w_stride;
            REAL* gwrow = gw ? gw + e * WDIM : nullptr;
            REAL gyl[NYP];
#pragma unroll
            for (int i = 0; i < NYP; ++i) gyl[i] = (REAL)0;
            gen_bwd<GY>(gxa, gyl, Ts, xr, gr, wrow, gwrow, ch, sc, mgx != 0, mgw);
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
}

#define CGTP_BWD_ENTRY(NAME, CONV, GY)                                                          \
    extern "C" __global__ void __launch_bounds__(BLOCK) NAME(                                 \
        long long n_items, const int* __restrict__ s_rowptr, const int* __restrict__ s_perm,  \
        const int* __restrict__ s_recv, const REAL* __restrict__ x,                           \
        const REAL* __restrict__ y, const REAL* __restrict__ w, long long w_stride,           \
        const REAL* __restrict__ g, REAL scale, REAL* __restrict__ gx, REAL* __restrict__ gy, \
        REAL* __restrict__ gw, int mgx, int mgy, int mgw) {                                   \
        bwd_body<CONV, GY>(n_items, s_rowptr, s_perm, s_recv, x, y, w, w_stride, g, scale,    \
                           gx, gy, gw, mgx, mgy, mgw);                                        \
    }

CGTP_BWD_ENTRY(cgtp_bwd_conv, true, true)
CGTP_BWD_ENTRY(cgtp_bwd_conv_nogy, true, false)
CGTP_BWD_ENTRY(cgtp_bwd_single, false, true)
CGTP_BWD_ENTRY(cgtp_bwd_single_nogy, false, false)
