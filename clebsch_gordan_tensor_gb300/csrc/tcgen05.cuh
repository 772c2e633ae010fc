// tcgen05 / bulk-copy / mbarrier helpers shared by the tensor-core kernels
// (sm_103a, inline PTX).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace cgtp {

__device__ __forceinline__ unsigned smem_addr(const void* p) {
    return (unsigned)__cvta_generic_to_shared(p);
}

// Canonical K-major layout without swizzle: 8-row x 16-byte core matrices;
// the 8-row groups of one 4-wide K slice are contiguous (128 B apart) and the
// K slices follow each other (rows / 8 * 128 B apart).
__device__ __forceinline__ unsigned kmajor_offset(int row, int k, int rows) {
    return (unsigned)((k >> 2) * (rows / 8) * 128 + (row >> 3) * 128 + (row & 7) * 16 + (k & 3) * 4);
}

// Shared-memory matrix descriptor (tcgen05): start >> 4 in bits 0-13, leading
// byte offset (between K-adjacent core matrices) >> 4 in 16-29, stride byte
// offset (between 8-row groups) >> 4 in 32-45, the fixed version value 1 in
// bits 46-47, no swizzle (bits 61-63 = 0).
__device__ __forceinline__ uint64_t smem_desc(unsigned addr, unsigned lbo, unsigned sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// The same for the K-major layout with 128-byte swizzle, as a 2D tile copy
// with CU_TENSOR_MAP_SWIZZLE_128B writes it: row r's 128 bytes at r * 128, its
// 16-byte piece j at (j ^ (r % 8)) * 16; the pattern repeats every 8 rows
// (1024 bytes, the stride byte offset); the leading byte offset is unused
// while an MMA's K extent stays inside one 128-byte row.  Layout type 2 in
// bits 61-63.  Advancing K inside the row adds its byte offset to `addr`;
// the tile itself must start on a 1024-byte boundary.
__device__ __forceinline__ uint64_t smem_desc_sw128(unsigned addr) {
    return smem_desc(addr, 16, 1024) | (2ull << 61);
}

// Byte offset of element (row, k) of a 32-bit K-major tile with 128-byte rows
// in the swizzled layout above (k < 32).
__device__ __forceinline__ unsigned sw128_offset(int row, int k) {
    return (unsigned)(row * 128 + ((((k >> 2) ^ row) & 7) << 4) + (k & 3) * 4);
}

// 2D tile copy through a tensor map into shared memory, completion on an
// mbarrier; coordinates: column c (innermost), row r.
__device__ __forceinline__ void tma_tile_g2s(void* dst, const CUtensorMap* map, int c, int r,
                                             unsigned long long* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c), "r"(r), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_commit(unsigned long long* b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(b))
                 : "memory");
}

__device__ __forceinline__ void tc_mbar_init(unsigned long long* b, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void tc_mbar_arrive(unsigned long long* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}

__device__ __forceinline__ void tc_expect_tx(unsigned long long* b, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tc_bulk_g2s(void* dst, const void* src, unsigned bytes,
                                            unsigned long long* b) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(b))
        : "memory");
}

// Bounded wait for phase `parity`: at most `polls` polls (the default is about a
// second; tests pass 0 to exercise the timeout path).
__device__ __forceinline__ bool tc_mbar_wait(unsigned long long* b, unsigned parity,
                                             unsigned polls = 1u << 24) {
    const unsigned a = smem_addr(b);
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

__device__ __forceinline__ void tmem_ld8(unsigned taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Instruction descriptor, kind::tf32: D fp32 (bits 4-5 = 1), A and B TF32
// (bits 7-9 and 10-12 = 2), both K-major, N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
__host__ __device__ constexpr uint32_t tf32_idesc(int m, int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32_n(unsigned tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                           unsigned acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// tcgen05.mma with the A operand in tensor memory (kind::tf32).
__device__ __forceinline__ void mma_tf32_tmem_a(unsigned d, unsigned a, uint64_t b, uint32_t idesc,
                                                unsigned acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// 16 consecutive 32-bit columns of this warp's 32 lanes (one row per lane).
__device__ __forceinline__ void tmem_st16(unsigned taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

}  // namespace cgtp
