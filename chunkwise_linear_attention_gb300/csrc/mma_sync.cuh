// mma_sync.cuh -- device helpers shared by the mma.sync kernels (chunk_la.cu,
// gla.cu): cp.async copies, ldmatrix, bf16 m16n8k16 products, exp2, bf16
// packing and the hi/lo split, and the XOR-swizzled row layout of tiles in
// shared memory.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace cla {
namespace {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(v);
}
// x = hi + lo + e as two bf16x2 words, by truncation: hi holds the upper 16 bits of each
// float (a bf16 rounded toward zero), the remainder x - hi is exact in fp32, and lo holds
// its upper 16 bits; |e| < 2^-16 |x|.  Integer and paired-float operations only (no
// conversion instructions); element .x goes to the low half of each word.
__device__ __forceinline__ void split_bf16x2(float2 x, uint32_t &hi, uint32_t &lo) {
    const uint32_t ux = __float_as_uint(x.x), uy = __float_as_uint(x.y);
    hi = __byte_perm(ux, uy, 0x7632);
    const float2 r = __ffma2_rn(make_float2(__uint_as_float(ux & 0xffff0000u), __uint_as_float(uy & 0xffff0000u)),
                                make_float2(-1.f, -1.f), x);  // x - hi, exact
    lo = __byte_perm(__float_as_uint(r.x), __float_as_uint(r.y), 0x7632);
}

// Byte offset of 16-byte chunk c16 of row `row` in a row-major tile with RB
// bytes per row; chunks are XOR-swizzled by the row's low 3 bits so that the
// 8 rows an ldmatrix reads fall in distinct banks.
template <int RB>
__device__ __forceinline__ uint32_t swz(int row, int c16) {
    return static_cast<uint32_t>(row * RB + ((c16 ^ (row & 7)) << 4));
}

}  // namespace
}  // namespace cla
