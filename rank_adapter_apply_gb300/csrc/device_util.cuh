// Small device helpers shared by the decode kernels.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace lora {

// D += A(16x16, row) * B(16x8, col), bf16 operands, fp32 accumulation.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16 pair in a 32-bit word: element 0 in the low half.
__device__ __forceinline__ float bf_lo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf_hi(uint32_t p) { return __uint_as_float(p & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float round_bf16(float f) {
    return __bfloat162float(__float2bfloat16_rn(f));
}

// Eight consecutive bf16 of a row starting at column c (zero past d or when !ok).
__device__ __forceinline__ uint4 load8_bf16(const uint16_t *row, int c, int d, bool ok, int vec) {
    uint4 r = make_uint4(0, 0, 0, 0);
    if (!ok) return r;
    if (vec && c + 8 <= d) return __ldg(reinterpret_cast<const uint4 *>(row + c));
    uint16_t e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] = (c + i < d) ? row[c + i] : (uint16_t)0;
    r.x = e[0] | ((uint32_t)e[1] << 16);
    r.y = e[2] | ((uint32_t)e[3] << 16);
    r.z = e[4] | ((uint32_t)e[5] << 16);
    r.w = e[6] | ((uint32_t)e[7] << 16);
    return r;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

}  // namespace lora
