// Warp-level tensor-core and conversion helpers shared by the attention
// kernels (bf16 tiles and INT2 windows).
#pragma once

#include <stdint.h>

namespace kvev {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// D = A B + C for one m16n8k16 block (bf16 in, fp32 accumulate); A rows
// 8..15 are zero (a1 = a3 = 0), so only d0, d1 (rows 0..7) are used.
__device__ __forceinline__ void mma_rows8(float& c0, float& c1, uint32_t a0, uint32_t a2,
                                          uint32_t b0, uint32_t b1) {
    float d2, d3;   // rows 8..15: discarded
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3},"
        " {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
        : "=f"(c0), "=f"(c1), "=f"(d2), "=f"(d3)
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(0.f),
          "f"(0.f));
    (void)d2;
    (void)d3;
}
// The same with fp16 operands (A and B both fp16).
__device__ __forceinline__ void mma_rows8_f16(float& c0, float& c1, uint32_t a0, uint32_t a2,
                                              uint32_t b0, uint32_t b1) {
    float d2, d3;   // rows 8..15: discarded
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3},"
        " {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
        : "=f"(c0), "=f"(c1), "=f"(d2), "=f"(d3)
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(0.f),
          "f"(0.f));
    (void)d2;
    (void)d3;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t w) {
    float2 r;
    asm("{\n .reg .f16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.f32.f16 %0, lo;\n"
        " cvt.f32.f16 %1, hi;\n}" : "=f"(r.x), "=f"(r.y) : "r"(w));
    return r;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace kvev
