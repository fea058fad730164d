// Packed fp32x2 arithmetic (sm_100-class mul/add.rn.f32x2: two independent
// round-to-nearest fp32 operations per instruction, so results are
// bit-identical to the scalar operations) and mixed-precision bf16 x bf16 +
// fp32 FMAs.
#pragma once

#include <cstdint>

namespace ccv {

using f32x2 = unsigned long long;  // (lo, hi) fp32 pair in one 64-bit register pair

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(f32x2 v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// acc + lo(x) * lo(w) and acc + hi(x) * hi(w) with bf16 sources and fp32
// accumulators (one rounding each; the bf16 product is exact in fp32, so this
// equals the fp32 fma of the widened values).
__device__ __forceinline__ void fma_bf16x2(float &acc_lo, float &acc_hi, uint32_t x, uint32_t w) {
    asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
        "mov.b32 {xl, xh}, %2;\n\t"
        "mov.b32 {wl, wh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, xl, wl, %0;\n\t"
        "fma.rn.f32.bf16 %1, xh, wh, %1;\n\t}"
        : "+f"(acc_lo), "+f"(acc_hi)
        : "r"(x), "r"(w));
}

// First tap: d = x * w + b per half (separate output, so b is not copied).
__device__ __forceinline__ void fma_bf16x2_init(float &d_lo, float &d_hi, uint32_t x, uint32_t w,
                                                float b_lo, float b_hi) {
    asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
        "mov.b32 {xl, xh}, %2;\n\t"
        "mov.b32 {wl, wh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, xl, wl, %4;\n\t"
        "fma.rn.f32.bf16 %1, xh, wh, %5;\n\t}"
        : "=f"(d_lo), "=f"(d_hi)
        : "r"(x), "r"(w), "f"(b_lo), "f"(b_hi));
}

// fp32 pair -> bf16x2 word, round-to-nearest-even.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(f32x2 v) {
    float lo, hi;
    unpack2(v, lo, hi);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float rcp_approx2(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// SiLU of a pair: v / (1 + 2^(-v log2 e)).  exp overflow for v < -88 gives
// 1/inf = 0 and a result of -0; NaN propagates.
__device__ __forceinline__ f32x2 silu2(f32x2 v) {
    const f32x2 kNegLog2e = pack2(-1.4426950408889634f, -1.4426950408889634f);
    const f32x2 kOne = pack2(1.0f, 1.0f);
    float t0, t1;
    unpack2(mul2(v, kNegLog2e), t0, t1);
    float d0, d1;
    unpack2(add2(pack2(ex2_approx(t0), ex2_approx(t1)), kOne), d0, d1);
    return mul2(v, pack2(rcp_approx2(d0), rcp_approx2(d1)));
}

}  // namespace ccv
