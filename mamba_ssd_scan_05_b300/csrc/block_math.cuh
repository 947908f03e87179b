// block_math.cuh -- float arithmetic shared by the conv1d and RMSNorm kernels (block.cu,
// block_staged.cu): SiLU from the hardware 2^x and reciprocal approximations, and Blackwell's
// packed two-lane fp32 instructions (fma / mul / add .rn.f32x2, one instruction for two
// independent IEEE round-to-nearest operations).  Every kernel that computes a SiLU uses silu1
// or silu2, which give the same bits for the same input, so the kernels agree bit for bit.
// Internal to libssd_scan.
#pragma once

#include <cuda_runtime.h>

namespace ssd {
namespace bm {

constexpr float kNegLog2e = -1.4426950408889634f;

__device__ __forceinline__ float ex2a(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcpa(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// d = a * b + c, lane-wise, each lane rounded once (fma.rn)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// silu(x) = x * sigmoid(x) = x / (1 + e^-x), as x * rcp(1 + 2^(-x log2 e)) with the hardware
// approximations (relative error a few 2^-23).  x < -88: 2^(...) = inf, rcp = 0, result -0;
// large x: the exponential is 0 and the result x.
__device__ __forceinline__ float silu1(float x) {
    const float t = x * kNegLog2e;
    const float d = 1.f + ex2a(t);
    return x * rcpa(d);
}
// silu1 of both lanes (the same bits as two silu1 calls)
__device__ __forceinline__ float2 silu2(float2 x) {
    const float2 t = fmul2(x, make_float2(kNegLog2e, kNegLog2e));
    const float2 d = fadd2(make_float2(ex2a(t.x), ex2a(t.y)), make_float2(1.f, 1.f));
    return fmul2(x, make_float2(rcpa(d.x), rcpa(d.y)));
}

}  // namespace bm
}  // namespace ssd
