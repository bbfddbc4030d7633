// Device helpers shared by the expert FFN kernels (number decoding, loads, reductions).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace ftmoe {
namespace ffn {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_stream32(const void *p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Four bytes of packed e2m1 codes -> eight floats (low nibble of each byte first).
__device__ __forceinline__ void e2m1x8(uint32_t w, float (&f)[8]) {
    uint32_t h0, h1, h2, h3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
    float2 a = __half22float2(*reinterpret_cast<__half2 *>(&h0));
    float2 b = __half22float2(*reinterpret_cast<__half2 *>(&h1));
    float2 c = __half22float2(*reinterpret_cast<__half2 *>(&h2));
    float2 d = __half22float2(*reinterpret_cast<__half2 *>(&h3));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

// One byte of packed e2m1 codes -> two floats (low nibble first).
__device__ __forceinline__ float2 e2m1x2(uint32_t byte) {
    uint32_t h;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
        : "=r"(h)
        : "r"(byte));
    return __half22float2(*reinterpret_cast<__half2 *>(&h));
}

// OCP e4m3fn byte -> float (bias 7, 3 mantissa bits, subnormals, S.1111.111 = NaN).
// The 7 magnitude bits placed at bit 20 of a binary32 give 2^(e-127)(1+m/8) for e > 0
// and the subnormal m * 2^-129 for e = 0; scaling by 2^120 (exact) rebiases both.
__device__ __forceinline__ float e4m3_to_f(uint32_t b) {
    const uint32_t mag = b & 0x7fu;
    float v = __uint_as_float(mag << 20) * 0x1p120f;
    if (mag == 0x7fu) v = __uint_as_float(0x7fc00000u);
    return __uint_as_float(__float_as_uint(v) | ((b & 0x80u) << 24));
}

// e8m0 byte -> 2^(b - 127); 0xFF is NaN.
__device__ __forceinline__ float e8m0_to_f(uint32_t b) {
    b &= 0xffu;
    if (b == 0xffu) return __uint_as_float(0x7fc00000u);
    return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ void unpack_bf16x8(uint4 v, float (&f)[8]) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

}  // namespace ffn
}  // namespace ftmoe
