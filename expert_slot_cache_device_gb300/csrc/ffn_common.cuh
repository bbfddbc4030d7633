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

// Eight packed e2m1 codes (one 32-bit word) -> four f16x2 registers, low nibble first.
// e2m1 values are exact in f16.
__device__ __forceinline__ void e2m1x8_h2(uint32_t w, uint32_t (&h)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// acc + w.lo * x.lo + w.hi * x.hi: f16 multiplicands, exact products, fp32 accumulation.
__device__ __forceinline__ float fma2_f16(uint32_t w2, uint32_t x2, float acc) {
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t"
        "mov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
        "fma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
        : "+f"(acc)
        : "r"(w2), "r"(x2));
    return acc;
}

// Packed fp32 fused multiply-add: (a.x * b.x + c.x, a.y * b.y + c.y).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%1, %2};\n\t"
        "mov.b64 rb, {%3, %4};\n\t"
        "mov.b64 rc, {%5, %6};\n\t"
        "fma.rn.f32x2 %0, ra, rb, rc;\n\t}"
        : "=l"(d)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
    return r;
}

__device__ __forceinline__ float2 h2_to_f2(uint32_t h) { return __half22float2(*reinterpret_cast<__half2 *>(&h)); }

// Two e4m3 bytes (low byte first) -> float2 via the f16x2 conversion (exact).
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t two_bytes) {
    uint32_t h;
    asm("{\n\t.reg .b16 s;\n\t"
        "cvt.u16.u32 s, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, s;\n\t}"
        : "=r"(h)
        : "r"(two_bytes & 0xffffu));
    return h2_to_f2(h);
}

// Dot product of one packed word of eight e2m1 codes with eight f16 activations
// (four f16x2 registers): products are exact in f16 (2 x 8 significant bits at most);
// each half accumulates four of them with f16 additions, then the two halves are
// summed in fp32. Callers keep |x| < 2^10 so no partial can overflow.
__device__ __forceinline__ float dot8_e2m1_f16(const uint32_t (&w)[4], const uint32_t (&x)[4]) {
    __half2 acc = __hmul2(*reinterpret_cast<const __half2 *>(&w[0]), *reinterpret_cast<const __half2 *>(&x[0]));
    acc = __hfma2(*reinterpret_cast<const __half2 *>(&w[1]), *reinterpret_cast<const __half2 *>(&x[1]), acc);
    acc = __hfma2(*reinterpret_cast<const __half2 *>(&w[2]), *reinterpret_cast<const __half2 *>(&x[2]), acc);
    acc = __hfma2(*reinterpret_cast<const __half2 *>(&w[3]), *reinterpret_cast<const __half2 *>(&x[3]), acc);
    const float2 f = __half22float2(acc);
    return f.x + f.y;
}

// Dot product of one 16-element block: sixteen e2m1 codes (eight f16x2 registers) with
// sixteen f16 activations. Each f16 half sums eight exact products (|x| < 2^10 keeps
// every partial below 8 * 6 * 2^10 = 49152 < 65504); the halves are added in fp32.
__device__ __forceinline__ float dot16_e2m1_f16(const uint32_t (&w)[8], const uint32_t (&x)[8]) {
    __half2 acc = __hmul2(*reinterpret_cast<const __half2 *>(&w[0]), *reinterpret_cast<const __half2 *>(&x[0]));
#pragma unroll
    for (int i = 1; i < 8; i++)
        acc = __hfma2(*reinterpret_cast<const __half2 *>(&w[i]), *reinterpret_cast<const __half2 *>(&x[i]), acc);
    const float2 f = __half22float2(acc);
    return f.x + f.y;
}

// Four e2m1 codes (16 bits) -> two f16x2 registers (low nibble first).
__device__ __forceinline__ void e2m1x4_h2(uint32_t v16, uint32_t (&h)[2]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t}"
        : "=r"(h[0]), "=r"(h[1])
        : "r"(v16));
}

// Eight fp32 values scaled by `sc` (a power of two) -> four f16x2 registers.
__device__ __forceinline__ void f32x8_to_h2(const float (&v)[8], float sc, uint32_t (&h)[4]) {
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const __half2 t = __floats2half2_rn(v[2 * i] * sc, v[2 * i + 1] * sc);
        h[i] = *reinterpret_cast<const uint32_t *>(&t);
    }
}

// Two e4m3 bytes (low byte first) -> f16x2 (exact: every e4m3 value is an f16 normal).
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t two_bytes) {
    uint32_t h;
    asm("{\n\t.reg .b16 s;\n\t"
        "cvt.u16.u32 s, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, s;\n\t}"
        : "=r"(h)
        : "r"(two_bytes & 0xffffu));
    return h;
}

// Low / high f16 of a packed pair as a 16-bit register value.
__device__ __forceinline__ uint16_t h2_lo(uint32_t h) { return static_cast<uint16_t>(h & 0xffffu); }
__device__ __forceinline__ uint16_t h2_hi(uint32_t h) { return static_cast<uint16_t>(h >> 16); }

// c + a.lo * s + a.hi * s with f16 multiplicands and fp32 addition (the f16 x f16
// products are exact in fp32): applies a block scale to an f16x2 partial sum.
__device__ __forceinline__ float fma_h2_scale(uint32_t a, uint16_t s, float c) {
    asm("{\n\t.reg .f16 a0, a1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t"
        "fma.rn.f32.f16 %0, a0, %2, %0;\n\t"
        "fma.rn.f32.f16 %0, a1, %2, %0;\n\t}"
        : "+f"(c)
        : "r"(a), "h"(s));
    return c;
}

// Sixteen e2m1 codes (eight f16x2 registers) against sixteen f16 activations, left as
// two f16 partial sums of eight exact products each (|x| < 2^10 keeps every partial
// below 8 * 6 * 2^10 = 49152 < 65504).
__device__ __forceinline__ uint32_t dot16_e2m1_h2(const uint32_t (&w)[8], const uint32_t (&x)[8]) {
    __half2 acc = __hmul2(*reinterpret_cast<const __half2 *>(&w[0]), *reinterpret_cast<const __half2 *>(&x[0]));
#pragma unroll
    for (int i = 1; i < 8; i++)
        acc = __hfma2(*reinterpret_cast<const __half2 *>(&w[i]), *reinterpret_cast<const __half2 *>(&x[i]), acc);
    return *reinterpret_cast<const uint32_t *>(&acc);
}

// (x * s, y * s) -> f16x2 (x in the low half): one packed fp32 multiply, one conversion.
__device__ __forceinline__ uint32_t f2_scale_to_h2(float x, float y, float s) {
    uint32_t h;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t.reg .f32 lo, hi;\n\t"
        "mov.b64 ra, {%1, %2};\n\t"
        "mov.b64 rb, {%3, %3};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {lo, hi}, rd;\n\t"
        "cvt.rn.f16x2.f32 %0, hi, lo;\n\t}"
        : "=r"(h)
        : "f"(x), "f"(y), "f"(s));
    return h;
}

// GGUF Q4_0 block b of a row staged in shared memory (18 bytes: binary16 scale d, then
// 16 bytes qs): blocks are only 2-byte aligned, so the block is read as five aligned
// 32-bit words and the qs words are funnel-shifted out of them. The row must start on a
// 4-byte boundary; the read may run up to 2 bytes past the block.
__device__ __forceinline__ void q4_block(const unsigned char *row, int b, uint32_t &d, uint32_t (&qs)[4]) {
    const int o = 18 * b, a = o & ~3, r = o - a;  // r is 0 or 2
    const uint32_t *w = reinterpret_cast<const uint32_t *>(row + a);
    const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3], w4 = w[4];
    d = (r ? (w0 >> 16) : w0) & 0xffffu;
    const uint32_t sh = 16u + 8u * (uint32_t)r;  // 32 (clamped funnel shift) selects the high word
    qs[0] = __funnelshift_rc(w0, w1, sh);
    qs[1] = __funnelshift_rc(w1, w2, sh);
    qs[2] = __funnelshift_rc(w2, w3, sh);
    qs[3] = __funnelshift_rc(w3, w4, sh);
}

// Four qs bytes -> (nibble - 8) as exact f16x2 pairs: lo = elements (0,1), (2,3) of the
// word's low nibbles, hi = the same elements of its high nibbles (element + 16). A nibble
// q placed under the f16 exponent of 1024 reads as 1024 + q; subtracting 1032 is exact.
__device__ __forceinline__ uint32_t sub_f16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ void q4_word_h2(uint32_t w, uint32_t (&lo)[2], uint32_t (&hi)[2]) {
    const uint32_t ml = w & 0x0F0F0F0Fu, mh = (w >> 4) & 0x0F0F0F0Fu;
    const uint32_t e = 0x64646464u, off = 0x64086408u;  // f16x2 (1032, 1032)
    lo[0] = sub_f16x2(__byte_perm(ml, e, 0x5140), off);
    lo[1] = sub_f16x2(__byte_perm(ml, e, 0x7362), off);
    hi[0] = sub_f16x2(__byte_perm(mh, e, 0x5140), off);
    hi[1] = sub_f16x2(__byte_perm(mh, e, 0x7362), off);
}

// A Q4_0 block (32 weights as sixteen f16x2 pairs, pair p = elements 2p, 2p + 1) against
// 32 f16 activations, left as two f16 partial sums of sixteen exact products each
// (|nibble - 8| <= 8 and |x| < 2^8 keep every partial below 2^15).
__device__ __forceinline__ uint32_t dot32_h2(const uint32_t (&w)[16], const uint32_t (&x)[16]) {
    __half2 acc = __hmul2(*reinterpret_cast<const __half2 *>(&w[0]), *reinterpret_cast<const __half2 *>(&x[0]));
#pragma unroll
    for (int i = 1; i < 16; i++)
        acc = __hfma2(*reinterpret_cast<const __half2 *>(&w[i]), *reinterpret_cast<const __half2 *>(&x[i]), acc);
    return *reinterpret_cast<const uint32_t *>(&acc);
}

// Decode a Q4_0 block's four qs words into the sixteen pairs of dot32_h2.
__device__ __forceinline__ void q4_decode(const uint32_t (&qs)[4], uint32_t (&w)[16]) {
#pragma unroll
    for (int i = 0; i < 4; i++) {
        uint32_t lo[2], hi[2];
        q4_word_h2(qs[i], lo, hi);
        w[2 * i] = lo[0];
        w[2 * i + 1] = lo[1];
        w[8 + 2 * i] = hi[0];
        w[9 + 2 * i] = hi[1];
    }
}

// Element layouts of the nvfp4 activation vectors staged in shared memory. A lane
// handles one 16-element block b per step; storing some of its 16-byte groups in a
// lane-dependent order makes the quarter-warp phases of 128-bit shared loads hit 32
// distinct banks without any data-dependent register selection:
//   f16 activations (32-byte blocks, two 16-byte halves): bit 3 of the element index
//   is flipped when bit 6 is set, i.e. blocks with b & 4 store their halves swapped;
//   fp32 h rows (64-byte blocks, four 16-byte quarters): quarter q of block b is stored
//   at quarter q ^ ((b >> 1) & 3).
__host__ __device__ __forceinline__ int swz_x16(int k) { return k ^ ((k >> 3) & 8); }
// Q4_0 (32-element blocks): f16 activations, 16-byte unit u of block b stored at
// u ^ ((b >> 1) & 3); fp32 h rows, unit u of block b stored at u ^ (b & 7).
__host__ __device__ __forceinline__ int swz_q4x16(int k) { return k ^ ((k >> 3) & 0x18); }
__host__ __device__ __forceinline__ int swz_q4h32(int n) { return n ^ ((n >> 3) & 0x1C); }

__host__ __device__ __forceinline__ int swz_h32(int n) { return n ^ ((n >> 3) & 12); }

// Distinct slot u owning pass `pi`: the largest u with upoff[u] <= pi (upoff ascending).
__device__ __forceinline__ int pass_owner(const int32_t *upoff, int nu, int pi) {
    int lo = 0, hi = nu - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (upoff[mid] <= pi)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

}  // namespace ffn
}  // namespace ftmoe
