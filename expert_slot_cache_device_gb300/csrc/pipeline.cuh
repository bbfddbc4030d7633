// Device helpers shared by the tensor-map pipelines: shared-memory addresses, bounded
// mbarrier waits, bulk and tensor copies, and the warp-level f16 / bf16 MMA.
#pragma once
#include <cuda.h>
#include <cstdint>

namespace ftmoe {
namespace pipe {

constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: far beyond any healthy wait

__device__ __forceinline__ uint32_t su32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void bar_init(uint64_t *b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_expect(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
// Bounded wait for the phase with the given parity: false once `limit_ns` of %globaltimer have
// passed (the default is far beyond any healthy wait; a shorter limit is a test setting).
__device__ __forceinline__ bool bar_wait(uint64_t *b, uint32_t parity, uint64_t limit_ns = kWaitNs) {
    const uint64_t t0 = gtimer();
    for (uint32_t i = 0;; i++) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(su32(b)), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((i & 255) == 255 && gtimer() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ void tma3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(su32(bar))
        : "memory");
}

// The same with an L2 cache policy (createpolicy), e.g. evict-first for weights read once:
// the lines a preceding copy left dirty in L2 then stay there instead of being written back
// while the weights stream through.
__device__ __forceinline__ void tma3d_hint(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar,
                                           uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3, %4}], [%5], %6;" ::"r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(su32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t evict_first_l2() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared with an L2 cache policy, completing on an mbarrier.
__device__ __forceinline__ void bulk1d_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(su32(dst)),
        "l"(src), "r"(bytes), "r"(su32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk1d(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     su32(dst)),
                 "l"(src), "r"(bytes), "r"(su32(bar))
                 : "memory");
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same with a zero accumulator input (d = A * B).
__device__ __forceinline__ void mma_f16_16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// d += A * B with bf16 operands and an fp32 accumulator (A 16 x 16 row, B 16 x 8 col).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four 8 x 8 matrices of 16-bit elements from shared memory (lane l gives the address of
// row l % 8 of matrix l / 8); lane (g, tig) receives elements (g, 2 tig) and (g, 2 tig + 1)
// of each matrix, which for the matrices (rows 0-7 | 8-15) x (k 0-7 | 8-15) of a 16 x 16
// tile is the A fragment of mma m16n8k16.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(su32(p)));
}

// Two e8m0 bytes (low byte first) -> their values 2^(b - 127) as floats, through the
// exact ue8m0 -> bf16 conversion (bf16 has f32's exponent range, so bf16 << 16 is the
// f32 value; 0 gives the bf16 subnormal 2^-127, 0xff NaN).
__device__ __forceinline__ float2 e8m0x2_to_f2(uint32_t two_bytes) {
    uint32_t b;
    asm("{\n\t.reg .b16 s;\n\t"
        "cvt.u16.u32 s, %1;\n\t"
        "cvt.rn.bf16x2.ue8m0x2 %0, s;\n\t}"
        : "=r"(b)
        : "r"(two_bytes & 0xffffu));
    return make_float2(__uint_as_float(b << 16), __uint_as_float(b & 0xffff0000u));
}

// (a0, a1) += (t0, t1) * s with one packed fp32 FMA.
__device__ __forceinline__ void ffma2_s(float &a0, float &a1, float t0, float t1, float s) {
    uint64_t r;
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%1, %2};\n\t"
        "mov.b64 rb, {%3, %3};\n\t"
        "mov.b64 rc, {%4, %5};\n\t"
        "fma.rn.f32x2 %0, ra, rb, rc;\n\t}"
        : "=l"(r)
        : "f"(t0), "f"(t1), "f"(s), "f"(a0), "f"(a1));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(r));
}

}  // namespace pipe
}  // namespace ftmoe
