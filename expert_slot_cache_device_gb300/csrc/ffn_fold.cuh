// Device helpers shared by the persistent FFN pipelines for small calls:
//   - the weighted combine folded into the down kernels: the CTA whose down item completes
//     the last routed pair of a token for a tile of output rows forms y for those rows
//     (y_t = addend_t + sum_j w_tj o_tj in routed order j, fp32, one round to bf16; the same
//     arithmetic and order as the separate combine kernel, so results are bitwise the same);
//   - the split reduction axis: the chunks of one (pass, tile) leave fp32 partial sums in
//     global scratch, the last chunk to arrive adds them in chunk order and finishes;
//   - the L2 prefetch of a call's down weights, issued by the gate_up kernel while it
//     streams its own weights, so that the down kernel reads them from L2.
// Every arrival counter is cleared by the routing kernel at the start of the call, and every
// "last to arrive" test is a single atomic: nothing here waits on another CTA.
#pragma once

#include "ffn_common.cuh"
#include "internal.cuh"
#include "pipeline.cuh"

namespace ftmoe {
namespace fold {

// Bounded barrier of the consumer warps on an mbarrier initialised with their count: every
// consumer thread calls it. False (status FTMOE_ERR_STATE recorded) if the wait expired.
__device__ __forceinline__ bool consumer_sync(uint64_t *bar, uint32_t phase, int32_t *status) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) pipe::bar_arrive(bar);
    if (!pipe::bar_wait(bar, phase)) {
        if ((threadIdx.x & 31) == 0) atomicCAS(status, 0, FTMOE_ERR_STATE);
        return false;
    }
    return true;
}

__device__ __forceinline__ uint32_t bf16_rn_bits(float v) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// y[t, n] for n in [n0, n1) (n0 even), lanes `lane` of `nl` striding over pairs of rows.
// o is read through L2 (__ldcg): other CTAs wrote it during this kernel.
__device__ __forceinline__ void combine_rows(const FfnParams &p, int t, int n0, int n1, int lane, int nl) {
    const int k = p.topk, H = p.H;
    const int64_t tq = (int64_t)t * k;
    for (int n = n0 + 2 * lane; n < n1; n += 2 * nl) {
        const bool two = n + 1 < n1;
        float a0 = 0.f, a1 = 0.f;
        if (p.addend) {
            a0 = p.addend[(int64_t)t * H + n];
            if (two) a1 = p.addend[(int64_t)t * H + n + 1];
        }
        for (int j = 0; j < k; j++) {
            if (p.slots[tq + j] < 0) continue;  // computed elsewhere (hybrid CPU executor)
            const float w = p.weights[tq + j];
            const float *orow = p.s.o + (tq + j) * H;
            a0 = fmaf(w, __ldcg(orow + n), a0);
            if (two) a1 = fmaf(w, __ldcg(orow + n + 1), a1);
        }
        uint16_t *yr = p.y + (int64_t)t * H;
        if (two && ((n & 1) == 0))
            *reinterpret_cast<uint32_t *>(yr + n) = bf16_rn_bits(a0) | (bf16_rn_bits(a1) << 16);
        else {
            yr[n] = (uint16_t)bf16_rn_bits(a0);
            if (two) yr[n + 1] = (uint16_t)bf16_rn_bits(a1);
        }
    }
}

// One thread, after the CTA's o rows of down tile `tile` for the routed pairs pairs[0..ntok)
// are stored and fenced by every thread that stored them: counts each pair for its token
// and returns the mask of positions i whose count completed the token (that CTA forms y for
// the token's rows of the tile). A completed count is followed by a fence, so the other
// CTAs' o rows (stored and fenced before their counts) are visible to the caller's group.
__device__ __forceinline__ uint32_t count_pairs(const FfnParams &p, const int32_t *pairs, int ntok, int tile) {
    uint32_t fin = 0;
    for (int i = 0; i < ntok; i++) {
        const int t = pairs[i] / p.topk;
        const int old = atomicAdd(p.s.ycnt + (int64_t)t * p.ytiles + tile, 1);
        if (old + 1 == p.s.gcnt[t]) fin |= 1u << i;
    }
    if (fin) __threadfence();
    return fin;
}

// Split reduction axis: one thread, after every consumer thread stored and fenced its partial
// sums of the item's chunk. True if this chunk is the last of the item's `ksplit` to arrive;
// then the caller's group reads all partials (fenced here).
__device__ __forceinline__ bool chunk_arrive(int32_t *counter, int ksplit) {
    const bool last = atomicAdd(counter, 1) == ksplit - 1;
    if (last) __threadfence();
    return last;
}

// Index of the partial sums of chunk kc, routed pair q, element e (see FfnScratch::part).
__device__ __forceinline__ int64_t part_index(const FfnParams &p, int kc, int q, int e) {
    return ((int64_t)kc * kSplitPairs + q) * p.split_row + e;
}

// L2 prefetch of the down weights of every distinct slot of the call, dealt round-robin over
// the CTAs in 64 KiB pieces, when they total at most p.l2_prefetch bytes. Prefetches are
// hints: nothing waits for them and they change no result.
__device__ __forceinline__ void prefetch_down(const FfnParams &p, int nu) {
    if (p.l2_prefetch <= 0 || nu <= 0) return;
    int64_t per = 0;
    for (int b = 0; b < p.dn_nb; b++) per += p.bank_bytes[p.dn_b0 + b];
    if ((int64_t)nu * per > p.l2_prefetch) return;
    constexpr int64_t kPiece = 64 * 1024;
    int64_t idx = 0;
    for (int u = 0; u < nu; u++) {
        const int slot = p.s.uslot[u];
        if (slot < 0 || slot >= p.S) continue;
        for (int b = 0; b < p.dn_nb; b++) {
            const int64_t bytes = p.bank_bytes[p.dn_b0 + b];
            const unsigned char *base = p.bank[p.dn_b0 + b] + (int64_t)slot * bytes;
            for (int64_t off = 0; off < bytes; off += kPiece, idx++) {
                if (idx % gridDim.x != blockIdx.x) continue;
                const int64_t len = (bytes - off < kPiece ? bytes - off : kPiece) & ~(int64_t)15;
                const unsigned char *a = base + off;
                if (len <= 0 || ((uintptr_t)a & 15)) continue;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"((uint32_t)len) : "memory");
            }
        }
    }
}

}  // namespace fold
}  // namespace ftmoe
