// The weighted combine folded into the down kernels of the persistent FFN pipelines.
//
// Every down CTA, once it has stored the o rows of all its work items, fences once, then
// counts each routed pair of its items for (token, row tile). The CTA whose count completes a
// token's tile (its last routed pair with a slot) forms y for those rows:
//     y_t = addend_t + sum_j w_tj o_tj   in routed order j, fp32, one round to bf16,
// the arithmetic and order of the separate combine kernel, so results are bitwise the same
// and reproducible. The counters are cleared by the routing kernel at the start of the call;
// each "last to arrive" test is one atomic, so no CTA waits on another. (Fencing per item
// instead costs about as much as the item itself under a full HBM stream; one fence per
// thread at exit does not.)
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

// y[t, n] for n in [n0, n1) (n0 even), `nl` threads (index `lane`) striding over pairs of
// rows. o is read through L2 (__ldcg): other CTAs wrote it during this kernel.
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
        if (two)
            *reinterpret_cast<uint32_t *>(yr + n) = bf16_rn_bits(a0) | (bf16_rn_bits(a1) << 16);
        else
            yr[n] = (uint16_t)bf16_rn_bits(a0);
    }
}

// Entries of the per-CTA queue of (token, tile) rows to form; a full queue falls back to the
// counting thread forming the rows itself.
constexpr int kQueue = 512;

struct ExitQueue {
    int n;
    int32_t tt[kQueue];  // token * ytiles + tile
};

// Called by every consumer thread (nthreads of them, index tid) of a down CTA after its last
// item, with the work-item decomposition of that kernel: items of `tiles` row tiles of
// `row_tile` rows per pass of at most `pass_tokens` pairs, dealt round-robin over the CTAs.
// Two consumer mbarriers (count = consumer warps, fresh phase `phase`) order the steps.
// False if a barrier wait expired (status recorded).
__device__ __forceinline__ bool fold_at_exit(const FfnParams &p, int tiles, int row_tile, int pass_tokens,
                                             uint64_t *bar0, uint64_t *bar1, uint32_t phase, ExitQueue *q,
                                             int tid, int nthreads) {
    __threadfence();  // this thread's o rows, before any item of the CTA is counted
    if (tid == 0) q->n = 0;
    if (!consumer_sync(bar0, phase, p.status)) return false;
    const int nu = *p.s.n_unique;
    const int npass = nu > 0 ? *p.s.n_passes : 0;
    const int items = npass * tiles;
    for (int it = blockIdx.x + tid * gridDim.x; it < items; it += nthreads * gridDim.x) {
        const int pi = it / tiles, tile = it - pi * tiles;
        const int u = ffn::pass_owner(p.s.upoff, nu, pi);
        const int pbase = (pi - p.s.upoff[u]) * pass_tokens;
        const int cnt = p.s.ucnt[u] - pbase < pass_tokens ? p.s.ucnt[u] - pbase : pass_tokens;
        const int off = p.s.uoff[u] + pbase;
        for (int i = 0; i < cnt; i++) {
            const int t = p.s.upairs[off + i] / p.topk;
            const int old = atomicAdd(p.s.ycnt + (int64_t)t * p.ytiles + tile, 1);
            if (old + 1 != p.s.gcnt[t]) continue;
            __threadfence();  // the other CTAs' o rows of this token (fenced before their counts)
            const int slot = atomicAdd(&q->n, 1);
            if (slot < kQueue) {
                q->tt[slot] = t * p.ytiles + tile;
            } else {
                const int n1 = (tile + 1) * row_tile < p.H ? (tile + 1) * row_tile : p.H;
                combine_rows(p, t, tile * row_tile, n1, 0, 1);
            }
        }
    }
    if (!consumer_sync(bar1, phase, p.status)) return false;
    const int nq = q->n < kQueue ? q->n : kQueue;
    const int warp = tid >> 5, nwarps = nthreads >> 5, lane = tid & 31;
    for (int e = warp; e < nq; e += nwarps) {
        const int tt = q->tt[e], t = tt / p.ytiles, tile = tt - t * p.ytiles;
        const int n1 = (tile + 1) * row_tile < p.H ? (tile + 1) * row_tile : p.H;
        combine_rows(p, t, tile * row_tile, n1, lane, 32);
    }
    return true;
}

}  // namespace fold
}  // namespace ftmoe
