// bf16 expert FFN phases on the 5th-generation tensor cores (tcgen05, accumulators in TMEM), as
// a persistent, warp-specialised pipeline for calls with several tokens per expert.
//
// bf16 banks (benchmark guide, section 4.2: gate_up and down) hold output-row-major weights
// [N, K]. A work item is (distinct slot u, pass of up to kTN = 16 tokens, tile of 128 rows of
// the MMA's M): down takes 128 output rows; gate_up takes 64 neurons, their 64 gate rows in
// rows 0-63 of the tile and their 64 up rows in rows 64-127, so one MMA forms both and the
// items are twice as many (fewer idle SMs in a call's last round). An item streams the
// reduction axis in stages of `boxes` 64-k boxes (128 bytes of each row). Warp roles of a CTA
// (one CTA per SM, items dealt round-robin as in the other pipelines):
//   warp 0 (one thread): 3-D tensor copies of the stage's weight boxes with the 128-byte
//       shared-memory swizzle (gate_up: two 64-row boxes, gate then up rows, per 128-row
//       tile), completing on the stage's full barrier; weights carry an L2 evict-first hint;
//   warp 6: the token operand of the stage: the pass's bf16 activations (gate_up) or the hi and
//       lo bf16 terms of its h rows (down), 16 rows x 128 bytes per box, written with generic
//       stores in the same swizzled K-major layout (rows past the pass's token count are zero),
//       made visible to the tensor cores with fence.proxy.async, then an arrive on the full
//       barrier;
//   warp 1: allocates the TMEM columns, and one elected thread issues
//       tcgen05.mma.cta_group::1.kind::f16 (bf16 x bf16 -> fp32, M = 128, N = 16, K = 16) from
//       shared-memory descriptors of both operands; tcgen05.commit releases each stage when its
//       MMAs are done and signals the item's accumulator when the item's last MMA is done;
//   warps 2-5: the epilogue; warp w reads TMEM lanes 32 (w % 4) .. + 31 (rows of the tile)
//       with tcgen05.ld, so each thread holds one row for the 16 tokens. gate_up: the warps
//       holding up rows hand them over through shared memory, and the warps holding the gate
//       rows store h = silu(gate) * up as two bf16 terms hi = bf16(h), lo = bf16(h - hi) (the
//       layout of the mma.sync pipeline, read by down as two operand terms, so every product is
//       exact and h keeps 16 significant bits); down stores o in fp32.
// The accumulators are double-buffered in TMEM, so the epilogue of an item overlaps the MMAs
// of the next.
//
// Every mbarrier wait is bounded (2 s); on expiry the thread records FTMOE_ERR_STATE and its
// role stops. The TMEM owner waits (bounded) for the other roles and for its own MMAs before it
// frees the columns, on every path.
#include <cuda.h>

#include "ffn_common.cuh"
#include "internal.cuh"
#include "pipeline.cuh"

namespace ftmoe {
namespace {

using namespace ffn;
using namespace pipe;

constexpr int kTM = 128;                  // output rows per item (UMMA M)
constexpr int kTN = 16;                   // tokens per pass (UMMA N)
constexpr int kBoxBytes = 128;            // one box row: 64 bf16 of k
constexpr int kABox = kTM * kBoxBytes;    // 16 KiB weight box
// token operand rows per box: gate_up the kTN tokens; down the kTN hi terms of h then their
// kTN lo terms, so one MMA of N = 2 kTN takes both (the epilogue adds the two column halves)
template <int PHASE>
constexpr int kBRows = PHASE == 0 ? kTN : 2 * kTN;
constexpr int kStagesMax = 4;
constexpr int kWarps = 7;                 // TMA, MMA, 4 epilogue, token operand
constexpr int kThreads = kWarps * 32;
constexpr int kTokWarp = 6;
constexpr uint32_t kTmemCols = 64;        // 2 buffers x 16 columns (gate_up) or 32 (down)
constexpr int kGuNeurons = kTM / 2;       // gate_up neurons per item (gate and up rows stacked)
static_assert(kTN == kTc05PassTokens, "the routing kernel cuts passes of kTN tokens");

enum { kGU = 0, kDN = 1 };

struct TcCfg {
    int32_t tiles, kst, boxes, stages, stage_bytes, b_off;
};

// UMMA instruction descriptor (kind::f16): fp32 D, bf16 A and B, both K-major, M = 128, N.
template <int N>
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
                            ((uint32_t)(kTM >> 4) << 24);

// Shared-memory matrix descriptor of a K-major tile stored with the 128-byte swizzle: rows of
// 128 bytes, groups of 8 rows 1024 bytes apart (stride byte offset), tile base 1024-byte
// aligned; a K = 16 step inside the 128-byte row advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

template <int N>
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(kIdesc<N>), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// The work item `it` of this call: its slot, pass token count and routed pairs.
struct ItemInfo {
    int slot, n0, cnt, off;
};

template <int PHASE>
__device__ __forceinline__ ItemInfo item_info(const FfnParams &p, int nu, int tiles, int it, int &u) {
    const int pi = it / tiles, tile = it - pi * tiles;
    while (u + 1 < nu && p.s.upoff[u + 1] <= pi) u++;  // increasing passes: walk forward
    ItemInfo f;
    f.slot = p.s.uslot[u];
    FTMOE_DCHECK(f.slot >= 0 && f.slot < p.S, p.status);
    f.slot = f.slot < 0 ? 0 : (f.slot >= p.S ? p.S - 1 : f.slot);
    const int pbase = (pi - p.s.upoff[u]) * kTN;
    f.cnt = p.s.ucnt[u] - pbase < kTN ? p.s.ucnt[u] - pbase : kTN;
    f.off = p.s.uoff[u] + pbase;
    f.n0 = tile * (PHASE == kGU ? kGuNeurons : kTM);  // first neuron (gate_up) or output row (down)
    return f;
}

template <int PHASE>
__global__ void __launch_bounds__(kThreads, 1)
    ffn_bf16_tc05_kernel(FfnParams p, TcCfg c, const __grid_constant__ CUtensorMap wmap) {
    constexpr int NB = kBRows<PHASE>;             // token-operand rows per box (the MMA's N)
    constexpr int BBOX = NB * kBoxBytes;          // bytes of one token-operand box
    extern __shared__ __align__(1024) unsigned char sm[];
    uint64_t *full = reinterpret_cast<uint64_t *>(sm);
    uint64_t *empty = full + kStagesMax;
    uint64_t *accf = empty + kStagesMax;  // [2] accumulator ready (MMA commit)
    uint64_t *acce = accf + 2;            // [2] accumulator read (epilogue warps)
    uint64_t *done = acce + 2;            // every role finished (TMEM may be freed)
    uint64_t *mdone = done + 1;           // the MMA issuer's last MMAs completed
    uint64_t *xsync = mdone + 1;          // gate_up epilogue: up rows handed over
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(xsync + 1);
    __shared__ float s_up[2][kTN][kGuNeurons];  // gate_up: up sums by token and neuron, per item parity
    // stages: the first 1024-byte aligned address past the barriers (256 bytes)
    const uint32_t base = (su32(sm) + 256u + 1023u) & ~1023u;
    unsigned char *stage0 = sm + (base - su32(sm));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H, I = p.I;
    const int K = PHASE == kGU ? H : I;

    if (threadIdx.x == 0) {
        for (int s = 0; s < c.stages; s++) {
            bar_init(&full[s], 2);   // the weight copies (arrive + bytes) and the token operand
            bar_init(&empty[s], 1);  // the MMA commit of the stage
        }
        for (int b = 0; b < 2; b++) {
            bar_init(&accf[b], 1);
            bar_init(&acce[b], 4);
        }
        bar_init(done, kWarps - 1);
        bar_init(mdone, 1);
        bar_init(xsync, 4);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {  // TMEM columns for the two accumulator buffers
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
    if (PHASE == kGU) asm volatile("griddepcontrol.wait;" ::: "memory");  // routing tables
    asm volatile("griddepcontrol.launch_dependents;" :::);

    const int nu = *p.s.n_unique;
    const int npass = nu > 0 ? *p.s.n_passes : 0;
    const int items = npass * c.tiles;
    const int first = blockIdx.x;
    const uint32_t stage_tx = (uint32_t)(c.boxes * kABox);

    if (warp == 0) {  // ------------------------------------------------ weight copies
        if (lane == 0) {
            const uint64_t pol = evict_first_l2();
            bool ok = true;
            int cnt = 0, u = items > first ? pass_owner(p.s.upoff, nu, first / c.tiles) : 0;
            for (int it = first; it < items && ok; it += gridDim.x) {
                const ItemInfo f = item_info<PHASE>(p, nu, c.tiles, it, u);
                for (int ks = 0; ks < c.kst; ks++, cnt++) {
                    const int s = cnt % c.stages;
                    if (!bar_wait(&empty[s], ((cnt / c.stages) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    bar_expect(&full[s], stage_tx);
                    unsigned char *st = stage0 + (size_t)s * c.stage_bytes;
                    for (int b = 0; b < c.boxes; b++) {
                        const int x = (ks * c.boxes + b) * kBoxBytes;
                        if (PHASE == kGU) {  // 64 gate rows, then the same neurons' 64 up rows
                            tma3d_hint(st + b * kABox, &wmap, x, f.n0, f.slot, &full[s], pol);
                            tma3d_hint(st + b * kABox + kABox / 2, &wmap, x, I + f.n0, f.slot, &full[s], pol);
                        } else {
                            tma3d_hint(st + b * kABox, &wmap, x, f.n0, f.slot, &full[s], pol);
                        }
                    }
                }
            }
            if (!ok) {
                atomicCAS(p.status, 0, FTMOE_ERR_STATE);
                // wait (bounded) until the copies already issued have landed
                for (int j = cnt - c.stages < 0 ? 0 : cnt - c.stages; j < cnt; j++)
                    bar_wait(&full[j % c.stages], (j / c.stages) & 1);
            }
        }
        __syncwarp();
        if (lane == 0) bar_arrive(done);
        return;
    }

    if (warp == kTokWarp) {  // ----------------------------------------- token operand
        // 16-byte asynchronous copies (cp.async, zero-filled past the pass's tokens), one commit
        // group per stage; a stage is signalled once the copies of the next stage are issued,
        // so the L2 latency of one stage's rows overlaps the issue of the next
        bool ok = true, waited = PHASE == kGU;
        int cnt = 0, pend = 0, u = items > first ? pass_owner(p.s.upoff, nu, first / c.tiles) : 0;
        for (int it = first; it < items && ok; it += gridDim.x) {
            const ItemInfo f = item_info<PHASE>(p, nu, c.tiles, it, u);
            if (!waited) {  // h rows come from the gate_up kernel
                asm volatile("griddepcontrol.wait;" ::: "memory");
                waited = true;
            }
            // lane l moves 16-byte chunks l, l + 32, ... of each box: row r = chunk / 8 of the
            // token operand (down: token r % kTN, term r / kTN), chunk j = chunk % 8 of its 128 bytes
            constexpr int CPL = NB / 4;  // chunks per lane and box
            const uint16_t *src[CPL];
#pragma unroll
            for (int i = 0; i < CPL; i++) {
                const int r = (lane + 32 * i) >> 3, tk = r % kTN;
                src[i] = PHASE == kGU ? p.x : reinterpret_cast<const uint16_t *>(p.s.h);  // valid, unread
                if (tk < f.cnt) {
                    const int q = p.s.upairs[f.off + tk];
                    src[i] = PHASE == kGU ? p.x + (int64_t)(q / p.topk) * H
                                          : reinterpret_cast<const uint16_t *>(p.s.h + (int64_t)q * I) + (r / kTN) * I;
                }
            }
            for (int ks = 0; ks < c.kst; ks++, cnt++) {
                const int s = cnt % c.stages;
                if (!bar_wait(&empty[s], ((cnt / c.stages) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                const uint32_t bt = base + (uint32_t)(s * c.stage_bytes + c.b_off);
                for (int b = 0; b < c.boxes; b++) {
                    const int k0 = (ks * c.boxes + b) * (kBoxBytes / 2);  // elements
                    const uint32_t box = bt + (uint32_t)(b * BBOX);
#pragma unroll
                    for (int i = 0; i < CPL; i++) {
                        const int ch = lane + 32 * i, r = ch >> 3, j = ch & 7;
                        const uint32_t bytes = (r % kTN) < f.cnt ? 16u : 0u;  // 0: zero-fill
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                                         box + (uint32_t)(r * kBoxBytes + ((j ^ (r & 7)) << 4))),
                                     "l"(src[i] + (bytes ? k0 + 8 * j : 0)), "r"(bytes)
                                     : "memory");
                    }
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
                if (++pend == 2) {  // the previous stage's copies have landed: signal it
                    asm volatile("cp.async.wait_group 1;" ::: "memory");
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor cores
                    __syncwarp();
                    if (lane == 0) bar_arrive(&full[(cnt - 1) % c.stages]);
                    pend = 1;
                }
            }
        }
        if (pend) {  // the last stage
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0 && ok) bar_arrive(&full[(cnt - 1) % c.stages]);
        }
        if (!ok && lane == 0) atomicCAS(p.status, 0, FTMOE_ERR_STATE);
        __syncwarp();
        if (lane == 0) bar_arrive(done);
        return;
    }

    if (warp == 1) {  // ------------------------------------------------ MMA issuer
        bool ok = true;
        if (lane == 0) {
            int cnt = 0, icnt = 0;
            for (int it = first; it < items && ok; it += gridDim.x, icnt++) {
                const int buf = icnt & 1;
                if (!bar_wait(&acce[buf], ((icnt >> 1) & 1) ^ 1)) {  // the epilogue has read it
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem + (uint32_t)(buf * NB);
                for (int ks = 0; ks < c.kst; ks++, cnt++) {
                    const int s = cnt % c.stages;
                    if (!bar_wait(&full[s], (cnt / c.stages) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = base + (uint32_t)(s * c.stage_bytes);
                    for (int b = 0; b < c.boxes; b++)
#pragma unroll
                        for (int kk = 0; kk < kBoxBytes / 32; kk++) {  // K = 16 steps: 32 bytes apart
                            const uint32_t acc = (ks | b | kk) ? 1u : 0u;
                            const uint64_t bd = sw128_desc(st + c.b_off + b * BBOX + 32 * kk);
                            const uint64_t ad = sw128_desc(st + b * kABox + 32 * kk);
                            umma_bf16<NB>(d0, ad, bd, acc);
                        }
                    umma_commit(&empty[s]);  // the stage is free once these MMAs are done
                }
                if (!ok) break;
                umma_commit(&accf[buf]);  // the item's accumulators are complete
            }
            if (!ok) atomicCAS(p.status, 0, FTMOE_ERR_STATE);
            umma_commit(mdone);  // every MMA issued above is done when this arrives
            bar_wait(mdone, 0);
        }
        __syncwarp();
        // the other roles are done with TMEM: free it (bounded wait; freed on every path)
        bar_wait(done, 0);
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
        return;
    }

    // ------------------------------------------------------------------ epilogue (warps 2-5)
    {
        const int quad = warp & 3;  // TMEM lanes 32 quad .. 32 quad + 31
        const int row = 32 * quad + lane;
        bool ok = true;
        int icnt = 0, u = items > first ? pass_owner(p.s.upoff, nu, first / c.tiles) : 0;
        for (int it = first; it < items && ok; it += gridDim.x, icnt++) {
            const ItemInfo f = item_info<PHASE>(p, nu, c.tiles, it, u);
            const int buf = icnt & 1;
            if (!bar_wait(&accf[buf], (icnt >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // gate_up: v[0] = the tile row's sums (gate rows in quadrants 0-1, up rows in 2-3);
            // down: v[0] the hi-term sums, v[1] the lo-term sums of the output row
            constexpr int NV = PHASE == kGU ? 1 : 2;
            float v[NV][16];
#pragma unroll
            for (int m = 0; m < NV; m++)
                tmem_ld16(tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(buf * NB + m * kTN), v[m]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive(&acce[buf]);  // the MMAs of a later item may overwrite it
            if (PHASE == kGU) {
                const int nr = 32 * (quad & 1) + lane;  // neuron of this row within the item
                if (quad >= 2) {                        // up rows: hand them to the gate rows' warps
#pragma unroll
                    for (int t = 0; t < kTN; t++) s_up[icnt & 1][t][nr] = v[0][t];
                }
                __syncwarp();
                if (lane == 0) bar_arrive(xsync);
                if (!bar_wait(xsync, icnt & 1)) {
                    ok = false;
                    break;
                }
                if (quad < 2) {
                    const int n = f.n0 + nr;
                    uint16_t *hr0 = reinterpret_cast<uint16_t *>(p.s.h);
#pragma unroll
                    for (int t = 0; t < kTN; t++) {
                        if (t >= f.cnt) break;
                        const int q = p.s.upairs[f.off + t];
                        const float hv = silu(v[0][t]) * s_up[icnt & 1][t][nr];
                        const __nv_bfloat16 hi = __float2bfloat16_rn(hv);
                        const __nv_bfloat16 lo = __float2bfloat16_rn(hv - __bfloat162float(hi));
                        uint16_t *hr = hr0 + (int64_t)q * 2 * I;
                        hr[n] = __bfloat16_as_ushort(hi);
                        hr[I + n] = __bfloat16_as_ushort(lo);
                    }
                }
            } else {
                const int n = f.n0 + row;
#pragma unroll
                for (int t = 0; t < kTN; t++) {
                    if (t >= f.cnt) break;
                    const int q = p.s.upairs[f.off + t];
                    p.s.o[(int64_t)q * H + n] = v[0][t] + v[1][t];
                }
            }
        }
        if (!ok && lane == 0) atomicCAS(p.status, 0, FTMOE_ERR_STATE);
        __syncwarp();
        if (lane == 0) bar_arrive(done);
    }
}

bool make_tc_cfg(const FfnParams &p, int phase, TcCfg &c, size_t &smem) {
    const int K = phase == kGU ? p.H : p.I;
    const int BBOX = (phase == kGU ? kBRows<kGU> : kBRows<kDN>) * kBoxBytes;
    const int rows = phase == kGU ? kGuNeurons : kTM, nout = phase == kGU ? p.I : p.H;
    if (K % (kBoxBytes / 2) || nout % rows) return false;
    const int kboxes = K / (kBoxBytes / 2);
    c.tiles = nout / rows;
    const size_t head = 256 + 1024;  // barriers and the TMEM address, + alignment slack
    const size_t cap = 227 * 1024 - 9 * 1024;  // dynamic; the static hand-over buffer takes 8 KiB
    // the widest stage (boxes along k dividing K) that still leaves three stages, else two
    for (int want = 3; want >= 2; want--) {
        for (int boxes = 4; boxes >= 1; boxes--) {
            if (kboxes % boxes) continue;
            const int stage = boxes * kABox + boxes * BBOX;  // multiples of 1024
            const int stages = (int)((cap - head) / (size_t)stage);
            if (stages < want) continue;
            c.boxes = boxes;
            c.kst = kboxes / boxes;
            c.stage_bytes = stage;
            c.b_off = boxes * kABox;
            c.stages = stages > kStagesMax ? kStagesMax : stages;
            smem = head + (size_t)c.stages * c.stage_bytes;
            return true;
        }
    }
    return false;
}

template <int PHASE>
cudaError_t launch_tc(const FfnParams &p, const MxTmaMaps &maps, int num_sms, cudaStream_t st) {
    TcCfg c;
    size_t smem;
    if (!make_tc_cfg(p, PHASE, c, smem)) return cudaErrorInvalidValue;
    auto kern = ffn_bf16_tc05_kernel<PHASE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // gate_up: the mma.sync pipeline's map (boxes of 64 rows); down: boxes of 128 rows
    const CUtensorMap *wm = reinterpret_cast<const CUtensorMap *>(PHASE == kGU ? maps.gu_blocks : maps.tc_dn);
    return cudaLaunchKernelEx(&cfg, kern, p, c, *wm);
}

}  // namespace

bool ffn_bf16_tc05_supported(const FfnParams &p, const MxTmaMaps *maps) {
    if (!maps || !maps->tc_valid || p.fmt != FTMOE_FMT_BF16 || !p.s.upoff || !p.s.n_passes) return false;
    TcCfg c;
    size_t smem;
    return make_tc_cfg(p, kGU, c, smem) && make_tc_cfg(p, kDN, c, smem);
}

cudaError_t launch_ffn_bf16_tc05(const FfnParams &p, const MxTmaMaps &maps, int num_sms, cudaStream_t st) {
    cudaError_t e = launch_tc<kGU>(p, maps, num_sms, st);
    if (e != cudaSuccess) return e;
    return launch_tc<kDN>(p, maps, num_sms, st);
}

}  // namespace ftmoe
