// bf16 expert FFN phases on the 5th-generation tensor cores (tcgen05, accumulators in TMEM), as
// a persistent, warp-specialised pipeline for calls with several tokens per expert.
//
// bf16 banks (benchmark guide, section 4.2: gate_up and down) hold output-row-major weights
// [N, K]. A work item is (distinct slot u, pass of up to kTN = 16 tokens, tile of kTM = 128
// output rows); it streams the reduction axis in stages of `boxes` 64-k boxes (128 bytes of
// each row). Warp roles of a CTA (one CTA per SM, items dealt round-robin as in the other
// pipelines):
//   warp 0 (one thread): 3-D tensor copies of the stage's weight boxes, 128 rows x 128 bytes
//       each with the 128-byte shared-memory swizzle (gate and up rows for gate_up), completing
//       on the stage's full barrier; weights carry an L2 evict-first hint;
//   warp 6: the token operand of the stage: the pass's bf16 activations (gate_up) or the hi and
//       lo bf16 terms of its h rows (down), 16 rows x 128 bytes per box, written with generic
//       stores in the same swizzled K-major layout (rows past the pass's token count are zero),
//       made visible to the tensor cores with fence.proxy.async, then an arrive on the full
//       barrier;
//   warp 1: allocates the TMEM columns, and one elected thread issues
//       tcgen05.mma.cta_group::1.kind::f16 (bf16 x bf16 -> fp32, M = 128, N = 16, K = 16) from
//       shared-memory descriptors of both operands; tcgen05.commit releases each stage when its
//       MMAs are done and signals the item's accumulator when the item's last MMA is done;
//   warps 2-5: the epilogue; warp w reads TMEM lanes 32 (w % 4) .. + 31 (output rows) with
//       tcgen05.ld, so each thread holds one output row for the 16 tokens: gate_up stores
//       h = silu(gate) * up as two bf16 terms hi = bf16(h), lo = bf16(h - hi) (the layout of the
//       mma.sync pipeline, read by down as two operand planes into one accumulator, so every
//       product is exact and h keeps 16 significant bits), down stores o in fp32.
// The accumulators are double-buffered in TMEM (gate_up: gate and up, 16 columns each, per
// buffer; down: one), so the epilogue of an item overlaps the MMAs of the next.
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
constexpr int kBBox = kTN * kBoxBytes;    // 2 KiB token box
constexpr int kStagesMax = 4;
constexpr int kWarps = 7;                 // TMA, MMA, 4 epilogue, token operand
constexpr int kThreads = kWarps * 32;
constexpr int kTokWarp = 6;
constexpr uint32_t kTmemCols = 64;        // 2 buffers x (gate, up) x 16 columns
static_assert(kTN == kTc05PassTokens, "the routing kernel cuts passes of kTN tokens");

enum { kGU = 0, kDN = 1 };

struct TcCfg {
    int32_t tiles, kst, boxes, stages, stage_bytes, b_off;
};

// UMMA instruction descriptor (kind::f16): fp32 D, bf16 A and B, both K-major, N = 16, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kTN >> 3) << 17) |
                            ((uint32_t)(kTM >> 4) << 24);

// Shared-memory matrix descriptor of a K-major tile stored with the 128-byte swizzle: rows of
// 128 bytes, groups of 8 rows 1024 bytes apart (stride byte offset), tile base 1024-byte
// aligned; a K = 16 step inside the 128-byte row advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate)
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

__device__ __forceinline__ ItemInfo item_info(const FfnParams &p, int nu, int tiles, int it, int &u) {
    const int pi = it / tiles, tile = it - pi * tiles;
    while (u + 1 < nu && p.s.upoff[u + 1] <= pi) u++;  // increasing passes: walk forward
    ItemInfo f;
    f.slot = p.s.uslot[u];
    f.slot = f.slot < 0 ? 0 : (f.slot >= p.S ? p.S - 1 : f.slot);
    const int pbase = (pi - p.s.upoff[u]) * kTN;
    f.cnt = p.s.ucnt[u] - pbase < kTN ? p.s.ucnt[u] - pbase : kTN;
    f.off = p.s.uoff[u] + pbase;
    f.n0 = tile * kTM;
    return f;
}

template <int PHASE>
__global__ void __launch_bounds__(kThreads, 1)
    ffn_bf16_tc05_kernel(FfnParams p, TcCfg c, const __grid_constant__ CUtensorMap wmap) {
    constexpr int NM = PHASE == kGU ? 2 : 1;      // weight matrices per item (gate, up) or down
    constexpr int NP = PHASE == kGU ? 1 : 2;      // token-operand planes: x, or h hi and lo
    extern __shared__ __align__(1024) unsigned char sm[];
    uint64_t *full = reinterpret_cast<uint64_t *>(sm);
    uint64_t *empty = full + kStagesMax;
    uint64_t *accf = empty + kStagesMax;  // [2] accumulator ready (MMA commit)
    uint64_t *acce = accf + 2;            // [2] accumulator read (epilogue warps)
    uint64_t *done = acce + 2;            // every role finished (TMEM may be freed)
    uint64_t *mdone = done + 1;           // the MMA issuer's last MMAs completed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mdone + 1);
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
    const uint32_t stage_tx = (uint32_t)(NM * c.boxes * kABox);

    if (warp == 0) {  // ------------------------------------------------ weight copies
        if (lane == 0) {
            const uint64_t pol = evict_first_l2();
            bool ok = true;
            int cnt = 0, u = items > first ? pass_owner(p.s.upoff, nu, first / c.tiles) : 0;
            for (int it = first; it < items && ok; it += gridDim.x) {
                const ItemInfo f = item_info(p, nu, c.tiles, it, u);
                for (int ks = 0; ks < c.kst; ks++, cnt++) {
                    const int s = cnt % c.stages;
                    if (!bar_wait(&empty[s], ((cnt / c.stages) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    bar_expect(&full[s], stage_tx);
                    unsigned char *st = stage0 + (size_t)s * c.stage_bytes;
                    for (int m = 0; m < NM; m++)
                        for (int b = 0; b < c.boxes; b++)
                            tma3d_hint(st + (m * c.boxes + b) * kABox, &wmap, (ks * c.boxes + b) * kBoxBytes,
                                       f.n0 + (m ? I : 0), f.slot, &full[s], pol);
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
        bool ok = true, waited = PHASE == kGU;
        int cnt = 0, u = items > first ? pass_owner(p.s.upoff, nu, first / c.tiles) : 0;
        for (int it = first; it < items && ok; it += gridDim.x) {
            const ItemInfo f = item_info(p, nu, c.tiles, it, u);
            if (!waited) {  // h rows come from the gate_up kernel
                asm volatile("griddepcontrol.wait;" ::: "memory");
                waited = true;
            }
            // lane l moves 16-byte chunks l, l + 32, l + 64, l + 96 of each box: row r = chunk / 8
            // of the token operand, chunk j = chunk % 8 of its 128 bytes
            const uint16_t *src[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int r = (lane + 32 * i) >> 3;
                src[i] = nullptr;
                if (r < f.cnt) {
                    const int q = p.s.upairs[f.off + r];
                    src[i] = PHASE == kGU ? p.x + (int64_t)(q / p.topk) * H
                                          : reinterpret_cast<const uint16_t *>(p.s.h + (int64_t)q * I);
                }
            }
            for (int ks = 0; ks < c.kst; ks++, cnt++) {
                const int s = cnt % c.stages;
                if (!bar_wait(&empty[s], ((cnt / c.stages) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                unsigned char *bt = stage0 + (size_t)s * c.stage_bytes + c.b_off;
                for (int pl = 0; pl < NP; pl++)
                    for (int b = 0; b < c.boxes; b++) {
                        const int k0 = (ks * c.boxes + b) * (kBoxBytes / 2) + pl * I;  // elements
                        unsigned char *box = bt + (pl * c.boxes + b) * kBBox;
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            const int ch = lane + 32 * i, r = ch >> 3, j = ch & 7;
                            uint4 v = make_uint4(0u, 0u, 0u, 0u);
                            if (src[i]) v = ldg_stream(src[i] + k0 + 8 * j);
                            *reinterpret_cast<uint4 *>(box + r * kBoxBytes + ((j ^ (r & 7)) << 4)) = v;
                        }
                    }
                // generic-proxy stores -> visible to the tensor cores (async proxy)
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) bar_arrive(&full[s]);
            }
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
                const uint32_t d0 = tmem + (uint32_t)(buf * NM * kTN);
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
#pragma unroll
                            for (int pl = 0; pl < NP; pl++) {
                                const uint64_t bd = sw128_desc(st + c.b_off + (pl * c.boxes + b) * kBBox + 32 * kk);
#pragma unroll
                                for (int m = 0; m < NM; m++) {
                                    const uint64_t ad = sw128_desc(st + (m * c.boxes + b) * kABox + 32 * kk);
                                    umma_bf16(d0 + m * kTN, ad, bd, acc | (uint32_t)pl);
                                }
                            }
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
            const ItemInfo f = item_info(p, nu, c.tiles, it, u);
            const int buf = icnt & 1;
            if (!bar_wait(&accf[buf], (icnt >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float v[NM][16];
#pragma unroll
            for (int m = 0; m < NM; m++)
                tmem_ld16(tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(buf * NM * kTN + m * kTN), v[m]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive(&acce[buf]);  // the MMAs of a later item may overwrite it
            const int n = f.n0 + row;
#pragma unroll
            for (int t = 0; t < kTN; t++) {
                if (t >= f.cnt) break;
                const int q = p.s.upairs[f.off + t];
                if (PHASE == kGU) {
                    const float hv = silu(v[0][t]) * v[NM - 1][t];
                    const __nv_bfloat16 hi = __float2bfloat16_rn(hv);
                    const __nv_bfloat16 lo = __float2bfloat16_rn(hv - __bfloat162float(hi));
                    uint16_t *hr = reinterpret_cast<uint16_t *>(p.s.h + (int64_t)q * I);
                    hr[n] = __bfloat16_as_ushort(hi);
                    hr[I + n] = __bfloat16_as_ushort(lo);
                } else {
                    p.s.o[(int64_t)q * H + n] = v[0][t];
                }
            }
        }
        if (!ok && lane == 0) atomicCAS(p.status, 0, FTMOE_ERR_STATE);
        __syncwarp();
        if (lane == 0) bar_arrive(done);
    }
}

bool make_tc_cfg(const FfnParams &p, int phase, TcCfg &c, size_t &smem) {
    const int K = phase == kGU ? p.H : p.I, nout = phase == kGU ? p.I : p.H;
    const int NM = phase == kGU ? 2 : 1, NP = phase == kGU ? 1 : 2;
    if (K % (kBoxBytes / 2) || nout % kTM) return false;
    const int kboxes = K / (kBoxBytes / 2);
    c.tiles = nout / kTM;
    const size_t head = 256 + 1024;  // barriers and the TMEM address, + alignment slack
    const size_t cap = 227 * 1024;
    // the widest stage (boxes along k dividing K) that still leaves three stages, else two
    for (int want = 3; want >= 2; want--) {
        for (int boxes = 4; boxes >= 1; boxes--) {
            if (kboxes % boxes) continue;
            const int stage = NM * boxes * kABox + NP * boxes * kBBox;  // multiples of 1024
            const int stages = (int)((cap - head) / (size_t)stage);
            if (stages < want) continue;
            c.boxes = boxes;
            c.kst = kboxes / boxes;
            c.stage_bytes = stage;
            c.b_off = NM * boxes * kABox;
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
    const CUtensorMap *wm = reinterpret_cast<const CUtensorMap *>(PHASE == kGU ? maps.tc_gu : maps.tc_dn);
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
