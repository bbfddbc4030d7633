// Transposed mxfp4 expert FFN phases as a persistent, warp-specialised bulk-tensor (TMA) pipeline.
//
// mxfp4 banks are stored transposed (benchmark guide, section 4.2: "_blocks /
// _scales / _bias"): blocks [K/2, N] (byte (i, n) holds k = 2i in the low nibble and
// k = 2i + 1 in the high nibble of output column n), scales [K/32, N] e8m0, bias [N].
// A work item is (distinct slot u, pass of up to four tokens, tile of 128 output
// columns); it streams the whole reduction axis in stages of kKp = 256 k-pair rows. A
// producer thread loads each stage with 3-D bulk tensor copies (cp.async.bulk.tensor
// over [slot, row, column], one box of 128 columns x 256 rows per matrix plus the 16
// matching scale rows, completion on an mbarrier; rows past the slot's end are
// zero-filled) and a 1-D bulk copy of the tokens' activations for those rows. Sixteen
// consumer warps each take one 16-row scale block of the stage: a lane owns 4 adjacent
// columns, decodes their code bytes to exact f16x2 (k even, k odd), and accumulates
// with packed f16 FMAs against the row's activation pair (a shared-memory broadcast):
// each f16 half sums 16 exact products of |e2m1| <= 6 and |x| < 2^9, so it stays below
// 2^15. The block's partial is scaled by 2^(e8m0 - 127) and accumulated in fp32. After
// the last stage of an item each warp writes its partials over its own (consumed) code
// block of that stage, the warps meet behind an mbarrier (bounded wait), the bias is
// added, and gate_up writes h = silu(g) * u while down writes o.
//
// Activations: gate_up uses the f16 copy of x (per-token power-of-two scale, max
// |x| < 2^9); down converts the fp32 h rows with the per-pair power-of-two scale
// derived from the max |h| recorded by gate_up.
#include <cuda.h>

#include "ffn_common.cuh"
#include "internal.cuh"

namespace ftmoe {
namespace {

using namespace ffn;

constexpr int kCW = 16;                     // consumer warps (one 16-row scale block each)
constexpr int kMxThreads = (kCW + 1) * 32;  // + producer warp
constexpr int kKp = 256;                    // k-pair rows per stage (16 blocks of 16)
constexpr int kCols = 128;                  // output columns per item
constexpr int kMxStagesMax = 4;
constexpr int kMxTokMax = 4;
static_assert(kMxTokMax * kCols * 4 <= 16 * kCols, "a warp's partials fit its 16-row code block");
constexpr uint64_t kWaitNs = 2000000000ull;

enum { kGU = 0, kDN = 1 };

struct MxHdr {
    int32_t slot, n0, kstage, rows, ntok, last, done, pad;
    int32_t pairs[kMxTokMax];
    int32_t texp[kMxTokMax];
};

struct MxCfg {
    int32_t tiles, kst, stages, stage_bytes, tok_off, tok_bytes, sc_off, tg;
};

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
__device__ __forceinline__ bool bar_wait(uint64_t *b, uint32_t parity) {
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
        if ((i & 255) == 255 && gtimer() - t0 > kWaitNs) return false;
    }
}

__device__ __forceinline__ void tma3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(su32(bar))
        : "memory");
}

__device__ __forceinline__ void bulk1d(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     su32(dst)),
                 "l"(src), "r"(bytes), "r"(su32(bar))
                 : "memory");
}

// Accumulate one 16-row scale block of the stage for NM matrices (gate, up) and NT tokens.
template <int NM, int NT, bool DOWN>
__device__ __forceinline__ void mx_block(const unsigned char *st, const MxCfg &c, int blk,
                                         float (&acc)[NM][4][kMxTokMax], const float (&hsc)[kMxTokMax]) {
    const int lane = threadIdx.x & 31;
    __half2 a16[NM][4][NT];
#pragma unroll
    for (int m = 0; m < NM; m++)
#pragma unroll
        for (int cc = 0; cc < 4; cc++)
#pragma unroll
            for (int t = 0; t < NT; t++) a16[m][cc][t] = __float2half2_rn(0.f);
    const int r0 = blk * 16;
#pragma unroll
    for (int r = r0; r < r0 + 16; r++) {
        uint32_t xp[NT];
#pragma unroll
        for (int t = 0; t < NT; t++) {
            if (DOWN) {
                const float2 hv = *reinterpret_cast<const float2 *>(st + c.tok_off + t * c.tok_bytes + 8 * r);
                const __half2 x2 = __floats2half2_rn(hv.x * hsc[t], hv.y * hsc[t]);
                xp[t] = *reinterpret_cast<const uint32_t *>(&x2);
            } else {
                xp[t] = *reinterpret_cast<const uint32_t *>(st + c.tok_off + t * c.tok_bytes + 4 * r);
            }
        }
#pragma unroll
        for (int m = 0; m < NM; m++) {
            const uint32_t cw = *reinterpret_cast<const uint32_t *>(st + m * kKp * kCols + r * kCols + 4 * lane);
            uint32_t w4[4];  // column cc: (k even, k odd) as exact f16x2
            e2m1x8_h2(cw, w4);
#pragma unroll
            for (int cc = 0; cc < 4; cc++) {
#pragma unroll
                for (int t = 0; t < NT; t++)
                    a16[m][cc][t] = __hfma2(*reinterpret_cast<const __half2 *>(&w4[cc]),
                                            *reinterpret_cast<const __half2 *>(&xp[t]), a16[m][cc][t]);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < NM; m++) {
        const uint32_t sw = *reinterpret_cast<const uint32_t *>(st + c.sc_off + m * (kKp / 16) * kCols + blk * kCols +
                                                                4 * lane);
#pragma unroll
        for (int cc = 0; cc < 4; cc++) {
            const float s = e8m0_to_f(sw >> (8 * cc));
#pragma unroll
            for (int t = 0; t < NT; t++) {
                const float2 f = __half22float2(a16[m][cc][t]);
                acc[m][cc][t] = fmaf(f.x + f.y, s, acc[m][cc][t]);
            }
        }
    }
}

template <int PHASE>
__global__ void __launch_bounds__(kMxThreads, 1)
    ffn_mx_tma_kernel(FfnParams p, MxCfg c, const __grid_constant__ CUtensorMap blocks_map,
                      const __grid_constant__ CUtensorMap scales_map) {
    constexpr int NM = PHASE == kGU ? 2 : 1;
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t *full = reinterpret_cast<uint64_t *>(sm);
    uint64_t *empty = full + kMxStagesMax;
    uint64_t *rbar = empty + kMxStagesMax;  // [2] consumer barriers around the reduction
    MxHdr *hdr = reinterpret_cast<MxHdr *>(sm + 256);
    unsigned char *stage0 = sm + 256 + kMxStagesMax * sizeof(MxHdr);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H, I = p.I;
    const int K2 = (PHASE == kGU ? H : I) / 2;  // k-pair rows
    const int nout = PHASE == kGU ? I : H;

    if (threadIdx.x == 0) {
        for (int s = 0; s < c.stages; s++) {
            bar_init(&full[s], 1);
            bar_init(&empty[s], kCW);
        }
        bar_init(&rbar[0], kCW);
        bar_init(&rbar[1], kCW);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (PHASE == kGU) asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" :::);

    if (warp == kCW) {  // producer
        if (lane != 0) return;
        const int nu = *p.s.n_unique;
        const int npass = nu > 0 ? *p.s.n_passes : 0;
        const int items = npass * c.tiles;
        const int first = (int)((int64_t)blockIdx.x * items / gridDim.x);
        const int last = (int)((int64_t)(blockIdx.x + 1) * items / gridDim.x);
        bool waited = PHASE == kGU, ok = true;
        int issued = 0;
        const uint32_t box_bytes = NM * (kKp * kCols + (kKp / 16) * kCols);
        int u = items > first ? pass_owner(p.s.upoff, nu, first / c.tiles) : 0;
        int cur_pi = -1, slot = 0, cnt = 0;
        int pairs_c[kMxTokMax], texp_c[kMxTokMax];
        for (int it = first; it < last && ok; it++) {
            const int pi = it / c.tiles, tile = it - pi * c.tiles;
            if (pi != cur_pi) {  // new pass: advance the owner and cache its tokens
                while (u + 1 < nu && p.s.upoff[u + 1] <= pi) u++;
                cur_pi = pi;
                slot = p.s.uslot[u];
                slot = slot < 0 ? 0 : (slot >= p.S ? p.S - 1 : slot);
                const int pbase = (pi - p.s.upoff[u]) * kPassTokens;
                cnt = p.s.ucnt[u] - pbase < kPassTokens ? p.s.ucnt[u] - pbase : kPassTokens;
                const int off = p.s.uoff[u] + pbase;
                if (!waited) {  // h rows and their maxima come from gate_up
                    asm volatile("griddepcontrol.wait;" ::: "memory");
                    waited = true;
                }
                for (int i = 0; i < kMxTokMax; i++) {
                    if (i >= cnt) break;
                    const int q = p.s.upairs[off + i];
                    pairs_c[i] = q;
                    int e = 0;
                    if (PHASE == kGU) {
                        e = p.s.xexp[q / p.topk];
                    } else {
                        const float mh = __uint_as_float(p.s.hmax[q]);
                        if (mh > 0.f && mh < INFINITY) {
                            frexpf(mh, &e);
                            e -= 9;
                        }
                    }
                    texp_c[i] = e;
                }
            }
            const int n0 = tile * kCols;
            {
                const int ntok = cnt;
                for (int ks = 0; ks < c.kst && ok; ks++) {
                    const int s = issued % c.stages;
                    if (!bar_wait(&empty[s], ((issued / c.stages) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    MxHdr &hh = hdr[s];
                    const int rows = K2 - ks * kKp < kKp ? K2 - ks * kKp : kKp;
                    hh.slot = slot; hh.n0 = n0; hh.kstage = ks; hh.rows = rows; hh.ntok = ntok;
                    hh.last = ks == c.kst - 1; hh.done = 0;
                    for (int i = 0; i < kMxTokMax; i++) {
                        if (i >= ntok) break;
                        hh.pairs[i] = pairs_c[i];
                        hh.texp[i] = texp_c[i];
                    }
                    const uint32_t tb = (uint32_t)rows * (PHASE == kGU ? 4u : 8u);
                    bar_expect(&full[s], box_bytes + (uint32_t)ntok * tb);
                    unsigned char *st = stage0 + (size_t)s * c.stage_bytes;
                    // rows past the slot's last k-pair row are zero-filled by the copy, not read
                    for (int m = 0; m < NM; m++) {
                        const int x = n0 + (m ? I : 0);
                        tma3d(st + m * kKp * kCols, &blocks_map, x, ks * kKp, slot, &full[s]);
                        tma3d(st + c.sc_off + m * (kKp / 16) * kCols, &scales_map, x, ks * (kKp / 16), slot, &full[s]);
                    }
                    for (int i = 0; i < ntok; i++) {
                        const int q = hh.pairs[i];
                        const void *src = PHASE == kGU
                                              ? static_cast<const void *>(p.s.x16 + (int64_t)(q / p.topk) * H +
                                                                          2 * ks * kKp)
                                              : static_cast<const void *>(p.s.h + (int64_t)q * I + 2 * ks * kKp);
                        bulk1d(st + c.tok_off + i * c.tok_bytes, src, tb, &full[s]);
                    }
                    issued++;
                }
            }
        }
        if (ok) {
            const int s = issued % c.stages;
            if (bar_wait(&empty[s], ((issued / c.stages) & 1) ^ 1)) {
                hdr[s].done = 1;
                bar_arrive(&full[s]);
            } else {
                ok = false;
            }
        }
        if (!ok) {
            atomicCAS(p.status, 0, FTMOE_ERR_STATE);
            for (int j = issued - c.stages < 0 ? 0 : issued - c.stages; j < issued; j++)
                bar_wait(&full[j % c.stages], (j / c.stages) & 1);
        }
        return;
    }

    // consumers
    float acc[NM][4][kMxTokMax];
#pragma unroll
    for (int m = 0; m < NM; m++)
#pragma unroll
        for (int cc = 0; cc < 4; cc++)
#pragma unroll
            for (int t = 0; t < kMxTokMax; t++) acc[m][cc][t] = 0.f;
    uint32_t rphase = 0;
    for (int k = 0;; k++) {
        const int s = k % c.stages;
        if (!bar_wait(&full[s], (k / c.stages) & 1)) {
            if (lane == 0) atomicCAS(p.status, 0, FTMOE_ERR_STATE);
            return;
        }
        const MxHdr &hs = hdr[s];  // stays valid until this warp releases the stage
        if (hs.done) return;
        const int ntok = hs.ntok, rows = hs.rows;
        const bool last = hs.last;
        const unsigned char *st = stage0 + (size_t)s * c.stage_bytes;
        float hsc[kMxTokMax];
#pragma unroll
        for (int t = 0; t < kMxTokMax; t++) hsc[t] = t < ntok ? ldexpf(1.f, -hs.texp[t]) : 0.f;
        if (warp * 16 < rows) {
            switch (ntok) {
                case 1: mx_block<NM, 1, PHASE == kDN>(st, c, warp, acc, hsc); break;
                case 2: mx_block<NM, 2, PHASE == kDN>(st, c, warp, acc, hsc); break;
                case 3: mx_block<NM, 3, PHASE == kDN>(st, c, warp, acc, hsc); break;
                default: mx_block<NM, 4, PHASE == kDN>(st, c, warp, acc, hsc); break;
            }
        }
        if (!last) {
            __syncwarp();
            if (lane == 0) bar_arrive(&empty[s]);
            continue;
        }

        // item end: the warps' partial sums meet in shared memory. Each warp writes its
        // partials [t][kCols] over its own 16-row code block of each matrix in this stage
        // (16 x 128 bytes = kMxTokMax x kCols floats), which no other warp reads. The
        // stage (and its header) is released afterwards.
#pragma unroll
        for (int m = 0; m < NM; m++)
#pragma unroll
            for (int t = 0; t < kMxTokMax; t++) {
                if (t < ntok) {
                    float4 v = make_float4(acc[m][0][t], acc[m][1][t], acc[m][2][t], acc[m][3][t]);
                    float *red = reinterpret_cast<float *>(const_cast<unsigned char *>(st) + m * kKp * kCols +
                                                           warp * 16 * kCols);
                    reinterpret_cast<float4 *>(red + t * kCols)[lane] = v;
                }
#pragma unroll
                for (int cc = 0; cc < 4; cc++) acc[m][cc][t] = 0.f;
            }
        __syncwarp();
        if (lane == 0) bar_arrive(&rbar[0]);
        if (!bar_wait(&rbar[0], rphase)) {
            if (lane == 0) atomicCAS(p.status, 0, FTMOE_ERR_STATE);
            return;
        }
        const int bi = PHASE == kGU ? 2 : 5;
        const uint16_t *bias = reinterpret_cast<const uint16_t *>(p.bank[bi] + (int64_t)hs.slot * p.bank_bytes[bi]);
        const int n0 = hs.n0;
        // ntok * kCols and the stride are multiples of 32, so a warp's 32 threads share
        // one token t here and take the max |h| over their columns before a single
        // atomic (every column doing its own atomic on the pair's word serialised on
        // one L2 slice)
        for (int i = threadIdx.x; i < ntok * kCols; i += kCW * 32) {
            const int t = i / kCols, col = i - t * kCols;
            const int n = n0 + col;
            const bool valid = n < nout;
            const float xs_t = ldexpf(1.f, hs.texp[t]);
            float v[NM];
#pragma unroll
            for (int m = 0; m < NM; m++) {
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kCW; w++)
                    sum += reinterpret_cast<const float *>(st + m * kKp * kCols + w * 16 * kCols)[t * kCols + col];
                v[m] = sum * xs_t;
            }
            const int q = hs.pairs[t];
            if (PHASE == kGU) {
                float hv = 0.f;
                if (valid) {
                    const float g = v[0] + __uint_as_float((uint32_t)bias[n] << 16);
                    const float uu = v[NM - 1] + __uint_as_float((uint32_t)bias[I + n] << 16);
                    hv = silu(g) * uu;
                    p.s.h[(int64_t)q * I + n] = hv;
                }
                const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv)));
                if (lane == 0 && wm) atomicMax(&p.s.hmax[q], wm);
            } else if (valid) {
                p.s.o[(int64_t)q * H + n] = v[0] + __uint_as_float((uint32_t)bias[n] << 16);
            }
        }
        __syncwarp();
        if (lane == 0) {
            bar_arrive(&rbar[1]);
            bar_arrive(&empty[s]);
        }
        if (!bar_wait(&rbar[1], rphase)) {
            if (lane == 0) atomicCAS(p.status, 0, FTMOE_ERR_STATE);
            return;
        }
        rphase ^= 1;
    }
}

bool make_mx_cfg(const FfnParams &p, int phase, MxCfg &c, size_t &smem) {
    const int K2 = (phase == kGU ? p.H : p.I) / 2;
    const int nout = phase == kGU ? p.I : p.H;
    const int NM = phase == kGU ? 2 : 1;
    c.tiles = (nout + kCols - 1) / kCols;
    c.kst = (K2 + kKp - 1) / kKp;
    c.tg = kMxTokMax;
    c.tok_bytes = kKp * (phase == kGU ? 4 : 8);
    c.sc_off = NM * kKp * kCols;
    c.tok_off = c.sc_off + NM * (kKp / 16) * kCols;
    c.stage_bytes = (c.tok_off + c.tg * c.tok_bytes + 127) & ~127;
    const size_t head = 256 + kMxStagesMax * sizeof(MxHdr);
    const size_t cap = 226 * 1024;
    int stages = kMxStagesMax;
    while (stages >= 2 && head + (size_t)stages * c.stage_bytes > cap) stages--;
    if (stages < 2) return false;
    c.stages = stages;
    smem = head + (size_t)stages * c.stage_bytes;
    return true;
}

template <int PHASE>
cudaError_t launch_mx(const FfnParams &p, const MxTmaMaps &maps, int num_sms, cudaStream_t st) {
    MxCfg c;
    size_t smem;
    if (!make_mx_cfg(p, PHASE, c, smem)) return cudaErrorInvalidValue;
    auto kern = ffn_mx_tma_kernel<PHASE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kMxThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const CUtensorMap *bm = reinterpret_cast<const CUtensorMap *>(PHASE == kGU ? maps.gu_blocks : maps.dn_blocks);
    const CUtensorMap *sm = reinterpret_cast<const CUtensorMap *>(PHASE == kGU ? maps.gu_scales : maps.dn_scales);
    return cudaLaunchKernelEx(&cfg, kern, p, c, *bm, *sm);
}

}  // namespace

bool ffn_mx_tma_supported(const FfnParams &p, const MxTmaMaps *maps) {
    return maps && maps->valid && p.fmt == FTMOE_FMT_MXFP4 && p.s.x16 && p.s.xexp && p.s.hmax && p.s.upoff &&
           p.s.n_passes &&
           p.H % 32 == 0 && p.I % 32 == 0;
}

cudaError_t launch_ffn_mx_tma(const FfnParams &p, const MxTmaMaps &maps, int num_sms, cudaStream_t st) {
    cudaError_t e = launch_mx<kGU>(p, maps, num_sms, st);
    if (e != cudaSuccess) return e;
    return launch_mx<kDN>(p, maps, num_sms, st);
}

// ---------------------------------------------------------------- tensor maps

namespace {
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
    static EncodeFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(f);
        else
            cudaGetLastError();
    }
    return fn;
}

// 3-D u8 map over [slots, rows, cols] bytes (one slot's rows contiguous, slots at a stride
// of rows * cols) with a box of 128 columns x box_rows rows x 1 slot. Rows past a slot's
// last row fall outside the map, so a ragged last box is zero-filled instead of reading
// the next slot.
bool encode_u8(void *out, const void *base, uint64_t cols, uint64_t rows, uint64_t slots, uint32_t box_rows) {
    EncodeFn fn = encode_fn();
    if (!fn || cols % 16 || ((uintptr_t)base % 16)) return false;
    const cuuint64_t dims[3] = {cols, rows, slots};
    const cuuint64_t strides[2] = {cols, cols * rows};
    const cuuint32_t box[3] = {(cuuint32_t)kCols, box_rows, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(reinterpret_cast<CUtensorMap *>(out), CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims,
              strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool make_mx_tma_maps(MxTmaMaps &m, const unsigned char *const *banks, int S, int H, int I) {
    static_assert(sizeof(CUtensorMap) <= sizeof(m.gu_blocks), "tensor map storage");
    m.valid = false;
    if (H % 32 || I % 32) return false;
    const uint64_t ngu = 2ull * I, ndn = (uint64_t)H;
    bool ok = encode_u8(m.gu_blocks, banks[0], ngu, (uint64_t)(H / 2), (uint64_t)S, kKp) &&
              encode_u8(m.gu_scales, banks[1], ngu, (uint64_t)(H / 32), (uint64_t)S, kKp / 16) &&
              encode_u8(m.dn_blocks, banks[3], ndn, (uint64_t)(I / 2), (uint64_t)S, kKp) &&
              encode_u8(m.dn_scales, banks[4], ndn, (uint64_t)(I / 32), (uint64_t)S, kKp / 16);
    m.valid = ok;
    return ok;
}

}  // namespace ftmoe
