// Output-row-major expert FFN phases on the tensor cores (block FP8 and bf16), as a
// persistent, warp-specialised bulk-tensor (TMA) pipeline.
//
// Block-FP8 banks (architecture deep-dive, section 五 lists "FP8 block" among the bank
// schemas; read here as) hold e4m3 weights [N, K] output-row-major and one binary32
// scale per 128 x 128 block ([N/128, K/128]); w = e4m3 * scale. bf16 banks (benchmark
// guide, section 4.2: gate_up and down) hold bf16 weights [N, K] output-row-major. A work
// item is (distinct slot u, pass of up to eight tokens, tile of 64 output rows); it
// streams the reduction axis in stages of 512 weight bytes per row (512 k of e4m3, 256 k
// of bf16). A producer thread loads each stage with 3-D tensor copies (cp.async.bulk.tensor
// over [slot, row, k byte], four boxes of 128 bytes x 64 rows per matrix, stored with the
// 128-byte shared-memory swizzle), 1-D bulk copies of the item's block-scale row per
// matrix (block FP8: a 64-row tile lies inside one 128-row block) and of the tokens'
// activations for the stage's k, all completing on the stage's mbarrier.
//
// Work split: items are dealt round-robin over the CTAs (item i to CTA i mod grid), so the
// passes of one hot expert run side by side and share L2. When a call has fewer items
// than SMs (batch 1) the idle SMs start the down kernel's weight stream early (the
// kernels are chained with programmatic dependent launch), which is why the items are not
// split further.
//
// The contraction runs on mma.sync m16n8k16 with fp32 accumulators: M = 16 output rows,
// N = 8 tokens, K = 16. Consumer warp w takes M tile w % 4 (rows 16 (w % 4) ..) and box
// w / 4 of every stage (block-FP8 down: k sixteenth w of the stage over all four M tiles, so
// the h pairs are converted to f16 once per stage).
//   block FP8 (f16 x f16): lane (g, tig) reads the 32-bit word at k = 4 tig of rows g and
//   g + 8 of the k step; with cvt.rn.f16x2.e4m3x2 (exact) its low half gives the fragment
//   registers of logical k (2 tig, 2 tig + 1) and its high half those of (2 tig + 8,
//   2 tig + 9), and the B fragment is the token's activations at the same four k (one
//   64-bit load). With the swizzle a warp's 32 weight loads hit 32 distinct banks. A warp's
//   k steps (one 128-k box = one scale block) are summed from zero on the tensor cores,
//   then multiplied by the block scale in fp32 and added to the item's accumulator.
//   bf16 (bf16 x bf16): the A fragment is one ldmatrix.x4 of the 16 x 16 tile (eight
//   16-byte rows per matrix, eight distinct bank groups under the swizzle); the B fragment
//   is the token's bf16 activations at k (2 tig, 2 tig + 1) and (2 tig + 8, 2 tig + 9).
// After the last stage of an item the warps' partials meet in shared memory behind an
// mbarrier (bounded wait); gate_up writes h = silu(g) * u, down writes o.
//
// Activations. Block FP8: gate_up uses the f16 copy of x (per-token power-of-two scale);
// down converts the fp32 h rows to f16 with the per-pair power-of-two scale from max |h|
// (gate_up records it, one atomic per warp). bf16: gate_up uses x itself; gate_up stores
// each h value as two bf16 terms, hi = bf16(h) and lo = bf16(h - hi) (hi + lo carries 16
// significant bits), in the pair's h row (hi in its first 2I bytes, lo in the next 2I), and
// down runs one MMA per term into the same accumulator, so every product is exact and all
// sums are fp32.
#include <cuda.h>

#include "ffn_common.cuh"
#include "internal.cuh"
#include "pipeline.cuh"

namespace ftmoe {
namespace {

using namespace ffn;
using namespace pipe;

enum { kWE4M3 = 0, kWBF16 = 1 };  // weight kinds

constexpr int kFCW = 16;                      // consumer warps
constexpr int kFThreads = (kFCW + 1) * 32;    // + producer warp
constexpr int kFRows = 64;                    // output rows per item (four M tiles)
constexpr int kFBox = 128;                    // weight bytes per box row (one 128-byte line)
constexpr int kFStageBytes = 512;             // weight bytes per row and stage (four boxes)
// k per stage: 512 e4m3 or 256 bf16. Consumer warp w takes box w / 4, so a block-FP8 warp
// covers 128 k (exactly one scale block) and a bf16 warp 64 k.
template <int WK>
constexpr int kfks() { return WK == kWE4M3 ? 512 : 256; }
constexpr int kRedStride = kFRows + 4;        // padded row of the reduction buffer
constexpr int kFStagesMax = 4;
constexpr int kFTok = 8;                      // tokens per pass = the MMA's N
static_assert(kFTok == kMxPassTokens, "the routing kernel cuts passes of kFTok tokens");
static_assert(kFCW == 16, "four M tiles x four boxes");
static_assert(kFTok * kFRows <= kFCW * 32, "one epilogue output per consumer thread at most");

enum { kGU = 0, kDN = 1 };

struct F8Hdr {
    int32_t slot, n0, kstage, ntok, last, done, pad0, pad1;
    int32_t pairs[kFTok];
    int32_t texp[kFTok];
};

// Stage layout (1024-byte aligned): weights [NM][4 boxes][kFRows][128 B] (swizzled),
// block-scale rows [NM][KB] f32 at sc_off (block FP8), tokens [planes][tg] at tok_off with a
// padded stride (bf16 down: planes hi and lo, tok_plane bytes apart).
struct F8Cfg {
    int32_t tiles, kst, stages, stage_bytes, sc_off, sc_bytes, tok_off, tok_stride, tok_plane, red_off;
};

__device__ __forceinline__ int swz(int row, int byte) { return row * kFBox + (byte ^ ((row & 7) << 4)); }

// Two e4m3 codes (low byte first) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_h2(uint32_t two) { return e4m3x2_to_h2(two); }

// Block-FP8 gate_up: box kq of the stage (128 k, one scale block) for M tile mt of both
// matrices; the B fragment is the token's f16 activations.
template <int NM>
__device__ __forceinline__ void f8_stage_mma(const unsigned char *st, const F8Cfg &c, int mt, int kq, int ntok,
                                             int kb_first, float (&acc)[NM][4]) {
    constexpr int KS = kfks<kWE4M3>();
    constexpr int KW = KS / 4;  // k of this warp in the stage: one 128-k scale block
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    const unsigned char *tokp = st + c.tok_off + g * c.tok_stride;
    const int box = (kq * KW) / kFBox, inbox = (kq * KW) % kFBox;
    float tmp[NM][4];
#pragma unroll
    for (int ks = 0; ks < KW / 16; ks++) {
        const int kk = kq * KW + ks * 16;      // k of this step inside the stage
        const int byte = inbox + 16 * ks + 4 * tig;  // inside the 128-byte box row
        uint32_t b0 = 0u, b1 = 0u;
        if (g < ntok) {
            const uint2 xv = *reinterpret_cast<const uint2 *>(tokp + 2 * (kk + 4 * tig));
            b0 = xv.x;
            b1 = xv.y;
        }
#pragma unroll
        for (int m = 0; m < NM; m++) {
            const unsigned char *tile = st + (m * (KS / kFBox) + box) * (kFRows * kFBox);
            const uint32_t wA = *reinterpret_cast<const uint32_t *>(tile + swz(16 * mt + g, byte));
            const uint32_t wB = *reinterpret_cast<const uint32_t *>(tile + swz(16 * mt + g + 8, byte));
            const uint32_t a0 = e4m3x2_h2(wA & 0xffffu), a2 = e4m3x2_h2(wA >> 16);
            const uint32_t a1 = e4m3x2_h2(wB & 0xffffu), a3 = e4m3x2_h2(wB >> 16);
            if (ks == 0)
                mma_f16_16816_z(tmp[m], a0, a1, a2, a3, b0, b1);
            else
                mma_f16_16816(tmp[m], a0, a1, a2, a3, b0, b1);
        }
    }
    // the warp's k steps lie in one 128 x 128 block: one binary32 scale per matrix
#pragma unroll
    for (int m = 0; m < NM; m++) {
        const float s = reinterpret_cast<const float *>(st + c.sc_off + m * c.sc_bytes)[kb_first + box];
        ffma2_s(acc[m][0], acc[m][1], tmp[m][0], tmp[m][1], s);
        ffma2_s(acc[m][2], acc[m][3], tmp[m][2], tmp[m][3], s);
    }
}

// Block-FP8 down: warp kp takes k [32 kp, 32 kp + 32) of the stage (two k steps, inside one
// 128-k scale block) for all four M tiles, so the fp32 -> f16 conversion of each token's h
// pair is done once per stage instead of once per M tile.
__device__ __forceinline__ void f8_stage_mma_kp16(const unsigned char *st, const F8Cfg &c, int kp, int ntok,
                                                  float tok_scale, int kb_first, float (&acc)[4][4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    const unsigned char *tokp = st + c.tok_off + g * c.tok_stride;
    const int box = kp >> 2, inbox = 32 * (kp & 3);
    const unsigned char *tile = st + box * (kFRows * kFBox);
    float tmp[4][4];
#pragma unroll
    for (int ks = 0; ks < 2; ks++) {
        const int kk = 32 * kp + 16 * ks;            // k of this step inside the stage
        const int byte = inbox + 16 * ks + 4 * tig;  // inside the 128-byte box row
        uint32_t b0 = 0u, b1 = 0u;
        if (g < ntok) {
            const float4 hv = *reinterpret_cast<const float4 *>(tokp + 4 * (kk + 4 * tig));
            b0 = f2_scale_to_h2(hv.x, hv.y, tok_scale);
            b1 = f2_scale_to_h2(hv.z, hv.w, tok_scale);
        }
#pragma unroll
        for (int mt = 0; mt < 4; mt++) {
            const uint32_t wA = *reinterpret_cast<const uint32_t *>(tile + swz(16 * mt + g, byte));
            const uint32_t wB = *reinterpret_cast<const uint32_t *>(tile + swz(16 * mt + g + 8, byte));
            const uint32_t a0 = e4m3x2_h2(wA & 0xffffu), a2 = e4m3x2_h2(wA >> 16);
            const uint32_t a1 = e4m3x2_h2(wB & 0xffffu), a3 = e4m3x2_h2(wB >> 16);
            if (ks == 0)
                mma_f16_16816_z(tmp[mt], a0, a1, a2, a3, b0, b1);
            else
                mma_f16_16816(tmp[mt], a0, a1, a2, a3, b0, b1);
        }
    }
    const float s = reinterpret_cast<const float *>(st + c.sc_off)[kb_first + box];
#pragma unroll
    for (int mt = 0; mt < 4; mt++) {
        ffma2_s(acc[mt][0], acc[mt][1], tmp[mt][0], tmp[mt][1], s);
        ffma2_s(acc[mt][2], acc[mt][3], tmp[mt][2], tmp[mt][3], s);
    }
}

// bf16: box kq of the stage (64 k in four k steps) for M tile mt of every matrix. Down runs
// the hi and the lo term of h through the same A fragment.
template <int NM, bool DOWN>
__device__ __forceinline__ void bf_stage_mma(const unsigned char *st, const F8Cfg &c, int mt, int kq, int ntok,
                                             float (&acc)[NM][4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    const unsigned char *tokp = st + c.tok_off + g * c.tok_stride;
    // ldmatrix row of this lane: matrices (rows 0-7 | 8-15) x (k 0-7 | 8-15) of the M tile
    const int lrow = 16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1);
    const int lbyte = 16 * (lane >> 4);
#pragma unroll
    for (int ks = 0; ks < 4; ks++) {
        const int kb = 2 * (64 * kq + 16 * ks + 2 * tig);  // byte of k (2 tig) of this step
        uint32_t b0 = 0u, b1 = 0u, l0 = 0u, l1 = 0u;
        if (g < ntok) {
            b0 = *reinterpret_cast<const uint32_t *>(tokp + kb);
            b1 = *reinterpret_cast<const uint32_t *>(tokp + kb + 16);
            if (DOWN) {
                l0 = *reinterpret_cast<const uint32_t *>(tokp + c.tok_plane + kb);
                l1 = *reinterpret_cast<const uint32_t *>(tokp + c.tok_plane + kb + 16);
            }
        }
#pragma unroll
        for (int m = 0; m < NM; m++) {
            const unsigned char *tile = st + (m * 4 + kq) * (kFRows * kFBox);
            uint32_t a[4];
            ldsm_x4(a, tile + swz(lrow, 32 * ks + lbyte));
            mma_bf16_16816(acc[m], a[0], a[1], a[2], a[3], b0, b1);
            if (DOWN) mma_bf16_16816(acc[m], a[0], a[1], a[2], a[3], l0, l1);
        }
    }
}

// hi = bf16(v), lo = bf16(v - hi): the two terms of one h value.
__device__ __forceinline__ void split_bf16(float v, uint16_t &hi, uint16_t &lo) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    hi = __bfloat16_as_ushort(h);
    lo = __bfloat16_as_ushort(__float2bfloat16_rn(v - __bfloat162float(h)));
}

// Final values v[NM] (gate and up, or down) of output row n for routed pair q: gate_up
// stores h (and, block FP8, the pair's max |h| with one atomic per warp; all 32 lanes of the
// warp take part), down stores o.
template <int WK, int PHASE, int NM>
__device__ __forceinline__ void rows_mma_store(const FfnParams &p, int q, int n, const float (&v)[NM], int lane) {
    const int nout = PHASE == kGU ? p.I : p.H;
    if (PHASE == kGU) {
        const float hv = n < nout ? silu(v[0]) * v[NM - 1] : 0.f;
        if (WK == kWE4M3) {
            if (n < nout) p.s.h[(int64_t)q * p.I + n] = hv;
            const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv)));
            if (lane == 0 && wm) atomicMax(&p.s.hmax[q], wm);
        } else if (n < nout) {
            uint16_t hi, lo;
            split_bf16(hv, hi, lo);
            uint16_t *hr = reinterpret_cast<uint16_t *>(p.s.h + (int64_t)q * p.I);
            hr[n] = hi;
            hr[p.I + n] = lo;
        }
    } else if (n < nout) {
        p.s.o[(int64_t)q * p.H + n] = v[0];
    }
}

template <int WK, int PHASE>
__device__ __forceinline__ void rows_mma_body(const FfnParams &p, const F8Cfg &c, const CUtensorMap *wmap) {
    constexpr int NM = PHASE == kGU ? 2 : 1;
    constexpr int kFKs = kfks<WK>();
    constexpr int kEs = WK == kWE4M3 ? 1 : 2;  // weight bytes per element
    extern __shared__ __align__(1024) unsigned char sm[];
    uint64_t *full = reinterpret_cast<uint64_t *>(sm);
    uint64_t *empty = full + kFStagesMax;
    uint64_t *rbar = empty + kFStagesMax;  // [2] consumer barriers around the reduction
    F8Hdr *hdr = reinterpret_cast<F8Hdr *>(sm + 256);
    const uint32_t hdr_end = su32(sm) + 256 + kFStagesMax * sizeof(F8Hdr);
    unsigned char *stage0 = sm + (((hdr_end + 1023u) & ~1023u) - su32(sm));
    float *red = reinterpret_cast<float *>(stage0 + c.red_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H, I = p.I;
    const int K = PHASE == kGU ? H : I;
    const int KB = K / 128;  // block-FP8 scale blocks along k

    if (threadIdx.x == 0) {
        for (int s = 0; s < c.stages; s++) {
            bar_init(&full[s], 1);
            bar_init(&empty[s], kFCW);
        }
        bar_init(&rbar[0], kFCW);
        bar_init(&rbar[1], kFCW);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (PHASE == kGU) asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" :::);

    if (warp == kFCW) {  // producer
        if (lane != 0) return;
        const int nu = *p.s.n_unique;
        const int npass = nu > 0 ? *p.s.n_passes : 0;
        const int items = npass * c.tiles;
        // items dealt round-robin: the passes of one expert run side by side and share L2
        const int first = blockIdx.x;
        bool waited = PHASE == kGU, ok = true;
        int issued = 0;
        const uint64_t pol = evict_first_l2();  // weights are read once
        const uint32_t box_bytes = NM * (kFStageBytes / kFBox) * kFRows * kFBox;
        // token bytes per stage and plane: f16 x / fp32 h (block FP8), bf16 x / h terms (bf16)
        const uint32_t tb = WK == kWE4M3 ? kFKs * (PHASE == kGU ? 2u : 4u) : kFKs * 2u;
        const int planes = WK == kWBF16 && PHASE == kDN ? 2 : 1;
        int u = items > first ? pass_owner(p.s.upoff, nu, first / c.tiles) : 0;
        int cur_pi = -1, slot = 0, cnt = 0;
        int pairs_c[kFTok], texp_c[kFTok];
        const unsigned char *scb = WK == kWE4M3 ? p.bank[PHASE == kGU ? 1 : 3] : nullptr;
        const int64_t scb_bytes = WK == kWE4M3 ? p.bank_bytes[PHASE == kGU ? 1 : 3] : 0;
        for (int it = first; it < items && ok; it += gridDim.x) {
            const int pi = it / c.tiles, tile = it - pi * c.tiles;
            if (pi != cur_pi) {  // new pass: advance the owner and cache its tokens
                while (u + 1 < nu && p.s.upoff[u + 1] <= pi) u++;
                cur_pi = pi;
                slot = p.s.uslot[u];
                FTMOE_DCHECK(slot >= 0 && slot < p.S, p.status);
                slot = slot < 0 ? 0 : (slot >= p.S ? p.S - 1 : slot);
                const int pbase = (pi - p.s.upoff[u]) * kFTok;
                cnt = p.s.ucnt[u] - pbase < kFTok ? p.s.ucnt[u] - pbase : kFTok;
                const int off = p.s.uoff[u] + pbase;
                if (!waited) {  // h rows (and their maxima) come from gate_up
                    asm volatile("griddepcontrol.wait;" ::: "memory");
                    waited = true;
                }
                for (int i = 0; i < kFTok; i++) {
                    if (i >= cnt) break;
                    const int q = p.s.upairs[off + i];
                    pairs_c[i] = q;
                    int e = 0;
                    if (WK == kWE4M3) {
                        if (PHASE == kGU) {
                            e = p.s.xexp[q / p.topk];
                        } else {
                            const float mh = __uint_as_float(p.s.hmax[q]);
                            if (mh > 0.f && mh < INFINITY) {
                                frexpf(mh, &e);
                                e -= 10;
                            }
                        }
                    }
                    texp_c[i] = e;
                }
            }
            const int n0 = tile * kFRows;
            for (int ks = 0; ks < c.kst && ok; ks++) {
                const int s = issued % c.stages;
                if (!bar_wait(&empty[s], ((issued / c.stages) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                F8Hdr &hh = hdr[s];
                hh.slot = slot; hh.n0 = n0; hh.kstage = ks; hh.ntok = cnt;
                hh.last = ks == c.kst - 1; hh.done = 0;
                for (int i = 0; i < kFTok; i++) {
                    if (i >= cnt) break;
                    hh.pairs[i] = pairs_c[i];
                    hh.texp[i] = texp_c[i];
                }
                bar_expect(&full[s], box_bytes + (uint32_t)(NM * c.sc_bytes) + (uint32_t)(cnt * planes) * tb);
                unsigned char *st = stage0 + (size_t)s * c.stage_bytes;
                const int k0 = ks * kFKs;
                for (int m = 0; m < NM; m++) {
                    const int row = n0 + (m ? I : 0);
                    for (int bx = 0; bx < kFStageBytes / kFBox; bx++)
                        tma3d_hint(st + (m * (kFStageBytes / kFBox) + bx) * (kFRows * kFBox), wmap,
                                   k0 * kEs + bx * kFBox, row, slot, &full[s], pol);
                    if (WK == kWE4M3)  // the 64-row tile lies in one 128-row block: its scale row
                        bulk1d(st + c.sc_off + m * c.sc_bytes,
                               scb + (int64_t)slot * scb_bytes + (int64_t)(row / 128) * KB * 4, (uint32_t)c.sc_bytes,
                               &full[s]);
                }
                for (int i = 0; i < cnt; i++) {
                    const int q = hh.pairs[i];
                    unsigned char *dst = st + c.tok_off + i * c.tok_stride;
                    if (PHASE == kGU) {
                        const uint16_t *xs = WK == kWE4M3 ? p.s.x16 : p.x;
                        bulk1d(dst, xs + (int64_t)(q / p.topk) * H + k0, tb, &full[s]);
                    } else if (WK == kWE4M3) {
                        bulk1d(dst, p.s.h + (int64_t)q * I + k0, tb, &full[s]);
                    } else {  // the pair's h row holds the hi terms, then the lo terms
                        const uint16_t *hr = reinterpret_cast<const uint16_t *>(p.s.h + (int64_t)q * I);
                        bulk1d(dst, hr + k0, tb, &full[s]);
                        bulk1d(dst + c.tok_plane, hr + I + k0, tb, &full[s]);
                    }
                }
                issued++;
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

    // consumers: warp = (M tile mt, box kq); block-FP8 down: warp = sixteenth kp of the
    // stage's k over all four M tiles (acc[a]: matrix a, or M tile a for block-FP8 down)
    constexpr bool KP16 = WK == kWE4M3 && PHASE == kDN;
    constexpr int NA = KP16 ? 4 : NM, NPART = KP16 ? 16 : 4;
    const int mt = warp & 3, kq = warp >> 2;
    const int g = lane >> 2, tig = lane & 3;
    float acc[NA][4];
#pragma unroll
    for (int m = 0; m < NA; m++)
#pragma unroll
        for (int i = 0; i < 4; i++) acc[m][i] = 0.f;
    uint32_t rphase = 0;
    for (int k = 0;; k++) {
        const int s = k % c.stages;
        if (!bar_wait(&full[s], (k / c.stages) & 1)) {
            if (lane == 0) atomicCAS(p.status, 0, FTMOE_ERR_STATE);
            return;
        }
        const F8Hdr &hs = hdr[s];  // stays valid until this warp releases the stage
        if (hs.done) return;
        const int ntok = hs.ntok;
        const bool last = hs.last;
        const unsigned char *st = stage0 + (size_t)s * c.stage_bytes;
        if constexpr (KP16) {
            const float tok_scale = g < ntok ? ldexpf(1.f, -hs.texp[g]) : 0.f;
            f8_stage_mma_kp16(st, c, warp, ntok, tok_scale, hs.kstage * (kFKs / 128), acc);
        } else if constexpr (WK == kWE4M3) {
            f8_stage_mma<NM>(st, c, mt, kq, ntok, hs.kstage * (kFKs / 128), acc);
        } else {
            bf_stage_mma<NM, PHASE == kDN>(st, c, mt, kq, ntok, acc);
        }
        if (!last) {
            __syncwarp();
            if (lane == 0) bar_arrive(&empty[s]);
            continue;
        }

        // item end: partials meet in red [NM][NPART][kFTok][kRedStride] (the padded row
        // keeps both the fragment stores and the row-wise sums free of bank conflicts)
#pragma unroll
        for (int a = 0; a < NA; a++) {
            const int m = KP16 ? 0 : a, part = KP16 ? warp : kq, mta = KP16 ? a : mt;
            float *r = red + ((m * NPART + part) * kFTok) * kRedStride;
            const int r0 = 16 * mta + g, t0 = 2 * tig;
            if (t0 < ntok) {
                r[t0 * kRedStride + r0] = acc[a][0];
                r[t0 * kRedStride + r0 + 8] = acc[a][2];
            }
            if (t0 + 1 < ntok) {
                r[(t0 + 1) * kRedStride + r0] = acc[a][1];
                r[(t0 + 1) * kRedStride + r0 + 8] = acc[a][3];
            }
#pragma unroll
            for (int i = 0; i < 4; i++) acc[a][i] = 0.f;
        }
        __syncwarp();
        if (lane == 0) bar_arrive(&rbar[0]);
        if (!bar_wait(&rbar[0], rphase)) {
            if (lane == 0) atomicCAS(p.status, 0, FTMOE_ERR_STATE);
            return;
        }
        // the epilogue needs only this thread's token from the header (ntok * kFRows <=
        // kFCW * 32, so every thread has at most one output), so the stage is released
        // now and the producer refills it while the outputs are formed
        const int n0 = hs.n0, i = threadIdx.x, t = i / kFRows, row = i - t * kFRows;
        const bool has = i < ntok * kFRows;  // whole warps: ntok * kFRows is a multiple of 32
        const int q_t = has ? hs.pairs[t] : 0, e_t = has ? hs.texp[t] : 0;
        __syncwarp();
        if (lane == 0) bar_arrive(&empty[s]);
        if (has) {
            const float xs_t = WK == kWE4M3 ? ldexpf(1.f, e_t) : 1.f;
            float v[NM];
#pragma unroll
            for (int m = 0; m < NM; m++) {
                float sum = 0.f;
#pragma unroll
                for (int q4 = 0; q4 < NPART; q4++) sum += red[((m * NPART + q4) * kFTok + t) * kRedStride + row];
                v[m] = sum * xs_t;
            }
            rows_mma_store<WK, PHASE, NM>(p, q_t, n0 + row, v, lane);
        }
        __syncwarp();
        if (lane == 0) bar_arrive(&rbar[1]);
        if (!bar_wait(&rbar[1], rphase)) {
            if (lane == 0) atomicCAS(p.status, 0, FTMOE_ERR_STATE);
            return;
        }
        rphase ^= 1;
    }
}

template <int PHASE>
__global__ void __launch_bounds__(kFThreads, 1)
    ffn_fp8_tma_kernel(FfnParams p, F8Cfg c, const __grid_constant__ CUtensorMap wmap) {
    rows_mma_body<kWE4M3, PHASE>(p, c, &wmap);
}

template <int PHASE>
__global__ void __launch_bounds__(kFThreads, 1)
    ffn_bf16_mma_kernel(FfnParams p, F8Cfg c, const __grid_constant__ CUtensorMap wmap) {
    rows_mma_body<kWBF16, PHASE>(p, c, &wmap);
}

bool make_f8_cfg(const FfnParams &p, int wk, int phase, F8Cfg &c, size_t &smem) {
    const int K = phase == kGU ? p.H : p.I;
    const int nout = phase == kGU ? p.I : p.H;
    const int NM = phase == kGU ? 2 : 1;
    const int kFKs = wk == kWE4M3 ? kfks<kWE4M3>() : kfks<kWBF16>();
    if (K % kFKs || nout % kFRows) return false;
    c.tiles = nout / kFRows;
    c.kst = K / kFKs;
    c.sc_bytes = wk == kWE4M3 ? (K / 128) * 4 : 0;  // one block-scale row (a multiple of 16 bytes)
    c.sc_off = NM * kFStageBytes * kFRows;
    // token rows, padded so that the eight tokens' B loads hit distinct banks: by 32 / 64
    // bytes for block FP8 (64-bit / 128-bit loads), by 16 bytes for bf16 (token g's 32-bit
    // words start at bank 4g)
    if (wk == kWE4M3)
        c.tok_stride = phase == kGU ? kFKs * 2 + 32 : kFKs * 4 + 64;
    else
        c.tok_stride = kFKs * 2 + 16;
    c.tok_plane = wk == kWBF16 && phase == kDN ? kFTok * c.tok_stride : 0;
    const int planes = c.tok_plane ? 2 : 1;
    c.tok_off = (c.sc_off + NM * c.sc_bytes + 15) & ~15;
    c.stage_bytes = (c.tok_off + planes * kFTok * c.tok_stride + 1023) & ~1023;
    const int npart = wk == kWE4M3 && phase == kDN ? 16 : 4;  // partial sums per output
    const size_t red = (size_t)NM * npart * kFTok * kRedStride * 4;
    const size_t head = 256 + kFStagesMax * sizeof(F8Hdr) + 1024;  // + alignment slack
    const size_t cap = 227 * 1024;
    int stages = kFStagesMax;
    while (stages >= 2 && head + (size_t)stages * c.stage_bytes + red > cap) stages--;
    if (stages < 2) return false;
    c.stages = stages;
    c.red_off = stages * c.stage_bytes;
    smem = head + (size_t)stages * c.stage_bytes + red;
    return true;
}

template <int WK, int PHASE>
cudaError_t launch_f8(const FfnParams &p, const MxTmaMaps &maps, int num_sms, cudaStream_t st) {
    F8Cfg c;
    size_t smem;
    if (!make_f8_cfg(p, WK, PHASE, c, smem)) return cudaErrorInvalidValue;
    auto kern = WK == kWE4M3 ? ffn_fp8_tma_kernel<PHASE> : ffn_bf16_mma_kernel<PHASE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const CUtensorMap *wm = reinterpret_cast<const CUtensorMap *>(PHASE == kGU ? maps.gu_blocks : maps.dn_blocks);
    return cudaLaunchKernelEx(&cfg, kern, p, c, *wm);
}

}  // namespace

bool ffn_fp8_tma_supported(const FfnParams &p, const MxTmaMaps *maps) {
    if (!maps || !maps->valid || p.fmt != FTMOE_FMT_FP8 || !p.s.x16 || !p.s.xexp || !p.s.hmax || !p.s.upoff ||
        !p.s.n_passes)
        return false;
    F8Cfg c;
    size_t smem;
    return make_f8_cfg(p, kWE4M3, kGU, c, smem) && make_f8_cfg(p, kWE4M3, kDN, c, smem);
}

cudaError_t launch_ffn_fp8_tma(const FfnParams &p, const MxTmaMaps &maps, int num_sms, cudaStream_t st) {
    cudaError_t e = launch_f8<kWE4M3, kGU>(p, maps, num_sms, st);
    if (e != cudaSuccess) return e;
    return launch_f8<kWE4M3, kDN>(p, maps, num_sms, st);
}

bool ffn_bf16_mma_supported(const FfnParams &p, const MxTmaMaps *maps) {
    if (!maps || !maps->valid || p.fmt != FTMOE_FMT_BF16 || !p.s.upoff || !p.s.n_passes) return false;
    F8Cfg c;
    size_t smem;
    return make_f8_cfg(p, kWBF16, kGU, c, smem) && make_f8_cfg(p, kWBF16, kDN, c, smem);
}

cudaError_t launch_ffn_bf16_mma(const FfnParams &p, const MxTmaMaps &maps, int num_sms, cudaStream_t st) {
    cudaError_t e = launch_f8<kWBF16, kGU>(p, maps, num_sms, st);
    if (e != cudaSuccess) return e;
    return launch_f8<kWBF16, kDN>(p, maps, num_sms, st);
}

}  // namespace ftmoe
