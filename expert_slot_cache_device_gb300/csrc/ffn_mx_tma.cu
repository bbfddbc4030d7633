// Transposed mxfp4 expert FFN phases as a persistent, warp-specialised bulk-tensor (TMA) pipeline.
//
// mxfp4 banks are stored transposed (benchmark guide, section 4.2: "_blocks /
// _scales / _bias"): blocks [K/2, N] (byte (i, n) holds k = 2i in the low nibble and
// k = 2i + 1 in the high nibble of output column n), scales [K/32, N] e8m0, bias [N].
// A work item is (distinct slot u, pass of up to eight tokens, tile of 128 output
// columns); it streams the whole reduction axis in stages of kKp = 256 k-pair rows. A
// producer thread loads each stage with 3-D bulk tensor copies (cp.async.bulk.tensor
// over [slot, row, column], one box of 128 columns x 256 rows per matrix stored with
// the 128-byte shared-memory swizzle, plus the 16 matching scale rows; completion on an
// mbarrier; rows past the slot's end are zero-filled) and a 1-D bulk copy of the
// tokens' activations for those rows.
//
// The contraction runs on the tensor cores with the warp-level mma.sync m16n8k16
// (f16 x f16 -> fp32): M = 16 output columns, N = 8 tokens, K = 16 (8 k-pair rows).
// Each consumer warp takes two 16-row scale blocks (32 k-pair rows) and one half of
// the 128 columns (four M tiles). A lane's A fragment is built directly from code bytes:
// one byte holds (k even, k odd) of one column, which is exactly an f16x2 register of
// the fragment after cvt.rn.f16x2.e2m1x2. The M index of a tile is a permutation of its
// columns (lane group g owns columns 4g..4g+3 of a 32-column group) and the k-pair rows
// of a k step are taken in the order 2*tig, 2*tig + 1, so every lane reads whole 32-bit
// words and, with the swizzle, the 32 lanes of a load hit 32 distinct banks. The B
// fragment of lane (g, tig) is token g's activation pairs of its two k-pair rows (one
// 64-bit load); tokens past the pass's count are zero. Each scale block is accumulated
// from zero on the tensor cores, multiplied by its e8m0 column scale in fp32 and added
// to the item's accumulator, so the block scale is exact. After the last stage of an
// item the warps' partials meet in a shared-memory buffer behind an mbarrier (bounded
// wait), the bias is added, and gate_up writes h = silu(g) * u while down writes o.
//
// Activations: gate_up uses the f16 copy of x (per-token power-of-two scale, max
// |x| < 2^9, so every bf16 value is exact in f16); down converts the fp32 h rows to
// f16 with the per-pair power-of-two scale derived from the max |h| recorded by gate_up.
#include <cuda.h>

#include "ffn_common.cuh"
#include "internal.cuh"
#include "pipeline.cuh"

namespace ftmoe {
namespace {

using namespace ffn;
using namespace pipe;

constexpr int kCW = 16;                     // consumer warps
constexpr int kMxThreads = (kCW + 1) * 32;  // + producer warp
constexpr int kKp = 256;                    // k-pair rows per stage (16 scale blocks of 16)
constexpr int kCols = 128;                  // output columns per item (one 128-byte box row)
constexpr int kMxStagesMax = 4;
constexpr int kMxTokMax = 8;                // tokens per pass = the MMA's N
constexpr int kBlkPairs = kKp / 32;         // consumer warps per column half
static_assert(kBlkPairs * 2 == kCW, "two column halves x eight pairs of scale blocks");
static_assert(kMxTokMax == kMxPassTokens, "the routing kernel cuts passes of kMxTokMax tokens");

enum { kGU = 0, kDN = 1 };

struct MxHdr {
    int32_t slot, n0, kstage, rows, ntok, last, done, pad;
    int32_t pairs[kMxTokMax];
    int32_t texp[kMxTokMax];
};

// Stage layout (each stage 1024-byte aligned for the swizzle): codes [NM][kKp][kCols],
// scales [NM][kKp / 16][kCols] at sc_off, tokens [tg] at tok_off with a padded stride,
// bias [NM][kCols] bf16 at bias_off (filled on an item's last stage).
struct MxCfg {
    int32_t tiles, kst, stages, stage_bytes, tok_off, tok_stride, sc_off, tg, red_off, bias_off;
};

// Shared-memory byte of logical (row, byte) of a 128-byte-swizzled code tile whose base
// is 1024-byte aligned: the 16-byte chunk index is XORed with the row's index mod 8.
__device__ __forceinline__ int swz128(int row, int byte) { return row * kCols + (byte ^ ((row & 7) << 4)); }

// One stage of one consumer warp: scale blocks 2bp and 2bp + 1 of the stage, column half
// hf (M tiles j = 4hf..4hf+3 of the item, here indexed 0..3), all NM matrices.
//   acc[m][j][0..1]: column 32jp + 4g + 2q,     tokens 2tig, 2tig + 1
//   acc[m][j][2..3]: column 32jp + 4g + 2q + 1, tokens 2tig, 2tig + 1
// with j = 2 * (jp - 2hf) + q, g = lane / 4, tig = lane % 4.
template <int NM, bool DOWN>
__device__ __forceinline__ void mx_stage_mma(const unsigned char *st, const MxCfg &c, int bp, int hf, int rows,
                                             int ntok, float tok_scale, float (&acc)[NM][4][4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    const unsigned char *tokp = st + c.tok_off + g * c.tok_stride;
#pragma unroll
    for (int bb = 0; bb < 2; bb++) {
        const int blk = 2 * bp + bb;
        if (blk * 16 >= rows) break;
        float tmp[NM][4][4];
#pragma unroll
        for (int ks = 0; ks < 2; ks++) {
            const int rA = blk * 16 + ks * 8 + 2 * tig, rB = rA + 1;  // k-pair rows of this lane
            uint32_t b0 = 0u, b1 = 0u;
            if (g < ntok) {
                if (DOWN) {
                    const float4 hv = *reinterpret_cast<const float4 *>(tokp + 8 * rA);
                    b0 = f2_scale_to_h2(hv.x, hv.y, tok_scale);
                    b1 = f2_scale_to_h2(hv.z, hv.w, tok_scale);
                } else {
                    const uint2 xv = *reinterpret_cast<const uint2 *>(tokp + 4 * rA);
                    b0 = xv.x;
                    b1 = xv.y;
                }
            }
#pragma unroll
            for (int m = 0; m < NM; m++) {
                const unsigned char *cm = st + m * kKp * kCols;
#pragma unroll
                for (int q2 = 0; q2 < 2; q2++) {
                    const int byte = 32 * (2 * hf + q2) + 4 * g;
                    const uint32_t wA = *reinterpret_cast<const uint32_t *>(cm + swz128(rA, byte));
                    const uint32_t wB = *reinterpret_cast<const uint32_t *>(cm + swz128(rB, byte));
                    uint32_t hA[4], hB[4];
                    e2m1x8_h2(wA, hA);
                    e2m1x8_h2(wB, hB);
                    if (ks == 0) {  // the block's sum starts from zero
                        mma_f16_16816_z(tmp[m][2 * q2], hA[0], hA[1], hB[0], hB[1], b0, b1);
                        mma_f16_16816_z(tmp[m][2 * q2 + 1], hA[2], hA[3], hB[2], hB[3], b0, b1);
                    } else {
                        mma_f16_16816(tmp[m][2 * q2], hA[0], hA[1], hB[0], hB[1], b0, b1);
                        mma_f16_16816(tmp[m][2 * q2 + 1], hA[2], hA[3], hB[2], hB[3], b0, b1);
                    }
                }
            }
        }
        // the block's e8m0 column scales: bytes 0..3 of the word are the columns of
        // (q = 0, row g), (q = 0, row g + 8), (q = 1, row g), (q = 1, row g + 8)
#pragma unroll
        for (int m = 0; m < NM; m++)
#pragma unroll
            for (int q2 = 0; q2 < 2; q2++) {
                const uint32_t sw = *reinterpret_cast<const uint32_t *>(
                    st + c.sc_off + (m * (kKp / 16) + blk) * kCols + 32 * (2 * hf + q2) + 4 * g);
#pragma unroll
                for (int q = 0; q < 2; q++) {
                    const float2 sc = e8m0x2_to_f2(sw >> (16 * q));  // (row g, row g + 8)
                    float *a = acc[m][2 * q2 + q];
                    const float *t = tmp[m][2 * q2 + q];
                    ffma2_s(a[0], a[1], t[0], t[1], sc.x);
                    ffma2_s(a[2], a[3], t[2], t[3], sc.y);
                }
            }
    }
}

template <int PHASE>
__global__ void __launch_bounds__(kMxThreads, 1)
    ffn_mx_tma_kernel(FfnParams p, MxCfg c, const __grid_constant__ CUtensorMap blocks_map,
                      const __grid_constant__ CUtensorMap scales_map) {
    constexpr int NM = PHASE == kGU ? 2 : 1;
    extern __shared__ __align__(1024) unsigned char sm[];
    uint64_t *full = reinterpret_cast<uint64_t *>(sm);
    uint64_t *empty = full + kMxStagesMax;
    uint64_t *rbar = empty + kMxStagesMax;  // [3] consumer barriers around the reduction
    MxHdr *hdr = reinterpret_cast<MxHdr *>(sm + 256);
    // stages start at the first 1024-byte aligned shared address after the headers (the
    // 128-byte swizzle pattern of the code tiles repeats every 1024 bytes)
    const uint32_t hdr_end = su32(sm) + 256 + kMxStagesMax * sizeof(MxHdr);
    unsigned char *stage0 = sm + (((hdr_end + 1023u) & ~1023u) - su32(sm));
    float *red = reinterpret_cast<float *>(stage0 + c.red_off);
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
        bar_init(&rbar[2], kCW);
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
        // items are dealt round-robin, so at any moment the CTAs hold neighbouring column
        // tiles of the same expert rows and a 128-byte line shared by two tiles (the up
        // half starts 64 bytes into a line when I is an odd multiple of 64) is still in L2
        // when the second tile asks for it
        const int first = blockIdx.x;
        bool waited = PHASE == kGU, ok = true;
        int issued = 0;
        const uint64_t pol = evict_first_l2();  // weights are read once
        const uint32_t box_bytes = NM * (kKp * kCols + (kKp / 16) * kCols);
        int u = items > first ? pass_owner(p.s.upoff, nu, first / c.tiles) : 0;
        int cur_pi = -1, slot = 0, cnt = 0;
        int pairs_c[kMxTokMax], texp_c[kMxTokMax];
        for (int it = first; it < items && ok; it += gridDim.x) {
            const int pi = it / c.tiles, tile = it - pi * c.tiles;
            if (pi != cur_pi) {  // new pass: advance the owner and cache its tokens
                while (u + 1 < nu && p.s.upoff[u + 1] <= pi) u++;
                cur_pi = pi;
                slot = p.s.uslot[u];
                FTMOE_DCHECK(slot >= 0 && slot < p.S, p.status);
                slot = slot < 0 ? 0 : (slot >= p.S ? p.S - 1 : slot);
                const int pbase = (pi - p.s.upoff[u]) * kMxTokMax;
                cnt = p.s.ucnt[u] - pbase < kMxTokMax ? p.s.ucnt[u] - pbase : kMxTokMax;
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
                    // the item's last stage also brings the bias of its columns (bf16; the
                    // column count is a multiple of 32, so 64-byte multiples)
                    const int ncol = nout - n0 < kCols ? nout - n0 : kCols;
                    const uint32_t bb = hh.last ? (uint32_t)(NM * ncol * 2) : 0u;
                    bar_expect(&full[s], box_bytes + (uint32_t)ntok * tb + bb);
                    unsigned char *st = stage0 + (size_t)s * c.stage_bytes;
                    // rows past the slot's last k-pair row are zero-filled by the copy, not read
                    for (int m = 0; m < NM; m++) {
                        const int x = n0 + (m ? I : 0);
                        tma3d_hint(st + m * kKp * kCols, &blocks_map, x, ks * kKp, slot, &full[s], pol);
                        tma3d_hint(st + c.sc_off + m * (kKp / 16) * kCols, &scales_map, x, ks * (kKp / 16), slot,
                                   &full[s], pol);
                    }
                    for (int i = 0; i < ntok; i++) {
                        const int q = hh.pairs[i];
                        const void *src = PHASE == kGU
                                              ? static_cast<const void *>(p.s.x16 + (int64_t)(q / p.topk) * H +
                                                                          2 * ks * kKp)
                                              : static_cast<const void *>(p.s.h + (int64_t)q * I + 2 * ks * kKp);
                        bulk1d(st + c.tok_off + i * c.tok_stride, src, tb, &full[s]);
                    }
                    if (hh.last) {
                        const int bi = PHASE == kGU ? 2 : 5;
                        const unsigned char *bsrc = p.bank[bi] + (int64_t)slot * p.bank_bytes[bi];
                        for (int m = 0; m < NM; m++)
                            bulk1d(st + c.bias_off + m * kCols * 2, bsrc + 2 * ((int64_t)n0 + (m ? I : 0)),
                                   (uint32_t)(ncol * 2), &full[s]);
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

    // consumers: warp = (pair of scale blocks bp, column half hf)
    const int bp = warp >> 1, hf = warp & 1;
    float acc[NM][4][4];
#pragma unroll
    for (int m = 0; m < NM; m++)
#pragma unroll
        for (int j = 0; j < 4; j++)
#pragma unroll
            for (int i = 0; i < 4; i++) acc[m][j][i] = 0.f;
    uint32_t rphase = 0;
    const int g = lane >> 2, tig = lane & 3;
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
        const float tok_scale = g < ntok ? ldexpf(1.f, -hs.texp[g]) : 0.f;
        mx_stage_mma<NM, PHASE == kDN>(st, c, bp, hf, rows, ntok, tok_scale, acc);
        if (!last) {
            __syncwarp();
            if (lane == 0) bar_arrive(&empty[s]);
            continue;
        }

        // item end: the warps' partials meet in red [NM][kBlkPairs][kMxTokMax][kCols]. Down
        // puts them over the last stage's code tile (the same 32 KB), once every warp is done
        // reading it, which leaves the shared memory for a fourth stage.
        float *red_i = red;
        if (PHASE == kDN) {
            __syncwarp();
            if (lane == 0) bar_arrive(&rbar[2]);
            if (!bar_wait(&rbar[2], rphase)) {
                if (lane == 0) atomicCAS(p.status, 0, FTMOE_ERR_STATE);
                return;
            }
            red_i = reinterpret_cast<float *>(stage0 + (size_t)s * c.stage_bytes);
        }
#pragma unroll
        for (int m = 0; m < NM; m++)
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int col = 32 * (2 * hf + (j >> 1)) + 4 * g + 2 * (j & 1);
                float *r = red_i + ((m * kBlkPairs + bp) * kMxTokMax) * kCols;
                const int t0 = 2 * tig, t1 = 2 * tig + 1;
                if (t0 < ntok) {
                    r[t0 * kCols + col] = acc[m][j][0];
                    r[t0 * kCols + col + 1] = acc[m][j][2];
                }
                if (t1 < ntok) {
                    r[t1 * kCols + col] = acc[m][j][1];
                    r[t1 * kCols + col + 1] = acc[m][j][3];
                }
#pragma unroll
                for (int i = 0; i < 4; i++) acc[m][j][i] = 0.f;
            }
        __syncwarp();
        if (lane == 0) bar_arrive(&rbar[0]);
        if (!bar_wait(&rbar[0], rphase)) {
            if (lane == 0) atomicCAS(p.status, 0, FTMOE_ERR_STATE);
            return;
        }
        const uint16_t *bias = reinterpret_cast<const uint16_t *>(st + c.bias_off);  // [NM][kCols], staged
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
                for (int w = 0; w < kBlkPairs; w++) sum += red_i[((m * kBlkPairs + w) * kMxTokMax + t) * kCols + col];
                v[m] = sum * xs_t;
            }
            const int q = hs.pairs[t];
            if (PHASE == kGU) {
                float hv = 0.f;
                if (valid) {
                    const float gg = v[0] + __uint_as_float((uint32_t)bias[col] << 16);
                    const float uu = v[NM - 1] + __uint_as_float((uint32_t)bias[(NM - 1) * kCols + col] << 16);
                    hv = silu(gg) * uu;
                    p.s.h[(int64_t)q * I + n] = hv;
                }
                const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv)));
                if (lane == 0 && wm) atomicMax(&p.s.hmax[q], wm);
            } else if (valid) {
                p.s.o[(int64_t)q * H + n] = v[0] + __uint_as_float((uint32_t)bias[col] << 16);
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
    // token rows: 4 bytes (f16 pair) or 8 bytes (fp32 pair) per k-pair row; the stride is
    // padded by 32 / 64 bytes so the B-fragment loads of eight tokens hit distinct banks
    c.tok_stride = phase == kGU ? kKp * 4 + 32 : kKp * 8 + 64;
    c.sc_off = NM * kKp * kCols;
    c.tok_off = c.sc_off + NM * (kKp / 16) * kCols;
    c.bias_off = c.tok_off + c.tg * c.tok_stride;
    c.stage_bytes = (c.bias_off + NM * kCols * 2 + 1023) & ~1023;
    // down's reduction reuses the last stage's code tile (NM * kKp * kCols bytes)
    static_assert(kBlkPairs * kMxTokMax * kCols * 4 == kKp * kCols, "down partials fill one code tile");
    const size_t red = phase == kDN ? 0 : (size_t)NM * kBlkPairs * kMxTokMax * kCols * 4;
    const size_t head = 256 + kMxStagesMax * sizeof(MxHdr) + 1024;  // + alignment slack
    const size_t cap = 227 * 1024;
    int stages = kMxStagesMax;
    while (stages >= 2 && head + (size_t)stages * c.stage_bytes + red > cap) stages--;
    if (stages < 2) return false;
    c.stages = stages;
    c.red_off = stages * c.stage_bytes;
    smem = head + (size_t)stages * c.stage_bytes + red;
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
// of rows * cols) with a box of 128 columns x box_rows rows x 1 slot and the given
// shared-memory swizzle. Rows past a slot's
// last row fall outside the map, so a ragged last box is zero-filled instead of reading
// the next slot.
bool encode_u8(void *out, const void *base, uint64_t cols, uint64_t rows, uint64_t slots, uint32_t box_rows,
               CUtensorMapSwizzle swizzle) {
    EncodeFn fn = encode_fn();
    if (!fn || cols % 16 || ((uintptr_t)base % 16)) return false;
    const cuuint64_t dims[3] = {cols, rows, slots};
    const cuuint64_t strides[2] = {cols, cols * rows};
    const cuuint32_t box[3] = {(cuuint32_t)kCols, box_rows, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(reinterpret_cast<CUtensorMap *>(out), CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims,
              strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool make_mx_tma_maps(MxTmaMaps &m, const unsigned char *const *banks, int S, int H, int I) {
    static_assert(sizeof(CUtensorMap) <= sizeof(m.gu_blocks), "tensor map storage");
    m.valid = false;
    if (H % 32 || I % 32) return false;
    const uint64_t ngu = 2ull * I, ndn = (uint64_t)H;
    // code tiles: 128-byte rows stored with the 128-byte swizzle; scale tiles plain
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B, none = CU_TENSOR_MAP_SWIZZLE_NONE;
    bool ok = encode_u8(m.gu_blocks, banks[0], ngu, (uint64_t)(H / 2), (uint64_t)S, kKp, sw) &&
              encode_u8(m.gu_scales, banks[1], ngu, (uint64_t)(H / 32), (uint64_t)S, kKp / 16, none) &&
              encode_u8(m.dn_blocks, banks[3], ndn, (uint64_t)(I / 2), (uint64_t)S, kKp, sw) &&
              encode_u8(m.dn_scales, banks[4], ndn, (uint64_t)(I / 32), (uint64_t)S, kKp / 16, none);
    m.valid = ok;
    return ok;
}

bool make_bf16_tma_maps(MxTmaMaps &m, const unsigned char *const *banks, int S, int H, int I) {
    m.valid = false;
    if (H % 256 || I % 256) return false;
    // bf16 weights [N rows, 2K bytes] per slot, boxes of 128 bytes (64 k) x 64 rows, 128-byte swizzle
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    bool ok = encode_u8(m.gu_blocks, banks[0], 2ull * H, 2ull * I, (uint64_t)S, 64, sw) &&
              encode_u8(m.dn_blocks, banks[1], 2ull * I, (uint64_t)H, (uint64_t)S, 64, sw);
    m.valid = ok;
    // the tcgen05 pipeline: boxes of 128 bytes x 128 rows (the UMMA's M)
    m.tc_valid = ok && encode_u8(m.tc_gu, banks[0], 2ull * H, 2ull * I, (uint64_t)S, 128, sw) &&
                 encode_u8(m.tc_dn, banks[1], 2ull * I, (uint64_t)H, (uint64_t)S, 128, sw);
    return ok;
}

bool make_fp8_tma_maps(MxTmaMaps &m, const unsigned char *const *banks, int S, int H, int I) {
    m.valid = false;
    if (H % 512 || I % 512) return false;
    // block-FP8 weights [N rows, K bytes] per slot, boxes of 128 k x 64 rows, 128-byte swizzle
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    bool ok = encode_u8(m.gu_blocks, banks[0], (uint64_t)H, 2ull * I, (uint64_t)S, 64, sw) &&
              encode_u8(m.dn_blocks, banks[2], (uint64_t)I, (uint64_t)H, (uint64_t)S, 64, sw);
    m.valid = ok;
    return ok;
}

}  // namespace ftmoe
