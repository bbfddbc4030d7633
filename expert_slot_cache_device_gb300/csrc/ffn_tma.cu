// Row-major expert FFN phases (bf16, nvfp4 and GGUF Q4_0 banks) on the CUDA cores, as a
// persistent, warp-specialised bulk-copy pipeline.
//
// Decode batches make the FFN a grouped GEMV that must stream every used expert's
// weights from HBM exactly once. Work items (pass of a distinct slot u, tile of R output
// rows) are dealt round-robin over the CTAs, so at any moment the CTAs read neighbouring
// rows and the passes of one hot expert side by side (its second pass hits L2). One
// producer thread fills a ring of shared-memory stages with 1-D bulk asynchronous copies
// (cp.async.bulk, completion counted on an mbarrier): the item's weight rows (gate and up
// rows of R neurons, or R down rows, plus the nvfp4 block scales and row globals) and the
// token vectors the item needs (bf16 activations, or their scaled f16 copy for nvfp4 and
// Q4_0, for gate_up; fp32 h rows for down). It also writes a small stage header (slot,
// rows, tokens). The consumer warps (8 for gate_up, 16 for down) wait on the stage's
// mbarrier, compute from shared memory (a warp per neuron in gate_up, per group of rows in
// down; lanes over 16-byte chunks or quantisation blocks, warp-shuffle reductions, fp32
// accumulation, nvfp4 and Q4_0 decoded in registers) and release the stage. Several stages
// stay in flight per SM, so the HBM stream never waits on a CTA's start-up latency; weight
// copies carry an L2 evict-first policy because they are read once.
//
// The kernels are chained with programmatic dependent launch: gate_up waits for the
// routing kernel, down's producer starts streaming its weights while gate_up drains
// and waits only before it copies the h rows gate_up writes.
//
// Every mbarrier wait is bounded (pipe::bar_wait): on expiry the waiting thread records
// FTMOE_ERR_STATE in the status word and leaves, and the producer waits (again bounded) for
// its own copies in flight before it exits. A test setting shortens the limit and leaves one
// stage unfilled to exercise that path.
#include "ffn_common.cuh"
#include "internal.cuh"
#include "pipeline.cuh"

namespace ftmoe {
namespace {

using namespace ffn;
using namespace pipe;

enum { kGateUp = 0, kDown = 1 };

// Consumer warps per CTA (the producer warp comes after them). Down has 16: its consumers are
// bound by instruction latency (one group of kDnRR rows per warp and stage at 64-row items),
// and with two rows per group Q4_0 fits the registers of a 544-thread CTA too. gate_up keeps
// 8, bound by the rows one stage holds (a warp per neuron).
template <int FMT, int PHASE>
constexpr int kConsumerWarps = PHASE == kDown ? 16 : 8;
// down rows sharing each h read (Q4_0: two, so that 16 warps fit the registers)
template <int FMT>
constexpr int kDnRR = FMT == FTMOE_FMT_Q4_0 ? 2 : 4;
template <int FMT, int PHASE>
constexpr int kTmaThreads = (kConsumerWarps<FMT, PHASE> + 1) * 32;
constexpr int kMaxStages = 4;
constexpr int kMaxTok = 4;  // tokens per stage

struct StageHdr {
    int32_t slot, n0, rows, ntok, done, pad0, pad1, pad2;
    int32_t pairs[kMaxTok];
    int32_t texp[kMaxTok];  // per-token exponent of the f16 activations (nvfp4 gate_up)
};

struct TmaCfg {
    int32_t R;           // rows (gate_up: neurons) per item
    int32_t tiles;       // items per distinct slot
    int32_t stages;
    int32_t stage_bytes;
    int32_t tok_off;     // offset of the token vectors inside a stage
    int32_t tok_bytes;   // bytes of one token vector
    int32_t tg;          // tokens per stage (<= kMaxTok)
};

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Bytes of the weight segments of an item with `rows` rows (R rows reserve the layout).
// Formats whose consumers use the power-of-two scaled f16 activation copy and f16 h.
template <int FMT>
constexpr bool kF16Act = FMT == FTMOE_FMT_NVFP4 || FMT == FTMOE_FMT_Q4_0;

template <int FMT, int PHASE>
struct Seg {
    // per-row bytes of the code/weight matrix and of the scale matrix
    __device__ __host__ static int64_t wrow(int H, int I) {
        const int64_t K = PHASE == kGateUp ? H : I;
        return FMT == FTMOE_FMT_BF16 ? 2 * K : (FMT == FTMOE_FMT_Q4_0 ? K / 32 * 18 : K / 2);
    }
    __device__ __host__ static int64_t srow(int H, int I) {
        const int64_t K = PHASE == kGateUp ? H : I;
        return FMT == FTMOE_FMT_NVFP4 ? K / 16 : 0;
    }
    static constexpr int mats = PHASE == kGateUp ? 2 : 1;  // gate + up, or down
    // offset of the nvfp4 per-row f16 globals (after the codes and scales of R rows)
    __device__ __host__ static int64_t goff(int R, int H, int I) {
        return (int64_t)mats * R * (wrow(H, I) + srow(H, I));
    }
    __device__ __host__ static int64_t bytes(int rows, int H, int I) {
        return (int64_t)mats * rows * (wrow(H, I) + srow(H, I) + (FMT == FTMOE_FMT_NVFP4 ? 2 : 0));
    }
};

// ---------------------------------------------------------------- consumers

// Running max |h| of one pair, kept by lane t for the pair in token slot t: the pair's max
// word is updated once per item (or run of items sharing the pair) instead of once per
// row (per-row atomics on a handful of words serialised on one L2 slice).
struct HMax {
    int pair = -1;
    float m = 0.f;
    __device__ __forceinline__ void flush(const FfnParams &p) {
        if (pair >= 0 && m > 0.f) atomicMax(&p.s.hmax[pair], __float_as_uint(m));
    }
    __device__ __forceinline__ void add(const FfnParams &p, int q, float v) {
        if (q != pair) {
            flush(p);
            pair = q;
            m = 0.f;
        }
        m = fmaxf(m, v);
    }
};

template <int FMT, int NT>
__device__ __forceinline__ void gu_consume(const FfnParams &p, const TmaCfg &c, const unsigned char *st,
                                           const StageHdr &h, HMax &hm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H, I = p.I, R = c.R;
    const int64_t wr = Seg<FMT, kGateUp>::wrow(H, I), sr = Seg<FMT, kGateUp>::srow(H, I);
    const uint4 *xs = reinterpret_cast<const uint4 *>(st + c.tok_off);
    const int nxv = H >> 3;  // 16-byte vectors per token (8 bf16)
    for (int j = warp; j < h.rows; j += kConsumerWarps<FMT, kGateUp>) {
        const int n = h.n0 + j;
        float g[NT], u[NT];
#pragma unroll
        for (int t = 0; t < NT; t++) g[t] = u[t] = 0.f;
        float gg = 1.f, gu = 1.f;
        if (FMT == FTMOE_FMT_NVFP4) {  // per-row f16 globals, staged after the scales
            const __half *gl = reinterpret_cast<const __half *>(st + Seg<FMT, kGateUp>::goff(R, H, I));
            gg = __half2float(gl[j]);
            gu = __half2float(gl[R + j]);
        }
        if (FMT == FTMOE_FMT_BF16) {
            const uint4 *wg = reinterpret_cast<const uint4 *>(st + j * wr);
            const uint4 *wu = reinterpret_cast<const uint4 *>(st + (R + j) * wr);
            const int nch = H >> 3;
#pragma unroll 2
            for (int ch = lane; ch < nch; ch += 32) {
                float fa[8], fb[8];
                unpack_bf16x8(wg[ch], fa);
                unpack_bf16x8(wu[ch], fb);
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    float fx[8];
                    unpack_bf16x8(xs[t * nxv + ch], fx);
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        g[t] = fmaf(fa[i], fx[i], g[t]);
                        u[t] = fmaf(fb[i], fx[i], u[t]);
                    }
                }
            }
        } else if (FMT == FTMOE_FMT_Q4_0) {
            // lane step = one 32-element Q4_0 block of the gate and of the up row, in integers:
            // w ^ 0x88888888 turns every nibble q into the 4-bit two's complement of q - 8, and
            // masked into the top half of a byte it reads as the int8 16 (q - 8); dp2a multiplies
            // two of them by two int16 activations (the token's block as int16 with one scale,
            // staged after the int16 row) and every block sums exactly in int32. The block's sum
            // is then scaled by the f16 weight scale times the activation scale (which carries
            // the 1/16). The int16 activations are staged in the swz_q4x16 layout: unit u of this
            // lane's block sits at u ^ ((b >> 1) & 3).
            const unsigned char *rg = st + j * wr, *ru = st + (R + j) * wr;
            const int nb = H >> 5;
            const int rot = (lane >> 1) & 3;
            for (int b = lane; b < nb; b += 32) {
                uint32_t dg, du, qg[4], qu[4];
                q4_block(rg, b, dg, qg);
                q4_block(ru, b, du, qu);
                uint32_t lg[4], hg[4], lu[4], hu[4];  // int8 16 (q - 8): elements 4i.. and 16 + 4i..
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const uint32_t a = qg[i] ^ 0x88888888u, e = qu[i] ^ 0x88888888u;
                    lg[i] = (a << 4) & 0xF0F0F0F0u;
                    hg[i] = a & 0xF0F0F0F0u;
                    lu[i] = (e << 4) & 0xF0F0F0F0u;
                    hu[i] = e & 0xF0F0F0F0u;
                }
                const float fdg = __half2float(__ushort_as_half((unsigned short)dg));
                const float fdu = __half2float(__ushort_as_half((unsigned short)du));
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    const unsigned char *tok = st + c.tok_off + t * c.tok_bytes;
                    const uint4 *xv = reinterpret_cast<const uint4 *>(tok);
                    uint32_t xw[16];  // xw[k] = int16 elements (2k, 2k + 1) of the block
#pragma unroll
                    for (int uu = 0; uu < 4; uu++) {
                        const uint4 v = xv[4 * b + (uu ^ rot)];
                        xw[4 * uu] = v.x;
                        xw[4 * uu + 1] = v.y;
                        xw[4 * uu + 2] = v.z;
                        xw[4 * uu + 3] = v.w;
                    }
                    const float xsc = reinterpret_cast<const float *>(tok + 2 * H)[b];
                    int g0 = 0, g1 = 0, u0 = 0, u1 = 0;
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        g0 = __dp2a_lo((int)xw[2 * i], (int)lg[i], g0);
                        g0 = __dp2a_hi((int)xw[2 * i + 1], (int)lg[i], g0);
                        g1 = __dp2a_lo((int)xw[8 + 2 * i], (int)hg[i], g1);
                        g1 = __dp2a_hi((int)xw[9 + 2 * i], (int)hg[i], g1);
                        u0 = __dp2a_lo((int)xw[2 * i], (int)lu[i], u0);
                        u0 = __dp2a_hi((int)xw[2 * i + 1], (int)lu[i], u0);
                        u1 = __dp2a_lo((int)xw[8 + 2 * i], (int)hu[i], u1);
                        u1 = __dp2a_hi((int)xw[9 + 2 * i], (int)hu[i], u1);
                    }
                    g[t] = fmaf((float)(g0 + g1), fdg * xsc, g[t]);
                    u[t] = fmaf((float)(u0 + u1), fdu * xsc, u[t]);
                }
            }
        } else {
            // lane step = one 16-element scale block (two 32-bit code words): codes ->
            // exact f16x2, sixteen exact f16 products summed in two f16 halves of eight,
            // then the block scale applied in fp32 (f16 x f16 products, fp32 sums). The
            // activations are staged in the swz_x16 layout: this lane's first 16-byte
            // half of block b sits at group 2b + rot, its second at 2b + (rot ^ 1).
            const uint2 *cg = reinterpret_cast<const uint2 *>(st + j * wr);
            const uint2 *cu = reinterpret_cast<const uint2 *>(st + (R + j) * wr);
            const unsigned char *sg = st + 2 * R * wr + j * sr, *su = st + 2 * R * wr + (R + j) * sr;
            const int nb = H >> 4;
            const int rot = (lane >> 2) & 1;
#pragma unroll 2
            for (int b = lane; b < nb; b += 32) {
                const uint2 ca = cg[b], cb = cu[b];
                uint32_t fa[8], fb[8];
                e2m1x8_h2(ca.x, *reinterpret_cast<uint32_t(*)[4]>(&fa[0]));
                e2m1x8_h2(ca.y, *reinterpret_cast<uint32_t(*)[4]>(&fa[4]));
                e2m1x8_h2(cb.x, *reinterpret_cast<uint32_t(*)[4]>(&fb[0]));
                e2m1x8_h2(cb.y, *reinterpret_cast<uint32_t(*)[4]>(&fb[4]));
                const uint32_t s2 = e4m3x2_to_h2((uint32_t)sg[b] | ((uint32_t)su[b] << 8));
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    const uint4 x0 = xs[t * nxv + 2 * b + rot], x1 = xs[t * nxv + 2 * b + (rot ^ 1)];
                    const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                    g[t] = fma_h2_scale(dot16_e2m1_h2(fa, xw), h2_lo(s2), g[t]);
                    u[t] = fma_h2_scale(dot16_e2m1_h2(fb, xw), h2_hi(s2), u[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < NT; t++) {
            const float xs_t = kF16Act<FMT> ? ldexpf(1.f, h.texp[t]) : 1.f;
            const float gs = warp_sum(g[t]) * gg * xs_t, us = warp_sum(u[t]) * gu * xs_t;
            if (lane == t) {
                const float hv = silu(gs) * us;
                const int hn = FMT == FTMOE_FMT_NVFP4 ? swz_h32(n) : (FMT == FTMOE_FMT_Q4_0 ? swz_q4h32(n) : n);
                p.s.h[(int64_t)h.pairs[t] * I + hn] = hv;
                if (kF16Act<FMT>) hm.add(p, h.pairs[t], fabsf(hv));
            }
        }
    }
}

template <int FMT, int NT>
__device__ __forceinline__ void dn_consume(const FfnParams &p, const TmaCfg &c, const unsigned char *st,
                                           const StageHdr &h) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H, I = p.I, R = c.R;
    const int64_t wr = Seg<FMT, kDown>::wrow(H, I), sr = Seg<FMT, kDown>::srow(H, I);
    const float4 *hs = reinterpret_cast<const float4 *>(st + c.tok_off);
    const int nh4 = I >> 2;
    constexpr int RR = kDnRR<FMT>;  // rows sharing each h read
    for (int j0 = warp * RR; j0 < h.rows; j0 += kConsumerWarps<FMT, kDown> * RR) {
        const int nr = h.rows - j0 < RR ? h.rows - j0 : RR;
        float o[RR][NT];
#pragma unroll
        for (int r = 0; r < RR; r++)
#pragma unroll
            for (int t = 0; t < NT; t++) o[r][t] = 0.f;
        float gl[RR];  // per-row f16 global scales (nvfp4), staged after the block scales
#pragma unroll
        for (int r = 0; r < RR; r++) {
            gl[r] = 1.f;
            if (FMT == FTMOE_FMT_NVFP4 && r < nr)
                gl[r] = __half2float(reinterpret_cast<const __half *>(st + Seg<FMT, kDown>::goff(R, H, I))[j0 + r]);
        }
        if (FMT == FTMOE_FMT_BF16) {
            // lane step = 4 consecutive k: 8-byte weight reads and 16-byte h reads are
            // contiguous across lanes (no bank conflicts)
            for (int q = lane; q < nh4; q += 32) {
                float fa[RR][4];
#pragma unroll
                for (int r = 0; r < RR; r++) {
                    const int jr = r < nr ? j0 + r : j0;
                    const uint2 v = *reinterpret_cast<const uint2 *>(st + jr * wr + 8 * q);
                    fa[r][0] = bf_lo(v.x); fa[r][1] = bf_hi(v.x); fa[r][2] = bf_lo(v.y); fa[r][3] = bf_hi(v.y);
                }
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    const float4 hv = hs[t * nh4 + q];
#pragma unroll
                    for (int r = 0; r < RR; r++) {
                        o[r][t] = fmaf(fa[r][0], hv.x, o[r][t]);
                        o[r][t] = fmaf(fa[r][1], hv.y, o[r][t]);
                        o[r][t] = fmaf(fa[r][2], hv.z, o[r][t]);
                        o[r][t] = fmaf(fa[r][3], hv.w, o[r][t]);
                    }
                }
            }
        } else if (FMT == FTMOE_FMT_Q4_0) {
            // lane step = one 32-element Q4_0 block of RR rows; h is converted once per
            // block and token to f16 with the token's power-of-two scale (max |h| < 2^8),
            // shared by the RR rows. The h rows are staged in the swz_q4h32 layout: unit u of
            // this lane's block sits at u ^ (b & 7), so the 8 lanes of a phase hit 8 units.
            const int nb = I >> 5;
            const int rot = lane & 7;
            float hsc[NT];
#pragma unroll
            for (int t = 0; t < NT; t++) hsc[t] = ldexpf(1.f, -h.texp[t]);
            for (int b = lane; b < nb; b += 32) {
                uint32_t fw[RR][16], dr[RR];
#pragma unroll
                for (int r = 0; r < RR; r++) {
                    const int jr = r < nr ? j0 + r : j0;
                    uint32_t qs[4];
                    q4_block(st + jr * wr, b, dr[r], qs);
                    q4_decode(qs, fw[r]);
                }
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    uint32_t hh[16];
#pragma unroll
                    for (int uu = 0; uu < 8; uu++) {
                        const float4 hv = hs[t * nh4 + 8 * b + (uu ^ rot)];
                        hh[2 * uu] = f2_scale_to_h2(hv.x, hv.y, hsc[t]);
                        hh[2 * uu + 1] = f2_scale_to_h2(hv.z, hv.w, hsc[t]);
                    }
#pragma unroll
                    for (int r = 0; r < RR; r++) o[r][t] = fma_h2_scale(dot32_h2(fw[r], hh), (uint16_t)dr[r], o[r][t]);
                }
            }
        } else {
            // lane step = one 16-element scale block (two code words); h is converted once
            // per block and token to f16 with the token's power-of-two scale (max |h| <
            // 2^10), shared by the RR rows; products summed as in gate_up. The h rows are
            // staged in the swz_h32 layout: quarter q of this lane's block sits at q ^ rot.
            const int nb = I >> 4;
            const int rot = (lane >> 1) & 3;
            float hsc[NT];
#pragma unroll
            for (int t = 0; t < NT; t++) hsc[t] = ldexpf(1.f, -h.texp[t]);
            for (int b = lane; b < nb; b += 32) {
                uint32_t fa[RR][8];
                uint32_t s2[RR / 2];
#pragma unroll
                for (int r = 0; r < RR; r += 2) {
                    const int j1 = r < nr ? j0 + r : j0, j2 = r + 1 < nr ? j0 + r + 1 : j0;
                    const uint2 c1 = *reinterpret_cast<const uint2 *>(st + j1 * wr + 8 * b);
                    const uint2 c2 = *reinterpret_cast<const uint2 *>(st + j2 * wr + 8 * b);
                    e2m1x8_h2(c1.x, *reinterpret_cast<uint32_t(*)[4]>(&fa[r][0]));
                    e2m1x8_h2(c1.y, *reinterpret_cast<uint32_t(*)[4]>(&fa[r][4]));
                    e2m1x8_h2(c2.x, *reinterpret_cast<uint32_t(*)[4]>(&fa[r + 1][0]));
                    e2m1x8_h2(c2.y, *reinterpret_cast<uint32_t(*)[4]>(&fa[r + 1][4]));
                    s2[r / 2] = e4m3x2_to_h2((uint32_t)st[R * wr + j1 * sr + b] |
                                             ((uint32_t)st[R * wr + j2 * sr + b] << 8));
                }
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    uint32_t hh[8];
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const float4 hv = hs[t * nh4 + 4 * b + (q ^ rot)];
                        hh[2 * q] = f2_scale_to_h2(hv.x, hv.y, hsc[t]);
                        hh[2 * q + 1] = f2_scale_to_h2(hv.z, hv.w, hsc[t]);
                    }
#pragma unroll
                    for (int r = 0; r < RR; r++) {
                        const uint32_t sr2 = s2[r / 2];
                        o[r][t] = fma_h2_scale(dot16_e2m1_h2(fa[r], hh), (r & 1) ? h2_hi(sr2) : h2_lo(sr2), o[r][t]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RR; r++) {
            if (r >= nr) break;
            const int n = h.n0 + j0 + r;
#pragma unroll
            for (int t = 0; t < NT; t++) {
                const float v = warp_sum(o[r][t]) * gl[r] * (kF16Act<FMT> ? ldexpf(1.f, h.texp[t]) : 1.f);
                if (lane == t) p.s.o[(int64_t)h.pairs[t] * H + n] = v;
            }
        }
    }
}

// ---------------------------------------------------------------- kernel

template <int FMT, int PHASE>
__global__ void __launch_bounds__(kTmaThreads<FMT, PHASE>, 1) ffn_rows_tma_kernel(FfnParams p, TmaCfg c) {
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t *full = reinterpret_cast<uint64_t *>(sm);
    uint64_t *empty = full + kMaxStages;
    StageHdr *hdr = reinterpret_cast<StageHdr *>(sm + 128);
    unsigned char *stage0 = sm + 128 + kMaxStages * sizeof(StageHdr);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t lim = p.wait_ns ? p.wait_ns : kWaitNs;  // limit of every bounded wait

    if (threadIdx.x == 0) {
        for (int s = 0; s < c.stages; s++) {
            bar_init(&full[s], 1);
            bar_init(&empty[s], kConsumerWarps<FMT, PHASE>);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (PHASE == kGateUp) griddep_wait();  // routing tables come from the previous kernel
    griddep_launch();

    if (warp == kConsumerWarps<FMT, PHASE>) {  // producer
        if (lane != 0) return;
        // Work items blockIdx.x, blockIdx.x + gridDim.x, ... of this CTA: dealt round-robin,
        // the CTAs hold neighbouring tiles and the passes of one expert at the same time,
        // so an expert read again by its next pass is still in L2.
        const int nu = *p.s.n_unique;
        const int npass = nu > 0 ? *p.s.n_passes : 0;
        const int items = npass * c.tiles;
        const int first = blockIdx.x;
        const uint64_t pol = evict_first_l2();
        const int H = p.H, I = p.I, R = c.R;
        const int nout = PHASE == kGateUp ? I : H;
        const int64_t wr = Seg<FMT, PHASE>::wrow(H, I), sr = Seg<FMT, PHASE>::srow(H, I);
        bool waited = PHASE == kGateUp, ok = true;
        int issued = 0;
        int u = items > first ? pass_owner(p.s.upoff, nu, first / c.tiles) : 0;
        for (int it = first; it < items && ok; it += gridDim.x) {
            const int pi = it / c.tiles, tile = it - pi * c.tiles;
            while (u + 1 < nu && p.s.upoff[u + 1] <= pi) u++;  // increasing passes: walk forward
            int slot = p.s.uslot[u];
            FTMOE_DCHECK(slot >= 0 && slot < p.S, p.status);
                slot = slot < 0 ? 0 : (slot >= p.S ? p.S - 1 : slot);
            const int pbase = (pi - p.s.upoff[u]) * kPassTokens;
            const int pcnt = p.s.ucnt[u] - pbase < kPassTokens ? p.s.ucnt[u] - pbase : kPassTokens;
            const int off = p.s.uoff[u] + pbase, cnt = pcnt;
            const int n0 = tile * R, rows = nout - n0 < R ? nout - n0 : R;
            for (int g0 = 0; g0 < cnt && ok; g0 += c.tg) {
                const int ntok = cnt - g0 < c.tg ? cnt - g0 : c.tg;
                const int s = issued % c.stages;
                const uint32_t ph = (issued / c.stages) & 1;
                if (!bar_wait(&empty[s], ph ^ 1, lim)) {
                    ok = false;
                    break;
                }
                if (PHASE == kGateUp && p.debug_skip_stage && blockIdx.x == 0 && issued == 0) {
                    // test setting: this CTA's first stage is left unfilled (no copies, no
                    // arrive), so its consumers' bounded wait runs out
                    issued++;
                    continue;
                }
                StageHdr &hh = hdr[s];
                hh.slot = slot; hh.n0 = n0; hh.rows = rows; hh.ntok = ntok; hh.done = 0;
                for (int i = 0; i < ntok; i++) {
                    hh.pairs[i] = p.s.upairs[off + g0 + i];
                    hh.texp[i] = (PHASE == kGateUp && kF16Act<FMT>) ? p.s.xexp[hh.pairs[i] / p.topk] : 0;
                }
                const uint32_t wbytes = (uint32_t)Seg<FMT, PHASE>::bytes(rows, H, I);
                bar_expect(&full[s], wbytes + (uint32_t)(ntok * c.tok_bytes));
                unsigned char *st = stage0 + (size_t)s * c.stage_bytes;
                if (PHASE == kGateUp) {
                    const unsigned char *wb = p.bank[0] + (int64_t)slot * p.bank_bytes[0];
                    bulk1d_hint(st, wb + n0 * wr, (uint32_t)(rows * wr), &full[s], pol);
                    bulk1d_hint(st + R * wr, wb + ((int64_t)I + n0) * wr, (uint32_t)(rows * wr), &full[s], pol);
                    if (FMT == FTMOE_FMT_NVFP4) {
                        const unsigned char *sb = p.bank[1] + (int64_t)slot * p.bank_bytes[1];
                        bulk1d_hint(st + 2 * R * wr, sb + n0 * sr, (uint32_t)(rows * sr), &full[s], pol);
                        bulk1d_hint(st + 2 * R * wr + R * sr, sb + ((int64_t)I + n0) * sr, (uint32_t)(rows * sr),
                                 &full[s], pol);
                        // per-row globals: rows * 2 bytes, a multiple of 16 (rows is a multiple of 8)
                        const unsigned char *gb = p.bank[2] + (int64_t)slot * p.bank_bytes[2];
                        unsigned char *gd = st + Seg<FMT, PHASE>::goff(R, H, I);
                        bulk1d_hint(gd, gb + 2 * (int64_t)n0, (uint32_t)(2 * rows), &full[s], pol);
                        bulk1d_hint(gd + 2 * R, gb + 2 * ((int64_t)I + n0), (uint32_t)(2 * rows), &full[s], pol);
                    }
                } else {
                    const int wb_i = FMT == FTMOE_FMT_NVFP4 ? 3 : 1;
                    const unsigned char *wb = p.bank[wb_i] + (int64_t)slot * p.bank_bytes[wb_i];
                    bulk1d_hint(st, wb + n0 * wr, (uint32_t)(rows * wr), &full[s], pol);
                    if (FMT == FTMOE_FMT_NVFP4) {
                        const unsigned char *sb = p.bank[4] + (int64_t)slot * p.bank_bytes[4];
                        bulk1d_hint(st + R * wr, sb + n0 * sr, (uint32_t)(rows * sr), &full[s], pol);
                        const unsigned char *gb = p.bank[5] + (int64_t)slot * p.bank_bytes[5];
                        bulk1d_hint(st + Seg<FMT, PHASE>::goff(R, H, I), gb + 2 * (int64_t)n0, (uint32_t)(2 * rows),
                                 &full[s], pol);
                    }
                }
                if (!waited) {  // h rows are written by the gate_up kernel
                    griddep_wait();
                    waited = true;
                }
                if (PHASE == kDown && kF16Act<FMT>) {
                    // power-of-two exponent for the f16 copy of each h row (max |h| < 2^10 for
                    // nvfp4's sums of 8 products, 2^8 for Q4_0's sums of 16)
                    for (int i = 0; i < ntok; i++) {
                        const float m = __uint_as_float(p.s.hmax[hh.pairs[i]]);
                        int e = 0;
                        if (m > 0.f && m < INFINITY) {
                            frexpf(m, &e);
                            e -= FMT == FTMOE_FMT_Q4_0 ? 8 : 10;
                        }
                        hh.texp[i] = e;
                    }
                }
                for (int i = 0; i < ntok; i++) {
                    const int q = hh.pairs[i];
                    const uint16_t *xsrc = kF16Act<FMT> ? p.s.x16 : p.x;
                    const void *src = PHASE == kGateUp
                                          ? (FMT == FTMOE_FMT_Q4_0  // prepared rows of tok_bytes each
                                                 ? static_cast<const void *>(reinterpret_cast<const unsigned char *>(p.s.x16) +
                                                                             (int64_t)(q / p.topk) * c.tok_bytes)
                                                 : static_cast<const void *>(xsrc + (int64_t)(q / p.topk) * H))
                                          : static_cast<const void *>(p.s.h + (int64_t)q * I);
                    bulk1d(st + c.tok_off + i * c.tok_bytes, src, (uint32_t)c.tok_bytes, &full[s]);
                }
                issued++;
            }
        }
        if (ok) {  // end marker
            const int s = issued % c.stages;
            if (bar_wait(&empty[s], ((issued / c.stages) & 1) ^ 1, lim)) {
                hdr[s].done = 1;
                bar_arrive(&full[s]);
            } else {
                ok = false;
            }
        }
        if (!ok) {
            atomicCAS(p.status, 0, FTMOE_ERR_STATE);
            // wait (bounded) until the copies already issued have landed
            for (int j = issued - c.stages < 0 ? 0 : issued - c.stages; j < issued; j++)
                bar_wait(&full[j % c.stages], (j / c.stages) & 1, lim);
        }
        return;
    }

    // consumers
    HMax hm;
    for (int k = 0;; k++) {
        const int s = k % c.stages;
        if (!bar_wait(&full[s], (k / c.stages) & 1, lim)) {
            if (lane == 0) atomicCAS(p.status, 0, FTMOE_ERR_STATE);
            return;
        }
        const StageHdr h = hdr[s];
        if (h.done) {
            hm.flush(p);
            return;
        }
        const unsigned char *st = stage0 + (size_t)s * c.stage_bytes;
        if (PHASE == kGateUp) {
            switch (h.ntok) {
                case 1: gu_consume<FMT, 1>(p, c, st, h, hm); break;
                case 2: gu_consume<FMT, 2>(p, c, st, h, hm); break;
                case 3: gu_consume<FMT, 3>(p, c, st, h, hm); break;
                default: gu_consume<FMT, 4>(p, c, st, h, hm); break;
            }
        } else {
            switch (h.ntok) {
                case 1: dn_consume<FMT, 1>(p, c, st, h); break;
                case 2: dn_consume<FMT, 2>(p, c, st, h); break;
                case 3: dn_consume<FMT, 3>(p, c, st, h); break;
                default: dn_consume<FMT, 4>(p, c, st, h); break;
            }
        }
        __syncwarp();
        if (lane == 0) bar_arrive(&empty[s]);
    }
}

constexpr size_t kSmemHeader = 128 + kMaxStages * sizeof(StageHdr);
constexpr size_t kSmemCap = 220 * 1024;

template <int FMT, int PHASE>
bool make_cfg(const FfnParams &p, TmaCfg &c) {
    const int H = p.H, I = p.I;
    const int nout = PHASE == kGateUp ? I : H;
    // gate_up token: f16 activations (2H bytes); Q4_0: int16 activations and fp32 block scales
    c.tok_bytes = PHASE == kGateUp ? (FMT == FTMOE_FMT_Q4_0 ? 2 * H + H / 8 : 2 * H) : 4 * I;
    const int rmax = PHASE == kGateUp ? 16 : 64;
    // Prefer enough rows per item to keep all consumer warps busy (gate_up: one neuron per
    // warp; down: four rows per warp), then as many token slots as fit.
    const int rmin_busy = PHASE == kGateUp ? kConsumerWarps<FMT, PHASE> : kDnRR<FMT> * kConsumerWarps<FMT, PHASE>;
    for (int pass = 0; pass < 2; pass++) {
        for (int tg = kMaxTok; tg >= 1; tg >>= 1) {
            // nvfp4 items stage their per-row f16 globals with bulk copies of 2R bytes: R >= 8
            const int rmin = pass == 0 ? rmin_busy : (FMT == FTMOE_FMT_NVFP4 ? 8 : 1);
            for (int R = rmax; R >= rmin; R >>= 1) {
                const int64_t wb = Seg<FMT, PHASE>::bytes(R, H, I);
                // weight bytes per stage: up to 80 KB (three or more stages), 100 KB for bf16
                // down, whose 64 rows of 2I bytes give two stages of 16 warps x 4 rows
                if (wb > (FMT == FTMOE_FMT_BF16 && PHASE == kDown ? 100 : 80) * 1024) continue;
                const int64_t stage = ((wb + 127) & ~(int64_t)127) + (int64_t)tg * c.tok_bytes;
                const int64_t stages = (int64_t)((kSmemCap - kSmemHeader) / (size_t)stage);
                if (stages < 2) continue;
                c.R = R;
                c.tiles = (nout + R - 1) / R;
                c.tg = tg;
                c.tok_off = (int32_t)((wb + 127) & ~(int64_t)127);
                c.stage_bytes = (int32_t)((stage + 127) & ~(int64_t)127);
                c.stages = stages > kMaxStages ? kMaxStages : (int32_t)stages;
                return true;
            }
        }
    }
    return false;
}

template <int FMT, int PHASE>
cudaError_t launch_one(const FfnParams &p, int num_sms, cudaStream_t st) {
    TmaCfg c;
    if (!make_cfg<FMT, PHASE>(p, c)) return cudaErrorInvalidValue;
    const size_t smem = kSmemHeader + (size_t)c.stages * c.stage_bytes;
    auto kern = ffn_rows_tma_kernel<FMT, PHASE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kTmaThreads<FMT, PHASE>);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, c);
}

}  // namespace

bool ffn_rows_tma_supported(const FfnParams &p) {
    if (!p.s.upoff || !p.s.n_passes) return false;
    if (p.fmt == FTMOE_FMT_BF16) return p.H % 8 == 0 && p.I % 8 == 0;
    TmaCfg c;
    if (p.fmt == FTMOE_FMT_NVFP4)
        return p.H % 256 == 0 && p.I % 256 == 0 && p.s.x16 && p.s.xexp && p.s.hmax &&
               make_cfg<FTMOE_FMT_NVFP4, kGateUp>(p, c) && make_cfg<FTMOE_FMT_NVFP4, kDown>(p, c);
    if (p.fmt == FTMOE_FMT_Q4_0)  // rows of 18-byte blocks: 16-byte multiples when K % 256 == 0
        return p.H % 256 == 0 && p.I % 256 == 0 && p.s.x16 && p.s.xexp && p.s.hmax &&
               make_cfg<FTMOE_FMT_Q4_0, kGateUp>(p, c) && make_cfg<FTMOE_FMT_Q4_0, kDown>(p, c);
    return false;
}

cudaError_t launch_ffn_rows_tma(const FfnParams &p, int num_sms, cudaStream_t st) {
    cudaError_t e;
    if (p.fmt == FTMOE_FMT_BF16) {
        if ((e = launch_one<FTMOE_FMT_BF16, kGateUp>(p, num_sms, st)) != cudaSuccess) return e;
        return launch_one<FTMOE_FMT_BF16, kDown>(p, num_sms, st);
    }
    if (p.fmt == FTMOE_FMT_Q4_0) {
        if ((e = launch_one<FTMOE_FMT_Q4_0, kGateUp>(p, num_sms, st)) != cudaSuccess) return e;
        return launch_one<FTMOE_FMT_Q4_0, kDown>(p, num_sms, st);
    }
    if ((e = launch_one<FTMOE_FMT_NVFP4, kGateUp>(p, num_sms, st)) != cudaSuccess) return e;
    return launch_one<FTMOE_FMT_NVFP4, kDown>(p, num_sms, st);
}

}  // namespace ftmoe
