// K3: expert FFN over resolved slots.
//
// FreeToken architecture deep-dive, section 五 (expert banks per format) and
// benchmark guide, section 一 (hit experts compute from the slot cache), 4.2
// (bank schemas: bf16 = gate_up + down; nvfp4 = packed e2m1 codes, one e4m3
// scale per 16 elements and one fp16 global per output row; mxfp4 = transposed
// blocks / e8m0 scales / bias). Layouts read as:
//   bf16   gate_up [2I, H] (rows [0, I) gate, [I, 2I) up), down [H, I];
//   nvfp4  codes [N, K/2] (low nibble = even k), scales [N, K/16], global [N];
//   mxfp4  blocks [K/2, N], scales [K/32, N] (2^(b-127)), bias [N].
// FFN: gu = W_gu x (+b), h = silu(gate) * up, o = W_d h (+b), y = sum_j w_j o_j.
//
// Decode batches are small, so the FFN is a grouped GEMV bound by HBM: every
// expert's weights must be read exactly once per call whatever its token count.
//   route   (1 CTA)  groups the bs*topk routed pairs by slot;
//   gate_up (grid = distinct slots x neuron tiles) streams the gate and up rows
//           of its tile once, for all the slot's tokens (staged in shared
//           memory), and writes h = silu(gate) * up in fp32;
//   down    (grid = distinct slots x output-row tiles) streams the down rows
//           once for all the slot's tokens and writes o in fp32;
//   combine sums o over each token's routed positions in a fixed order, weighted
//           by the router probabilities, and rounds once to bf16.
// Row-major formats (bf16, nvfp4) give each warp whole rows, lanes striding over
// 16-byte chunks, and reduce with warp shuffles. The transposed mxfp4 layout gives
// each lane four adjacent output columns (coalesced 4-byte loads), splits the
// reduction axis across the warps and reduces in shared memory. fp4 codes are
// decoded in registers (cvt e2m1x2 -> f16x2), the block scales are applied to
// per-block partial sums, and all accumulation is fp32. Nothing is atomic, so
// results are bitwise reproducible.
#include "ffn_common.cuh"
#include "internal.cuh"

namespace ftmoe {
namespace {

using namespace ffn;

constexpr int kThreads = 256;  // 8 warps
constexpr int kRowsTgMax = 4;  // tokens per pass, row-major kernels
constexpr int kColsGuTgMax = 2;  // tokens per pass, transposed gate_up kernel
constexpr int kColsDnTgMax = 4;  // tokens per pass, transposed down kernel
constexpr int kGuNeurons = 16; // gate_up rows kernel: neurons per CTA (2 per warp)
constexpr int kDnRows = 32;    // down rows kernel: output rows per CTA
constexpr int kColTile = 128;  // transposed kernels: columns per CTA (4 per lane)

// ------------------------------------------------------------------------ route

__device__ int block_scan_sum(int v, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += u;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? warp_tot[lane] : 0;
        int wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int u = __shfl_up_sync(0xffffffffu, wi, d);
            if (lane >= d) wi += u;
        }
        warp_tot[lane] = wi - w;
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    int r = warp_tot[warp] + incl - v;
    __syncthreads();
    return r;
}

// The routing tables of a call of at most 32 routed pairs, by warp 0 of the routing CTA with
// register shuffles (no block barriers): lane q holds the key slot * 32 + q of pair q (slot -1,
// computed elsewhere, and lanes past P sort last), a bitonic network sorts the keys ascending,
// runs of equal slots become the distinct slots (ascending, their pairs grouped), and a warp
// scan of each slot's pass count gives its first pass. Same tables as the block path below.
__device__ void route_warp(const FfnParams &p) {
    const int lane = threadIdx.x & 31;
    const int s0 = lane < p.P ? p.slots[lane] : -1;
    const bool bad = s0 != -1 && (unsigned)s0 >= (unsigned)p.S;
    if (__any_sync(0xffffffffu, bad)) {
        if (lane == 0) {
            *p.s.n_unique = -1;
            atomicCAS(p.status, 0, FTMOE_ERR_INVALID_ARG);
        }
        return;
    }
    if (p.s.hmax && lane < p.P) p.s.hmax[lane] = 0u;
    constexpr int kNone = 0x7fffffff;
    int key = s0 >= 0 ? (s0 << 5) | lane : kNone;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const int other = __shfl_xor_sync(0xffffffffu, key, j);
            const bool up = (lane & k) == 0, low = (lane & j) == 0;
            key = (low == up) ? min(key, other) : max(key, other);
        }
    const bool valid = key != kNone;
    const int slot = key >> 5, q = key & 31;
    const int prev = __shfl_up_sync(0xffffffffu, slot, 1);
    const bool start = valid && (lane == 0 || prev != slot);
    const unsigned starts = __ballot_sync(0xffffffffu, start);
    const int nvalid = __popc(__ballot_sync(0xffffffffu, valid));
    const unsigned below = (1u << lane) - 1u;
    const unsigned after = starts & ~(below | (1u << lane));
    const int run = start ? ((after ? __ffs(after) - 1 : nvalid) - lane) : 0;
    const int np = start ? (run + p.pass_tokens - 1) / p.pass_tokens : 0;
    int incl = np;  // inclusive scan of the pass counts over the lanes
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    if (valid) p.s.upairs[lane] = q;
    if (start) {
        const int u = __popc(starts & below);
        p.s.uslot[u] = slot;
        p.s.ucnt[u] = run;
        p.s.uoff[u] = lane;
        if (p.s.upoff) p.s.upoff[u] = incl - np;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
        if (p.s.n_passes) *p.s.n_passes = total;
        *p.s.n_unique = __popc(starts);
    }
}

// CTA 0 groups the routed pairs by slot (and clears the per-pair max |h| words). CTAs
// 1..bs (launched only when the fp4 activation copy is wanted) convert token
// t = blockIdx.x - 1 to f16 with a power-of-two scale 2^-e chosen so that
// max|x_t| * 2^-e < 2^10: bf16 values (8 significant bits) land exactly in f16 except
// below the f16 normal range, and the f16 partial sums of the fp4 dot products (four
// products of |e2m1| <= 6) stay below 2^15.
__global__ void __launch_bounds__(1024) ffn_route_kernel(FfnParams p) {
    extern __shared__ int cnt[];  // [S], later the placement cursor
    __shared__ int warp_tot[32];
    __shared__ int s_bad, s_tot_u, s_tot_c;
    __shared__ float s_wmax[32];
    const int tid = threadIdx.x, nt = blockDim.x;
    asm volatile("griddepcontrol.launch_dependents;" :::);
    // launched as a programmatic dependent of the previous kernel (the copy of the missed
    // experts, whose bytes the FFN reads): wait for it before reading slots or x
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (blockIdx.x > 0 && p.x16_swz == 2) {
        // Q4_0: token t as int16 with one scale per 32-element block (the Q4_0 block), so the
        // gate_up kernel multiplies integer nibbles by integer activations (dp2a): warp w takes
        // block k / 32, d = max |x| over the block / 32767, x_int = rint(x / d); stored after
        // the int16 row is d / 16 (the weights enter as 16 (q - 8)).
        const int t = blockIdx.x - 1;
        const uint16_t *xr = p.x + (int64_t)t * p.H;
        unsigned char *row = reinterpret_cast<unsigned char *>(p.s.x16) + (int64_t)t * (2 * (int64_t)p.H + p.H / 8);
        int16_t *xi = reinterpret_cast<int16_t *>(row);
        float *xs = reinterpret_cast<float *>(row + 2 * (int64_t)p.H);
        for (int k = tid; k < p.H; k += nt) {  // nt is a multiple of 32 and H of 256: whole blocks per warp
            const float v = __uint_as_float((uint32_t)xr[k] << 16);
            const float m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
            const float d = m > 0.f && m < INFINITY ? m * (1.f / 32767.f) : 0.f;
            int q = d > 0.f ? __float2int_rn(v / d) : 0;
            q = q > 32767 ? 32767 : (q < -32767 ? -32767 : q);
            xi[swz_q4x16(k)] = (int16_t)q;
            if ((tid & 31) == 0) xs[k >> 5] = d * 0.0625f;
        }
        if (tid == 0) p.s.xexp[t] = 0;
        return;
    }
    if (blockIdx.x > 0) {
        const int t = blockIdx.x - 1;
        const uint16_t *xr = p.x + (int64_t)t * p.H;
        float m = 0.f;
        for (int k = tid; k < p.H; k += nt) m = fmaxf(m, fabsf(__uint_as_float((uint32_t)xr[k] << 16)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((tid & 31) == 0) s_wmax[tid >> 5] = m;
        __syncthreads();
        if (tid < 32) {
            float v = tid < (nt >> 5) ? s_wmax[tid] : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (tid == 0) s_wmax[0] = v;
        }
        __syncthreads();
        int e = 0;
        if (s_wmax[0] > 0.f && s_wmax[0] < INFINITY) {
            frexpf(s_wmax[0], &e);  // max < 2^e
            e -= p.x16_emax;
        }
        const float sc = ldexpf(1.f, -e);
        uint16_t *dst = p.s.x16 + (int64_t)t * p.H;
        for (int k = tid; k < p.H; k += nt)
            dst[p.x16_swz == 1 ? swz_x16(k) : (p.x16_swz == 2 ? swz_q4x16(k) : k)] =
                __half_as_ushort(__float2half_rn(__uint_as_float((uint32_t)xr[k] << 16) * sc));
        if (tid == 0) p.s.xexp[t] = e;
        return;
    }
    if (p.P <= 32) {  // one warp routes small calls (every decode step of one token)
        if (tid < 32) route_warp(p);
        return;
    }
    if (tid == 0) s_bad = 0;
    for (int s = tid; s < p.S; s += nt) cnt[s] = 0;
    if (p.s.hmax)
        for (int q = tid; q < p.P; q += nt) p.s.hmax[q] = 0u;
    __syncthreads();
    for (int q = tid; q < p.P; q += nt) {
        int s = p.slots[q];
        if (s == -1) continue;  // computed elsewhere (hybrid CPU executor)
        if ((unsigned)s >= (unsigned)p.S)
            s_bad = 1;
        else
            atomicAdd(&cnt[s], 1);
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            *p.s.n_unique = -1;
            atomicCAS(p.status, 0, FTMOE_ERR_INVALID_ARG);
        }
        return;
    }
    int base_u = 0, base_c = 0, base_p = 0;
    __shared__ int s_tot_p;
    for (int s0 = 0; s0 < p.S; s0 += nt) {
        int s = s0 + tid;
        int c = s < p.S ? cnt[s] : 0;
        int ru = block_scan_sum(c > 0, warp_tot, &s_tot_u);
        int rc = block_scan_sum(c, warp_tot, &s_tot_c);
        int rp = block_scan_sum((c + p.pass_tokens - 1) / p.pass_tokens, warp_tot, &s_tot_p);
        if (c > 0) {
            int u = base_u + ru;
            p.s.uslot[u] = s;
            p.s.ucnt[u] = c;
            p.s.uoff[u] = base_c + rc;
            if (p.s.upoff) p.s.upoff[u] = base_p + rp;
            cnt[s] = base_c + rc;
        }
        base_u += s_tot_u;
        base_c += s_tot_c;
        base_p += s_tot_p;
        __syncthreads();
    }
    if (tid == 0 && p.s.n_passes) *p.s.n_passes = base_p;
    for (int q = tid; q < p.P; q += nt) {
        const int s = p.slots[q];
        if (s < 0) continue;
        int pos = atomicAdd(&cnt[s], 1);
        p.s.upairs[pos] = q;
    }
    if (tid == 0) *p.s.n_unique = base_u;
}

// Stage the bf16 activations of `ntok` tokens (pairs upairs[first..]) into shared
// memory as [ntok, H] bf16.
__device__ __forceinline__ void stage_x_bf16(const FfnParams &p, const int *pairs, int ntok, uint4 *xs) {
    const int nv = p.H >> 3;
    for (int i = 0; i < ntok; i++) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.x) + (int64_t)(pairs[i] / p.topk) * nv;
        for (int v = threadIdx.x; v < nv; v += kThreads) xs[i * nv + v] = src[v];
    }
}

// ------------------------------------------------- gate_up, row-major formats

// One neuron n: gate row n and up row I + n against NT staged tokens.
template <int FMT, int NT>
__device__ __forceinline__ void gu_neuron(const FfnParams &p, int slot, int n, const uint4 *xs, float (&g)[NT],
                                          float (&u)[NT]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int t = 0; t < NT; t++) g[t] = u[t] = 0.f;
    if (FMT == FTMOE_FMT_BF16) {
        const int nch = p.H >> 3;  // 16-byte chunks per row
        const uint4 *wg = reinterpret_cast<const uint4 *>(p.bank[0] + (int64_t)slot * p.bank_bytes[0]) + (int64_t)n * nch;
        const uint4 *wu = wg + (int64_t)p.I * nch;
        constexpr int U = NT <= 2 ? 4 : (NT <= 4 ? 2 : 1);
        for (int c0 = lane; c0 < nch; c0 += 32 * U) {
            uint4 a[U], b[U];
#pragma unroll
            for (int k = 0; k < U; k++) {
                int c = c0 + 32 * k;
                if (c < nch) {
                    a[k] = ldg_stream(wg + c);
                    b[k] = ldg_stream(wu + c);
                }
            }
#pragma unroll
            for (int k = 0; k < U; k++) {
                int c = c0 + 32 * k;
                if (c < nch) {
                    float fa[8], fb[8];
                    unpack_bf16x8(a[k], fa);
                    unpack_bf16x8(b[k], fb);
#pragma unroll
                    for (int t = 0; t < NT; t++) {
                        float fx[8];
                        unpack_bf16x8(xs[t * nch + c], fx);
#pragma unroll
                        for (int i = 0; i < 8; i++) {
                            g[t] = fmaf(fa[i], fx[i], g[t]);
                            u[t] = fmaf(fb[i], fx[i], u[t]);
                        }
                    }
                }
            }
        }
    } else {  // NVFP4
        const int H = p.H;
        const int nch = H >> 5;  // 16-byte code chunks (32 weights) per row
        const int nxv = H >> 3;  // staged x: 16-byte vectors (8 bf16) per token
        const unsigned char *cg = p.bank[0] + (int64_t)slot * p.bank_bytes[0] + (int64_t)n * (H >> 1);
        const unsigned char *cu = cg + (int64_t)p.I * (H >> 1);
        const unsigned char *sg = p.bank[1] + (int64_t)slot * p.bank_bytes[1] + (int64_t)n * (H >> 4);
        const unsigned char *su = sg + (int64_t)p.I * (H >> 4);
        constexpr int U = NT <= 2 ? 2 : 1;
        for (int c0 = lane; c0 < nch; c0 += 32 * U) {
            uint4 a[U], b[U];
            uint32_t sa[U], sb[U];
#pragma unroll
            for (int k = 0; k < U; k++) {
                int c = c0 + 32 * k;
                if (c < nch) {
                    a[k] = ldg_stream(cg + 16 * (int64_t)c);
                    b[k] = ldg_stream(cu + 16 * (int64_t)c);
                    sa[k] = *reinterpret_cast<const unsigned short *>(sg + 2 * c);
                    sb[k] = *reinterpret_cast<const unsigned short *>(su + 2 * c);
                }
            }
#pragma unroll
            for (int k = 0; k < U; k++) {
                int c = c0 + 32 * k;
                if (c < nch) {
                    const uint32_t wa[4] = {a[k].x, a[k].y, a[k].z, a[k].w};
                    const uint32_t wb[4] = {b[k].x, b[k].y, b[k].z, b[k].w};
#pragma unroll
                    for (int blk = 0; blk < 2; blk++) {
                        float pg[NT], pu[NT];
#pragma unroll
                        for (int t = 0; t < NT; t++) pg[t] = pu[t] = 0.f;
#pragma unroll
                        for (int q = 0; q < 2; q++) {
                            float fa[8], fb[8];
                            e2m1x8(wa[2 * blk + q], fa);
                            e2m1x8(wb[2 * blk + q], fb);
#pragma unroll
                            for (int t = 0; t < NT; t++) {
                                float fx[8];
                                unpack_bf16x8(xs[t * nxv + 4 * c + 2 * blk + q], fx);
#pragma unroll
                                for (int i = 0; i < 8; i++) {
                                    pg[t] = fmaf(fa[i], fx[i], pg[t]);
                                    pu[t] = fmaf(fb[i], fx[i], pu[t]);
                                }
                            }
                        }
                        const float scg = e4m3_to_f(sa[k] >> (8 * blk));
                        const float scu = e4m3_to_f(sb[k] >> (8 * blk));
#pragma unroll
                        for (int t = 0; t < NT; t++) {
                            g[t] = fmaf(pg[t], scg, g[t]);
                            u[t] = fmaf(pu[t], scu, u[t]);
                        }
                    }
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; t++) {
        g[t] = warp_sum(g[t]);
        u[t] = warp_sum(u[t]);
    }
    if (FMT == FTMOE_FMT_NVFP4) {
        const unsigned char *gl = p.bank[2] + (int64_t)slot * p.bank_bytes[2];
        const float gg = __half2float(*reinterpret_cast<const __half *>(gl + 2 * (int64_t)n));
        const float gu = __half2float(*reinterpret_cast<const __half *>(gl + 2 * ((int64_t)p.I + n)));
#pragma unroll
        for (int t = 0; t < NT; t++) {
            g[t] *= gg;
            u[t] *= gu;
        }
    }
}

template <int FMT, int NT>
__device__ __forceinline__ void gu_rows_pass(const FfnParams &p, int slot, int tile, const int *pairs,
                                             const uint4 *xs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int w = warp; w < kGuNeurons; w += kThreads / 32) {
        const int n = tile * kGuNeurons + w;
        if (n >= p.I) break;
        float g[NT], u[NT];
        gu_neuron<FMT, NT>(p, slot, n, xs, g, u);
#pragma unroll
        for (int t = 0; t < NT; t++)
            if (lane == t) p.s.h[(int64_t)pairs[t] * p.I + n] = silu(g[t]) * u[t];
    }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) ffn_gate_up_rows_kernel(FfnParams p, int tiles, int tg) {
    extern __shared__ uint4 xs[];
    const int u = blockIdx.x / tiles, tile = blockIdx.x - u * tiles;
    if (u >= *p.s.n_unique) return;
    const int slot = p.s.uslot[u], cnt = p.s.ucnt[u];
    const int *pairs = p.s.upairs + p.s.uoff[u];
    for (int g0 = 0; g0 < cnt; g0 += tg) {
        const int ntok = cnt - g0 < tg ? cnt - g0 : tg;
        if (g0) __syncthreads();
        stage_x_bf16(p, pairs + g0, ntok, xs);
        __syncthreads();
        switch (ntok) {
            case 1: gu_rows_pass<FMT, 1>(p, slot, tile, pairs + g0, xs); break;
            case 2: gu_rows_pass<FMT, 2>(p, slot, tile, pairs + g0, xs); break;
            case 3: gu_rows_pass<FMT, 3>(p, slot, tile, pairs + g0, xs); break;
            default: gu_rows_pass<FMT, 4>(p, slot, tile, pairs + g0, xs); break;
        }
    }
}

// ---------------------------------------------------- down, row-major formats

// R output rows n0..n0+R-1 against NT staged h vectors (fp32 [NT, I]).
template <int FMT, int NT, int R>
__device__ __forceinline__ void dn_rows(const FfnParams &p, int slot, int n0, const float4 *hs, float (&o)[R][NT]) {
    const int lane = threadIdx.x & 31;
    const int I = p.I;
#pragma unroll
    for (int r = 0; r < R; r++)
#pragma unroll
        for (int t = 0; t < NT; t++) o[r][t] = 0.f;
    const int nh4 = I >> 2;  // float4 per staged h row
    if (FMT == FTMOE_FMT_BF16) {
        const int nch = I >> 3;
        const uint4 *w = reinterpret_cast<const uint4 *>(p.bank[1] + (int64_t)slot * p.bank_bytes[1]) + (int64_t)n0 * nch;
        for (int c = lane; c < nch; c += 32) {
            uint4 a[R];
#pragma unroll
            for (int r = 0; r < R; r++) a[r] = ldg_stream(w + (int64_t)r * nch + c);
            float fa[R][8];
#pragma unroll
            for (int r = 0; r < R; r++) unpack_bf16x8(a[r], fa[r]);
#pragma unroll
            for (int t = 0; t < NT; t++) {
                const float4 h0 = hs[t * nh4 + 2 * c], h1 = hs[t * nh4 + 2 * c + 1];
                const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
                for (int r = 0; r < R; r++)
#pragma unroll
                    for (int i = 0; i < 8; i++) o[r][t] = fmaf(fa[r][i], hv[i], o[r][t]);
            }
        }
    } else {  // NVFP4
        const int nch = I >> 5;
        const unsigned char *cw = p.bank[3] + (int64_t)slot * p.bank_bytes[3] + (int64_t)n0 * (I >> 1);
        const unsigned char *sw = p.bank[4] + (int64_t)slot * p.bank_bytes[4] + (int64_t)n0 * (I >> 4);
        for (int c = lane; c < nch; c += 32) {
            uint4 a[R];
            uint32_t sc[R];
#pragma unroll
            for (int r = 0; r < R; r++) {
                a[r] = ldg_stream(cw + (int64_t)r * (I >> 1) + 16 * (int64_t)c);
                sc[r] = *reinterpret_cast<const unsigned short *>(sw + (int64_t)r * (I >> 4) + 2 * c);
            }
#pragma unroll
            for (int blk = 0; blk < 2; blk++) {
                float part[R][NT];
#pragma unroll
                for (int r = 0; r < R; r++)
#pragma unroll
                    for (int t = 0; t < NT; t++) part[r][t] = 0.f;
#pragma unroll
                for (int q = 0; q < 2; q++) {
                    float fa[R][8];
#pragma unroll
                    for (int r = 0; r < R; r++) {
                        const uint32_t wr[4] = {a[r].x, a[r].y, a[r].z, a[r].w};
                        e2m1x8(wr[2 * blk + q], fa[r]);
                    }
#pragma unroll
                    for (int t = 0; t < NT; t++) {
                        const int hb = t * nh4 + 8 * c + 4 * blk + 2 * q;
                        const float4 h0 = hs[hb], h1 = hs[hb + 1];
                        const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
                        for (int r = 0; r < R; r++)
#pragma unroll
                            for (int i = 0; i < 8; i++) part[r][t] = fmaf(fa[r][i], hv[i], part[r][t]);
                    }
                }
#pragma unroll
                for (int r = 0; r < R; r++) {
                    const float sc_f = e4m3_to_f(sc[r] >> (8 * blk));
#pragma unroll
                    for (int t = 0; t < NT; t++) o[r][t] = fmaf(part[r][t], sc_f, o[r][t]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; r++)
#pragma unroll
        for (int t = 0; t < NT; t++) o[r][t] = warp_sum(o[r][t]);
    if (FMT == FTMOE_FMT_NVFP4) {
        const unsigned char *gl = p.bank[5] + (int64_t)slot * p.bank_bytes[5];
#pragma unroll
        for (int r = 0; r < R; r++) {
            const float gg = __half2float(*reinterpret_cast<const __half *>(gl + 2 * ((int64_t)n0 + r)));
#pragma unroll
            for (int t = 0; t < NT; t++) o[r][t] *= gg;
        }
    }
}

template <int FMT, int NT>
__device__ __forceinline__ void dn_rows_pass(const FfnParams &p, int slot, int tile, const int *pairs,
                                             const float4 *hs) {
    constexpr int R = 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int w = warp * R; w < kDnRows; w += (kThreads / 32) * R) {
        const int n0 = tile * kDnRows + w;
        if (n0 >= p.H) break;
        float o[R][NT];
        if (n0 + R <= p.H) {
            dn_rows<FMT, NT, R>(p, slot, n0, hs, o);
#pragma unroll
            for (int r = 0; r < R; r++)
#pragma unroll
                for (int t = 0; t < NT; t++)
                    if (lane == t) p.s.o[(int64_t)pairs[t] * p.H + n0 + r] = o[r][t];
        } else {
            float o1[1][NT];
            dn_rows<FMT, NT, 1>(p, slot, n0, hs, o1);
#pragma unroll
            for (int t = 0; t < NT; t++)
                if (lane == t) p.s.o[(int64_t)pairs[t] * p.H + n0] = o1[0][t];
        }
    }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) ffn_down_rows_kernel(FfnParams p, int tiles, int tg) {
    extern __shared__ float4 hs[];
    const int u = blockIdx.x / tiles, tile = blockIdx.x - u * tiles;
    if (u >= *p.s.n_unique) return;
    const int slot = p.s.uslot[u], cnt = p.s.ucnt[u];
    const int *pairs = p.s.upairs + p.s.uoff[u];
    const int nh4 = p.I >> 2;
    for (int g0 = 0; g0 < cnt; g0 += tg) {
        const int ntok = cnt - g0 < tg ? cnt - g0 : tg;
        if (g0) __syncthreads();
        for (int i = 0; i < ntok; i++) {
            const float4 *src = reinterpret_cast<const float4 *>(p.s.h) + (int64_t)pairs[g0 + i] * nh4;
            for (int v = threadIdx.x; v < nh4; v += kThreads) hs[i * nh4 + v] = src[v];
        }
        __syncthreads();
        switch (ntok) {
            case 1: dn_rows_pass<FMT, 1>(p, slot, tile, pairs + g0, hs); break;
            case 2: dn_rows_pass<FMT, 2>(p, slot, tile, pairs + g0, hs); break;
            case 3: dn_rows_pass<FMT, 3>(p, slot, tile, pairs + g0, hs); break;
            default: dn_rows_pass<FMT, 4>(p, slot, tile, pairs + g0, hs); break;
        }
    }
}

// ------------------------------------------------------- transposed (mxfp4)
//
// Matrix view: blocks [K/2, N] bytes, scales [K/32, N] e8m0, bias [N] bf16.
// A lane owns 4 adjacent columns c0..c0+3 of `NCOL` matrices (1 for down, 2 for
// gate_up: gate column n and up column I + n); warp w reduces the scale blocks
// [w*nsb/8, (w+1)*nsb/8); partial sums meet in shared memory.
template <int NT, int NCOL>
__device__ __forceinline__ void cols_partial(const unsigned char *blocks, const unsigned char *scales, int N,
                                             int K, const int (&col0)[NCOL], bool valid, const float2 *vs,
                                             float (&acc)[NCOL][4][NT]) {
    const int warp = threadIdx.x >> 5;
    const int nsb = K >> 5;                      // scale blocks along K
    const int b0 = (warp * nsb) >> 3, b1 = ((warp + 1) * nsb) >> 3;
    const int nkp = K >> 1;                      // k-pairs per staged vector
#pragma unroll
    for (int m = 0; m < NCOL; m++)
#pragma unroll
        for (int c = 0; c < 4; c++)
#pragma unroll
            for (int t = 0; t < NT; t++) acc[m][c][t] = 0.f;
    if (!valid) return;
    for (int sb = b0; sb < b1; sb++) {
        float part[NCOL][4][NT];
#pragma unroll
        for (int m = 0; m < NCOL; m++)
#pragma unroll
            for (int c = 0; c < 4; c++)
#pragma unroll
                for (int t = 0; t < NT; t++) part[m][c][t] = 0.f;
        uint32_t sw[NCOL];
#pragma unroll
        for (int m = 0; m < NCOL; m++) sw[m] = ldg_stream32(scales + (int64_t)sb * N + col0[m]);
        constexpr int RU = 8;  // k-pair rows loaded ahead
#pragma unroll
        for (int r0 = 0; r0 < 16; r0 += RU) {
            uint32_t wv[NCOL][RU];
#pragma unroll
            for (int m = 0; m < NCOL; m++)
#pragma unroll
                for (int r = 0; r < RU; r++)
                    wv[m][r] = ldg_stream32(blocks + (int64_t)(sb * 16 + r0 + r) * N + col0[m]);
#pragma unroll
            for (int r = 0; r < RU; r++) {
                const int kp = sb * 16 + r0 + r;
                float2 xv[NT];
#pragma unroll
                for (int t = 0; t < NT; t++) xv[t] = vs[t * nkp + kp];
#pragma unroll
                for (int m = 0; m < NCOL; m++) {
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const float2 w = e2m1x2((wv[m][r] >> (8 * c)) & 0xffu);
#pragma unroll
                        for (int t = 0; t < NT; t++)
                            part[m][c][t] = fmaf(w.x, xv[t].x, fmaf(w.y, xv[t].y, part[m][c][t]));
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < NCOL; m++)
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const float s = e8m0_to_f(sw[m] >> (8 * c));
#pragma unroll
                for (int t = 0; t < NT; t++) acc[m][c][t] = fmaf(part[m][c][t], s, acc[m][c][t]);
            }
    }
}

// Stage NT vectors of length K as float2 pairs: bf16 activations (gate_up) or fp32 h (down).
__device__ __forceinline__ void stage_x_f32(const FfnParams &p, const int *pairs, int ntok, float *vs) {
    const int H = p.H;
    for (int i = 0; i < ntok; i++) {
        const uint16_t *src = p.x + (int64_t)(pairs[i] / p.topk) * H;
        for (int k = threadIdx.x; k < H; k += kThreads) vs[i * H + k] = __uint_as_float((uint32_t)src[k] << 16);
    }
}

template <int NT>
__device__ __forceinline__ void gu_cols_pass(const FfnParams &p, int slot, int tile, const int *pairs,
                                             const float *vs, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int I = p.I, N = 2 * I;
    const int n = tile * kColTile + lane * 4;
    const bool valid = n < I;
    const int col0[2] = {n, I + n};
    float acc[2][4][NT];
    cols_partial<NT, 2>(p.bank[0] + (int64_t)slot * p.bank_bytes[0], p.bank[1] + (int64_t)slot * p.bank_bytes[1],
                        N, p.H, col0, valid, reinterpret_cast<const float2 *>(vs), acc);
    // red[warp][t][m][128 columns]
#pragma unroll
    for (int t = 0; t < NT; t++)
#pragma unroll
        for (int m = 0; m < 2; m++)
#pragma unroll
            for (int c = 0; c < 4; c++) red[((warp * NT + t) * 2 + m) * kColTile + lane * 4 + c] = acc[m][c][t];
    __syncthreads();
    const unsigned char *bias = p.bank[2] + (int64_t)slot * p.bank_bytes[2];
    for (int i = threadIdx.x; i < NT * kColTile; i += kThreads) {
        const int t = i / kColTile, col = i - t * kColTile;
        const int nn = tile * kColTile + col;
        if (nn >= I) continue;
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; w++) {
            g += red[((w * NT + t) * 2 + 0) * kColTile + col];
            u += red[((w * NT + t) * 2 + 1) * kColTile + col];
        }
        g += __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(bias)[nn] << 16);
        u += __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(bias)[I + nn] << 16);
        p.s.h[(int64_t)pairs[t] * I + nn] = silu(g) * u;
    }
}

__global__ void __launch_bounds__(kThreads, 2) ffn_gate_up_cols_kernel(FfnParams p, int tiles, int tg) {
    extern __shared__ float smf[];
    const int u = blockIdx.x / tiles, tile = blockIdx.x - u * tiles;
    if (u >= *p.s.n_unique) return;
    const int slot = p.s.uslot[u], cnt = p.s.ucnt[u];
    const int *pairs = p.s.upairs + p.s.uoff[u];
    float *vs = smf;
    float *red = smf + (size_t)tg * p.H;
    for (int g0 = 0; g0 < cnt; g0 += tg) {
        const int ntok = cnt - g0 < tg ? cnt - g0 : tg;
        if (g0) __syncthreads();
        stage_x_f32(p, pairs + g0, ntok, vs);
        __syncthreads();
        if (ntok == 1)
            gu_cols_pass<1>(p, slot, tile, pairs + g0, vs, red);
        else
            gu_cols_pass<2>(p, slot, tile, pairs + g0, vs, red);
    }
}

template <int NT>
__device__ __forceinline__ void dn_cols_pass(const FfnParams &p, int slot, int tile, const int *pairs,
                                             const float *vs, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = p.H;
    const int n = tile * kColTile + lane * 4;
    const bool valid = n < H;
    const int col0[1] = {n};
    float acc[1][4][NT];
    cols_partial<NT, 1>(p.bank[3] + (int64_t)slot * p.bank_bytes[3], p.bank[4] + (int64_t)slot * p.bank_bytes[4], H,
                        p.I, col0, valid, reinterpret_cast<const float2 *>(vs), acc);
#pragma unroll
    for (int t = 0; t < NT; t++)
#pragma unroll
        for (int c = 0; c < 4; c++) red[(warp * NT + t) * kColTile + lane * 4 + c] = acc[0][c][t];
    __syncthreads();
    const uint16_t *bias = reinterpret_cast<const uint16_t *>(p.bank[5] + (int64_t)slot * p.bank_bytes[5]);
    for (int i = threadIdx.x; i < NT * kColTile; i += kThreads) {
        const int t = i / kColTile, col = i - t * kColTile;
        const int nn = tile * kColTile + col;
        if (nn >= H) continue;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; w++) o += red[(w * NT + t) * kColTile + col];
        o += __uint_as_float((uint32_t)bias[nn] << 16);
        p.s.o[(int64_t)pairs[t] * H + nn] = o;
    }
}

__global__ void __launch_bounds__(kThreads, 2) ffn_down_cols_kernel(FfnParams p, int tiles, int tg) {
    extern __shared__ float smf[];
    const int u = blockIdx.x / tiles, tile = blockIdx.x - u * tiles;
    if (u >= *p.s.n_unique) return;
    const int slot = p.s.uslot[u], cnt = p.s.ucnt[u];
    const int *pairs = p.s.upairs + p.s.uoff[u];
    const int I = p.I;
    float *vs = smf;
    float *red = smf + (size_t)tg * I;
    for (int g0 = 0; g0 < cnt; g0 += tg) {
        const int ntok = cnt - g0 < tg ? cnt - g0 : tg;
        if (g0) __syncthreads();
        for (int i = 0; i < ntok; i++) {
            const float *src = p.s.h + (int64_t)pairs[g0 + i] * I;
            for (int k = threadIdx.x; k < I; k += kThreads) vs[i * I + k] = src[k];
        }
        __syncthreads();
        switch (ntok) {
            case 1: dn_cols_pass<1>(p, slot, tile, pairs + g0, vs, red); break;
            case 2: dn_cols_pass<2>(p, slot, tile, pairs + g0, vs, red); break;
            case 3: dn_cols_pass<3>(p, slot, tile, pairs + g0, vs, red); break;
            default: dn_cols_pass<4>(p, slot, tile, pairs + g0, vs, red); break;
        }
    }
}

// --------------------------------------------------------------------- combine

__global__ void __launch_bounds__(kThreads) ffn_combine_kernel(FfnParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // o comes from the down kernel
    if (*p.s.n_unique < 0) return;  // a bad slot: y is left untouched
    const int t = blockIdx.y;
    const int n4 = blockIdx.x * kThreads + threadIdx.x;  // 4 outputs per thread
    const int H = p.H;
    if (4 * n4 >= H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 *o4 = reinterpret_cast<const float4 *>(p.s.o);
    const int64_t h4 = H >> 2;
    // load a group of routed positions before using any of them (independent L2 reads)
    if (p.addend) acc = reinterpret_cast<const float4 *>(p.addend + (int64_t)t * H)[n4];
    for (int j0 = 0; j0 < p.topk; j0 += 8) {
        float4 ov[8];
        float wv[8];
#pragma unroll
        for (int jj = 0; jj < 8; jj++) {
            const int j = j0 + jj;
            wv[jj] = 0.f;
            ov[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < p.topk) {
                const int q = t * p.topk + j;
                if (p.slots[q] >= 0) {  // slot -1: the pair is computed elsewhere
                    wv[jj] = p.weights[q];
                    ov[jj] = o4[(int64_t)q * h4 + n4];
                }
            }
        }
#pragma unroll
        for (int jj = 0; jj < 8; jj++) {
            if (j0 + jj < p.topk) {
                acc.x = fmaf(wv[jj], ov[jj].x, acc.x);
                acc.y = fmaf(wv[jj], ov[jj].y, acc.y);
                acc.z = fmaf(wv[jj], ov[jj].z, acc.z);
                acc.w = fmaf(wv[jj], ov[jj].w, acc.w);
            }
        }
    }
    __nv_bfloat16 b0 = __float2bfloat16_rn(acc.x), b1 = __float2bfloat16_rn(acc.y);
    __nv_bfloat16 b2 = __float2bfloat16_rn(acc.z), b3 = __float2bfloat16_rn(acc.w);
    uint2 v;
    v.x = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
    v.y = (uint32_t)__bfloat16_as_ushort(b2) | ((uint32_t)__bfloat16_as_ushort(b3) << 16);
    reinterpret_cast<uint2 *>(p.y + (int64_t)t * H)[n4] = v;
}

int pick_tg(int tg_max, size_t per_token, size_t fixed_per_token, size_t budget) {
    int tg = tg_max;
    while (tg > 1 && (size_t)tg * (per_token + fixed_per_token) > budget) tg >>= 1;
    return tg;
}

template <typename K>
cudaError_t launch_dyn(K kernel, int grid, size_t smem, cudaStream_t st, const FfnParams &p, int tiles, int tg) {
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kernel<<<grid, kThreads, smem, st>>>(p, tiles, tg);
    return cudaGetLastError();
}

}  // namespace

int ffn_bf16_family(const FfnParams &p, int num_sms, const MxTmaMaps *mx, int kernels) {
    if (num_sms <= 0 || p.fmt != FTMOE_FMT_BF16) return FTMOE_FFN_ROWS;
    if (kernels == FTMOE_FFN_ROWS) return FTMOE_FFN_ROWS;
    if (kernels == FTMOE_FFN_MMA) return ffn_bf16_mma_supported(p, mx) ? FTMOE_FFN_MMA : FTMOE_FFN_ROWS;
    const bool tc05 = ffn_bf16_tc05_supported(p, mx);
    if (kernels == FTMOE_FFN_TC05 && tc05) return FTMOE_FFN_TC05;
    // AUTO: the tensor cores, except around one routed token per expert (E/4 <= P < 2E), where
    // the CUDA-core pipeline is 3-6% faster (c2 bs 16: 194 us against 206 us tcgen05 and
    // 210 us mma.sync); from two tokens per expert up tcgen05 wins (bs 32: 207 / 221 / 218 us,
    // bs 64: 209 / 242 / 330 us for tcgen05 / mma.sync / CUDA cores) and at bs 1 tcgen05 and
    // mma.sync tie (28 us)
    const bool one_per_expert = 4 * (int64_t)p.P >= p.E && p.P < 2 * (int64_t)p.E;
    if (kernels == FTMOE_FFN_AUTO && one_per_expert) return FTMOE_FFN_ROWS;
    if (tc05) return FTMOE_FFN_TC05;
    return ffn_bf16_mma_supported(p, mx) ? FTMOE_FFN_MMA : FTMOE_FFN_ROWS;
}

cudaError_t launch_ffn(const FfnParams &p_in, int num_sms, cudaStream_t st, const MxTmaMaps *mx, int kernels) {
    FfnParams p = p_in;
    cudaError_t e;
    size_t route_smem = (size_t)p.S * sizeof(int);
    if (route_smem > 48 * 1024) {
        e = cudaFuncSetAttribute(ffn_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)route_smem);
        if (e != cudaSuccess) return e;
    }
    const int bf16_family = ffn_bf16_family(p, num_sms, mx, kernels);
    const bool bf16_tc05 = bf16_family == FTMOE_FFN_TC05;
    const bool bf16_mma = bf16_family == FTMOE_FFN_MMA;
    const bool fp4_rows_tma = num_sms > 0 && !bf16_mma && !bf16_tc05 && ffn_rows_tma_supported(p);
    const bool mx_tma = num_sms > 0 && ffn_mx_tma_supported(p, mx);
    const bool fp8_tma = num_sms > 0 && ffn_fp8_tma_supported(p, mx);
    if (p.fmt == FTMOE_FMT_FP8 && !fp8_tma) return cudaErrorNotSupported;  // block FP8 has one pipeline only
    if (p.fmt == FTMOE_FMT_Q4_0 && !fp4_rows_tma) return cudaErrorNotSupported;  // so has Q4_0
    const bool want_x16 =
        (fp4_rows_tma && (p.fmt == FTMOE_FMT_NVFP4 || p.fmt == FTMOE_FMT_Q4_0)) || mx_tma || fp8_tma;
    p.x16_emax = p.fmt == FTMOE_FMT_MXFP4 ? 9 : (p.fmt == FTMOE_FMT_Q4_0 ? 8 : 10);
    p.x16_swz = fp4_rows_tma && p.fmt == FTMOE_FMT_NVFP4 ? 1 : (fp4_rows_tma && p.fmt == FTMOE_FMT_Q4_0 ? 2 : 0);
    p.pass_tokens = bf16_tc05 ? kTc05PassTokens : ((mx_tma || fp8_tma || bf16_mma) ? kMxPassTokens : kPassTokens);
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1 + (want_x16 ? p.bs : 0));
        cfg.blockDim = dim3(1024);
        cfg.dynamicSmemBytes = route_smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, ffn_route_kernel, p)) != cudaSuccess) return e;
    }

    const int umax = p.P < p.S ? p.P : p.S;  // distinct slots at most
    const size_t budget = 64 * 1024;
    bool pdl_combine = false;
    if (bf16_tc05) {
        if ((e = launch_ffn_bf16_tc05(p, *mx, num_sms, st)) != cudaSuccess) return e;
        pdl_combine = true;
    } else if (bf16_mma) {
        if ((e = launch_ffn_bf16_mma(p, *mx, num_sms, st)) != cudaSuccess) return e;
        pdl_combine = true;
    } else if (fp4_rows_tma) {
        if ((e = launch_ffn_rows_tma(p, num_sms, st)) != cudaSuccess) return e;
        pdl_combine = true;
    } else if (mx_tma) {
        if ((e = launch_ffn_mx_tma(p, *mx, num_sms, st)) != cudaSuccess) return e;
        pdl_combine = true;
    } else if (fp8_tma) {
        if ((e = launch_ffn_fp8_tma(p, *mx, num_sms, st)) != cudaSuccess) return e;
        pdl_combine = true;
    } else if (p.fmt == FTMOE_FMT_BF16 || p.fmt == FTMOE_FMT_NVFP4) {
        const int tiles_gu = (p.I + kGuNeurons - 1) / kGuNeurons;
        const int tg_gu = pick_tg(kRowsTgMax, (size_t)p.H * 2, 0, budget);
        const int tiles_dn = (p.H + kDnRows - 1) / kDnRows;
        const int tg_dn = pick_tg(kRowsTgMax, (size_t)p.I * 4, 0, budget);
        if (p.fmt == FTMOE_FMT_BF16) {
            e = launch_dyn(ffn_gate_up_rows_kernel<FTMOE_FMT_BF16>, umax * tiles_gu, (size_t)tg_gu * p.H * 2, st, p,
                           tiles_gu, tg_gu);
            if (e != cudaSuccess) return e;
            e = launch_dyn(ffn_down_rows_kernel<FTMOE_FMT_BF16>, umax * tiles_dn, (size_t)tg_dn * p.I * 4, st, p,
                           tiles_dn, tg_dn);
        } else {
            e = launch_dyn(ffn_gate_up_rows_kernel<FTMOE_FMT_NVFP4>, umax * tiles_gu, (size_t)tg_gu * p.H * 2, st, p,
                           tiles_gu, tg_gu);
            if (e != cudaSuccess) return e;
            e = launch_dyn(ffn_down_rows_kernel<FTMOE_FMT_NVFP4>, umax * tiles_dn, (size_t)tg_dn * p.I * 4, st, p,
                           tiles_dn, tg_dn);
        }
        if (e != cudaSuccess) return e;
    } else {  // MXFP4
        const int tiles_gu = (p.I + kColTile - 1) / kColTile;
        const size_t red_gu = (size_t)(kThreads / 32) * 2 * kColTile * 4;  // per token
        const int tg_gu = pick_tg(kColsGuTgMax, (size_t)p.H * 4, red_gu, 96 * 1024);
        const int tiles_dn = (p.H + kColTile - 1) / kColTile;
        const size_t red_dn = (size_t)(kThreads / 32) * kColTile * 4;
        const int tg_dn = pick_tg(kColsDnTgMax, (size_t)p.I * 4, red_dn, 96 * 1024);
        e = launch_dyn(ffn_gate_up_cols_kernel, umax * tiles_gu, (size_t)tg_gu * ((size_t)p.H * 4 + red_gu), st, p,
                       tiles_gu, tg_gu);
        if (e != cudaSuccess) return e;
        e = launch_dyn(ffn_down_cols_kernel, umax * tiles_dn, (size_t)tg_dn * ((size_t)p.I * 4 + red_dn), st, p,
                       tiles_dn, tg_dn);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.H / 4 + kThreads - 1) / kThreads, p.bs);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_combine ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, ffn_combine_kernel, p);
}

}  // namespace ftmoe
