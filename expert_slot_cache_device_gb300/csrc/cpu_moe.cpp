// Host CPU expert executor of the hybrid decode path.
//
// FreeToken benchmark guide, section 5.4: in hybrid mode the misses beyond the fetch
// cap are not copied to the GPU; their routed positions get slot -1 and a CPU MoE
// executor computes those experts from the page-locked host banks while the GPU
// computes the resident and fetched ones (architecture deep-dive, section 五: the CPU
// side runs a GEMV over the host expert banks). This is that executor for the bf16,
// nvfp4 and transposed mxfp4 bank schemas, with fp32 accumulation, split over std::thread
// workers (gate_up + SiLU * up for every CPU pair, then down); on the Grace host the inner
// loops are NEON (bf16 rows 16 weights per step in four accumulators; e2m1 codes through a
// table lookup of twice their values as int8, so the block scale takes the factor one half).
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "ftmoe.h"

// The Grace host (aarch64) runs the executor's inner loops on NEON (ARMv8-A base SIMD: 16-bit
// widening shifts, table lookups, fp32 fused multiply-adds); other hosts run the plain loops.
#if defined(__aarch64__) && defined(__ARM_NEON)
#include <arm_neon.h>
#define FTMOE_CPU_NEON 1
#else
#define FTMOE_CPU_NEON 0
#endif

// records the library's thread-local error message (defined with the other entry points)
int ftmoe_probe_report(int code, const char *msg);

namespace {

float bf16_to_f(uint16_t b) {
    const uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return f;
}

float f16_to_f(uint16_t h) {
    const int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    float v;
    if (e == 0)
        v = std::ldexp(static_cast<float>(m), -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = std::ldexp(static_cast<float>(1024 + m), e - 25);
    return s ? -v : v;
}

struct Tables {
    float e2m1[16];
    float e4m3[256];
    Tables() {
        for (int c = 0; c < 16; c++) {
            const int mag = c & 7;
            const float v = mag < 2 ? 0.5f * mag : std::ldexp(1.0f + 0.5f * (mag & 1), (mag >> 1) - 1);
            e2m1[c] = (c & 8) ? -v : v;
        }
        for (int b = 0; b < 256; b++) {
            const int e = (b >> 3) & 15, m = b & 7;
            float v = e == 0 ? std::ldexp(static_cast<float>(m), -9) : std::ldexp(1.0f + m / 8.0f, e - 7);
            if (e == 15 && m == 7) v = NAN;
            e4m3[b] = (b & 0x80) ? -v : v;
        }
    }
};

const Tables &tables() {
    static const Tables t;
    return t;
}

float silu(float z) { return z / (1.0f + std::exp(-z)); }

template <typename F>
void parallel_for(int64_t n, int threads, F &&fn) {
    if (n <= 0) return;
    const int nt = static_cast<int>(std::min<int64_t>(threads, n));
    if (nt <= 1) {
        fn(0, n);
        return;
    }
    std::vector<std::thread> pool;
    pool.reserve(nt);
    for (int i = 0; i < nt; i++) {
        const int64_t a = n * i / nt, b = n * (i + 1) / nt;
        pool.emplace_back([&fn, a, b] { fn(a, b); });
    }
    for (auto &th : pool) th.join();
}

#if FTMOE_CPU_NEON
// Twice the e2m1 values, exact in int8, indexed by the 4-bit code (sign in bit 3).
const int8_t kE2m1x2[16] = {0, 1, 2, 3, 4, 6, 8, 12, 0, -1, -2, -3, -4, -6, -8, -12};

// bf16 row . v: 16 weights per step (bf16 -> fp32 by a 16-bit widening shift), four
// independent accumulators.
float dot_bf16_neon(const uint16_t *w, const float *v, int64_t K) {
    float32x4_t a0 = vdupq_n_f32(0.f), a1 = a0, a2 = a0, a3 = a0;
    int64_t k = 0;
    for (; k + 16 <= K; k += 16) {
        const uint16x8_t p = vld1q_u16(w + k), q = vld1q_u16(w + k + 8);
        a0 = vfmaq_f32(a0, vreinterpretq_f32_u32(vshll_n_u16(vget_low_u16(p), 16)), vld1q_f32(v + k));
        a1 = vfmaq_f32(a1, vreinterpretq_f32_u32(vshll_high_n_u16(p, 16)), vld1q_f32(v + k + 4));
        a2 = vfmaq_f32(a2, vreinterpretq_f32_u32(vshll_n_u16(vget_low_u16(q), 16)), vld1q_f32(v + k + 8));
        a3 = vfmaq_f32(a3, vreinterpretq_f32_u32(vshll_high_n_u16(q, 16)), vld1q_f32(v + k + 12));
    }
    float acc = vaddvq_f32(vaddq_f32(vaddq_f32(a0, a1), vaddq_f32(a2, a3)));
    for (; k < K; k++) acc += bf16_to_f(w[k]) * v[k];
    return acc;
}

// Sixteen e2m1 codes (eight bytes, low nibble = even k) of one nvfp4 scale block against
// v[0..16): the codes become twice their values as int8 by a table lookup, then fp32; the
// partial sum comes back as four lanes (the caller scales and accumulates them).
inline float32x4_t block16_e2m1_neon(const uint8_t *codes, const float *v, int8x16_t tbl) {
    const uint8x8_t c = vld1_u8(codes);
    const int8x8_t lo = vqtbl1_s8(tbl, vand_u8(c, vdup_n_u8(15)));
    const int8x8_t hi = vqtbl1_s8(tbl, vshr_n_u8(c, 4));
    const int16x8_t s0 = vmovl_s8(vzip1_s8(lo, hi)), s1 = vmovl_s8(vzip2_s8(lo, hi));  // k 0..7, 8..15
    float32x4_t p = vmulq_f32(vcvtq_f32_s32(vmovl_s16(vget_low_s16(s0))), vld1q_f32(v));
    p = vfmaq_f32(p, vcvtq_f32_s32(vmovl_high_s16(s0)), vld1q_f32(v + 4));
    p = vfmaq_f32(p, vcvtq_f32_s32(vmovl_s16(vget_low_s16(s1))), vld1q_f32(v + 8));
    p = vfmaq_f32(p, vcvtq_f32_s32(vmovl_high_s16(s1)), vld1q_f32(v + 12));
    return p;
}

// Sixteen columns of one transposed mxfp4 k-pair row: codes (16 bytes, one column each, low
// nibble = even k) against the pair (x0, x1), accumulated into four column vectors.
inline void cols16_e2m1_neon(const uint8_t *codes, float x0, float x1, int8x16_t tbl, float32x4_t (&acc)[4]) {
    const uint8x16_t c = vld1q_u8(codes);
    const int8x16_t lo = vqtbl1q_s8(tbl, vandq_u8(c, vdupq_n_u8(15)));
    const int8x16_t hi = vqtbl1q_s8(tbl, vshrq_n_u8(c, 4));
    const int16x8_t l0 = vmovl_s8(vget_low_s8(lo)), l1 = vmovl_high_s8(lo);
    const int16x8_t h0 = vmovl_s8(vget_low_s8(hi)), h1 = vmovl_high_s8(hi);
    acc[0] = vfmaq_n_f32(vfmaq_n_f32(acc[0], vcvtq_f32_s32(vmovl_s16(vget_low_s16(l0))), x0),
                         vcvtq_f32_s32(vmovl_s16(vget_low_s16(h0))), x1);
    acc[1] = vfmaq_n_f32(vfmaq_n_f32(acc[1], vcvtq_f32_s32(vmovl_high_s16(l0)), x0),
                         vcvtq_f32_s32(vmovl_high_s16(h0)), x1);
    acc[2] = vfmaq_n_f32(vfmaq_n_f32(acc[2], vcvtq_f32_s32(vmovl_s16(vget_low_s16(l1))), x0),
                         vcvtq_f32_s32(vmovl_s16(vget_low_s16(h1))), x1);
    acc[3] = vfmaq_n_f32(vfmaq_n_f32(acc[3], vcvtq_f32_s32(vmovl_high_s16(l1)), x0),
                         vcvtq_f32_s32(vmovl_high_s16(h1)), x1);
}
#endif

// Dot product of output row n of a row-major expert matrix (bf16 or nvfp4) with v[K].
float row_dot(int fmt, const uint8_t *const *b, int which, int64_t n, int64_t K, const float *v) {
    const Tables &T = tables();
#if FTMOE_CPU_NEON
    if (fmt == FTMOE_FMT_BF16)
        return dot_bf16_neon(reinterpret_cast<const uint16_t *>(b[which]) + n * K, v, K);
    {
        const uint8_t *codes = b[3 * which] + n * (K / 2);
        const uint8_t *sc = b[3 * which + 1] + n * (K / 16);
        const uint16_t g = reinterpret_cast<const uint16_t *>(b[3 * which + 2])[n];
        const int8x16_t tbl = vld1q_s8(kE2m1x2);
        float32x4_t a0 = vdupq_n_f32(0.f), a1 = a0;
        int64_t blk = 0;
        for (; blk + 2 <= K / 16; blk += 2) {  // two blocks per step, two accumulators
            a0 = vfmaq_n_f32(a0, block16_e2m1_neon(codes + blk * 8, v + blk * 16, tbl), 0.5f * T.e4m3[sc[blk]]);
            a1 = vfmaq_n_f32(a1, block16_e2m1_neon(codes + blk * 8 + 8, v + blk * 16 + 16, tbl),
                             0.5f * T.e4m3[sc[blk + 1]]);
        }
        if (blk < K / 16)
            a0 = vfmaq_n_f32(a0, block16_e2m1_neon(codes + blk * 8, v + blk * 16, tbl), 0.5f * T.e4m3[sc[blk]]);
        return vaddvq_f32(vaddq_f32(a0, a1)) * f16_to_f(g);
    }
#endif
    if (fmt == FTMOE_FMT_BF16) {
        const uint16_t *w = reinterpret_cast<const uint16_t *>(b[which]) + n * K;
        float acc = 0.f;
        for (int64_t k = 0; k < K; k++) acc += bf16_to_f(w[k]) * v[k];
        return acc;
    }
    const uint8_t *codes = b[3 * which] + n * (K / 2);
    const uint8_t *sc = b[3 * which + 1] + n * (K / 16);
    const uint16_t g = reinterpret_cast<const uint16_t *>(b[3 * which + 2])[n];
    float acc = 0.f;
    for (int64_t blk = 0; blk < K / 16; blk++) {
        float part = 0.f;
        for (int i = 0; i < 8; i++) {
            const uint8_t c = codes[blk * 8 + i];
            part += T.e2m1[c & 15] * v[blk * 16 + 2 * i] + T.e2m1[c >> 4] * v[blk * 16 + 2 * i + 1];
        }
        acc += part * T.e4m3[sc[blk]];
    }
    return acc * f16_to_f(g);
}

// Columns [n0, n1) of a transposed mxfp4 matrix (blocks [K/2, N], scales [K/32, N],
// bias [N]) against v[K]: out[n] = sum_k w(n, k) v[k] + bias[n].
void cols_dot(const uint8_t *const *b, int which, int64_t N, int64_t K, const float *v, int64_t n0, int64_t n1,
              float *out) {
    const Tables &T = tables();
    const uint8_t *blocks = b[3 * which], *scales = b[3 * which + 1];
    const uint16_t *bias = reinterpret_cast<const uint16_t *>(b[3 * which + 2]);
    std::vector<float> part(static_cast<size_t>(n1 - n0));
    for (int64_t n = n0; n < n1; n++) out[n - n0] = 0.f;
    for (int64_t blk = 0; blk < K / 32; blk++) {
        std::fill(part.begin(), part.end(), 0.f);
#if FTMOE_CPU_NEON
        // sixteen columns at a time: the block's 16 k-pair rows into four column vectors
        const int8x16_t tbl = vld1q_s8(kE2m1x2);
        int64_t n = n0;
        for (; n + 16 <= n1; n += 16) {
            float32x4_t acc[4] = {vdupq_n_f32(0.f), vdupq_n_f32(0.f), vdupq_n_f32(0.f), vdupq_n_f32(0.f)};
            for (int64_t i = blk * 16; i < blk * 16 + 16; i++)
                cols16_e2m1_neon(blocks + i * N + n, 0.5f * v[2 * i], 0.5f * v[2 * i + 1], tbl, acc);
            for (int q = 0; q < 4; q++) vst1q_f32(&part[n - n0 + 4 * q], acc[q]);
        }
        for (int64_t i = blk * 16; n < n1 && i < blk * 16 + 16; i++) {  // ragged columns
            const uint8_t *row = blocks + i * N;
            const float x0 = v[2 * i], x1 = v[2 * i + 1];
            for (int64_t m = n; m < n1; m++) {
                const uint8_t c = row[m];
                part[m - n0] += T.e2m1[c & 15] * x0 + T.e2m1[c >> 4] * x1;
            }
        }
#else
        for (int64_t i = blk * 16; i < blk * 16 + 16; i++) {
            const uint8_t *row = blocks + i * N;
            const float x0 = v[2 * i], x1 = v[2 * i + 1];
            for (int64_t n = n0; n < n1; n++) {
                const uint8_t c = row[n];
                part[n - n0] += T.e2m1[c & 15] * x0 + T.e2m1[c >> 4] * x1;
            }
        }
#endif
        const uint8_t *srow = scales + blk * N;
        for (int64_t n = n0; n < n1; n++) out[n - n0] += part[n - n0] * std::ldexp(1.0f, static_cast<int>(srow[n]) - 127);
    }
    for (int64_t n = n0; n < n1; n++) out[n - n0] += bf16_to_f(bias[n]);
}

}  // namespace

extern "C" int ftmoe_cpu_expert_ffn(int32_t format, int32_t H, int32_t I, int32_t bs, int32_t topk,
                                    const int32_t *h_topk_ids, const int32_t *h_slots,
                                    const void *const *h_layer_banks, const int64_t *bank_bytes,
                                    const uint16_t *h_x, const float *h_weights, float *h_y,
                                    int32_t threads) {
    if (format != FTMOE_FMT_BF16 && format != FTMOE_FMT_NVFP4 && format != FTMOE_FMT_MXFP4) return FTMOE_ERR_FORMAT;
    if (H <= 0 || I <= 0 || bs < 0 || topk <= 0 || !h_topk_ids || !h_slots || !h_layer_banks || !bank_bytes ||
        !h_x || !h_weights || !h_y)
        return FTMOE_ERR_INVALID_ARG;
    const int q = format == FTMOE_FMT_BF16 ? 8 : 32;
    if (H % q || I % q) return FTMOE_ERR_FORMAT;
    const int nb = format == FTMOE_FMT_BF16 ? 2 : 6;
    if (threads <= 0) threads = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));

    // pairs computed here: routed positions whose slot is -1
    std::vector<int> pairs;
    for (int64_t p = 0; p < (int64_t)bs * topk; p++)
        if (h_slots[p] == -1) pairs.push_back(static_cast<int>(p));
    std::fill(h_y, h_y + (int64_t)bs * H, 0.f);
    if (pairs.empty()) return FTMOE_OK;
    const int64_t np = static_cast<int64_t>(pairs.size());
    std::vector<const uint8_t *> eb(static_cast<size_t>(np * nb));
    for (int64_t i = 0; i < np; i++) {
        const int e = h_topk_ids[pairs[i]];
        if (e < 0) return FTMOE_ERR_ID_RANGE;
        for (int b = 0; b < nb; b++)
            eb[i * nb + b] = static_cast<const uint8_t *>(h_layer_banks[b]) + (int64_t)e * bank_bytes[b];
    }
    std::vector<float> xs(static_cast<size_t>(np * H)), hs(static_cast<size_t>(np * I)),
        os(static_cast<size_t>(np * H));
    for (int64_t i = 0; i < np; i++) {
        const int64_t t = pairs[i] / topk;
        for (int64_t k = 0; k < H; k++) xs[i * H + k] = bf16_to_f(h_x[t * H + k]);
    }
    if (format == FTMOE_FMT_MXFP4) {
        // gate_up: columns split over the workers, in chunks of 64 columns per pair
        const int64_t chunk = 64, nch = (I + chunk - 1) / chunk;
        parallel_for(np * nch, threads, [&](int64_t a, int64_t b) {
            std::vector<float> g(chunk), u(chunk);
            for (int64_t w = a; w < b; w++) {
                const int64_t i = w / nch, c0 = (w % nch) * chunk, c1 = std::min<int64_t>(I, c0 + chunk);
                const uint8_t *const *bk = &eb[i * nb];
                cols_dot(bk, 0, 2 * (int64_t)I, H, &xs[i * H], c0, c1, g.data());
                cols_dot(bk, 0, 2 * (int64_t)I, H, &xs[i * H], I + c0, I + c1, u.data());
                for (int64_t n = c0; n < c1; n++) hs[i * I + n] = silu(g[n - c0]) * u[n - c0];
            }
        });
        const int64_t nchd = (H + chunk - 1) / chunk;
        parallel_for(np * nchd, threads, [&](int64_t a, int64_t b) {
            for (int64_t w = a; w < b; w++) {
                const int64_t i = w / nchd, c0 = (w % nchd) * chunk, c1 = std::min<int64_t>(H, c0 + chunk);
                cols_dot(&eb[i * nb], 1, H, I, &hs[i * I], c0, c1, &os[i * H + c0]);
            }
        });
    } else {
        parallel_for(np * I, threads, [&](int64_t a, int64_t b) {
            for (int64_t w = a; w < b; w++) {
                const int64_t i = w / I, n = w % I;
                const uint8_t *const *bk = &eb[i * nb];
                const float g = row_dot(format, bk, 0, n, H, &xs[i * H]);
                const float u = row_dot(format, bk, 0, I + n, H, &xs[i * H]);
                hs[i * I + n] = silu(g) * u;
            }
        });
        parallel_for(np * H, threads, [&](int64_t a, int64_t b) {
            for (int64_t w = a; w < b; w++) {
                const int64_t i = w / H, n = w % H;
                os[i * H + n] = row_dot(format, &eb[i * nb], 1, n, I, &hs[i * I]);
            }
        });
    }
    // combine in routed order (fixed summation order)
    for (int64_t i = 0; i < np; i++) {
        const int64_t p = pairs[i], t = p / topk;
        const float w = h_weights[p];
        for (int64_t n = 0; n < H; n++) h_y[t * H + n] += w * os[i * H + n];
    }
    return FTMOE_OK;
}

// STREAM-style read ceiling of the host memory the CPU executor reads (benchmark guide,
// section 5.2: the bandwidth probe reports the CPU's memory read ceiling beside the link's).
// Each worker sums its contiguous share of the buffer as 64-bit words into eight independent
// accumulators (no dependency chain, so the loads stream at the memory system's rate); the
// result is folded into a volatile sink so the reads cannot be dropped.
extern "C" int ftmoe_measure_cpu_read(const void *h_buf, size_t bytes, int32_t threads, int32_t reps,
                                      double *gbps) {
    if (!h_buf || !gbps || bytes < 64 || reps <= 0)
        return ftmoe_probe_report(FTMOE_ERR_INVALID_ARG, "measure_cpu_read: NULL pointer, bytes < 64 or reps <= 0");
    if (threads <= 0) threads = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
    const uint64_t *w = static_cast<const uint64_t *>(h_buf);
    const int64_t nw = static_cast<int64_t>(bytes / 64) * 8;  // whole 64-byte lines
    static volatile uint64_t sink;
    double best = 1e30;
    for (int r = 0; r < reps; r++) {
        std::vector<uint64_t> part(static_cast<size_t>(threads), 0);
        const auto t0 = std::chrono::steady_clock::now();
        parallel_for(threads, threads, [&](int64_t a, int64_t b) {
            for (int64_t t = a; t < b; t++) {
                const int64_t lo = nw / 8 * t / threads * 8, hi = nw / 8 * (t + 1) / threads * 8;
                uint64_t s0 = 0, s1 = 0, s2 = 0, s3 = 0, s4 = 0, s5 = 0, s6 = 0, s7 = 0;
                for (int64_t i = lo; i < hi; i += 8) {
                    s0 += w[i]; s1 += w[i + 1]; s2 += w[i + 2]; s3 += w[i + 3];
                    s4 += w[i + 4]; s5 += w[i + 5]; s6 += w[i + 6]; s7 += w[i + 7];
                }
                part[static_cast<size_t>(t)] = s0 ^ s1 ^ s2 ^ s3 ^ s4 ^ s5 ^ s6 ^ s7;
            }
        });
        const auto t1 = std::chrono::steady_clock::now();
        uint64_t x = 0;
        for (uint64_t v : part) x ^= v;
        sink = x;
        best = std::min(best, std::chrono::duration<double>(t1 - t0).count());
    }
    *gbps = static_cast<double>(nw) * 8.0 / best / 1e9;
    return FTMOE_OK;
}
