/*
 * Oracle: number formats and the expert FFN — TEST INFRASTRUCTURE ONLY.
 *
 * The pages name the bank formats ([BENCH] section 4.2: bf16 = gate_up and
 * down; nvfp4 = packed e2m1 codes, one e4m3 scale per 16 elements and one fp16
 * global per output row, for gate_up and for down; mxfp4 = transposed
 * _blocks / _scales / _bias) and that hit experts compute from the slot cache
 * ([BENCH] section 一). They give no element layout and no FFN formula; the
 * readings used here:
 *   bf16   gate_up [2I, H] output-row-major, rows [0, I) gate and [I, 2I) up;
 *          down [H, I] output-row-major.
 *   nvfp4  codes [N, K/2] (byte (n, i) holds k = 2i in the low nibble and
 *          k = 2i + 1 in the high nibble), scales [N, K/16] e4m3fn,
 *          global [N] fp16; w = e2m1 * e4m3 * f16.
 *   mxfp4  blocks [K/2, N] (transposed; low nibble = even k), scales [K/32, N]
 *          e8m0 (2^(b - 127)), bias [N] bf16; w = e2m1 * 2^(b - 127).
 *   fp8    block FP8 ([ARCH] section 五 lists "FP8 block" among the bank schemas):
 *          weight [N, K] e4m3fn output-row-major, scale [N/128, K/128] binary32
 *          row-major, one per 128 x 128 block; w = e4m3 * scale[n / 128][k / 128].
 *   q4_0   GGUF Q4_0 ([ARCH] sections 五 and 六 name a GGUF Q4_0 bank schema and MoE):
 *          each output row is K/32 blocks of 18 bytes, a binary16 scale d then 16
 *          bytes qs; element j < 16 of a block is the low nibble of qs[j], element
 *          j + 16 the high nibble; w = (nibble - 8) * d (the ggml Q4_0 block).
 *   FFN    gu = W_gu x (+ b_gu), h = silu(gu[0:I]) * gu[I:2I],
 *          o = W_d h (+ b_d), y_t = sum_j w_{t,j} o_{t,j}; all in fp64.
 * Number formats follow their published definitions: OCP 8-bit floating point
 * (E4M3, bias 7, no infinities, S.1111.111 = NaN), OCP Microscaling v1.0
 * (E2M1 with bias 1, E8M0 = 2^(e - 127), 0xFF = NaN), IEEE 754 binary16 and
 * binary32 (little-endian bytes), and bfloat16 = the upper half of a binary32.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#include "oracle.h"

/* ---------------------------------------------------------------- numbers */

static double dec_e2m1(uint32_t c) {
    int sign = (c >> 3) & 1, ex = (c >> 1) & 3, man = c & 1;
    double v = ex == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, ex - 1);
    return sign ? -v : v;
}

static double dec_e4m3(uint32_t b) {
    int sign = (b >> 7) & 1, ex = (b >> 3) & 15, man = b & 7;
    double v;
    if (ex == 15 && man == 7)
        v = NAN;
    else if (ex == 0)
        v = ldexp(man / 8.0, -6);
    else
        v = ldexp(1.0 + man / 8.0, ex - 7);
    return sign ? -v : v;
}

static double dec_e8m0(uint32_t b) {
    if ((b & 0xFF) == 0xFF) return NAN;
    return ldexp(1.0, (int)(b & 0xFF) - 127);
}

static double dec_f16(uint32_t h) {
    int sign = (h >> 15) & 1, ex = (h >> 10) & 31, man = h & 1023;
    double v;
    if (ex == 31)
        v = man ? NAN : INFINITY;
    else if (ex == 0)
        v = ldexp(man / 1024.0, -14);
    else
        v = ldexp(1.0 + man / 1024.0, ex - 15);
    return sign ? -v : v;
}

static double dec_bf16(uint32_t h) {
    uint32_t u = (h & 0xFFFFu) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double orc_decode(int32_t kind, uint32_t bits) {
    switch (kind) {
        case ORC_NUM_E2M1: return dec_e2m1(bits & 15);
        case ORC_NUM_E4M3: return dec_e4m3(bits & 255);
        case ORC_NUM_E8M0: return dec_e8m0(bits & 255);
        case ORC_NUM_F16: return dec_f16(bits & 0xFFFF);
        case ORC_NUM_BF16: return dec_bf16(bits & 0xFFFF);
        default: return NAN;
    }
}

static uint32_t rd16(const uint8_t *p, int64_t i) { return (uint32_t)p[2 * i] | ((uint32_t)p[2 * i + 1] << 8); }

static double rdf32(const uint8_t *p, int64_t i) {
    uint32_t u = (uint32_t)p[4 * i] | ((uint32_t)p[4 * i + 1] << 8) | ((uint32_t)p[4 * i + 2] << 16) |
                 ((uint32_t)p[4 * i + 3] << 24);
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static uint32_t nibble(uint8_t byte, int64_t k) { return (k % 2 == 0) ? (byte & 15u) : (byte >> 4); }

int32_t orc_num_banks(int32_t fmt) {
    switch (fmt) {
        case ORC_FMT_BF16: return 2;
        case ORC_FMT_NVFP4: return 6;
        case ORC_FMT_MXFP4: return 6;
        case ORC_FMT_FP8: return 4;
        case ORC_FMT_Q4_0: return 2;
        default: return -1;
    }
}

/* --------------------------------------------------------------- weights */

double orc_weight(int32_t fmt, int32_t which, const uint8_t *const *banks, int32_t H,
                  int32_t I, int64_t n, int64_t k) {
    int64_t N = which == 0 ? 2 * (int64_t)I : H; /* outputs */
    int64_t K = which == 0 ? H : I;              /* reduction length */
    if (fmt == ORC_FMT_BF16) {
        const uint8_t *w = banks[which];
        return dec_bf16(rd16(w, n * K + k));
    }
    if (fmt == ORC_FMT_NVFP4) {
        const uint8_t *codes = banks[3 * which + 0];
        const uint8_t *scales = banks[3 * which + 1];
        const uint8_t *global = banks[3 * which + 2];
        double c = dec_e2m1(nibble(codes[n * (K / 2) + k / 2], k));
        double s = dec_e4m3(scales[n * (K / 16) + k / 16]);
        double g = dec_f16(rd16(global, n));
        return c * s * g;
    }
    if (fmt == ORC_FMT_MXFP4) {
        const uint8_t *blocks = banks[3 * which + 0];
        const uint8_t *scales = banks[3 * which + 1];
        double c = dec_e2m1(nibble(blocks[(k / 2) * N + n], k));
        double s = dec_e8m0(scales[(k / 32) * N + n]);
        return c * s;
    }
    if (fmt == ORC_FMT_FP8) {
        const uint8_t *wq = banks[2 * which + 0];
        const uint8_t *sc = banks[2 * which + 1];
        int64_t kb = (K + 127) / 128; /* scale blocks along k */
        return dec_e4m3(wq[n * K + k]) * rdf32(sc, (n / 128) * kb + k / 128);
    }
    if (fmt == ORC_FMT_Q4_0) {
        const uint8_t *blk = banks[which] + (n * (K / 32) + k / 32) * 18;
        int64_t j = k % 32;
        uint32_t q = j < 16 ? (blk[2 + j] & 15u) : (blk[2 + j - 16] >> 4);
        return ((double)q - 8.0) * dec_f16(rd16(blk, 0));
    }
    return NAN;
}

double orc_bias(int32_t fmt, int32_t which, const uint8_t *const *banks, int32_t H,
                int32_t I, int64_t n) {
    (void)H;
    (void)I;
    if (fmt != ORC_FMT_MXFP4) return 0.0;
    return dec_bf16(rd16(banks[3 * which + 2], n));
}

/* ------------------------------------------------------------------ FFN */

static double silu(double z) { return z / (1.0 + exp(-z)); }

int orc_expert_ffn(int32_t fmt, int32_t H, int32_t I, int32_t bs, int32_t k,
                   int32_t num_banks, const uint8_t *const *pair_banks, const uint16_t *x,
                   const float *w, double *y, int32_t threads) {
    if (orc_num_banks(fmt) != num_banks || H <= 0 || I <= 0 || bs < 0 || k <= 0) return ORC_ERR_INVALID_ARG;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
    double *xt = (double *)malloc(sizeof(double) * (size_t)H);
    double *gu = (double *)malloc(sizeof(double) * 2 * (size_t)I);
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    double *o = (double *)malloc(sizeof(double) * (size_t)H);
    for (int32_t t = 0; t < bs; t++) {
        for (int32_t c = 0; c < H; c++) xt[c] = dec_bf16(x[(int64_t)t * H + c]);
        for (int32_t c = 0; c < H; c++) y[(int64_t)t * H + c] = 0.0;
        for (int32_t j = 0; j < k; j++) {
            const uint8_t *const *banks = pair_banks + ((int64_t)t * k + j) * num_banks;
            /* gate_up: gu[n] = sum_c W_gu[n, c] x[c] (+ bias) */
#pragma omp parallel for schedule(static)
            for (int64_t n = 0; n < 2 * (int64_t)I; n++) {
                double acc = 0.0;
                for (int64_t c = 0; c < H; c++) acc += orc_weight(fmt, 0, banks, H, I, n, c) * xt[c];
                gu[n] = acc + orc_bias(fmt, 0, banks, H, I, n);
            }
            for (int32_t i = 0; i < I; i++) h[i] = silu(gu[i]) * gu[I + i];
            /* down: o[n] = sum_i W_d[n, i] h[i] (+ bias) */
#pragma omp parallel for schedule(static)
            for (int64_t n = 0; n < H; n++) {
                double acc = 0.0;
                for (int64_t i = 0; i < I; i++) acc += orc_weight(fmt, 1, banks, H, I, n, i) * h[i];
                o[n] = acc + orc_bias(fmt, 1, banks, H, I, n);
            }
            double wt = (double)w[(int64_t)t * k + j];
            for (int32_t c = 0; c < H; c++) y[(int64_t)t * H + c] += wt * o[c];
        }
    }
    free(xt);
    free(gu);
    free(h);
    free(o);
    return ORC_OK;
}
