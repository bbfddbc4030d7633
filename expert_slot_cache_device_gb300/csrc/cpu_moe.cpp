// Host CPU expert executor of the hybrid decode path.
//
// FreeToken benchmark guide, section 5.4: in hybrid mode the misses beyond the fetch
// cap are not copied to the GPU; their routed positions get slot -1 and a CPU MoE
// executor computes those experts from the page-locked host banks while the GPU
// computes the resident and fetched ones (architecture deep-dive, section 五: the CPU
// side runs a GEMV over the host expert banks). This is that executor for the bf16,
// nvfp4 and transposed mxfp4 bank schemas, with fp32 accumulation, split over std::thread
// workers (gate_up + SiLU * up for every CPU pair, then down). On the Grace host the inner
// loops use the BF16 extension's dot product (BFDOT: fp32 += two bf16 products per lane): bf16
// weights and activations enter unchanged, e2m1 codes become their exact bf16 values by two
// byte-table lookups, and the fp32 h rows of down enter as two bf16 vectors hi + lo (hi = h
// rounded to bf16, lo = the remainder rounded), about 16 significant bits. nvfp4 rows read their
// vectors in the even/odd order of each 16-element scale block, so that a code byte's two nibbles
// need no interleaving. Arm hosts without
// it run NEON fp32 loops (bf16 rows 16 weights per step in four accumulators; e2m1 codes
// through a table lookup of twice their values as int8, so the block scale takes the factor
// one half); other hosts run the plain loops.
#include <algorithm>
#include <chrono>
#include <cmath>
#include <condition_variable>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

#include <unistd.h>

#include "ftmoe.h"

// The Grace host (aarch64) runs the executor's inner loops on NEON (ARMv8-A base SIMD: 16-bit
// widening shifts, table lookups, fp32 fused multiply-adds); other hosts run the plain loops.
#if defined(__aarch64__) && defined(__ARM_NEON)
#include <arm_neon.h>
#include <sys/auxv.h>
#define FTMOE_CPU_NEON 1
#ifndef HWCAP2_BF16
#define HWCAP2_BF16 (1UL << 14)  // Linux aarch64 hwcap bit of the BF16 extension
#endif
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
    float e8m0[256];          // 2^(b - 127), as ldexp gives it (b = 255: infinity)
    uint8_t e2m1_lo[16], e2m1_hi[16];  // low and high byte of each e2m1 value as bf16 (exact)
    Tables() {
        for (int b = 0; b < 256; b++) e8m0[b] = std::ldexp(1.0f, b - 127);
        for (int c = 0; c < 16; c++) {
            const int mag = c & 7;
            const float v = mag < 2 ? 0.5f * mag : std::ldexp(1.0f + 0.5f * (mag & 1), (mag >> 1) - 1);
            e2m1[c] = (c & 8) ? -v : v;
            uint32_t u;
            std::memcpy(&u, &e2m1[c], sizeof u);  // two significant bits: the bf16 is the top half
            e2m1_lo[c] = static_cast<uint8_t>(u >> 16);
            e2m1_hi[c] = static_cast<uint8_t>(u >> 24);
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

// Persistent workers of parallel_for: started on first use (and grown on demand), then parked
// on a condition variable between calls, so a call pays a wake-up instead of a thread start
// per worker. One call runs at a time (calls from several host threads queue on the mutex).
// The pool belongs to the process that made it: a forked child has none of its threads, so it
// leaves the inherited pool untouched (never destroyed, never joined) and makes its own. Pools
// are never destroyed; their parked workers end with the process.
class WorkerPool {
  public:
    static WorkerPool &get() {
        static std::mutex mu;
        static WorkerPool *pool = nullptr;
        static pid_t owner = 0;
        std::lock_guard<std::mutex> lk(mu);
        if (!pool || owner != getpid()) {
            pool = new WorkerPool();
            owner = getpid();
        }
        return *pool;
    }
    // fn(a, b) over [0, n) split into nt contiguous ranges; range 0 runs on the calling thread.
    void run(int64_t n, int nt, const std::function<void(int64_t, int64_t)> &fn) {
        std::lock_guard<std::mutex> call(call_mu_);
        {
            std::unique_lock<std::mutex> lk(mu_);
            while (static_cast<int>(workers_.size()) < nt - 1) {
                const int id = static_cast<int>(workers_.size()) + 1;
                workers_.emplace_back([this, id] { loop(id); });
            }
            fn_ = &fn;
            n_ = n;
            nt_ = nt;
            pending_ = nt - 1;
            gen_++;
        }
        cv_.notify_all();
        fn(0, n / nt);
        std::unique_lock<std::mutex> lk(mu_);
        done_cv_.wait(lk, [this] { return pending_ == 0; });
        fn_ = nullptr;
    }
  private:
    void loop(int id) {
        uint64_t seen = 0;
        for (;;) {
            const std::function<void(int64_t, int64_t)> *fn;
            int64_t a, b;
            {
                std::unique_lock<std::mutex> lk(mu_);
                cv_.wait(lk, [&] { return gen_ != seen; });
                seen = gen_;
                if (id >= nt_) continue;  // not part of this call
                fn = fn_;
                a = n_ * id / nt_;
                b = n_ * (id + 1) / nt_;
            }
            (*fn)(a, b);
            std::lock_guard<std::mutex> lk(mu_);
            if (--pending_ == 0) done_cv_.notify_one();
        }
    }
    std::mutex call_mu_, mu_;
    std::condition_variable cv_, done_cv_;
    std::vector<std::thread> workers_;
    const std::function<void(int64_t, int64_t)> *fn_ = nullptr;
    int64_t n_ = 0;
    int nt_ = 0, pending_ = 0;
    uint64_t gen_ = 0;
};

template <typename F>
void parallel_for(int64_t n, int threads, F &&fn) {
    if (n <= 0) return;
    const int nt = static_cast<int>(std::min<int64_t>(threads, n));
    if (nt <= 1) {
        fn(0, n);
        return;
    }
    const std::function<void(int64_t, int64_t)> f = fn;
    WorkerPool::get().run(n, nt, f);
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

bool host_has_bf16() {
    static const bool has = (getauxval(AT_HWCAP2) & HWCAP2_BF16) != 0;
    return has;
}

#define FTMOE_BF16_FN __attribute__((target("+bf16")))

FTMOE_BF16_FN inline bfloat16x8_t ld_bf16(const uint16_t *p) {
    return vld1q_bf16(reinterpret_cast<const bfloat16_t *>(p));
}

// bf16 row . (vh + vl), vl only when LO: 32 weights per step, four accumulators (K % 8 == 0).
template <bool LO>
FTMOE_BF16_FN float dot_bf16_bfdot(const uint16_t *w, const uint16_t *vh, const uint16_t *vl, int64_t K) {
    float32x4_t a0 = vdupq_n_f32(0.f), a1 = a0, a2 = a0, a3 = a0;
    int64_t k = 0;
    for (; k + 32 <= K; k += 32) {
        const bfloat16x8_t w0 = ld_bf16(w + k), w1 = ld_bf16(w + k + 8), w2 = ld_bf16(w + k + 16),
                           w3 = ld_bf16(w + k + 24);
        a0 = vbfdotq_f32(a0, w0, ld_bf16(vh + k));
        a1 = vbfdotq_f32(a1, w1, ld_bf16(vh + k + 8));
        a2 = vbfdotq_f32(a2, w2, ld_bf16(vh + k + 16));
        a3 = vbfdotq_f32(a3, w3, ld_bf16(vh + k + 24));
        if (LO) {
            a0 = vbfdotq_f32(a0, w0, ld_bf16(vl + k));
            a1 = vbfdotq_f32(a1, w1, ld_bf16(vl + k + 8));
            a2 = vbfdotq_f32(a2, w2, ld_bf16(vl + k + 16));
            a3 = vbfdotq_f32(a3, w3, ld_bf16(vl + k + 24));
        }
    }
    for (; k + 8 <= K; k += 8) {
        const bfloat16x8_t w0 = ld_bf16(w + k);
        a0 = vbfdotq_f32(a0, w0, ld_bf16(vh + k));
        if (LO) a1 = vbfdotq_f32(a1, w0, ld_bf16(vl + k));
    }
    return vaddvq_f32(vaddq_f32(vaddq_f32(a0, a1), vaddq_f32(a2, a3)));
}

// nvfp4 rows run against activation vectors in the even/odd order of each 16-element scale block
// (its eight even elements, then its eight odd ones; see eo16_permute): a block's low nibbles are
// its even elements and its high nibbles its odd ones, so the nibbles need no interleaving, and
// BFDOT's lane pairs meet matching elements on both sides. Sixteen code bytes (two blocks) per
// step: nibbles split, bf16 low and high bytes looked up and interleaved.
FTMOE_BF16_FN inline void e2m1x32_bf16_eo(const uint8_t *codes, uint8x16_t tlo, uint8x16_t thi, bfloat16x8_t (&w)[4]) {
    const uint8x16_t c = vld1q_u8(codes);
    const uint8x16_t ev = vandq_u8(c, vdupq_n_u8(15)), od = vshrq_n_u8(c, 4);
    const uint8x16_t le = vqtbl1q_u8(tlo, ev), he = vqtbl1q_u8(thi, ev);
    const uint8x16_t lo = vqtbl1q_u8(tlo, od), ho = vqtbl1q_u8(thi, od);
    w[0] = vreinterpretq_bf16_u8(vzip1q_u8(le, he));  // first block, even elements
    w[1] = vreinterpretq_bf16_u8(vzip1q_u8(lo, ho));  // first block, odd elements
    w[2] = vreinterpretq_bf16_u8(vzip2q_u8(le, he));  // second block, even elements
    w[3] = vreinterpretq_bf16_u8(vzip2q_u8(lo, ho));  // second block, odd elements
}

// nvfp4 row . (vh + vl) over even/odd-ordered vectors (K % 32 == 0): per block two BFDOTs into a
// fresh partial (two more for vl, a second chain), scaled by the block's e4m3 scale into one of
// four accumulators; the row's f16 global last.
template <bool LO>
FTMOE_BF16_FN float row_nvfp4_bfdot(const uint8_t *codes, const uint8_t *sc, float g, const uint16_t *vh,
                                    const uint16_t *vl, int64_t K, const float *e4m3, uint8x16_t tlo,
                                    uint8x16_t thi) {
    float32x4_t acc[4] = {vdupq_n_f32(0.f), vdupq_n_f32(0.f), vdupq_n_f32(0.f), vdupq_n_f32(0.f)};
    for (int64_t b2 = 0; b2 < K / 32; b2++) {
        bfloat16x8_t w[4];
        e2m1x32_bf16_eo(codes + b2 * 16, tlo, thi, w);
        const uint16_t *v = vh + b2 * 32;
        const float s0 = e4m3[sc[2 * b2]], s1 = e4m3[sc[2 * b2 + 1]];
        const float32x4_t p0 = vbfdotq_f32(vbfdotq_f32(vdupq_n_f32(0.f), w[0], ld_bf16(v)), w[1], ld_bf16(v + 8));
        const float32x4_t p1 =
            vbfdotq_f32(vbfdotq_f32(vdupq_n_f32(0.f), w[2], ld_bf16(v + 16)), w[3], ld_bf16(v + 24));
        acc[0] = vfmaq_n_f32(acc[0], p0, s0);
        acc[1] = vfmaq_n_f32(acc[1], p1, s1);
        if (LO) {
            const uint16_t *u = vl + b2 * 32;
            const float32x4_t q0 =
                vbfdotq_f32(vbfdotq_f32(vdupq_n_f32(0.f), w[0], ld_bf16(u)), w[1], ld_bf16(u + 8));
            const float32x4_t q1 =
                vbfdotq_f32(vbfdotq_f32(vdupq_n_f32(0.f), w[2], ld_bf16(u + 16)), w[3], ld_bf16(u + 24));
            acc[2] = vfmaq_n_f32(acc[2], q0, s0);
            acc[3] = vfmaq_n_f32(acc[3], q1, s1);
        }
    }
    return vaddvq_f32(vaddq_f32(vaddq_f32(acc[0], acc[1]), vaddq_f32(acc[2], acc[3]))) * g;
}

// The gate and the up row of one nvfp4 neuron against the same even/odd-ordered bf16
// activations (each activation vector loaded once for both rows): out = {gate . v, up . v}.
FTMOE_BF16_FN void row2_nvfp4_bfdot(const uint8_t *cg, const uint8_t *sg, float gg, const uint8_t *cu,
                                    const uint8_t *su, float gu, const uint16_t *vh, int64_t K, const float *e4m3,
                                    uint8x16_t tlo, uint8x16_t thi, float (&out)[2]) {
    float32x4_t ag[2] = {vdupq_n_f32(0.f), vdupq_n_f32(0.f)}, au[2] = {vdupq_n_f32(0.f), vdupq_n_f32(0.f)};
    for (int64_t b2 = 0; b2 < K / 32; b2++) {
        bfloat16x8_t wg[4], wu[4];
        e2m1x32_bf16_eo(cg + b2 * 16, tlo, thi, wg);
        e2m1x32_bf16_eo(cu + b2 * 16, tlo, thi, wu);
        const uint16_t *v = vh + b2 * 32;
        const bfloat16x8_t x0 = ld_bf16(v), x1 = ld_bf16(v + 8), x2 = ld_bf16(v + 16), x3 = ld_bf16(v + 24);
        const float32x4_t pg0 = vbfdotq_f32(vbfdotq_f32(vdupq_n_f32(0.f), wg[0], x0), wg[1], x1);
        const float32x4_t pg1 = vbfdotq_f32(vbfdotq_f32(vdupq_n_f32(0.f), wg[2], x2), wg[3], x3);
        const float32x4_t pu0 = vbfdotq_f32(vbfdotq_f32(vdupq_n_f32(0.f), wu[0], x0), wu[1], x1);
        const float32x4_t pu1 = vbfdotq_f32(vbfdotq_f32(vdupq_n_f32(0.f), wu[2], x2), wu[3], x3);
        ag[0] = vfmaq_n_f32(ag[0], pg0, e4m3[sg[2 * b2]]);
        ag[1] = vfmaq_n_f32(ag[1], pg1, e4m3[sg[2 * b2 + 1]]);
        au[0] = vfmaq_n_f32(au[0], pu0, e4m3[su[2 * b2]]);
        au[1] = vfmaq_n_f32(au[1], pu1, e4m3[su[2 * b2 + 1]]);
    }
    out[0] = vaddvq_f32(vaddq_f32(ag[0], ag[1])) * gg;
    out[1] = vaddvq_f32(vaddq_f32(au[0], au[1])) * gu;
}

// One k-pair row of 16 columns of a transposed mxfp4 matrix (16 code bytes, low nibble = even
// k) against the k pair (vh[0], vh[1]) (and (vl[0], vl[1]) when LO), into the hi / lo
// accumulators of the four 4-column groups.
template <bool LO>
FTMOE_BF16_FN inline void mx_row16_bfdot(const uint8_t *codes, const uint16_t *vh, const uint16_t *vl, uint8x16_t tlo,
                                         uint8x16_t thi, float32x4_t (&ah)[4], float32x4_t (&al)[4]) {
    const uint8x16_t c = vld1q_u8(codes);
    const uint8x16_t ev = vandq_u8(c, vdupq_n_u8(15)), od = vshrq_n_u8(c, 4);
    const uint8x16_t z0 = vzip1q_u8(ev, od), z1 = vzip2q_u8(ev, od);
    const uint8x16_t l0 = vqtbl1q_u8(tlo, z0), h0 = vqtbl1q_u8(thi, z0);
    const uint8x16_t l1 = vqtbl1q_u8(tlo, z1), h1 = vqtbl1q_u8(thi, z1);
    const bfloat16x8_t w[4] = {vreinterpretq_bf16_u8(vzip1q_u8(l0, h0)), vreinterpretq_bf16_u8(vzip2q_u8(l0, h0)),
                               vreinterpretq_bf16_u8(vzip1q_u8(l1, h1)), vreinterpretq_bf16_u8(vzip2q_u8(l1, h1))};
    uint32_t xp;
    std::memcpy(&xp, vh, sizeof xp);  // (v[2i], v[2i+1]), v[2i] in the low half
    const bfloat16x8_t xh = vreinterpretq_bf16_u32(vdupq_n_u32(xp));
    for (int q = 0; q < 4; q++) ah[q] = vbfdotq_f32(ah[q], w[q], xh);
    if (LO) {
        std::memcpy(&xp, vl, sizeof xp);
        const bfloat16x8_t xl = vreinterpretq_bf16_u32(vdupq_n_u32(xp));
        for (int q = 0; q < 4; q++) al[q] = vbfdotq_f32(al[q], w[q], xl);
    }
}

// Columns [n0, n1) of a transposed mxfp4 matrix over the scale blocks [blk0, blk1) of the
// reduction axis, against vh + vl (see cols_dot): per k-pair row and 16 columns, the 16 code
// bytes become four bf16x8 vectors (4 columns x (even k, odd k)) and meet the k pair of v
// broadcast to every lane. out[n - n0] = the range's partial sum (no bias).
template <bool LO>
FTMOE_BF16_FN void cols_mx_bfdot(const uint8_t *const *b, int which, int64_t N, int64_t blk0, int64_t blk1,
                                 const uint16_t *vh, const uint16_t *vl, int64_t n0, int64_t n1, float *out) {
    const Tables &T = tables();
    const uint8x16_t tlo = vld1q_u8(T.e2m1_lo), thi = vld1q_u8(T.e2m1_hi);
    const uint8_t *blocks = b[3 * which], *scales = b[3 * which + 1];
    for (int64_t n = n0; n < n1; n++) out[n - n0] = 0.f;
    for (int64_t blk = blk0; blk < blk1; blk++) {
        const uint8_t *srow = scales + blk * N;
        int64_t n = n0;
        for (; n + 16 <= n1; n += 16) {
            // accumulators per (row parity, hi / lo, 4-column group): short dependency chains
            float32x4_t ah0[4], ah1[4], al0[4], al1[4];
            for (int q = 0; q < 4; q++) ah0[q] = ah1[q] = al0[q] = al1[q] = vdupq_n_f32(0.f);
            for (int64_t i = blk * 16; i < blk * 16 + 16; i += 2) {
                mx_row16_bfdot<LO>(blocks + i * N + n, vh + 2 * i, LO ? vl + 2 * i : nullptr, tlo, thi, ah0, al0);
                mx_row16_bfdot<LO>(blocks + (i + 1) * N + n, vh + 2 * i + 2, LO ? vl + 2 * i + 2 : nullptr, tlo, thi,
                                   ah1, al1);
            }
            float s[16];
            for (int j = 0; j < 16; j++) s[j] = T.e8m0[srow[n + j]];
            for (int q = 0; q < 4; q++) {
                float32x4_t a = vaddq_f32(ah0[q], ah1[q]);
                if (LO) a = vaddq_f32(a, vaddq_f32(al0[q], al1[q]));
                vst1q_f32(out + (n - n0) + 4 * q,
                          vfmaq_f32(vld1q_f32(out + (n - n0) + 4 * q), a, vld1q_f32(s + 4 * q)));
            }
        }
        for (; n < n1; n++) {  // ragged columns
            float part = 0.f;
            for (int64_t i = blk * 16; i < blk * 16 + 16; i++) {
                const uint8_t c = blocks[i * N + n];
                const float x0 = bf16_to_f(vh[2 * i]) + (LO ? bf16_to_f(vl[2 * i]) : 0.f);
                const float x1 = bf16_to_f(vh[2 * i + 1]) + (LO ? bf16_to_f(vl[2 * i + 1]) : 0.f);
                part += T.e2m1[c & 15] * x0 + T.e2m1[c >> 4] * x1;
            }
            out[n - n0] += part * T.e8m0[srow[n]];
        }
    }
}
#endif

#if FTMOE_CPU_NEON
// out = v in the even/odd order of each 16-element block (n % 16 == 0): out[16b + i] =
// v[16b + 2i], out[16b + 8 + i] = v[16b + 2i + 1], i < 8.
void eo16_permute(const uint16_t *v, int64_t n, uint16_t *out) {
    for (int64_t b = 0; b < n; b += 16)
        for (int i = 0; i < 8; i++) {
            out[b + i] = v[b + 2 * i];
            out[b + 8 + i] = v[b + 2 * i + 1];
        }
}

// fp32 -> bf16 bits, rounded to nearest even (finite inputs).
uint16_t f_to_bf16(float f) {
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    return static_cast<uint16_t>((u + 0x7fffu + ((u >> 16) & 1u)) >> 16);
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
        for (int64_t n = n0; n < n1; n++) out[n - n0] += part[n - n0] * T.e8m0[srow[n]];
    }
    for (int64_t n = n0; n < n1; n++) out[n - n0] += bf16_to_f(bias[n]);
}

#if FTMOE_CPU_NEON
// Row n of a row-major expert matrix (bf16 or nvfp4) . (vh + vl) on the BF16 dot product.
template <bool LO>
float row_dot_bfdot(int fmt, const uint8_t *const *b, int which, int64_t n, int64_t K, const uint16_t *vh,
                    const uint16_t *vl) {
    if (fmt == FTMOE_FMT_BF16)
        return dot_bf16_bfdot<LO>(reinterpret_cast<const uint16_t *>(b[which]) + n * K, vh, vl, K);
    const Tables &T = tables();
    const uint16_t g = reinterpret_cast<const uint16_t *>(b[3 * which + 2])[n];
    return row_nvfp4_bfdot<LO>(b[3 * which] + n * (K / 2), b[3 * which + 1] + n * (K / 16), f16_to_f(g), vh, vl, K,
                               T.e4m3, vld1q_u8(T.e2m1_lo), vld1q_u8(T.e2m1_hi));
}

// gate_up + SiLU * up, then down, of every CPU pair on the BF16 dot product: the activations
// enter as they are (bf16), the h rows as hi + lo bf16 vectors. Same work split as the fp32
// paths of ftmoe_cpu_expert_ffn.
void expert_ffn_bfdot(int format, int64_t H, int64_t I, int topk, const std::vector<int> &pairs,
                      const std::vector<const uint8_t *> &eb, int nb, const uint16_t *h_x, std::vector<float> &hs,
                      std::vector<float> &os, int threads) {
    const int64_t np = static_cast<int64_t>(pairs.size());
    auto xrow = [&](int64_t i) { return h_x + (int64_t)(pairs[static_cast<size_t>(i)] / topk) * H; };
    // nvfp4 rows read even/odd-ordered activation and h vectors (see row_nvfp4_bfdot)
    const bool eo = format == FTMOE_FMT_NVFP4;
    std::vector<uint16_t> xp(eo ? static_cast<size_t>(np * H) : 0);
    for (int64_t i = 0; i < np && eo; i++) eo16_permute(xrow(i), H, &xp[static_cast<size_t>(i * H)]);
    auto xv = [&](int64_t i) { return eo ? &xp[static_cast<size_t>(i * H)] : xrow(i); };
    // mxfp4 (transposed [K/2, N] codes): a work item is one pair's range of scale blocks over all
    // N columns, so a worker reads whole contiguous rows (16 rows x N bytes per block) instead of
    // one line per row at a stride of N bytes; the ranges' partial sums are added in range order.
    auto mx_matrix = [&](int which, int64_t N, int64_t K, const uint16_t *const *vh, const uint16_t *const *vl,
                         float *outp) {
        const int64_t KB = K / 32;
        const int64_t R = std::max<int64_t>(1, std::min<int64_t>(KB, (2 * threads + np - 1) / np));
        std::vector<float> part(static_cast<size_t>(np * R * N));
        parallel_for(np * R, threads, [&](int64_t a, int64_t b) {
            for (int64_t w = a; w < b; w++) {
                const int64_t i = w / R, r = w % R;
                const uint8_t *const *bk = &eb[static_cast<size_t>(i * nb)];
                float *dst = &part[static_cast<size_t>(w * N)];
                if (vl)
                    cols_mx_bfdot<true>(bk, which, N, KB * r / R, KB * (r + 1) / R, vh[i], vl[i], 0, N, dst);
                else
                    cols_mx_bfdot<false>(bk, which, N, KB * r / R, KB * (r + 1) / R, vh[i], nullptr, 0, N, dst);
            }
        });
        parallel_for(np, threads, [&](int64_t a, int64_t b) {
            for (int64_t i = a; i < b; i++) {
                const uint16_t *bias = reinterpret_cast<const uint16_t *>(eb[static_cast<size_t>(i * nb + 3 * which + 2)]);
                for (int64_t n = 0; n < N; n++) {
                    float v = 0.f;
                    for (int64_t r = 0; r < R; r++) v += part[static_cast<size_t>((i * R + r) * N + n)];
                    outp[i * N + n] = v + bf16_to_f(bias[n]);
                }
            }
        });
    };
    if (format == FTMOE_FMT_MXFP4) {
        std::vector<const uint16_t *> xr(static_cast<size_t>(np));
        for (int64_t i = 0; i < np; i++) xr[static_cast<size_t>(i)] = xrow(i);
        std::vector<float> gu(static_cast<size_t>(np * 2 * I));
        mx_matrix(0, 2 * I, H, xr.data(), nullptr, gu.data());
        for (int64_t i = 0; i < np; i++)
            for (int64_t n = 0; n < I; n++) hs[i * I + n] = silu(gu[i * 2 * I + n]) * gu[i * 2 * I + I + n];
    } else {
        const Tables &T = tables();
        parallel_for(np * I, threads, [&](int64_t a, int64_t b) {
            for (int64_t w = a; w < b; w++) {
                const int64_t i = w / I, n = w % I;
                const uint8_t *const *bk = &eb[static_cast<size_t>(i * nb)];
                float gu[2];
                if (format == FTMOE_FMT_BF16) {
                    gu[0] = row_dot_bfdot<false>(format, bk, 0, n, H, xv(i), nullptr);
                    gu[1] = row_dot_bfdot<false>(format, bk, 0, I + n, H, xv(i), nullptr);
                } else {
                    const uint16_t *gl = reinterpret_cast<const uint16_t *>(bk[2]);
                    row2_nvfp4_bfdot(bk[0] + n * (H / 2), bk[1] + n * (H / 16), f16_to_f(gl[n]),
                                     bk[0] + (I + n) * (H / 2), bk[1] + (I + n) * (H / 16), f16_to_f(gl[I + n]),
                                     xv(i), H, T.e4m3, vld1q_u8(T.e2m1_lo), vld1q_u8(T.e2m1_hi), gu);
                }
                hs[i * I + n] = silu(gu[0]) * gu[1];
            }
        });
    }
    std::vector<uint16_t> hh(static_cast<size_t>(np * I)), hl(static_cast<size_t>(np * I));
    for (size_t k = 0; k < hh.size(); k++) {
        hh[k] = f_to_bf16(hs[k]);
        hl[k] = f_to_bf16(hs[k] - bf16_to_f(hh[k]));
    }
    if (eo) {
        std::vector<uint16_t> t(static_cast<size_t>(I));
        for (int64_t i = 0; i < np; i++)
            for (std::vector<uint16_t> *v : {&hh, &hl}) {
                eo16_permute(v->data() + i * I, I, t.data());
                std::copy(t.begin(), t.end(), v->begin() + i * I);
            }
    }
    if (format == FTMOE_FMT_MXFP4) {
        std::vector<const uint16_t *> hr(static_cast<size_t>(np)), lr(static_cast<size_t>(np));
        for (int64_t i = 0; i < np; i++) {
            hr[static_cast<size_t>(i)] = &hh[static_cast<size_t>(i * I)];
            lr[static_cast<size_t>(i)] = &hl[static_cast<size_t>(i * I)];
        }
        mx_matrix(1, H, I, hr.data(), lr.data(), os.data());
    } else {
        parallel_for(np * H, threads, [&](int64_t a, int64_t b) {
            for (int64_t w = a; w < b; w++) {
                const int64_t i = w / H, n = w % H;
                os[i * H + n] = row_dot_bfdot<true>(format, &eb[static_cast<size_t>(i * nb)], 1, n, I, &hh[i * I],
                                                    &hl[i * I]);
            }
        });
    }
}
#endif

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
    std::vector<float> hs(static_cast<size_t>(np * I)), os(static_cast<size_t>(np * H));
#if FTMOE_CPU_NEON
    const bool bfdot = host_has_bf16();
    if (bfdot) expert_ffn_bfdot(format, H, I, topk, pairs, eb, nb, h_x, hs, os, threads);
#else
    const bool bfdot = false;
#endif
    std::vector<float> xs(bfdot ? 0 : static_cast<size_t>(np * H));
    for (int64_t i = 0; i < np && !bfdot; i++) {
        const int64_t t = pairs[i] / topk;
        for (int64_t k = 0; k < H; k++) xs[i * H + k] = bf16_to_f(h_x[t * H + k]);
    }
    if (bfdot) {
        // computed above
    } else if (format == FTMOE_FMT_MXFP4) {
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
