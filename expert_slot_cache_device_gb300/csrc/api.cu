// Host side of the C-ABI: argument checks, workspace layout, host-bank mapping and
// kernel launches. See include/ftmoe.h for the contract of every entry point.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "internal.cuh"

using namespace ftmoe;

namespace {

// NVTX range around a hot-path call (K1 ensure, K2 copy, K3 FFN, prefetch, prefill): shown by
// Nsight tools on the host timeline; without a tool attached it costs two no-op calls.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(FTMOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CK(call, what)                            \
    do {                                          \
        cudaError_t e_ = (call);                  \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct Layout {
    size_t hdr, id2slot, owner, stamp, miss_ids, miss_slots, all_ids, pf_slots;
    size_t n_unique, uslot, ucnt, uoff, upairs, h, o, x16, xexp, hmax, upoff, pipe_slots;
    size_t total;
    bool ffn;
};

int schema_banks(int fmt) {
    switch (fmt) {
        case FTMOE_FMT_BF16: return 2;
        case FTMOE_FMT_NVFP4: return 6;
        case FTMOE_FMT_MXFP4: return 6;
        case FTMOE_FMT_FP8: return 4;
        case FTMOE_FMT_Q4_0: return 2;
        default: return -1;
    }
}

// Per-expert bytes of bank b of a format's schema.
int64_t schema_bytes(int fmt, int b, int64_t H, int64_t I) {
    if (fmt == FTMOE_FMT_BF16) return b == 0 ? 2 * I * H * 2 : H * I * 2;
    const int64_t N = b < 3 ? 2 * I : H, K = b < 3 ? H : I;
    if (fmt == FTMOE_FMT_NVFP4) {
        switch (b % 3) {
            case 0: return N * K / 2;
            case 1: return N * K / 16;
            default: return N * 2;
        }
    }
    if (fmt == FTMOE_FMT_MXFP4) {
        switch (b % 3) {
            case 0: return K / 2 * N;
            case 1: return K / 32 * N;
            default: return N * 2;
        }
    }
    if (fmt == FTMOE_FMT_FP8) {
        const int64_t Nf = b < 2 ? 2 * I : H, Kf = b < 2 ? H : I;
        return b % 2 == 0 ? Nf * Kf : ((Nf + 127) / 128) * ((Kf + 127) / 128) * 4;
    }
    if (fmt == FTMOE_FMT_Q4_0) return b == 0 ? 2 * I * (H / 32) * 18 : H * (I / 32) * 18;
    return -1;
}

int schema_dtype(int fmt, int b) {
    if (fmt == FTMOE_FMT_BF16) return FTMOE_DT_BF16;
    if (fmt == FTMOE_FMT_NVFP4) {
        const int d[3] = {FTMOE_DT_U8, FTMOE_DT_E4M3, FTMOE_DT_F16};
        return d[b % 3];
    }
    if (fmt == FTMOE_FMT_FP8) return b % 2 == 0 ? FTMOE_DT_E4M3 : FTMOE_DT_F32;
    if (fmt == FTMOE_FMT_Q4_0) return FTMOE_DT_Q4_0;
    const int d[3] = {FTMOE_DT_U8, FTMOE_DT_E8M0, FTMOE_DT_BF16};
    return d[b % 3];
}

Layout make_layout(int fmt, int E, int L, int S, int H, int I, int max_pairs) {
    Layout l{};
    size_t off = 0;
    const int maxm = E < S ? E : S;
    l.hdr = off; off += 256;
    l.id2slot = off; off += align256((size_t)E * L * 4);
    l.owner = off; off += align256((size_t)S * 4);
    l.stamp = off; off += align256((size_t)S * 4);
    l.miss_ids = off; off += align256((size_t)maxm * 4);
    l.miss_slots = off; off += align256((size_t)maxm * 4);
    l.all_ids = off; off += align256((size_t)E * 4);   // 0..E-1: the ids of a whole-layer prefetch
    l.pf_slots = off; off += align256((size_t)E * 4);  // slots written by a whole-layer prefetch
    l.ffn = fmt != FTMOE_FMT_RAW && max_pairs > 0;
    if (l.ffn) {
        const size_t P = (size_t)max_pairs;
        l.n_unique = off; off += 256;
        l.uslot = off; off += align256(P * 4);
        l.ucnt = off; off += align256(P * 4);
        l.uoff = off; off += align256(P * 4);
        l.upairs = off; off += align256(P * 4);
        l.h = off; off += align256(P * (size_t)I * 4);
        l.o = off; off += align256(P * (size_t)H * 4);
        // f16 activations [P, H], or for Q4_0 per token int16 [H] + fp32 block scales [H / 32]
        l.x16 = off; off += align256(P * ((size_t)H * 2 + (size_t)H / 8));
        l.xexp = off; off += align256(P * 4);
        l.hmax = off; off += align256(P * 4);
        l.upoff = off; off += align256(P * 4);
        l.pipe_slots = off; off += 2 * align256(P * 4);  // two routed-slot buffers of the prefill pipeline
    }
    l.total = off;
    return l;
}

int check_geometry(int fmt, int nb, int E, int L, int S, int H, int I, int max_pairs) {
    if (E <= 0 || E > FTMOE_MAX_EXPERTS) return fail(FTMOE_ERR_INVALID_ARG, "E=%d outside [1, %d]", E, FTMOE_MAX_EXPERTS);
    if (S <= 0 || S > FTMOE_MAX_SLOTS) return fail(FTMOE_ERR_INVALID_ARG, "S=%d outside [1, %d]", S, FTMOE_MAX_SLOTS);
    if (L <= 0 || (int64_t)L * E > (int64_t)1 << 30) return fail(FTMOE_ERR_INVALID_ARG, "L=%d invalid", L);
    if (nb <= 0 || nb > FTMOE_MAX_BANKS) return fail(FTMOE_ERR_INVALID_ARG, "num_banks=%d outside [1, %d]", nb, FTMOE_MAX_BANKS);
    if (max_pairs < 0) return fail(FTMOE_ERR_INVALID_ARG, "max_pairs < 0");
    if (fmt == FTMOE_FMT_RAW) return FTMOE_OK;
    if (schema_banks(fmt) < 0) return fail(FTMOE_ERR_FORMAT, "unknown format %d", fmt);
    if (nb != schema_banks(fmt))
        return fail(FTMOE_ERR_FORMAT, "format %d needs %d banks, got %d", fmt, schema_banks(fmt), nb);
    if (H <= 0 || I <= 0) return fail(FTMOE_ERR_INVALID_ARG, "H=%d, I=%d must be positive", H, I);
    const int q = fmt == FTMOE_FMT_BF16 ? 8 : (fmt == FTMOE_FMT_FP8 ? 512 : (fmt == FTMOE_FMT_Q4_0 ? 256 : 32));
    if (H % q || I % q)
        return fail(FTMOE_ERR_FORMAT, "format %d needs H and I multiples of %d (H=%d, I=%d)", fmt, q, H, I);
    return FTMOE_OK;
}

}  // namespace

int ftmoe::report_error(int code, const char *msg) { return fail(code, "%s", msg); }
int ftmoe_probe_report(int code, const char *msg) { return fail(code, "%s", msg); }

struct ftmoe_cache {
    int fmt, E, L, S, H, I, max_pairs, nb;
    int num_sms;
    int copy_mode = FTMOE_COPY_FUSED;
    int ffn_kernels = FTMOE_FFN_AUTO;
    int64_t dbg_wait_ns = 0;  // test settings (ftmoe_set_debug)
    int dbg_skip_stage = 0;
    int last_layer = -1;
    bool vec16 = true;
    std::vector<std::vector<const void *>> host;      // [nb][L] host addresses
    std::vector<std::vector<const unsigned char *>> dev_view;  // [nb][L] device views
    unsigned char *dev_slots[FTMOE_MAX_BANKS];
    int64_t bytes[FTMOE_MAX_BANKS];
    Tables t;
    FfnScratch s;
    bool ffn;
    MxTmaMaps mx;
    int32_t *all_ids = nullptr, *pf_slots = nullptr, *pipe_slots[2] = {nullptr, nullptr};
    cudaStream_t aux = nullptr;  // copy-engine stream of the prefill pipeline (created on first use)
    ~ftmoe_cache() {
        if (aux) cudaStreamDestroy(aux);
    }
};

namespace {
__global__ void iota_kernel(int32_t *p, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = i;
}
}  // namespace

extern "C" {

const char *ftmoe_last_error(void) { return g_err; }

int ftmoe_cache_workspace_bytes(int32_t format, int32_t num_banks, int32_t E, int32_t L, int32_t S, int32_t H,
                                int32_t I, int32_t max_pairs, size_t *bytes) {
    if (!bytes) return fail(FTMOE_ERR_INVALID_ARG, "bytes is NULL");
    int rc = check_geometry(format, num_banks, E, L, S, H, I, max_pairs);
    if (rc) return rc;
    *bytes = make_layout(format, E, L, S, H, I, max_pairs).total;
    return FTMOE_OK;
}

int ftmoe_cache_create(const ftmoe_bank_spec *banks, int32_t num_banks, int32_t format, int32_t E, int32_t L,
                       int32_t S, int32_t H, int32_t I, int32_t max_pairs, void *d_workspace,
                       size_t workspace_bytes, void *stream, ftmoe_cache_t **out) {
    if (!out) return fail(FTMOE_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!banks) return fail(FTMOE_ERR_INVALID_ARG, "banks is NULL");
    int rc = check_geometry(format, num_banks, E, L, S, H, I, max_pairs);
    if (rc) return rc;
    const Layout lay = make_layout(format, E, L, S, H, I, max_pairs);
    if (!d_workspace || ((uintptr_t)d_workspace & 255))
        return fail(FTMOE_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device pointer");
    if (workspace_bytes < lay.total)
        return fail(FTMOE_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes, lay.total);

    ftmoe_cache *c = new ftmoe_cache();
    c->fmt = format; c->E = E; c->L = L; c->S = S; c->H = H; c->I = I;
    c->max_pairs = max_pairs; c->nb = num_banks; c->ffn = lay.ffn;
    c->host.assign(num_banks, std::vector<const void *>(L, nullptr));
    c->dev_view.assign(num_banks, std::vector<const unsigned char *>(L, nullptr));
    for (int b = 0; b < num_banks; b++) {
        const ftmoe_bank_spec &bs = banks[b];
        const int64_t nbytes = bs.rows * bs.row_bytes;
        if (bs.rows <= 0 || bs.row_bytes <= 0) {
            delete c;
            return fail(FTMOE_ERR_INVALID_ARG, "bank %d: rows and row_bytes must be positive", b);
        }
        if (format != FTMOE_FMT_RAW) {
            const int64_t want = schema_bytes(format, b, H, I);
            if (nbytes != want) {
                delete c;
                return fail(FTMOE_ERR_FORMAT, "bank %d (%s): %lld bytes per expert, schema needs %lld", b,
                            bs.name ? bs.name : "?", (long long)nbytes, (long long)want);
            }
            if (bs.dtype != schema_dtype(format, b)) {
                delete c;
                return fail(FTMOE_ERR_FORMAT, "bank %d (%s): dtype %d, schema needs %d", b, bs.name ? bs.name : "?",
                            bs.dtype, schema_dtype(format, b));
            }
        }
        if (!bs.dev_slots || !bs.host_src) {
            delete c;
            return fail(FTMOE_ERR_INVALID_ARG, "bank %d: NULL dev_slots or host_src", b);
        }
        c->dev_slots[b] = static_cast<unsigned char *>(bs.dev_slots);
        c->bytes[b] = nbytes;
        if (nbytes % 16 || (uintptr_t)bs.dev_slots % 16) c->vec16 = false;
    }
    // map the host banks only once every bank passed the host-side checks
    for (int b = 0; b < num_banks; b++) {
        for (int l = 0; l < L; l++) {
            const void *h = banks[b].host_src[l];
            c->host[b][l] = h;
            if (!h) continue;
            if ((uintptr_t)h % 16) c->vec16 = false;
            cudaPointerAttributes attr;
            cudaError_t e = cudaPointerGetAttributes(&attr, h);
            if (e != cudaSuccess || attr.type != cudaMemoryTypeHost || !attr.devicePointer) {
                cudaGetLastError();
                delete c;
                return fail(FTMOE_ERR_INVALID_ARG, "bank %d layer %d: host pointer is not page-locked mapped memory", b,
                            l);
            }
            c->dev_view[b][l] = static_cast<const unsigned char *>(attr.devicePointer);
        }
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        delete c;
        return cuda_fail(e, "device query");
    }

    unsigned char *ws = static_cast<unsigned char *>(d_workspace);
    c->t.clock = reinterpret_cast<uint32_t *>(ws + lay.hdr);
    c->t.status = reinterpret_cast<int32_t *>(ws + lay.hdr + 4);
    c->t.num_miss = reinterpret_cast<int32_t *>(ws + lay.hdr + 8);
    c->t.stats = reinterpret_cast<unsigned long long *>(ws + lay.hdr + 16);
    c->t.id2slot = reinterpret_cast<int32_t *>(ws + lay.id2slot);
    c->t.owner = reinterpret_cast<int32_t *>(ws + lay.owner);
    c->t.stamp = reinterpret_cast<uint32_t *>(ws + lay.stamp);
    c->t.miss_ids = reinterpret_cast<int32_t *>(ws + lay.miss_ids);
    c->t.miss_slots = reinterpret_cast<int32_t *>(ws + lay.miss_slots);
    c->all_ids = reinterpret_cast<int32_t *>(ws + lay.all_ids);
    c->pf_slots = reinterpret_cast<int32_t *>(ws + lay.pf_slots);
    if (lay.ffn) {
        c->pipe_slots[0] = reinterpret_cast<int32_t *>(ws + lay.pipe_slots);
        c->pipe_slots[1] = reinterpret_cast<int32_t *>(ws + lay.pipe_slots + align256((size_t)max_pairs * 4));
        c->s.n_unique = reinterpret_cast<int32_t *>(ws + lay.n_unique);
        c->s.uslot = reinterpret_cast<int32_t *>(ws + lay.uslot);
        c->s.ucnt = reinterpret_cast<int32_t *>(ws + lay.ucnt);
        c->s.uoff = reinterpret_cast<int32_t *>(ws + lay.uoff);
        c->s.upairs = reinterpret_cast<int32_t *>(ws + lay.upairs);
        c->s.h = reinterpret_cast<float *>(ws + lay.h);
        c->s.o = reinterpret_cast<float *>(ws + lay.o);
        c->s.x16 = reinterpret_cast<uint16_t *>(ws + lay.x16);
        c->s.xexp = reinterpret_cast<int32_t *>(ws + lay.xexp);
        c->s.hmax = reinterpret_cast<uint32_t *>(ws + lay.hmax);
        c->s.upoff = reinterpret_cast<int32_t *>(ws + lay.upoff);
        c->s.n_passes = c->s.n_unique + 1;  // second word of the 256-byte n_unique block
    }
    if (format == FTMOE_FMT_MXFP4 && lay.ffn) {
        const unsigned char *sb[6];
        for (int b = 0; b < 6; b++) sb[b] = c->dev_slots[b];
        make_mx_tma_maps(c->mx, sb, S, H, I);  // on failure the FFN uses the register path
    }
    if (format == FTMOE_FMT_BF16 && lay.ffn) {
        const unsigned char *sb[2] = {c->dev_slots[0], c->dev_slots[1]};
        make_bf16_tma_maps(c->mx, sb, S, H, I);  // on failure the FFN uses the CUDA-core pipeline
    }
    if (format == FTMOE_FMT_FP8 && lay.ffn) {
        const unsigned char *sb[4];
        for (int b = 0; b < 4; b++) sb[b] = c->dev_slots[b];
        if (!make_fp8_tma_maps(c->mx, sb, S, H, I)) {  // block FP8 has no other FFN path
            delete c;
            return fail(FTMOE_ERR_FORMAT, "block FP8: tensor maps over the slot banks could not be encoded");
        }
    }
    e = launch_init_state(c->t, E, L, S, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) {
        iota_kernel<<<(E + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(c->all_ids, E);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        delete c;
        return cuda_fail(e, "init state");
    }
    *out = c;
    return FTMOE_OK;
}

int ftmoe_cache_destroy(ftmoe_cache_t *cache) {
    delete cache;
    return FTMOE_OK;
}

int ftmoe_set_copy_mode(ftmoe_cache_t *c, int32_t mode) {
    if (!c) return fail(FTMOE_ERR_INVALID_ARG, "cache is NULL");
    if (mode != FTMOE_COPY_FUSED && mode != FTMOE_COPY_PER_BANK && mode != FTMOE_COPY_ENGINE)
        return fail(FTMOE_ERR_INVALID_ARG, "unknown copy mode %d", mode);
    c->copy_mode = mode;
    return FTMOE_OK;
}

int ftmoe_set_debug(ftmoe_cache_t *c, int32_t what, int64_t value) {
    if (!c) return fail(FTMOE_ERR_INVALID_ARG, "cache is NULL");
    if (what == FTMOE_DEBUG_WAIT_NS) {
        if (value < 0) return fail(FTMOE_ERR_INVALID_ARG, "wait limit must be >= 0");
        c->dbg_wait_ns = value;
        return FTMOE_OK;
    }
    if (what == FTMOE_DEBUG_FFN_SKIP_STAGE) {
        if (value != 0 && value != 1) return fail(FTMOE_ERR_INVALID_ARG, "skip setting must be 0 or 1");
        c->dbg_skip_stage = (int)value;
        return FTMOE_OK;
    }
    return fail(FTMOE_ERR_INVALID_ARG, "unknown debug setting %d", what);
}

int ftmoe_set_ffn_kernels(ftmoe_cache_t *c, int32_t kind) {
    if (!c) return fail(FTMOE_ERR_INVALID_ARG, "cache is NULL");
    if (kind != FTMOE_FFN_AUTO && kind != FTMOE_FFN_ROWS && kind != FTMOE_FFN_MMA && kind != FTMOE_FFN_TC05)
        return fail(FTMOE_ERR_INVALID_ARG, "unknown FFN kernel kind %d", kind);
    if (kind != FTMOE_FFN_AUTO && c->fmt != FTMOE_FMT_BF16)
        return fail(FTMOE_ERR_FORMAT, "only bf16 caches have several FFN kernel families");
    if (kind == FTMOE_FFN_MMA && !c->mx.valid)
        return fail(FTMOE_ERR_FORMAT, "no tensor-core FFN for this cache (H, I multiples of 256 and FFN scratch)");
    if (kind == FTMOE_FFN_TC05 && !c->mx.tc_valid)
        return fail(FTMOE_ERR_FORMAT, "no tcgen05 FFN for this cache (H, I multiples of 256 and FFN scratch)");
    c->ffn_kernels = kind;
    return FTMOE_OK;
}

int ftmoe_ffn_kernels_for(ftmoe_cache_t *c, int32_t bs, int32_t topk, int32_t *kind) {
    if (!c || !kind) return fail(FTMOE_ERR_INVALID_ARG, "NULL argument");
    if (bs < 0 || topk <= 0 || (int64_t)bs * topk > FTMOE_MAX_IDS_PER_CALL)
        return fail(FTMOE_ERR_INVALID_ARG, "bs=%d, topk=%d", bs, topk);
    if (!c->ffn) return fail(FTMOE_ERR_STATE, "the cache was created without FFN scratch");
    FfnParams p;
    memset(&p, 0, sizeof p);
    p.s = c->s;
    p.fmt = c->fmt; p.H = c->H; p.I = c->I; p.S = c->S; p.bs = bs; p.topk = topk; p.P = bs * topk;
    p.E = c->E;
    if (c->fmt == FTMOE_FMT_BF16)
        *kind = ffn_bf16_family(p, c->num_sms, &c->mx, c->ffn_kernels);
    else  // block FP8 and mxfp4 run on the tensor cores, nvfp4 and Q4_0 on the CUDA cores
        *kind = (c->fmt == FTMOE_FMT_FP8 || (c->fmt == FTMOE_FMT_MXFP4 && c->mx.valid)) ? FTMOE_FFN_MMA
                                                                                        : FTMOE_FFN_ROWS;
    return FTMOE_OK;
}

static int ensure_impl(ftmoe_cache_t *c, int32_t layer, const int32_t *d_topk_ids, int32_t bs, int32_t topk,
                       int32_t *d_slots_out, int hybrid, int32_t max_fetch, float fetch_fraction, int32_t *d_counts,
                       void *stream) {
    if (!c) return fail(FTMOE_ERR_INVALID_ARG, "cache is NULL");
    if (layer < 0 || layer >= c->L) return fail(FTMOE_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, c->L);
    if (bs < 0 || topk < 0) return fail(FTMOE_ERR_INVALID_ARG, "bs and topk must be >= 0");
    const int64_t n = (int64_t)bs * topk;
    if (n > FTMOE_MAX_IDS_PER_CALL) return fail(FTMOE_ERR_INVALID_ARG, "bs*topk=%lld above %d", (long long)n, FTMOE_MAX_IDS_PER_CALL);
    if (n > 0 && (!d_topk_ids || !d_slots_out)) return fail(FTMOE_ERR_INVALID_ARG, "NULL ids or slots_out");
    for (int b = 0; b < c->nb; b++)
        if (!c->dev_view[b][layer])
            return fail(FTMOE_ERR_INVALID_ARG, "layer %d of bank %d has no host source", layer, b);
    EnsureParams p;
    p.t = c->t;
    p.ids = d_topk_ids;
    p.slots_out = d_slots_out;
    p.E = c->E; p.L = c->L; p.S = c->S; p.layer = layer; p.n = (int)n;
    int spad = 2;
    while (spad < c->S) spad <<= 1;
    p.Spad = spad;
    p.maxm = c->E < c->S ? c->E : c->S;
    p.hybrid = hybrid;
    p.max_fetch = max_fetch;
    p.fetch_fraction = fetch_fraction;
    p.counts = d_counts;
    cudaError_t e = launch_ensure(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ensure kernel");
    c->last_layer = layer;
    return FTMOE_OK;
}

int ftmoe_ensure_experts(ftmoe_cache_t *c, int32_t layer, const int32_t *d_topk_ids, int32_t bs, int32_t topk,
                         int32_t *d_slots_out, void *stream) {
    NvtxRange nvtx_range("ftmoe_ensure_experts");
    return ensure_impl(c, layer, d_topk_ids, bs, topk, d_slots_out, 0, -1, 0.f, nullptr, stream);
}

int ftmoe_ensure_experts_hybrid(ftmoe_cache_t *c, int32_t layer, const int32_t *d_topk_ids, int32_t bs,
                                int32_t topk, int32_t max_fetch, float fetch_fraction, int32_t *d_slots_out,
                                int32_t *d_counts, void *stream) {
    NvtxRange nvtx_range("ftmoe_ensure_experts_hybrid");
    return ensure_impl(c, layer, d_topk_ids, bs, topk, d_slots_out, 1, max_fetch, fetch_fraction, d_counts, stream);
}

int ftmoe_hybrid_fetch_fraction(double pcie_gbps, double cpu_gbps, float *out) {
    if (!out) return fail(FTMOE_ERR_INVALID_ARG, "out is NULL");
    if (!(pcie_gbps > 0.0) || !(cpu_gbps > 0.0))
        *out = 0.f;
    else if (cpu_gbps <= pcie_gbps)
        *out = 1.f;
    else
        *out = (float)(pcie_gbps / cpu_gbps);
    return FTMOE_OK;
}

static void fill_copy_params(const ftmoe_cache *c, int b_first, int b_count, CopyParams &p) {
    memset(&p, 0, sizeof p);
    p.nb = b_count;
    p.E = c->E;
    p.L = c->L;
    p.S = c->S;
    p.maxm = c->E < c->S ? c->E : c->S;
    p.status = c->t.status;
    p.miss_ids = c->t.miss_ids;
    p.miss_slots = c->t.miss_slots;
    p.num_miss = c->t.num_miss;
    int64_t tiles = 0;
    for (int i = 0; i < b_count; i++) {
        const int b = b_first + i;
        p.src[i] = c->dev_view[b][c->last_layer];
        p.dst[i] = c->dev_slots[b];
        p.bytes[i] = c->bytes[b];
        p.tile0[i] = tiles;
        tiles += (c->bytes[b] + kCopyTile - 1) / kCopyTile;
    }
    p.tile0[b_count] = tiles;
}

// Copy-engine arm of copy_missing: reads the last ensure's miss list back (waiting on
// read_st) and issues one cudaMemcpyAsync per (miss, bank) on copy_st.
static int copy_engine(ftmoe_cache_t *c, cudaStream_t read_st, cudaStream_t copy_st) {
    const int maxm = c->E < c->S ? c->E : c->S;
    std::vector<int32_t> ids(maxm), slots(maxm);
    int32_t m = 0;
    CK(cudaMemcpyAsync(&m, c->t.num_miss, 4, cudaMemcpyDeviceToHost, read_st), "read miss count");
    CK(cudaStreamSynchronize(read_st), "sync");
    if (m > 0) {
        CK(cudaMemcpyAsync(ids.data(), c->t.miss_ids, (size_t)m * 4, cudaMemcpyDeviceToHost, read_st), "read miss ids");
        CK(cudaMemcpyAsync(slots.data(), c->t.miss_slots, (size_t)m * 4, cudaMemcpyDeviceToHost, read_st),
           "read miss slots");
        CK(cudaStreamSynchronize(read_st), "sync");
    }
    // misses come in ascending expert id; a run of consecutive experts landing in
    // consecutive slots is contiguous on both sides, so it is one transfer per bank (split
    // into transfers of at most kEngineChunk bytes)
    constexpr size_t kEngineChunk = (size_t)256 << 20;
    for (int j = 0; j < m;) {
        const int64_t e = ids[j] % c->E, s = slots[j];
        int run = 1;
        while (j + run < m && ids[j + run] == ids[j] + run && slots[j + run] == slots[j] + run) run++;
        for (int b = 0; b < c->nb; b++) {
            const unsigned char *src = static_cast<const unsigned char *>(c->host[b][c->last_layer]) + e * c->bytes[b];
            unsigned char *dst = c->dev_slots[b] + s * c->bytes[b];
            const size_t total = (size_t)run * c->bytes[b];
            for (size_t off = 0; off < total; off += kEngineChunk) {
                const size_t n = total - off < kEngineChunk ? total - off : kEngineChunk;
                CK(cudaMemcpyAsync(dst + off, src + off, n, cudaMemcpyHostToDevice, copy_st), "copy engine");
            }
        }
        j += run;
    }
    return FTMOE_OK;
}

int ftmoe_copy_missing(ftmoe_cache_t *c, void *stream) {
    NvtxRange nvtx_range("ftmoe_copy_missing");
    if (!c) return fail(FTMOE_ERR_INVALID_ARG, "cache is NULL");
    if (c->last_layer < 0) return fail(FTMOE_ERR_STATE, "copy_missing before any ensure_experts call");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int grid = c->num_sms * 4;
    if (c->copy_mode == FTMOE_COPY_FUSED) {
        CopyParams p;
        fill_copy_params(c, 0, c->nb, p);
        CK(launch_copy(p, c->vec16, grid, st), "copy kernel");
    } else if (c->copy_mode == FTMOE_COPY_PER_BANK) {
        for (int b = 0; b < c->nb; b++) {
            CopyParams p;
            fill_copy_params(c, b, 1, p);
            CK(launch_copy(p, c->vec16, grid, st), "copy kernel (per bank)");
        }
    } else {
        return copy_engine(c, st, st);
    }
    return FTMOE_OK;
}

int ftmoe_expert_ffn(ftmoe_cache_t *c, const void *d_x_bf16, int32_t bs, const int32_t *d_slots,
                     const float *d_weights, int32_t topk, void *d_y_bf16, void *stream) {
    NvtxRange nvtx_range("ftmoe_expert_ffn");
    return ftmoe_expert_ffn_hybrid(c, d_x_bf16, bs, d_slots, d_weights, topk, nullptr, d_y_bf16, stream);
}

int ftmoe_expert_ffn_hybrid(ftmoe_cache_t *c, const void *d_x_bf16, int32_t bs, const int32_t *d_slots,
                            const float *d_weights, int32_t topk, const float *d_addend, void *d_y_bf16,
                            void *stream) {
    NvtxRange nvtx_range("ftmoe_expert_ffn_hybrid");
    if (!c) return fail(FTMOE_ERR_INVALID_ARG, "cache is NULL");
    if (c->fmt == FTMOE_FMT_RAW) return fail(FTMOE_ERR_FORMAT, "a raw-format cache has no FFN");
    if (!c->ffn) return fail(FTMOE_ERR_INVALID_ARG, "cache created with max_pairs = 0");
    if (bs < 0 || topk <= 0) return fail(FTMOE_ERR_INVALID_ARG, "bs >= 0 and topk > 0 required");
    const int64_t P = (int64_t)bs * topk;
    if (P > c->max_pairs) return fail(FTMOE_ERR_INVALID_ARG, "bs*topk=%lld above max_pairs=%d", (long long)P, c->max_pairs);
    if (P == 0) return FTMOE_OK;
    if (!d_x_bf16 || !d_slots || !d_weights || !d_y_bf16) return fail(FTMOE_ERR_INVALID_ARG, "NULL FFN argument");
    if (((uintptr_t)d_x_bf16 | (uintptr_t)d_y_bf16 | (uintptr_t)d_addend) % 16)
        return fail(FTMOE_ERR_INVALID_ARG, "x, y and the addend must be 16-byte aligned");
    FfnParams p;
    memset(&p, 0, sizeof p);
    p.s = c->s;
    for (int b = 0; b < c->nb && b < 6; b++) {
        p.bank[b] = c->dev_slots[b];
        p.bank_bytes[b] = c->bytes[b];
    }
    p.x = static_cast<const uint16_t *>(d_x_bf16);
    p.slots = d_slots;
    p.weights = d_weights;
    p.addend = d_addend;
    p.y = static_cast<uint16_t *>(d_y_bf16);
    p.status = c->t.status;
    p.fmt = c->fmt; p.H = c->H; p.I = c->I; p.S = c->S; p.bs = bs; p.topk = topk; p.P = (int)P;
    p.E = c->E;
    p.wait_ns = (uint64_t)c->dbg_wait_ns;
    p.debug_skip_stage = c->dbg_skip_stage;
    CK(launch_ffn(p, c->num_sms, static_cast<cudaStream_t>(stream), &c->mx, c->ffn_kernels), "ffn kernels");
    return FTMOE_OK;
}

int ftmoe_prefetch_layer(ftmoe_cache_t *c, int32_t layer, void *stream) {
    NvtxRange nvtx_range("ftmoe_prefetch_layer");
    if (!c) return fail(FTMOE_ERR_INVALID_ARG, "cache is NULL");
    int rc = ensure_impl(c, layer, c->all_ids, 1, c->E, c->pf_slots, 0, -1, 0.f, nullptr, stream);
    if (rc) return rc;
    return ftmoe_copy_missing(c, stream);
}

int ftmoe_prefill_layers(ftmoe_cache_t *c, int32_t num_layers, const int32_t *h_layers,
                         const int32_t *const *d_topk_ids, int32_t bs, int32_t topk, const void *const *d_x_bf16,
                         const float *const *d_weights, void *const *d_y_bf16, void *compute_stream,
                         void *copy_stream) {
    NvtxRange nvtx_range("ftmoe_prefill_layers");
    if (!c) return fail(FTMOE_ERR_INVALID_ARG, "cache is NULL");
    if (!c->ffn || c->fmt == FTMOE_FMT_RAW) return fail(FTMOE_ERR_INVALID_ARG, "the cache has no FFN");
    if (num_layers <= 0) return FTMOE_OK;
    if (!h_layers || !d_topk_ids || !d_x_bf16 || !d_weights || !d_y_bf16)
        return fail(FTMOE_ERR_INVALID_ARG, "NULL per-layer array");
    if ((int64_t)c->S < 2 * (int64_t)c->E)
        return fail(FTMOE_ERR_INVALID_ARG, "whole-layer double buffering needs S >= 2E (S=%d, E=%d)", c->S, c->E);
    if (bs <= 0 || topk <= 0 || (int64_t)bs * topk > c->max_pairs)
        return fail(FTMOE_ERR_INVALID_ARG, "bs*topk must be in [1, max_pairs=%d]", c->max_pairs);
    for (int i = 0; i < num_layers; i++) {
        if (h_layers[i] < 0 || h_layers[i] >= c->L)
            return fail(FTMOE_ERR_INVALID_ARG, "layer %d outside [0, %d)", h_layers[i], c->L);
        if (!d_topk_ids[i] || !d_x_bf16[i] || !d_weights[i] || !d_y_bf16[i])
            return fail(FTMOE_ERR_INVALID_ARG, "NULL pointer for pipeline step %d", i);
    }
    cudaStream_t cs = static_cast<cudaStream_t>(compute_stream), ps = static_cast<cudaStream_t>(copy_stream);
    const bool engine = c->copy_mode == FTMOE_COPY_ENGINE;
    if (engine && !c->aux) {
        cudaError_t e = cudaStreamCreateWithFlags(&c->aux, cudaStreamNonBlocking);
        if (e != cudaSuccess) {
            c->aux = nullptr;
            return cuda_fail(e, "stream create");
        }
    }
    cudaEvent_t ready[2] = {nullptr, nullptr}, done[2] = {nullptr, nullptr}, cdone[2] = {nullptr, nullptr};
    int rc = FTMOE_OK;
    for (int k = 0; k < 2 && !rc; k++) {
        cudaError_t e = cudaEventCreateWithFlags(&ready[k], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&done[k], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&cdone[k], cudaEventDisableTiming);
        if (e != cudaSuccess) rc = cuda_fail(e, "event create");
    }
    auto record = [&](cudaEvent_t ev, cudaStream_t st) -> int {
        cudaError_t e = cudaEventRecord(ev, st);
        return e == cudaSuccess ? FTMOE_OK : cuda_fail(e, "event record");
    };
    auto wait = [&](cudaStream_t st, cudaEvent_t ev) -> int {
        cudaError_t e = cudaStreamWaitEvent(st, ev, 0);
        return e == cudaSuccess ? FTMOE_OK : cuda_fail(e, "stream wait");
    };
    // Step i's slots replace those of step i - 2 (S >= 2E and LRU order), so its copies and
    // its routed-slot buffer (i % 2) wait for the FFN of step i - 2.
    // SM-copy modes, all on copy_stream: prefetch(i) (ensure of every expert + copy kernel),
    // routed ensure -> ready[i % 2]; the FFN of step i waits for ready[i % 2].
    // Copy-engine mode: the ensures stay on copy_stream (the miss list is read back from it
    // at once, not behind the previous step's transfers) while the transfers queue on an
    // internal stream -> cdone[i % 2]; the FFN of step i waits for ready and cdone.
    auto stage = [&](int i) -> int {
        int r = FTMOE_OK;
        if (i >= 2) r = wait(ps, done[i & 1]);
        if (!r) r = ensure_impl(c, h_layers[i], c->all_ids, 1, c->E, c->pf_slots, 0, -1, 0.f, nullptr, ps);
        if (!r) {
            if (engine) {
                if (i >= 2) r = wait(c->aux, done[i & 1]);
                if (!r) r = copy_engine(c, ps, c->aux);
                if (!r) r = record(cdone[i & 1], c->aux);
            } else {
                r = ftmoe_copy_missing(c, ps);
            }
        }
        if (!r) r = ensure_impl(c, h_layers[i], d_topk_ids[i], bs, topk, c->pipe_slots[i & 1], 0, -1, 0.f, nullptr, ps);
        if (!r) r = record(ready[i & 1], ps);
        return r;
    };
    if (!rc) rc = stage(0);
    for (int i = 0; !rc && i < num_layers; i++) {
        rc = wait(cs, ready[i & 1]);
        if (!rc && engine) rc = wait(cs, cdone[i & 1]);
        if (!rc) rc = ftmoe_expert_ffn(c, d_x_bf16[i], bs, c->pipe_slots[i & 1], d_weights[i], topk, d_y_bf16[i], cs);
        if (!rc) rc = record(done[i & 1], cs);
        if (!rc && i + 1 < num_layers) rc = stage(i + 1);
    }
    for (int k = 0; k < 2; k++) {  // released once their pending work completes
        if (ready[k]) cudaEventDestroy(ready[k]);
        if (done[k]) cudaEventDestroy(done[k]);
        if (cdone[k]) cudaEventDestroy(cdone[k]);
    }
    return rc;
}

int ftmoe_cache_get_state(ftmoe_cache_t *c, int32_t *h_owner, uint32_t *h_stamp, uint32_t *h_clock, void *stream) {
    if (!c || !h_owner || !h_stamp || !h_clock) return fail(FTMOE_ERR_INVALID_ARG, "NULL argument");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CK(cudaMemcpyAsync(h_owner, c->t.owner, (size_t)c->S * 4, cudaMemcpyDeviceToHost, st), "read owner");
    CK(cudaMemcpyAsync(h_stamp, c->t.stamp, (size_t)c->S * 4, cudaMemcpyDeviceToHost, st), "read stamp");
    CK(cudaMemcpyAsync(h_clock, c->t.clock, 4, cudaMemcpyDeviceToHost, st), "read clock");
    CK(cudaStreamSynchronize(st), "sync");
    return FTMOE_OK;
}

int ftmoe_cache_set_state(ftmoe_cache_t *c, const int32_t *h_owner, const uint32_t *h_stamp, uint32_t clock,
                          void *stream) {
    if (!c || !h_owner || !h_stamp) return fail(FTMOE_ERR_INVALID_ARG, "NULL argument");
    const int64_t LE = (int64_t)c->L * c->E;
    std::vector<char> seen((size_t)LE, 0);
    for (int s = 0; s < c->S; s++) {
        const int32_t f = h_owner[s];
        if (f < -1 || f >= LE) return fail(FTMOE_ERR_STATE, "owner[%d]=%d outside [-1, %lld)", s, f, (long long)LE);
        if (f >= 0) {
            if (seen[f]) return fail(FTMOE_ERR_STATE, "id %d owns two slots", f);
            seen[f] = 1;
        }
        if (h_stamp[s] > clock) return fail(FTMOE_ERR_STATE, "stamp[%d]=%u above clock %u", s, h_stamp[s], clock);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // pageable sources: cudaMemcpyAsync stages them before it returns
    CK(cudaMemcpyAsync(c->t.owner, h_owner, (size_t)c->S * 4, cudaMemcpyHostToDevice, st), "write owner");
    CK(cudaMemcpyAsync(c->t.stamp, h_stamp, (size_t)c->S * 4, cudaMemcpyHostToDevice, st), "write stamp");
    CK(cudaMemcpyAsync(c->t.clock, &clock, 4, cudaMemcpyHostToDevice, st), "write clock");
    CK(launch_rebuild_id2slot(c->t, c->E, c->L, c->S, st), "rebuild id2slot");
    CK(cudaStreamSynchronize(st), "sync");
    return FTMOE_OK;
}

int ftmoe_get_miss_list(ftmoe_cache_t *c, int32_t *h_ids, int32_t *h_slots, int32_t *h_m, void *stream) {
    if (!c || !h_ids || !h_slots || !h_m) return fail(FTMOE_ERR_INVALID_ARG, "NULL argument");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CK(cudaMemcpyAsync(h_m, c->t.num_miss, 4, cudaMemcpyDeviceToHost, st), "read miss count");
    CK(cudaStreamSynchronize(st), "sync");
    if (*h_m > 0) {
        CK(cudaMemcpyAsync(h_ids, c->t.miss_ids, (size_t)*h_m * 4, cudaMemcpyDeviceToHost, st), "read miss ids");
        CK(cudaMemcpyAsync(h_slots, c->t.miss_slots, (size_t)*h_m * 4, cudaMemcpyDeviceToHost, st), "read miss slots");
        CK(cudaStreamSynchronize(st), "sync");
    }
    return FTMOE_OK;
}

int ftmoe_get_counters(ftmoe_cache_t *c, uint64_t *h_counters, int32_t reset, void *stream) {
    if (!c || !h_counters) return fail(FTMOE_ERR_INVALID_ARG, "NULL argument");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned long long v[3];
    CK(cudaMemcpyAsync(v, c->t.stats, sizeof v, cudaMemcpyDeviceToHost, st), "read counters");
    CK(cudaStreamSynchronize(st), "sync");
    for (int i = 0; i < 3; i++) h_counters[i] = (uint64_t)v[i];
    if (reset) {
        CK(cudaMemsetAsync(c->t.stats, 0, sizeof v, st), "reset counters");
        CK(cudaStreamSynchronize(st), "sync");
    }
    return FTMOE_OK;
}

int ftmoe_get_device_status(ftmoe_cache_t *c, int32_t *h_status, void *stream) {
    if (!c || !h_status) return fail(FTMOE_ERR_INVALID_ARG, "NULL argument");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CK(cudaMemcpyAsync(h_status, c->t.status, 4, cudaMemcpyDeviceToHost, st), "read status");
    CK(cudaMemsetAsync(c->t.status, 0, 4, st), "clear status");
    CK(cudaStreamSynchronize(st), "sync");
    return FTMOE_OK;
}

int ftmoe_h2d_stream_copy(void *d_dst, const void *h_src, size_t bytes, void *stream) {
    if (!d_dst || !h_src) return fail(FTMOE_ERR_INVALID_ARG, "NULL argument");
    if (bytes == 0) return FTMOE_OK;
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, h_src);
    if (e != cudaSuccess || attr.type != cudaMemoryTypeHost || !attr.devicePointer) {
        cudaGetLastError();
        return fail(FTMOE_ERR_INVALID_ARG, "source is not page-locked mapped host memory");
    }
    int dev = 0, sms = 0;
    CK(cudaGetDevice(&dev), "device");
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "device query");
    const bool vec = ((uintptr_t)d_dst % 16 == 0) && ((uintptr_t)attr.devicePointer % 16 == 0) && (bytes % 16 == 0);
    CK(launch_linear_copy(static_cast<unsigned char *>(d_dst), static_cast<const unsigned char *>(attr.devicePointer),
                          (int64_t)bytes, vec, sms * 4, static_cast<cudaStream_t>(stream)),
       "linear copy");
    return FTMOE_OK;
}

}  // extern "C"
