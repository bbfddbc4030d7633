// Expert FFN without any device allocation: the routing tables and the fp32
// intermediates that the FFN kernels need live in one file-scope device array
// instead of a caller-provided workspace.
//
// Who needs this: code that runs inside a host runtime which already owns all of the
// GPU's memory (a serving engine that reserved HBM up front for weights and KV cache,
// so a cudaMalloc would fail or break its accounting), and code on a latency-critical
// path that must not pay for cudaMalloc/cudaFree, which can synchronise the device.
// Such a caller passes only its inputs (slot banks, activations, slots, router
// weights) and the output buffer.
//
// The array is kStaticScratchBytes (FTMOE_NOALLOC_SCRATCH_BYTES) large. Every GPU that
// loads the library reserves it until the process exits. All calls share it and it
// keeps the previous call's contents; calls that overlap on the GPU (two streams, two
// threads) race on it and must be serialised by the caller.
#include <cstring>
#include <mutex>

#include "internal.cuh"

namespace ftmoe {
namespace {

constexpr size_t kStaticScratchBytes = FTMOE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_ffn_scratch[kStaticScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

size_t round256(size_t v) { return (v + 255) & ~(size_t)255; }

// Device address of g_ffn_scratch on the current device. In host code the symbol
// name is only a host-side stand-in, so the address is looked up once per device
// (on that device's first call) and cached.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_ffn_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

int64_t bank_bytes_of(int fmt, int b, int64_t H, int64_t I) {
    if (fmt == FTMOE_FMT_BF16) return b == 0 ? 4 * I * H : 2 * H * I;
    const int64_t N = b < 3 ? 2 * I : H, K = b < 3 ? H : I;
    if (fmt == FTMOE_FMT_NVFP4) return b % 3 == 0 ? N * K / 2 : (b % 3 == 1 ? N * K / 16 : 2 * N);
    return b % 3 == 0 ? K / 2 * N : (b % 3 == 1 ? K / 32 * N : 2 * N);
}

}  // namespace
}  // namespace ftmoe

using namespace ftmoe;

extern "C" int ftmoe_expert_ffn_noalloc(int32_t format, const void *const *d_slot_banks, int32_t num_banks,
                                        int32_t S, int32_t H, int32_t I, const void *d_x_bf16, int32_t bs,
                                        const int32_t *d_slots, const float *d_weights, int32_t topk,
                                        void *d_y_bf16, void *stream) {
    const int want_banks = format == FTMOE_FMT_BF16 ? 2 : (format == FTMOE_FMT_NVFP4 || format == FTMOE_FMT_MXFP4 ? 6 : -1);
    if (want_banks < 0) return report_error(FTMOE_ERR_INVALID_ARG, "format must be FTMOE_FMT_BF16, NVFP4 or MXFP4");
    if (num_banks != want_banks || !d_slot_banks) return report_error(FTMOE_ERR_INVALID_ARG, "wrong number of slot banks for the format");
    const int q = format == FTMOE_FMT_BF16 ? 8 : 32;
    if (H <= 0 || I <= 0 || H % q || I % q) return report_error(FTMOE_ERR_INVALID_ARG, "H and I must be positive multiples of 8 (bf16) or 32 (fp4)");
    if (S <= 0 || S > FTMOE_MAX_SLOTS) return report_error(FTMOE_ERR_INVALID_ARG, "S outside [1, FTMOE_MAX_SLOTS]");
    if (bs < 0 || topk <= 0) return report_error(FTMOE_ERR_INVALID_ARG, "bs >= 0 and topk > 0 required");
    if (bs > 65535) return report_error(FTMOE_ERR_INVALID_ARG, "bs above 65535 (one grid row per token)");
    const int64_t P = (int64_t)bs * topk;
    if (P == 0) return FTMOE_OK;
    // P fits the fixed scratch only if P * (H + I) * 4 < its size: checked before any size
    // is formed, so no product below can wrap
    if (P > (int64_t)(kStaticScratchBytes / (4 * ((uint64_t)H + (uint64_t)I))))
        return report_error(FTMOE_ERR_INVALID_ARG, "bs * topk * (H + I) too large for the fixed FFN scratch (FTMOE_NOALLOC_SCRATCH_BYTES)");
    if (!d_x_bf16 || !d_slots || !d_weights || !d_y_bf16) return report_error(FTMOE_ERR_INVALID_ARG, "NULL FFN argument");
    if (((uintptr_t)d_x_bf16 | (uintptr_t)d_y_bf16) % 16) return report_error(FTMOE_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
    for (int b = 0; b < num_banks; b++)
        if (!d_slot_banks[b]) return report_error(FTMOE_ERR_INVALID_ARG, "NULL slot bank");

    // scratch layout: [status, n_unique] | uslot | ucnt | uoff | upairs | h [P, I] | o [P, H]
    const size_t tab = round256((size_t)P * 4);
    const size_t need = 256 + 4 * tab + round256((size_t)P * I * 4) + round256((size_t)P * H * 4);
    if (need > kStaticScratchBytes)
        return report_error(FTMOE_ERR_INVALID_ARG, "bs * topk * (H + I) too large for the fixed FFN scratch (FTMOE_NOALLOC_SCRATCH_BYTES)");

    void *base = nullptr;
    cudaError_t e = scratch_address(&base);
    if (e != cudaSuccess) return report_error(FTMOE_ERR_CUDA, cudaGetErrorString(e));
    unsigned char *ws = static_cast<unsigned char *>(base);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    FfnParams p;
    memset(&p, 0, sizeof p);
    p.status = reinterpret_cast<int32_t *>(ws);
    p.s.n_unique = reinterpret_cast<int32_t *>(ws + 4);
    size_t off = 256;
    p.s.uslot = reinterpret_cast<int32_t *>(ws + off); off += tab;
    p.s.ucnt = reinterpret_cast<int32_t *>(ws + off); off += tab;
    p.s.uoff = reinterpret_cast<int32_t *>(ws + off); off += tab;
    p.s.upairs = reinterpret_cast<int32_t *>(ws + off); off += tab;
    p.s.h = reinterpret_cast<float *>(ws + off); off += round256((size_t)P * I * 4);
    p.s.o = reinterpret_cast<float *>(ws + off);
    for (int b = 0; b < num_banks; b++) {
        p.bank[b] = static_cast<const unsigned char *>(d_slot_banks[b]);
        p.bank_bytes[b] = bank_bytes_of(format, b, H, I);
    }
    p.x = static_cast<const uint16_t *>(d_x_bf16);
    p.slots = d_slots;
    p.weights = d_weights;
    p.y = static_cast<uint16_t *>(d_y_bf16);
    p.fmt = format; p.H = H; p.I = I; p.S = S; p.bs = bs; p.topk = topk; p.P = (int)P;
    // the status word is the only thing that must start at zero; everything else the
    // kernels read is written earlier in the same call
    e = cudaMemsetAsync(p.status, 0, 4, st);
    if (e == cudaSuccess) e = launch_ffn(p, 0, st);
    if (e != cudaSuccess) return report_error(FTMOE_ERR_CUDA, cudaGetErrorString(e));
    return FTMOE_OK;
}
