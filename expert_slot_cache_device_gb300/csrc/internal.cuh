// Internal declarations of libftmoe (not part of the C-ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ftmoe.h"

namespace ftmoe {

// Bounds-checked debug builds (compiled with -DFTMOE_CHECK, see build.build(check=True)) test
// device-side indices before they are used: a failed test records FTMOE_ERR_STATE in the
// status word and the access is skipped; nothing traps. Release builds compile the tests out.
#ifdef FTMOE_CHECK
#define FTMOE_DCHECK(cond, status) ((cond) || (atomicCAS((status), 0, FTMOE_ERR_STATE), false))
#else
#define FTMOE_DCHECK(cond, status) true
#endif

// ---------------------------------------------------------------- cache tables
// Device-resident state of one cache; all pointers point into the caller's
// workspace.
struct Tables {
    uint32_t *clock;      // [1]
    int32_t *status;      // [1] sticky device error
    int32_t *num_miss;    // [1] misses of the last ensure call
    int32_t *id2slot;     // [L * E]
    int32_t *owner;       // [S]
    uint32_t *stamp;      // [S]
    int32_t *miss_ids;    // [min(E, S)] flat ids, ascending
    int32_t *miss_slots;  // [min(E, S)]
    unsigned long long *stats;  // [3] successful ensure calls, distinct ids looked up, fetched misses
};

// ---------------------------------------------------------------- K1 ensure
struct EnsureParams {
    Tables t;
    const int32_t *ids;   // [n] routed local ids
    int32_t *slots_out;   // [n]
    int32_t E, L, S, layer, n;
    int32_t Spad;         // power of two >= S (bitonic sort width)
    int32_t maxm;         // min(E, S)
    // hybrid fetch cap: hybrid = 0 fetches every miss; otherwise cap = max_fetch when
    // max_fetch >= 0, else rint(float(misses) * fetch_fraction) when fetch_fraction > 0,
    // else 1. counts (nullable): [fetched, misses before the cap].
    int32_t hybrid, max_fetch;
    float fetch_fraction;
    int32_t *counts;
};
size_t ensure_smem_bytes(int E, int S, int Spad, int maxm);
cudaError_t launch_ensure(const EnsureParams &p, cudaStream_t st);

// ---------------------------------------------------------------- K2 copy
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 8;
constexpr int64_t kCopyTile = (int64_t)kCopyThreads * 16 * kCopyUnroll;  // 32 KiB

struct CopyParams {
    const unsigned char *src[FTMOE_MAX_BANKS];  // device view of the layer's host bank
    unsigned char *dst[FTMOE_MAX_BANKS];        // slot bank
    int64_t bytes[FTMOE_MAX_BANKS];             // per-expert bytes of each bank
    int64_t tile0[FTMOE_MAX_BANKS + 1];         // prefix of tiles per expert over banks
    const int32_t *miss_ids;
    const int32_t *miss_slots;
    const int32_t *num_miss;
    int32_t nb, E;
    int32_t L, S, maxm;  // bounds of the miss list (checked in -DFTMOE_CHECK builds)
    int32_t *status;
};
cudaError_t launch_copy(const CopyParams &p, bool vec16, int grid, cudaStream_t st);
cudaError_t launch_linear_copy(unsigned char *dst, const unsigned char *src, int64_t bytes, bool vec16,
                               int grid, cudaStream_t st);

// ---------------------------------------------------------------- state rebuild
cudaError_t launch_init_state(Tables t, int E, int L, int S, cudaStream_t st);
cudaError_t launch_rebuild_id2slot(Tables t, int E, int L, int S, cudaStream_t st);

// ---------------------------------------------------------------- K3 expert FFN
struct FfnScratch {
    int32_t *n_unique;  // [1] distinct slots of the call (0 on a bad slot)
    int32_t *uslot;     // [P] distinct slots, ascending
    int32_t *ucnt;      // [P] routed pairs per distinct slot
    int32_t *uoff;      // [P] first entry of the slot's pairs in upairs
    int32_t *upairs;    // [P] pair indices t * topk + j grouped by slot
    float *h;           // [P, I] SiLU(gate) * up per pair
    float *o;           // [P, H] down output per pair
    uint16_t *x16;      // [bs, H] activations as f16, scaled by 2^-xexp[t] (nullptr: not prepared);
                        // Q4_0: per token 2H + H/8 bytes, int16 [H] then fp32 [H/32] block scales / 16
    int32_t *xexp;      // [bs] per-token power-of-two exponent of x16
    uint32_t *hmax;     // [P] bit pattern of max |h| per pair (order-independent atomicMax)
    int32_t *upoff;     // [P] first pass (group of pass_tokens pairs) of each distinct slot
    int32_t *n_passes;  // [1] passes over all distinct slots
};

// Pipelined FFN kernels split each slot's routed pairs into passes of at most
// FfnParams::pass_tokens tokens; every (pass, tile) is a separate work item so hot experts
// spread over the SMs. The CUDA-core row-major kernels use kPassTokens, the tensor-core
// kernels (mxfp4, block FP8, bf16; the MMA's N = 8) kMxPassTokens.
constexpr int kPassTokens = 4;
constexpr int kMxPassTokens = 8;
constexpr int kTc05PassTokens = 16;  // bf16 tcgen05 pipeline: the UMMA's N

struct FfnParams {
    FfnScratch s;
    // slot banks (schema order of the format)
    const unsigned char *bank[6];
    int64_t bank_bytes[6];
    const uint16_t *x;      // [bs, H] bf16
    const int32_t *slots;   // [P]
    const float *weights;   // [P]
    const float *addend;    // [bs, H] fp32 added before the final round (nullable)
    uint16_t *y;            // [bs, H] bf16
    int32_t *status;
    int32_t fmt, H, I, S, bs, topk, P;
    int32_t E;         // experts per layer (0: unknown; used only to choose kernels)
    int32_t x16_emax;  // f16 activation copy keeps max |x| < 2^x16_emax
    int32_t x16_swz;   // activation copy layout: 0 plain, 1 swz_x16 (nvfp4), 2 int16 in swz_q4x16 (Q4_0)
    int32_t pass_tokens;  // tokens per pass of the pipelined kernels (kPassTokens / kMxPassTokens)
    // test settings (ftmoe_set_debug): limit of the CUDA-core pipeline's bounded waits (0: the
    // default), and 1 to leave CTA 0's first gate_up stage unfilled so that a wait runs out
    uint64_t wait_ns;
    int32_t debug_skip_stage;
};

// Tensor maps (CUtensorMap, 128 bytes each) of the tensor-map pipelines: the transposed
// mxfp4 banks, or the block-FP8 / bf16 weight banks (gu_blocks / dn_blocks).
struct MxTmaMaps {
    alignas(128) unsigned char gu_blocks[128];
    alignas(128) unsigned char gu_scales[128];
    alignas(128) unsigned char dn_blocks[128];
    alignas(128) unsigned char dn_scales[128];
    bool valid = false;
    // bf16 weight maps of the tcgen05 pipeline (boxes of 128 bytes x 128 rows)
    alignas(128) unsigned char tc_gu[128];
    alignas(128) unsigned char tc_dn[128];
    bool tc_valid = false;
};
bool make_mx_tma_maps(MxTmaMaps &m, const unsigned char *const *banks, int S, int H, int I);
// kernels: FTMOE_FFN_* (bf16 caches: see ffn_bf16_family; other formats ignore it).
// The kernel family a bf16 call runs: FTMOE_FFN_ROWS, FTMOE_FFN_MMA or FTMOE_FFN_TC05 (the
// AUTO rule lives here).
int ffn_bf16_family(const FfnParams &p, int num_sms, const MxTmaMaps *mx, int kernels);
cudaError_t launch_ffn(const FfnParams &p, int num_sms, cudaStream_t st, const MxTmaMaps *mx = nullptr,
                       int kernels = FTMOE_FFN_AUTO);
// Persistent bulk-copy pipeline for the row-major formats (bf16; nvfp4 with H, I multiples of 256).
bool ffn_rows_tma_supported(const FfnParams &p);
cudaError_t launch_ffn_rows_tma(const FfnParams &p, int num_sms, cudaStream_t st);
// 2-D tensor-map pipeline for the transposed mxfp4 format.
bool ffn_mx_tma_supported(const FfnParams &p, const MxTmaMaps *maps);
cudaError_t launch_ffn_mx_tma(const FfnParams &p, const MxTmaMaps &maps, int num_sms, cudaStream_t st);
// Tensor-map pipeline for block FP8 (its weight maps sit in gu_blocks / dn_blocks).
bool make_fp8_tma_maps(MxTmaMaps &m, const unsigned char *const *banks, int S, int H, int I);
bool ffn_fp8_tma_supported(const FfnParams &p, const MxTmaMaps *maps);
cudaError_t launch_ffn_fp8_tma(const FfnParams &p, const MxTmaMaps &maps, int num_sms, cudaStream_t st);
// Tensor-core pipeline for bf16 (weight maps in gu_blocks / dn_blocks; H, I multiples of 256).
bool make_bf16_tma_maps(MxTmaMaps &m, const unsigned char *const *banks, int S, int H, int I);
bool ffn_bf16_mma_supported(const FfnParams &p, const MxTmaMaps *maps);
cudaError_t launch_ffn_bf16_mma(const FfnParams &p, const MxTmaMaps &maps, int num_sms, cudaStream_t st);
// tcgen05 pipeline for bf16 (maps tc_gu / tc_dn; H a multiple of 64, I of 128, both phases fit).
bool ffn_bf16_tc05_supported(const FfnParams &p, const MxTmaMaps *maps);
cudaError_t launch_ffn_bf16_tc05(const FfnParams &p, const MxTmaMaps &maps, int num_sms, cudaStream_t st);

// Record `msg` as the thread's last error message and return `code`.
int report_error(int code, const char *msg);

}  // namespace ftmoe
