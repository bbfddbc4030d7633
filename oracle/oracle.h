/*
 * CPU oracle of the offloaded expert slot cache — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct restatement of what the decode step of the
 * offloaded MoE expert cache computes, used to check the CUDA path. Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product path never calls it. It shares no code, header, table or constant
 * with the CUDA library.
 *
 * Sources (FreeToken pages):
 *   [ARCH]  "深入FreeToken架构：从HTTP API到CUDA内核的本地MoE推理引擎全链路剖析",
 *           section 五 (MoE engine): expert banks per quantisation format,
 *           one global LRU expert cache.
 *   [BENCH] "FreeToken MoE 离线推理基准完全指南", section 一 (hit experts
 *           compute from the slot cache, misses are copied over PCIe),
 *           section 4.1 (ensure_experts = LRU slot remap + per-bank gather),
 *           4.2 (bank schemas; the cache is layout-agnostic and only moves
 *           rows), 4.3 (flat id = layer * E + expert; prepared state),
 *           4.4 (copy_MiB = misses * bytes per expert; per-layer source lists).
 *
 * Parity status: every function here is pinned by CPU tests against values
 * the pages or the format specifications fix (brute-force LRU traces, the
 * worked tiny case, the miss-count closed form, spec tables of the number
 * formats, closed-form FFN special cases).
 */
#ifndef FTMOE_ORACLE_H
#define FTMOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes (same numeric meaning as the library's, defined independently) */
#define ORC_OK 0
#define ORC_ERR_INVALID_ARG (-1)
#define ORC_ERR_CAPACITY (-2)
#define ORC_ERR_ID_RANGE (-3)
#define ORC_ERR_STATE (-6)

/* formats */
#define ORC_FMT_BF16 0
#define ORC_FMT_NVFP4 1
#define ORC_FMT_MXFP4 2
#define ORC_FMT_FP8 3
#define ORC_FMT_Q4_0 4

/* number kinds for orc_decode */
#define ORC_NUM_E2M1 0
#define ORC_NUM_E4M3 1
#define ORC_NUM_E8M0 2
#define ORC_NUM_F16 3
#define ORC_NUM_BF16 4

/* LRU ensure_experts on a caller-owned state (owner[S], stamp[S], id2slot[L*E], *clock).
 * topk_ids: n local ids of layer `layer`. Outputs slots_out[n], miss_ids[m] (flat ids,
 * ascending), miss_slots[m], *num_miss. On error the state is untouched, slots_out is
 * filled with -1 and *num_miss = 0. */
int orc_ensure(int32_t E, int32_t L, int32_t S, int32_t *owner, uint32_t *stamp,
               int32_t *id2slot, uint32_t *clock, int32_t layer, const int32_t *topk_ids,
               int32_t n, int32_t *slots_out, int32_t *miss_ids, int32_t *miss_slots,
               int32_t *num_miss);

/* Hybrid ensure_experts (benchmark guide, section 5.4): as orc_ensure, but only the
 * first `cap` misses in ascending flat id get slots; the others keep slot -1 and leave
 * the cache untouched. cap = max_fetch when max_fetch >= 0; otherwise the fetch share
 * of the measured bandwidths, round-half-even(float(misses) * fetch_fraction) computed
 * in binary32, when fetch_fraction > 0; otherwise 1. counts[0] = misses fetched
 * (num_indices), counts[1] = misses before the cap (num_missing_full). */
int orc_ensure_hybrid(int32_t E, int32_t L, int32_t S, int32_t *owner, uint32_t *stamp,
                      int32_t *id2slot, uint32_t *clock, int32_t layer, const int32_t *topk_ids,
                      int32_t n, int32_t max_fetch, float fetch_fraction, int32_t *slots_out,
                      int32_t *miss_ids, int32_t *miss_slots, int32_t *num_miss, int32_t *counts);

/* Rebuild id2slot[L*E] from owner[S]; returns ORC_ERR_STATE on duplicate / bad owners. */
int orc_rebuild_id2slot(int32_t E, int32_t L, int32_t S, const int32_t *owner, int32_t *id2slot);

/* copy_missing: for each miss j and bank b, copy bank_bytes[b] bytes of expert
 * (miss_ids[j] mod E) from host_layer[b] to slot row miss_slots[j] of slots[b]. */
void orc_copy_missing(int32_t num_banks, const int64_t *bank_bytes,
                      const uint8_t *const *host_layer, uint8_t *const *slots, int32_t E,
                      const int32_t *miss_ids, const int32_t *miss_slots, int32_t m);

/* Decode one stored number of the given kind to double. */
double orc_decode(int32_t kind, uint32_t bits);

/* Weight (n, k) of an expert's gate_up (which = 0: N = 2I, K = H) or down
 * (which = 1: N = H, K = I) matrix; `banks` points at this expert's bytes in each bank. */
double orc_weight(int32_t fmt, int32_t which, const uint8_t *const *banks, int32_t H,
                  int32_t I, int64_t n, int64_t k);

/* Bias of output n (mxfp4 only; 0 for the other formats). */
double orc_bias(int32_t fmt, int32_t which, const uint8_t *const *banks, int32_t H,
                int32_t I, int64_t n);

/* Expert FFN of `bs` tokens: y[t, :] = sum_j w[t, j] * down(silu(gate) * up)(x_t)
 * with every pair's expert bytes given by pair_banks[(t * k + j) * num_banks + b].
 * x is bf16 bit patterns [bs, H]; y is fp64 [bs, H]. Runs its row loops on
 * `threads` OpenMP threads (<= 0: runtime default). */
int orc_expert_ffn(int32_t fmt, int32_t H, int32_t I, int32_t bs, int32_t k,
                   int32_t num_banks, const uint8_t *const *pair_banks, const uint16_t *x,
                   const float *w, double *y, int32_t threads);

/* Number of banks of a format's schema (2, 6, 6). */
int32_t orc_num_banks(int32_t fmt);

#ifdef __cplusplus
}
#endif
#endif
