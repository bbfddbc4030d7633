/*
 * ftmoe — offloaded MoE expert slot cache for one GB300 (sm_103a).
 *
 * C-ABI of the per-layer decode step of an offloaded mixture-of-experts expert
 * cache: expert weights live in page-locked host "banks"; a fixed pool of GPU
 * slots caches them under one global LRU over the flat id space
 * id = layer * E + expert. A decode step of one layer is
 *
 *   ftmoe_ensure_experts  -> dedup the routed ids, look them up, evict LRU slots
 *                            for the misses (one kernel, no host sync);
 *   ftmoe_copy_missing    -> copy every missed expert's bytes of every bank from
 *                            the host banks into its new slot (one fused kernel);
 *   ftmoe_expert_ffn      -> gate_up -> SiLU * up -> down over the resolved slots,
 *                            combined with the router probabilities.
 *
 * Sources (FreeToken pages): the architecture deep-dive "深入FreeToken架构：从HTTP
 * API到CUDA内核的本地MoE推理引擎全链路剖析", section 五 (expert banks per
 * quantisation format, a global LRU expert cache), and the benchmark guide
 * "FreeToken MoE 离线推理基准完全指南", sections 一 (hit experts compute from the
 * slot cache, misses are copied over the host link), 4.1 (ensure_experts = LRU
 * slot remap plus a gather of the bank rows), 4.2 (bank schemas; the cache is
 * layout-agnostic and only moves rows), 4.3 (flat id space, prepared state,
 * miss counts) and 4.4 (copy_MiB, per-layer source lists, a fused multi-bank
 * copy with a per-bank path kept for A/B comparison).
 *
 * Conventions for every entry point:
 *   - returns FTMOE_OK (0) or a negative FTMOE_ERR_* code; on error
 *     ftmoe_last_error() gives a message (thread-local, valid until the next call
 *     on the same thread);
 *   - pointers named d_* are device pointers, h_* host pointers;
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream); work is enqueued on it and the call returns without waiting,
 *     unless the entry point says it synchronises;
 *   - errors found on the host return before anything is enqueued; errors found
 *     on the device (an expert id out of range, more misses than free slots)
 *     leave the cache state untouched, make the kernel write nothing else, and
 *     are recorded in a sticky device status word read by
 *     ftmoe_get_device_status. No kernel traps, asserts or spin-waits.
 *   - ftmoe_ensure_experts, ftmoe_copy_missing (FTMOE_COPY_FUSED / PER_BANK) and
 *     ftmoe_expert_ffn only enqueue kernels, so a sequence of them can be captured
 *     into a CUDA graph (stream capture) and replayed: the graph reads the id, weight
 *     and activation buffers and the cache tables at replay time. Calls that read
 *     back to the host (FTMOE_COPY_ENGINE, the get_* and measure_* entry points)
 *     cannot be captured.
 */
#ifndef FTMOE_H
#define FTMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define FTMOE_OK 0
#define FTMOE_ERR_INVALID_ARG (-1) /* bad argument found on the host */
#define FTMOE_ERR_CAPACITY (-2)    /* more distinct missing experts than evictable slots */
#define FTMOE_ERR_ID_RANGE (-3)    /* a routed expert id outside [0, E) */
#define FTMOE_ERR_CUDA (-4)        /* a CUDA runtime call failed */
#define FTMOE_ERR_FORMAT (-5)      /* banks do not match the format's schema */
#define FTMOE_ERR_STATE (-6)       /* inconsistent cache state, clock exhausted, call order */

/* bank formats (schemas of the benchmark guide, section 4.2) */
#define FTMOE_FMT_RAW 0   /* any banks; copy only, no FFN */
#define FTMOE_FMT_BF16 1  /* banks: gate_up [2I, H] bf16, down [H, I] bf16 */
#define FTMOE_FMT_NVFP4 2 /* banks: gate_up codes [2I, H/2] u8, scales [2I, H/16] e4m3,
                             global [2I] f16, down codes [H, I/2], scales [H, I/16], global [H] */
#define FTMOE_FMT_MXFP4 3 /* banks (transposed): gate_up blocks [H/2, 2I] u8, scales [H/32, 2I]
                             e8m0, bias [2I] bf16, down blocks [I/2, H], scales [I/32, H], bias [H] */
#define FTMOE_FMT_FP8 4   /* block FP8 (architecture deep-dive, section 五 lists it among the
                             bank schemas): gate_up weight [2I, H] e4m3, scale [2I/128, H/128]
                             f32 (one per 128 x 128 block), down weight [H, I] e4m3, scale
                             [H/128, I/128] f32; H and I multiples of 512. No CPU MoE path. */
#define FTMOE_FMT_Q4_0 5  /* GGUF Q4_0 (architecture deep-dive, sections 五 and 六): gate_up
                             [2I rows][H/32 blocks] and down [H rows][I/32 blocks] of 18-byte
                             blocks (binary16 d, 16 bytes qs; element j < 16 = low nibble of
                             qs[j], j + 16 = high nibble; w = (nibble - 8) * d); H and I
                             multiples of 256. */

/* element types of a bank (informative; FFN formats check them against the schema) */
#define FTMOE_DT_U8 0
#define FTMOE_DT_BF16 1
#define FTMOE_DT_F16 2
#define FTMOE_DT_E4M3 3
#define FTMOE_DT_E8M0 4
#define FTMOE_DT_F32 5
#define FTMOE_DT_Q4_0 6

/* copy_missing implementations (benchmark guide, section 4.4: the fused multi-bank
 * copy is the main path; the per-bank path is kept for A/B comparison) */
#define FTMOE_COPY_FUSED 0    /* one kernel for all banks (default) */
#define FTMOE_COPY_PER_BANK 1 /* one kernel launch per bank */
#define FTMOE_COPY_ENGINE 2   /* copy engines: reads the miss list back to the host
                                 (synchronises the stream), then one cudaMemcpyAsync
                                 per bank and run of consecutive experts landing in
                                 consecutive slots (a single miss is a run of one),
                                 in transfers of at most 256 MiB */

/* Expert FFN kernel families of a bf16 cache (other formats have one family each and
 * accept FTMOE_FFN_AUTO only) */
#define FTMOE_FFN_AUTO 0   /* TC05 where the shape has it (else MMA), except ROWS when the
                              call has about one routed pair per expert
                              (E/4 <= bs*topk < 2E); default */
#define FTMOE_FFN_ROWS 1   /* CUDA-core bulk-copy pipeline: fp32 FMAs, passes of 4 tokens */
#define FTMOE_FFN_MMA 2    /* tensor-core pipeline: bf16 mma.sync, passes of 8 tokens,
                              h kept as two bf16 terms; needs H and I multiples of 256 */
#define FTMOE_FFN_TC05 3   /* 5th-generation tensor cores: tcgen05.mma with accumulators in
                              TMEM (M = 128 rows, N = 16 tokens), passes of 16 tokens, h kept
                              as two bf16 terms; needs H and I multiples of 256 */

/* Limits of one cache. */
#define FTMOE_MAX_BANKS 8
#define FTMOE_MAX_EXPERTS 8192      /* E */
#define FTMOE_MAX_SLOTS 8192        /* S */
#define FTMOE_MAX_IDS_PER_CALL 65536 /* bs * topk of one ensure call */

typedef struct ftmoe_cache ftmoe_cache_t;

/* One bank of the per-expert weights.
 *   rows, row_bytes : per-expert geometry as declared; one expert occupies
 *                     rows * row_bytes bytes (a multiple of 16 is fastest);
 *   host_src        : host array of L pointers; host_src[l] points at layer l's
 *                     [E, rows * row_bytes] bytes in PAGE-LOCKED host memory
 *                     (cudaHostAlloc, cudaHostRegister, torch pin_memory). NULL
 *                     entries mark layers whose banks are not filled (ensure on
 *                     such a layer fails with FTMOE_ERR_INVALID_ARG). Entries may
 *                     alias. The array is copied at create; the memory it points
 *                     at must outlive the cache and must not change while a copy
 *                     reads it;
 *   dev_slots       : device [S, rows * row_bytes] slot bank, caller-owned. */
typedef struct {
    const char *name;
    int32_t dtype;
    int64_t rows;
    int64_t row_bytes;
    const void *const *host_src;
    void *dev_slots;
} ftmoe_bank_spec;

/* Bytes of device workspace a cache with these sizes needs (cache tables, miss
 * list and FFN scratch for up to max_pairs = bs * topk routed pairs per FFN call;
 * max_pairs = 0 disables the FFN). H and I are ignored for FTMOE_FMT_RAW. */
int ftmoe_cache_workspace_bytes(int32_t format, int32_t num_banks, int32_t E, int32_t L,
                                int32_t S, int32_t H, int32_t I, int32_t max_pairs,
                                size_t *bytes);

/* Create a cache over caller-owned banks and workspace (d_workspace: device,
 * 256-byte aligned, at least ftmoe_cache_workspace_bytes). Maps every non-NULL host
 * bank pointer for device access and initialises the state on `stream` to empty:
 * every slot free, stamp 0, clock 0, status 0. format FTMOE_FMT_BF16/NVFP4/MXFP4
 * checks the number of banks and each bank's per-expert bytes against the schema
 * for (H, I) (FTMOE_ERR_FORMAT on mismatch; the declared rows/row_bytes may be any
 * factorisation). The library owns only the returned host handle. */
int ftmoe_cache_create(const ftmoe_bank_spec *banks, int32_t num_banks, int32_t format,
                       int32_t E, int32_t L, int32_t S, int32_t H, int32_t I,
                       int32_t max_pairs, void *d_workspace, size_t workspace_bytes,
                       void *stream, ftmoe_cache_t **out);

/* Destroy the host handle (the caller frees banks and workspace). NULL is a no-op. */
int ftmoe_cache_destroy(ftmoe_cache_t *cache);

/* ensure_experts (benchmark guide, section 4.1: "LRU slot remap"; architecture
 * deep-dive, section 五: one global LRU for all layers) for the bs * topk routed
 * local expert ids d_topk_ids[bs, topk] (int32, device) of `layer`:
 *   1. clock += 1;
 *   2. U = ascending distinct flat ids layer * E + id;
 *   3. resident members of U (hits) get stamp = clock;
 *   4. the misses, in ascending flat id, take the slots not hit in this call in
 *      ascending (stamp, slot) order — least recently used first, lowest slot on
 *      equal stamps; an evicted owner loses its slot, the new owner gets stamp =
 *      clock;
 *   5. d_slots_out[bs, topk] (int32, device) = slot of every routed position.
 * The miss list (flat ids and slots, ascending id) stays on the device for
 * ftmoe_copy_missing. One kernel, no host synchronisation. Device-detected errors
 * (FTMOE_ERR_ID_RANGE, FTMOE_ERR_CAPACITY, clock exhausted = FTMOE_ERR_STATE) leave
 * the state and clock untouched, fill d_slots_out with -1, empty the miss list and
 * set the device status. bs * topk = 0 only advances the clock. */
int ftmoe_ensure_experts(ftmoe_cache_t *cache, int32_t layer, const int32_t *d_topk_ids,
                         int32_t bs, int32_t topk, int32_t *d_slots_out, void *stream);

/* copy_missing (benchmark guide, sections 4.1, 4.2, 4.4): for every miss of the
 * last ensure call and every bank b, copy the expert's rows * row_bytes bytes from
 * host_src[layer] + expert * bytes to dev_slots + slot * bytes, unchanged. The
 * miss count is read on the device: no host synchronisation (except in
 * FTMOE_COPY_ENGINE mode). Must be stream-ordered after that ensure call;
 * FTMOE_ERR_STATE if no ensure call was made yet. */
int ftmoe_copy_missing(ftmoe_cache_t *cache, void *stream);

/* Expert FFN over resolved slots (architecture deep-dive, section 五; benchmark
 * guide, section 一: hit experts compute from the slot cache). For every token t
 * and routed position j with slot s = d_slots[t, j]:
 *     gu = W_gu[s] x_t (+ b_gu), h = silu(gu[0:I]) * gu[I:2I],
 *     o  = W_d[s] h (+ b_d),     y_t = sum_j d_weights[t, j] * o
 * with fp32 accumulation and one final round to bf16. d_x_bf16 [bs, H] bf16,
 * d_slots [bs, topk] int32, d_weights [bs, topk] fp32, d_y_bf16 [bs, H] bf16 (all
 * device). Slots must be in [0, S), or -1 for a position computed elsewhere (the hybrid
 * CPU executor), which then contributes nothing; any other slot is a device error
 * (y left unwritten, status FTMOE_ERR_INVALID_ARG). bs * topk <= max_pairs of create.
 * Uses the FFN scratch of the cache workspace, so FFN calls on one cache must not
 * overlap. */
int ftmoe_expert_ffn(ftmoe_cache_t *cache, const void *d_x_bf16, int32_t bs,
                     const int32_t *d_slots, const float *d_weights, int32_t topk,
                     void *d_y_bf16, void *stream);

/* Hybrid ensure_experts (benchmark guide, section 5.4: in hybrid mode only a capped
 * number of misses is fetched per step; the overflow is rewritten to -1 and computed by
 * the CPU executor; num_indices and num_missing_full count the capped and the uncapped
 * misses). As ftmoe_ensure_experts, except that only the first `cap` misses in
 * ascending flat id get slots (and are copied by the next ftmoe_copy_missing); the
 * other misses leave the cache untouched and their routed positions get slot -1.
 *   cap = max_fetch                                     if max_fetch >= 0,
 *       = rint(float(misses) * fetch_fraction) (binary32, half to even)
 *                                                       if max_fetch < 0 and fetch_fraction > 0,
 *       = 1                                             otherwise (no bandwidth profile).
 * d_counts (device int32[2], may be NULL) receives {fetched, misses before the cap}. */
int ftmoe_ensure_experts_hybrid(ftmoe_cache_t *cache, int32_t layer, const int32_t *d_topk_ids,
                                int32_t bs, int32_t topk, int32_t max_fetch, float fetch_fraction,
                                int32_t *d_slots_out, int32_t *d_counts, void *stream);

/* Fetch share of the hybrid split (benchmark guide, section 5.4: PCIe-fetched experts :
 * CPU-computed experts = pcie_bw : (cpu_bw - pcie_bw), i.e. pcie_bw / cpu_bw of the
 * misses are fetched). *out = pcie_gbps / cpu_gbps when cpu_gbps > pcie_gbps > 0, 1 when
 * 0 < cpu_gbps <= pcie_gbps (the link is the faster path), 0 when either is <= 0 (no
 * profile: ftmoe_ensure_experts_hybrid then falls back to a cap of 1). Host only. */
int ftmoe_hybrid_fetch_fraction(double pcie_gbps, double cpu_gbps, float *out);

/* Expert FFN of the hybrid path: as ftmoe_expert_ffn (which is this call with
 * d_addend = NULL), plus an optional device fp32 [bs, H] addend (the CPU executor's
 * partial output) added to every token's sum before the single round to bf16. Routed
 * positions with slot -1 contribute nothing here. */
int ftmoe_expert_ffn_hybrid(ftmoe_cache_t *cache, const void *d_x_bf16, int32_t bs,
                            const int32_t *d_slots, const float *d_weights, int32_t topk,
                            const float *d_addend, void *d_y_bf16, void *stream);

/* CPU expert executor of the hybrid path (benchmark guide, section 5.4; architecture
 * deep-dive, section 五: the CPU side computes experts by GEMV from the host banks).
 * Host-side, synchronous, multi-threaded (threads <= 0: all hardware threads). For every
 * routed position (t, j) with h_slots[t, j] == -1 it computes the expert FFN of expert
 * h_topk_ids[t, j] from the layer's host banks and accumulates it into h_y:
 *     h_y[t, :] = sum over those j of h_weights[t, j] * down(silu(gate) * up)(x_t)
 * in fp32 (h_y [bs, H] fp32 is overwritten; tokens without CPU pairs get 0).
 * h_layer_banks[b] points at the layer's [E, bank_bytes[b]] host bank b in the schema
 * order of `format` (FTMOE_FMT_BF16 / NVFP4 / MXFP4); h_x is bf16 [bs, H]. All pointers
 * are host pointers. */
int ftmoe_cpu_expert_ffn(int32_t format, int32_t H, int32_t I, int32_t bs, int32_t topk,
                         const int32_t *h_topk_ids, const int32_t *h_slots,
                         const void *const *h_layer_banks, const int64_t *bank_bytes,
                         const uint16_t *h_x, const float *h_weights, float *h_y,
                         int32_t threads);

/* Whole-layer prefetch (architecture deep-dive, section 五: the global LRU expert cache
 * streams prefill layer by layer through a double buffer so that copies overlap compute).
 * Enqueues on `stream` an ensure_experts of all E experts of `layer` (as if every expert
 * were routed once, ids 0..E-1 in ascending order) followed by ftmoe_copy_missing in the
 * cache's copy mode. The slots it assigns are written to workspace scratch, not returned.
 * Same errors as those two calls; with FTMOE_COPY_ENGINE the call waits on the host for
 * the ensure to finish (the miss list is read back) and then issues copy-engine transfers,
 * which leave the SMs free for work on other streams. */
int ftmoe_prefetch_layer(ftmoe_cache_t *cache, int32_t layer, void *stream);

/* Double-buffered prefill over a sequence of layers (architecture deep-dive, section 五:
 * whole-layer double-buffered prefill streaming, copy overlapped with compute). Step i
 * runs layer h_layers[i] (host array, num_layers entries) for one batch: bs tokens,
 * routed ids d_topk_ids[i] (device int32 [bs, topk]), activations d_x_bf16[i] (device
 * bf16 [bs, H]), router weights d_weights[i] (device fp32 [bs, topk]), output
 * d_y_bf16[i] (device bf16 [bs, H]); the four arrays of device pointers are host arrays.
 * Schedule: on copy_stream, step i's ftmoe_prefetch_layer then its routed ensure (all hits)
 * into one of two workspace slot buffers; on compute_stream, step i's expert FFN waits for
 * that and runs while step i + 1 is prefetched. Step i's copies and slot buffer wait for the
 * FFN of step i - 2, whose slots they replace. With FTMOE_COPY_ENGINE the ensures stay on
 * copy_stream, the miss list of each prefetch is read back from it right away, and the
 * transfers queue on a stream the cache creates on first use (destroyed with the cache), so
 * the copy engines stay busy back to back while the SMs run the FFN; the FFN of a step then
 * also waits for its transfers. The LRU sequence equals the calls prefetch(0), ensure(0),
 * prefetch(1), ensure(1), ... made one after another. Needs S >= 2E (one layer computing,
 * the next arriving) and 1 <= bs * topk <= max_pairs; -> FTMOE_ERR_INVALID_ARG otherwise.
 * Returns once everything is enqueued (the host waits for the miss lists in copy-engine
 * mode); the caller synchronises compute_stream for the outputs. Device-detected errors land
 * in the status word as for the single calls. */
int ftmoe_prefill_layers(ftmoe_cache_t *cache, int32_t num_layers, const int32_t *h_layers,
                         const int32_t *const *d_topk_ids, int32_t bs, int32_t topk,
                         const void *const *d_x_bf16, const float *const *d_weights, void *const *d_y_bf16,
                         void *compute_stream, void *copy_stream);

/* Cumulative ensure statistics since cache creation (or the last reset): h_counters[0] =
 * successful ensure calls (plain and hybrid, prefetches included), [1] = distinct ids looked
 * up (hits + misses before any hybrid cap), [2] = misses given a slot (fetched). Hits =
 * [1] - misses before the cap; for plain calls the hit rate is 1 - [2] / [1]. Calls that
 * fail on the device do not count. reset != 0 zeroes them after the read. Synchronises the
 * stream. This library's observability; the pages define no such counters. */
int ftmoe_get_counters(ftmoe_cache_t *cache, uint64_t *h_counters, int32_t reset, void *stream);

/* MoE backends of the decision below. */
#define FTMOE_BACKEND_OFFLOAD 0  /* fetch every miss over the host link */
#define FTMOE_BACKEND_HYBRID 1   /* fetch a share, compute the rest on the host CPU */

/* Host -> device link probe (benchmark guide, section 5.2: the pinned -> device gather
 * bandwidth, the linear pinned <-> device copy ceiling). Times `bytes` from the page-locked
 * host buffer h_src to the device buffer d_dst on `stream`, best of `reps`, once with
 * cudaMemcpyAsync (copy engines) and once with the SM zero-copy read kernel of
 * ftmoe_h2d_stream_copy; writes both rates in GB/s (1e9 bytes/s). Synchronises the stream.
 * Caller-owned buffers; FTMOE_ERR_INVALID_ARG for NULL pointers, bytes == 0 or reps <= 0. */
int ftmoe_measure_link(const void *h_src, void *d_dst, size_t bytes, int32_t reps, void *stream,
                       double *memcpy_gbps, double *sm_read_gbps);

/* CPU MoE probe (benchmark guide, section 5.2: the bandwidth the CPU MoE kernel reaches on
 * the host's memory). Runs ftmoe_cpu_expert_ffn on `experts` tokens, each routed to a
 * different expert of the layer banks h_layer_banks (host, schema order, bank_bytes per
 * expert): repetition r routes token t to expert (r * experts + t) % E, so repetitions read
 * different experts while E allows. Best of `reps`; *gbps = experts * bytes per expert /
 * time. Host only.
 * FTMOE_ERR_FORMAT for formats without a CPU MoE path. */
int ftmoe_measure_cpu_moe(int32_t format, int32_t H, int32_t I, int32_t E, const void *const *h_layer_banks,
                          const int64_t *bank_bytes, int32_t experts, int32_t threads, int32_t reps,
                          double *gbps);

/* CPU memory read ceiling (benchmark guide, section 5.2: the bandwidth probe reports the
 * host CPU's memory read ceiling, the bound of the CPU MoE kernel, beside the link's).
 * `threads` workers (<= 0: all hardware threads) each sum a contiguous share of the host
 * buffer h_buf (whole 64-byte lines of its first `bytes` bytes; any host memory, e.g. a
 * layer's bank) as 64-bit words; best of `reps`; *gbps = bytes read / time / 1e9. Host
 * only, synchronous. FTMOE_ERR_INVALID_ARG for NULL pointers, bytes < 64 or reps <= 0. */
int ftmoe_measure_cpu_read(const void *h_buf, size_t bytes, int32_t threads, int32_t reps, double *gbps);

/* Backend decision (benchmark guide, section 5.2): FTMOE_BACKEND_HYBRID when the format has
 * a CPU MoE path and cpu_gbps > threshold * link_gbps (threshold <= 0: the default 2.0),
 * with *fetch_fraction from ftmoe_hybrid_fetch_fraction; otherwise FTMOE_BACKEND_OFFLOAD
 * with *fetch_fraction = 1. Formats without a CPU path (raw) always offload. Host only. */
int ftmoe_moe_backend_decision(int32_t format, double link_gbps, double cpu_gbps, double threshold,
                               int32_t *backend, float *fetch_fraction);

/* Select the copy_missing implementation (FTMOE_COPY_*). */
int ftmoe_set_copy_mode(ftmoe_cache_t *cache, int32_t mode);

/* Select the expert FFN kernels (FTMOE_FFN_*) of later ftmoe_expert_ffn calls. Both
 * families compute the same FFN (hit experts read from the slot cache: benchmark guide,
 * section 1; bf16 gate_up and down banks: section 4.2). FTMOE_ERR_INVALID_ARG for an
 * unknown kind; FTMOE_ERR_FORMAT for ROWS or MMA on a cache that is not bf16, or for MMA
 * when the shape has no tensor-core pipeline (H or I not a multiple of 256, or the cache
 * was created without FFN scratch). Host only. */
int ftmoe_set_ffn_kernels(ftmoe_cache_t *cache, int32_t kind);

/* The kernel family (FTMOE_FFN_ROWS: CUDA cores, FTMOE_FFN_MMA: tensor cores) that
 * ftmoe_expert_ffn on this cache runs for a call of bs tokens x topk experts, under the
 * current ftmoe_set_ffn_kernels choice. FTMOE_ERR_INVALID_ARG for NULL, bs < 0, topk <= 0
 * or bs * topk above FTMOE_MAX_IDS_PER_CALL; FTMOE_ERR_STATE for a cache created without
 * FFN scratch. Host only. */
int ftmoe_ffn_kernels_for(ftmoe_cache_t *cache, int32_t bs, int32_t topk, int32_t *kind);

/* Test settings of one cache, for exercising the bounded-wait error path (the pages define
 * nothing of the kind; production callers leave them at 0):
 *   FTMOE_DEBUG_WAIT_NS        value = the limit, in ns, of every bounded wait of the CUDA-core
 *                              FFN pipeline (0 restores the default of 2 s);
 *   FTMOE_DEBUG_FFN_SKIP_STAGE value = 1: later FFN calls that run the CUDA-core pipeline leave
 *                              the first gate_up stage of CTA 0 unfilled (no copies issued, no
 *                              arrive), so that CTA's consumers stop when their wait runs out:
 *                              the call records FTMOE_ERR_STATE in the status word, leaves y
 *                              undefined and returns with nothing in flight; 0 turns it off.
 * FTMOE_ERR_INVALID_ARG for an unknown setting or value. Host only. */
#define FTMOE_DEBUG_WAIT_NS 1
#define FTMOE_DEBUG_FFN_SKIP_STAGE 2
int ftmoe_set_debug(ftmoe_cache_t *cache, int32_t what, int64_t value);

/* Read the state into host arrays h_owner[S] (flat id or -1), h_stamp[S], *h_clock.
 * Synchronises the stream. */
int ftmoe_cache_get_state(ftmoe_cache_t *cache, int32_t *h_owner, uint32_t *h_stamp,
                          uint32_t *h_clock, void *stream);

/* Replace the state from host arrays (owner flat ids in [-1, L*E), no id twice,
 * stamps <= clock); id2slot is rebuilt on the device. FTMOE_ERR_STATE if the arrays
 * are inconsistent. The host arrays may be reused when the call returns. */
int ftmoe_cache_set_state(ftmoe_cache_t *cache, const int32_t *h_owner,
                          const uint32_t *h_stamp, uint32_t clock, void *stream);

/* Read the last ensure call's miss list into host arrays h_ids[], h_slots[] (room
 * for min(E, S) entries) and *h_m. Synchronises the stream. */
int ftmoe_get_miss_list(ftmoe_cache_t *cache, int32_t *h_ids, int32_t *h_slots,
                        int32_t *h_m, void *stream);

/* Read and clear the sticky device status word (FTMOE_OK or the first device error
 * since the last read). Synchronises the stream. */
int ftmoe_get_device_status(ftmoe_cache_t *cache, int32_t *h_status, void *stream);

/* Linear copy of `bytes` from page-locked host memory to device memory by SM loads
 * of the mapped host pointer (the copy kernel's data path without the cache; used to
 * measure the host-to-device link ceiling, as the pinned-to-device copy ceiling of
 * the benchmark guide, section 5.2). */
int ftmoe_h2d_stream_copy(void *d_dst, const void *h_src, size_t bytes, void *stream);

/* Bytes of the fixed device scratch behind ftmoe_expert_ffn_noalloc (16 MiB). */
#define FTMOE_NOALLOC_SCRATCH_BYTES (16u << 20)

/* Expert FFN that allocates nothing. The FreeToken pages have no counterpart of this
 * call; it is for callers that cannot call cudaMalloc: code embedded in a host runtime
 * that already owns all of the GPU's memory (a serving engine that reserved HBM for its
 * weights and KV cache up front, where an allocation would fail or break its
 * accounting), and code on a latency-critical path that must not pay for
 * cudaMalloc/cudaFree and the device synchronisation they can cause.
 *
 * Computes the FFN of ftmoe_expert_ffn, without a cache handle, to within the FFN
 * tolerance of that call (max abs 2e-2, relative L2 1e-2 on bf16 outputs; it runs the
 * general register-path kernels, not the bulk-copy or tensor-core pipelines, so it is
 * slower at decode sizes and its rounding differs). Formats FTMOE_FMT_BF16, NVFP4 and
 * MXFP4 only (block FP8 and Q4_0 have no register-path kernels): FTMOE_ERR_INVALID_ARG
 * otherwise. The caller passes its slot banks d_slot_banks[num_banks] (device
 * [S, per-expert bytes] each, in the schema order of `format`), the activations, slots,
 * router weights and the output, with the same layouts as ftmoe_expert_ffn; a slot of
 * -1 marks a position computed elsewhere, which contributes nothing. The routing tables
 * and fp32 intermediates live in one file-scope device array of
 * FTMOE_NOALLOC_SCRATCH_BYTES that every GPU loading the library reserves until the
 * process exits; calls needing more (about bs * topk * (H + I) * 4 bytes), or with bs
 * above 65535, fail with FTMOE_ERR_INVALID_ARG. The first call on a device looks up that
 * array's device address (cudaGetSymbolAddress) and keeps it for the life of the
 * process, so a device reset (cudaDeviceReset, or a reset of the primary context) while
 * the library is loaded is not supported; make that first call before any stream
 * capture. All calls share the array and it keeps the previous call's contents: calls
 * that overlap on the GPU race on it and must be serialised by the caller. A slot
 * outside [-1, S) leaves d_y_bf16 unwritten (there is no status to read back). */
int ftmoe_expert_ffn_noalloc(int32_t format, const void *const *d_slot_banks, int32_t num_banks,
                             int32_t S, int32_t H, int32_t I, const void *d_x_bf16, int32_t bs,
                             const int32_t *d_slots, const float *d_weights, int32_t topk,
                             void *d_y_bf16, void *stream);

/* Message of the last failing call on this thread. */
const char *ftmoe_last_error(void);

#ifdef __cplusplus
}
#endif
#endif
