/*
 * Oracle: global LRU expert slot cache (ensure_experts) — TEST INFRASTRUCTURE ONLY.
 *
 * Follows the FreeToken pages: one unified GPU slot cache shared by all layers
 * with LRU eviction ([ARCH] section 五), ensure_experts performs the "LRU slot
 * remap" of a layer's routed experts ([BENCH] section 4.1), over the flat id
 * space id = layer * E + expert ([BENCH] section 4.3).
 *
 * The pages give no tie rule and no clock; the readings used here are:
 *   - clock advances by one at the start of every ensure call (one tick per
 *     (step, layer) call, shared by all layers);
 *   - a slot hit or filled in the current call is never evicted in that call;
 *   - misses, taken in ascending flat id, receive the untouched slots in
 *     ascending (stamp, slot) order: least recently used first, lowest slot on
 *     equal stamps; empty slots keep stamp 0 and therefore go first;
 *   - more misses than untouched slots is a capacity error that leaves the
 *     state untouched.
 * Hybrid variant ([BENCH] section 5.4): only the first `cap` misses in ascending
 * flat id are fetched; the overflow keeps slot -1 for the CPU executor.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"

int orc_rebuild_id2slot(int32_t E, int32_t L, int32_t S, const int32_t *owner, int32_t *id2slot) {
    int64_t n = (int64_t)E * L;
    for (int64_t f = 0; f < n; f++) id2slot[f] = -1;
    for (int32_t s = 0; s < S; s++) {
        int32_t f = owner[s];
        if (f < 0) continue;
        if (f >= n) return ORC_ERR_STATE;
        if (id2slot[f] != -1) return ORC_ERR_STATE; /* one id in two slots */
        id2slot[f] = s;
    }
    return ORC_OK;
}

typedef struct {
    uint32_t stamp;
    int32_t slot;
} cand_t;

static int cand_cmp(const void *a, const void *b) {
    const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
    if (x->stamp != y->stamp) return x->stamp < y->stamp ? -1 : 1;
    return x->slot < y->slot ? -1 : (x->slot > y->slot ? 1 : 0);
}

static void fail_outputs(int32_t n, int32_t *slots_out, int32_t *num_miss) {
    for (int32_t t = 0; t < n; t++) slots_out[t] = -1;
    *num_miss = 0;
}

/* Fetch cap of the hybrid rule (see oracle.h); the product is formed in binary32. */
static int32_t hybrid_cap(int32_t misses, int32_t max_fetch, float fetch_fraction) {
    if (max_fetch >= 0) return max_fetch;
    if (fetch_fraction > 0.0f) {
        float want = (float)misses * fetch_fraction;
        return (int32_t)rintf(want);
    }
    return 1;
}

static int ensure_core(int32_t E, int32_t L, int32_t S, int32_t *owner, uint32_t *stamp,
                       int32_t *id2slot, uint32_t *clock, int32_t layer, const int32_t *topk_ids,
                       int32_t n, int hybrid, int32_t max_fetch, float fetch_fraction,
                       int32_t *slots_out, int32_t *miss_ids, int32_t *miss_slots,
                       int32_t *num_miss, int32_t *counts) {
    if (E <= 0 || L <= 0 || S <= 0 || n < 0 || layer < 0 || layer >= L) {
        fail_outputs(n < 0 ? 0 : n, slots_out, num_miss);
        return ORC_ERR_INVALID_ARG;
    }
    /* 1. every routed id must be a local expert id */
    for (int32_t t = 0; t < n; t++) {
        if (topk_ids[t] < 0 || topk_ids[t] >= E) {
            fail_outputs(n, slots_out, num_miss);
            return ORC_ERR_ID_RANGE;
        }
    }
    if (*clock == 0xFFFFFFFFu) {
        fail_outputs(n, slots_out, num_miss);
        return ORC_ERR_STATE;
    }
    uint32_t now = *clock + 1;

    /* 2. U = ascending unique flat ids of this call */
    char *present = (char *)calloc((size_t)E, 1);
    for (int32_t t = 0; t < n; t++) present[topk_ids[t]] = 1;

    /* 3. split U into hits (slot found) and misses (ascending) */
    char *hit_slot = (char *)calloc((size_t)S, 1);
    int32_t *misses = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    int32_t m = 0;
    for (int32_t e = 0; e < E; e++) {
        if (!present[e]) continue;
        int32_t f = layer * E + e;
        int32_t s = id2slot[f];
        if (s >= 0)
            hit_slot[s] = 1;
        else
            misses[m++] = f;
    }

    /* 4. candidates: every slot not hit by this call, ascending (stamp, slot) */
    cand_t *cand = (cand_t *)malloc(sizeof(cand_t) * (size_t)S);
    int32_t nc = 0;
    for (int32_t s = 0; s < S; s++) {
        if (hit_slot[s]) continue;
        cand[nc].stamp = stamp[s];
        cand[nc].slot = s;
        nc++;
    }
    qsort(cand, (size_t)nc, sizeof(cand_t), cand_cmp);

    int32_t m_full = m;
    if (hybrid) {
        int32_t cap = hybrid_cap(m_full, max_fetch, fetch_fraction);
        if (cap < 0) cap = 0;
        if (m > cap) m = cap; /* the first `cap` misses in ascending id are fetched */
    }
    int rc = ORC_OK;
    if (m > nc) {
        fail_outputs(n, slots_out, num_miss);
        rc = ORC_ERR_CAPACITY;
        goto done;
    }

    /* 5. commit: clock, hit stamps, then the j-th miss takes the j-th candidate */
    *clock = now;
    for (int32_t s = 0; s < S; s++)
        if (hit_slot[s]) stamp[s] = now;
    for (int32_t j = 0; j < m; j++) {
        int32_t s = cand[j].slot;
        int32_t old = owner[s];
        if (old >= 0) id2slot[old] = -1;
        owner[s] = misses[j];
        id2slot[misses[j]] = s;
        stamp[s] = now;
        miss_ids[j] = misses[j];
        miss_slots[j] = s;
    }
    *num_miss = m;
    if (counts) {
        counts[0] = m;
        counts[1] = m_full;
    }

    /* 6. slot of every routed (token, j) position (-1 for misses left to the CPU) */
    for (int32_t t = 0; t < n; t++) slots_out[t] = id2slot[layer * E + topk_ids[t]];

done:
    if (rc != ORC_OK && counts) counts[0] = counts[1] = 0;
    free(present);
    free(hit_slot);
    free(misses);
    free(cand);
    return rc;
}

int orc_ensure(int32_t E, int32_t L, int32_t S, int32_t *owner, uint32_t *stamp,
               int32_t *id2slot, uint32_t *clock, int32_t layer, const int32_t *topk_ids,
               int32_t n, int32_t *slots_out, int32_t *miss_ids, int32_t *miss_slots,
               int32_t *num_miss) {
    return ensure_core(E, L, S, owner, stamp, id2slot, clock, layer, topk_ids, n, 0, -1, 0.0f,
                       slots_out, miss_ids, miss_slots, num_miss, NULL);
}

int orc_ensure_hybrid(int32_t E, int32_t L, int32_t S, int32_t *owner, uint32_t *stamp,
                      int32_t *id2slot, uint32_t *clock, int32_t layer, const int32_t *topk_ids,
                      int32_t n, int32_t max_fetch, float fetch_fraction, int32_t *slots_out,
                      int32_t *miss_ids, int32_t *miss_slots, int32_t *num_miss, int32_t *counts) {
    return ensure_core(E, L, S, owner, stamp, id2slot, clock, layer, topk_ids, n, 1, max_fetch,
                       fetch_fraction, slots_out, miss_ids, miss_slots, num_miss, counts);
}
