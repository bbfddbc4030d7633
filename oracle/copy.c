/*
 * Oracle: copy_missing — TEST INFRASTRUCTURE ONLY.
 *
 * [BENCH] section 4.2: the cache is layout-agnostic and only moves rows, so a
 * miss copies, for every bank, the expert's bytes unchanged from the host bank
 * of its layer into the slot row; section 4.4: the sources are per-layer
 * lists and copy_MiB = misses * bytes per expert.
 */
#include <string.h>

#include "oracle.h"

void orc_copy_missing(int32_t num_banks, const int64_t *bank_bytes,
                      const uint8_t *const *host_layer, uint8_t *const *slots, int32_t E,
                      const int32_t *miss_ids, const int32_t *miss_slots, int32_t m) {
    for (int32_t j = 0; j < m; j++) {
        int64_t e = miss_ids[j] % E;
        int64_t s = miss_slots[j];
        for (int32_t b = 0; b < num_banks; b++) {
            int64_t nb = bank_bytes[b];
            memcpy(slots[b] + s * nb, host_layer[b] + e * nb, (size_t)nb);
        }
    }
}
