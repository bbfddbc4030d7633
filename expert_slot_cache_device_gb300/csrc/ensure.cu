// K1: ensure_experts — dedup, slot lookup and LRU eviction in one CTA.
//
// FreeToken benchmark guide ("FreeToken MoE 离线推理基准完全指南"), section 4.1:
// ensure_experts is the LRU slot remap of a layer's routed experts; section 4.3:
// flat id = layer * E + expert. Architecture deep-dive, section 五: one global
// LRU cache shared by all layers. Victim rule: the misses, ascending by flat id,
// take the slots not hit in this call in ascending (stamp, slot) order.
//
// One CTA of 1024 threads does the whole call so that the miss list is ready on
// the device for the copy kernel without a host round trip. Every independent
// global load (ids, the layer's id2slot row, stamps, owners, clock) is issued
// up front, so a call costs about one memory latency plus the sort:
//   1. mark the routed local ids in a shared table over E (dedup; scanning the
//      table in index order yields the distinct ids already ascending);
//   2. probe id2slot for every distinct id; hits mark their slot as used;
//   3. block-wide prefix sum over the miss flags gives every miss its rank;
//   4. 64-bit keys (stamp << 32 | slot) of the unused slots are sorted by a
//      bitonic network (one key per thread in registers for S <= 1024: warp
//      shuffles for distances below 32, shared memory above; a shared-memory
//      network for larger S); the j-th smallest key is the j-th victim —
//      exactly the lowest-(stamp, slot) rule;
//   5. tables are updated and every routed position gets its slot.
// The hybrid variant (benchmark guide, section 5.4) fetches only the first `cap`
// misses in ascending flat id; the overflow keeps slot -1 for the CPU executor.
// Errors (id out of range, clock exhausted, too many misses) write only the
// status word, -1 slots and an empty miss list.
#include "internal.cuh"

namespace ftmoe {
namespace {

constexpr int kThreads = 1024;

__device__ __forceinline__ void set_status(int32_t *status, int err) { atomicCAS(status, 0, err); }

// Exclusive prefix sum of `flag` over the block (deterministic, in thread order).
__device__ __forceinline__ int block_excl_scan(int flag, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned ball = __ballot_sync(0xffffffffu, flag);
    int pre = __popc(ball & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[warp] = __popc(ball);
    __syncthreads();
    if (warp == 0) {
        int v = (lane < (int)(blockDim.x >> 5)) ? warp_tot[lane] : 0;
        int incl = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int u = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += u;
        }
        warp_tot[lane] = incl - v;  // exclusive warp offsets
        if (lane == 31) *total = incl;
    }
    __syncthreads();
    int r = warp_tot[warp] + pre;
    __syncthreads();  // warp_tot reused by the next call
    return r;
}

// In-place ascending bitonic sort of n (power of two) keys in shared memory.
__device__ void bitonic_sort_smem(uint64_t *keys, int n) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < (n >> 1); i += blockDim.x) {
                int lo = ((i & ~(j - 1)) << 1) | (i & (j - 1));
                int hi = lo + j;
                bool up = (lo & k) == 0;
                uint64_t a = keys[lo], b = keys[hi];
                if ((a > b) == up) {
                    keys[lo] = b;
                    keys[hi] = a;
                }
            }
            __syncthreads();
        }
    }
}

// Ascending bitonic sort of n <= blockDim.x keys, one per thread (thread i ends with
// the i-th smallest). Exchange distances below 32 use warp shuffles, larger ones go
// through shared memory `xbuf` (blockDim.x entries). Every thread must call it.
__device__ uint64_t bitonic_sort_regs(uint64_t key, int n, uint64_t *xbuf) {
    const int i = threadIdx.x;
    const bool active = (i & ~31) < n;  // whole warps past the sort width only join the barriers
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            uint64_t other = key;
            if (j >= 32) {
                if (active) xbuf[i] = key;
                __syncthreads();
                if (active) other = xbuf[i ^ j];
                __syncthreads();
            } else if (active) {
                other = __shfl_xor_sync(0xffffffffu, key, j);
            }
            const bool keep_min = ((i & j) == 0) == ((i & k) == 0);
            key = keep_min ? (other < key ? other : key) : (other > key ? other : key);
        }
    }
    return key;
}

constexpr int kPerThread = 8;  // slots and experts per thread: 8 x blockDim covers S and E

__global__ void __launch_bounds__(kThreads) ensure_kernel(EnsureParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int xn = p.Spad > (int)blockDim.x ? p.Spad : (int)blockDim.x;
    uint64_t *keys = reinterpret_cast<uint64_t *>(smem);          // [max(Spad, blockDim)]
    int32_t *s_slot = reinterpret_cast<int32_t *>(keys + xn);      // [E]: -2 absent, -1 miss, >=0 slot
    int32_t *s_miss = s_slot + p.E;                               // [maxm] flat ids by rank
    int32_t *s_owner = s_miss + p.maxm;                           // [S]
    unsigned char *s_hit = reinterpret_cast<unsigned char *>(s_owner + p.S);  // [S]
    __shared__ int warp_tot[32];
    __shared__ int s_bad_id, s_m, s_mfull, s_h, s_tmp;

    const int tid = threadIdx.x, nt = blockDim.x;
    const int E = p.E, S = p.S;
    // the copy kernel behind this one may become resident now; it waits for this grid to
    // finish before it reads the miss list
    asm volatile("griddepcontrol.launch_dependents;" :::);
    // Prologue: issue every independent global load before the first use, so the
    // call pays about one memory latency instead of one per step.
    const int32_t *row = p.t.id2slot + (int64_t)p.layer * E;
    int32_t rowv[kPerThread];
    uint32_t stampv[kPerThread];
#pragma unroll
    for (int k = 0; k < kPerThread; k++) {
        const int e = tid + k * nt, s = tid + k * nt;
        rowv[k] = e < E ? row[e] : -1;
        stampv[k] = s < S ? p.t.stamp[s] : 0u;
        if (s < S) s_owner[s] = p.t.owner[s];
    }
    const uint32_t clock = *p.t.clock;
    if (tid == 0) {
        s_bad_id = 0;
        s_h = 0;
    }
    for (int e = tid; e < E; e += nt) s_slot[e] = -2;
    for (int s = tid; s < S; s += nt) s_hit[s] = 0;
    __syncthreads();

    // 1. dedup (benign races: every writer stores the same value)
    for (int t = tid; t < p.n; t += nt) {
        int id = p.ids[t];
        if ((unsigned)id >= (unsigned)E)
            s_bad_id = 1;
        else
            s_slot[id] = -1;
    }
    __syncthreads();

    int err = s_bad_id ? FTMOE_ERR_ID_RANGE : (clock == 0xFFFFFFFFu ? FTMOE_ERR_STATE : 0);
    if (err == 0) {
        // 2. probe (the row was prefetched; each thread handles the ids it loaded)
        int hits = 0;
#pragma unroll
        for (int k = 0; k < kPerThread; k++) {
            const int e = tid + k * nt;
            if (e < E && s_slot[e] == -1 && rowv[k] >= 0) {
                s_slot[e] = rowv[k];
                s_hit[rowv[k]] = 1;
                hits++;
            }
        }
        if (hits) atomicAdd(&s_h, hits);
        // 3. miss ranks in ascending id (each s_slot entry is read by the thread that wrote it)
        int base = 0;
        for (int e0 = 0; e0 < E; e0 += nt) {
            int e = e0 + tid;
            int flag = (e < E) && (s_slot[e] == -1);
            int r = block_excl_scan(flag, warp_tot, &s_tmp);
            // more than min(E, S) misses is a capacity error found below; never write past the list
            if (flag && base + r < p.maxm) s_miss[base + r] = p.layer * E + e;
            base += s_tmp;  // every thread reads the same total (synchronised in the scan)
            __syncthreads();
        }
        if (tid == 0) {
            s_mfull = base;
            int m = base;
            if (p.hybrid) {  // fetch only the first `cap` misses (ascending flat id)
                int cap = p.max_fetch >= 0 ? p.max_fetch
                                           : (p.fetch_fraction > 0.f ? (int)rintf((float)base * p.fetch_fraction) : 1);
                if (cap < 0) cap = 0;
                if (m > cap) m = cap;
            }
            s_m = m;
        }
        __syncthreads();
        if (s_m > S - s_h) err = FTMOE_ERR_CAPACITY;
    }
    if (err != 0) {
        for (int t = tid; t < p.n; t += nt) p.slots_out[t] = -1;
        if (tid == 0) {
            *p.t.num_miss = 0;
            if (p.counts) p.counts[0] = p.counts[1] = 0;
            set_status(p.t.status, err);
        }
        return;
    }

    const int m = s_m;
    const uint32_t now = clock + 1;
    // 4. victims: the m smallest (stamp, slot) keys among the slots not hit in this call
    uint64_t victim = ~0ull;
    if (m > 0) {
        if (p.Spad <= nt) {
            const uint64_t key = (tid < S && !s_hit[tid]) ? ((uint64_t)stampv[0] << 32) | (uint32_t)tid : ~0ull;
            victim = bitonic_sort_regs(key, p.Spad, keys);
        } else {
#pragma unroll
            for (int k = 0; k < kPerThread; k++) {
                const int s = tid + k * nt;
                if (s < p.Spad) keys[s] = (s < S && !s_hit[s]) ? ((uint64_t)stampv[k] << 32) | (uint32_t)s : ~0ull;
            }
            __syncthreads();
            bitonic_sort_smem(keys, p.Spad);
        }
    }
    // 5. update: hit stamps, then victims (hit and victim slots are disjoint; an
    //    evicted owner is never one of this call's misses, whose id2slot is -1)
    for (int s = tid; s < S; s += nt)
        if (s_hit[s]) p.t.stamp[s] = now;
    for (int j = tid; j < m; j += nt) {
        const uint64_t key = p.Spad <= nt ? victim : keys[j];
        int s = (int)(uint32_t)(key & 0xffffffffu);
        int f = s_miss[j];
        int old = s_owner[s];
        if (old >= 0) p.t.id2slot[old] = -1;
        p.t.owner[s] = f;
        p.t.id2slot[f] = s;
        p.t.stamp[s] = now;
        p.t.miss_ids[j] = f;
        p.t.miss_slots[j] = s;
        s_slot[f - p.layer * E] = s;
    }
    __syncthreads();
    for (int t = tid; t < p.n; t += nt) p.slots_out[t] = s_slot[p.ids[t]];
    if (tid == 0) {
        *p.t.clock = now;
        *p.t.num_miss = m;
        if (p.counts) {
            p.counts[0] = m;
            p.counts[1] = s_mfull;
        }
        if (p.t.stats) {  // cumulative: calls, distinct ids (hits + all misses), fetched misses
            p.t.stats[0] += 1ull;
            p.t.stats[1] += (unsigned long long)(s_h + s_mfull);
            p.t.stats[2] += (unsigned long long)m;
        }
    }
}

__global__ void init_state_kernel(Tables t, int LE, int S) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    int stride = gridDim.x * blockDim.x;
    for (int f = i; f < LE; f += stride) t.id2slot[f] = -1;
    for (int s = i; s < S; s += stride) {
        t.owner[s] = -1;
        t.stamp[s] = 0;
    }
    if (i == 0) {
        *t.clock = 0;
        *t.status = 0;
        *t.num_miss = 0;
        if (t.stats) t.stats[0] = t.stats[1] = t.stats[2] = 0ull;
    }
}

__global__ void clear_id2slot_kernel(Tables t, int LE) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    for (int f = i; f < LE; f += gridDim.x * blockDim.x) t.id2slot[f] = -1;
}

__global__ void scatter_owner_kernel(Tables t, int S) {
    int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s < S) {
        int f = t.owner[s];
        if (f >= 0) t.id2slot[f] = s;
    }
    if (s == 0) *t.num_miss = 0;
}

}  // namespace

// Smallest power-of-two block (256..1024) whose threads cover the sort width, S and E / 8.
int ensure_threads(int E, int S, int Spad) {
    int need = Spad > S ? Spad : S;
    const int e8 = (E + kPerThread - 1) / kPerThread;
    if (e8 > need) need = e8;
    int nt = 256;
    while (nt < need && nt < kThreads) nt <<= 1;
    return nt;
}

size_t ensure_smem_bytes(int E, int S, int Spad, int maxm) {
    const int nt = ensure_threads(E, S, Spad);
    const size_t xn = Spad > nt ? Spad : nt;
    size_t b = xn * 8 + (size_t)E * 4 + (size_t)maxm * 4 + (size_t)S * 4 + (size_t)S;
    return (b + 15) & ~(size_t)15;
}

cudaError_t launch_ensure(const EnsureParams &p, cudaStream_t st) {
    size_t smem = ensure_smem_bytes(p.E, p.S, p.Spad, p.maxm);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(ensure_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    ensure_kernel<<<1, ensure_threads(p.E, p.S, p.Spad), smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_init_state(Tables t, int E, int L, int S, cudaStream_t st) {
    int LE = E * L;
    int n = LE > S ? LE : S;
    int grid = (n + 255) / 256;
    if (grid > 1024) grid = 1024;
    init_state_kernel<<<grid, 256, 0, st>>>(t, LE, S);
    return cudaGetLastError();
}

cudaError_t launch_rebuild_id2slot(Tables t, int E, int L, int S, cudaStream_t st) {
    int LE = E * L;
    int grid = (LE + 255) / 256;
    if (grid > 1024) grid = 1024;
    clear_id2slot_kernel<<<grid, 256, 0, st>>>(t, LE);
    scatter_owner_kernel<<<(S + 255) / 256, 256, 0, st>>>(t, S);
    return cudaGetLastError();
}

}  // namespace ftmoe
