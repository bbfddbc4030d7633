// K2: copy_missing — one fused kernel for every (miss, bank) segment.
//
// FreeToken benchmark guide, section 4.2: the cache is layout-agnostic and only
// moves rows; section 4.4: the multi-bank copy is fused (a per-bank path is kept
// for A/B comparison); section 一: misses travel from page-locked host memory to
// the GPU slot cache over the host link.
//
// The SMs read the mapped host banks directly (zero-copy) with 16-byte loads and
// write 16-byte stores into the slot banks. The work is cut into 32 KiB tiles,
// each inside one (miss, bank) segment; a persistent grid (a multiple of the SM
// count) strides over the tiles. The number of misses is read on the device, so
// the launch needs no host round trip after ensure_experts; surplus CTAs find no
// tile and exit. Each thread issues all its loads of a tile before its stores so
// that every SM keeps ~kCopyUnroll x 4 KiB per CTA of host reads in flight, which
// the link's latency needs.
#include "internal.cuh"

namespace ftmoe {
namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_vec(uint4 *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Copy `nbytes` (<= kCopyTile) from src to dst with the whole CTA.
template <bool VEC>
__device__ __forceinline__ void copy_tile(unsigned char *dst, const unsigned char *src, int64_t nbytes) {
    if (VEC) {
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
        const int nvec = (int)(nbytes >> 4);
        uint4 v[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; u++) {
            int i = u * kCopyThreads + threadIdx.x;
            if (i < nvec) v[u] = ld_stream(s4 + i);
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; u++) {
            int i = u * kCopyThreads + threadIdx.x;
            if (i < nvec) st_vec(d4 + i, v[u]);
        }
    } else {
        for (int64_t i = threadIdx.x; i < nbytes; i += kCopyThreads) dst[i] = src[i];
    }
}

template <bool VEC>
__global__ void __launch_bounds__(kCopyThreads) copy_missing_kernel(CopyParams p) {
    // launched as a programmatic dependent of ensure_experts: the CTAs become resident while
    // it runs and wait here until its miss list is complete and visible; the FFN's routing
    // kernel may in turn launch early behind this grid
    asm volatile("griddepcontrol.launch_dependents;" :::);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int m = *p.num_miss;
    if (!FTMOE_DCHECK(m >= 0 && m <= p.maxm, p.status)) return;
    const int64_t tpe = p.tile0[p.nb];  // tiles per expert over all banks
    const int64_t total = (int64_t)m * tpe;
    for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
        const int j = (int)(t / tpe);
        const int64_t r = t - (int64_t)j * tpe;
        int b = 0;
        while (b + 1 < p.nb && r >= p.tile0[b + 1]) b++;
        const int64_t off = (r - p.tile0[b]) * kCopyTile;
        const int64_t bb = p.bytes[b];
        const int64_t n = bb - off < kCopyTile ? bb - off : kCopyTile;
        const int64_t e = p.miss_ids[j] % p.E;
        const int64_t s = p.miss_slots[j];
        if (!FTMOE_DCHECK(s >= 0 && s < p.S && p.miss_ids[j] >= 0 && p.miss_ids[j] < (int64_t)p.L * p.E, p.status))
            continue;
        copy_tile<VEC>(p.dst[b] + s * bb + off, p.src[b] + e * bb + off, n);
    }
}

template <bool VEC>
__global__ void __launch_bounds__(kCopyThreads) linear_copy_kernel(unsigned char *dst, const unsigned char *src,
                                                                   int64_t bytes) {
    const int64_t tiles = (bytes + kCopyTile - 1) / kCopyTile;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t off = t * kCopyTile;
        const int64_t n = bytes - off < kCopyTile ? bytes - off : kCopyTile;
        copy_tile<VEC>(dst + off, src + off, n);
    }
}

}  // namespace

cudaError_t launch_copy(const CopyParams &p, bool vec16, int grid, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kCopyThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return vec16 ? cudaLaunchKernelEx(&cfg, copy_missing_kernel<true>, p)
                 : cudaLaunchKernelEx(&cfg, copy_missing_kernel<false>, p);
}

cudaError_t launch_linear_copy(unsigned char *dst, const unsigned char *src, int64_t bytes, bool vec16, int grid,
                               cudaStream_t st) {
    if (vec16)
        linear_copy_kernel<true><<<grid, kCopyThreads, 0, st>>>(dst, src, bytes);
    else
        linear_copy_kernel<false><<<grid, kCopyThreads, 0, st>>>(dst, src, bytes);
    return cudaGetLastError();
}

}  // namespace ftmoe
