// Bandwidth probes and the offload / hybrid backend decision.
//
// FreeToken benchmark guide, section 5.2: the engine measures the host memory bandwidth
// the CPU MoE kernel reaches and the pinned -> device gather bandwidth, and recommends
// hybrid for a (workload, format) when the CPU MoE bandwidth exceeds a threshold (2x by
// default) times the gather bandwidth, offload otherwise; formats without a CPU MoE
// weight path always offload. Section 5.4 sets the fetch share of a hybrid step to
// pcie : (cpu - pcie) of the misses.
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cstdint>
#include <vector>

#include "ftmoe.h"

// records the library's thread-local error message (defined with the other entry points)
int ftmoe_probe_report(int code, const char *msg);

namespace {
int probe_fail(int code, const char *msg) { return ftmoe_probe_report(code, msg); }

bool has_cpu_path(int32_t format) {
    return format == FTMOE_FMT_BF16 || format == FTMOE_FMT_NVFP4 || format == FTMOE_FMT_MXFP4;
}
}  // namespace

extern "C" {

int ftmoe_measure_link(const void *h_src, void *d_dst, size_t bytes, int32_t reps, void *stream,
                       double *memcpy_gbps, double *sm_read_gbps) {
    if (!h_src || !d_dst || !memcpy_gbps || !sm_read_gbps || bytes == 0 || reps <= 0)
        return probe_fail(FTMOE_ERR_INVALID_ARG, "measure_link: NULL pointer, zero bytes or reps <= 0");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaEvent_t a = nullptr, b = nullptr;
    if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) {
        if (a) cudaEventDestroy(a);
        cudaGetLastError();
        return probe_fail(FTMOE_ERR_CUDA, "measure_link: event create failed");
    }
    double best[2] = {1e30, 1e30};
    int rc = FTMOE_OK;
    for (int arm = 0; arm < 2 && rc == FTMOE_OK; arm++) {
        for (int r = 0; r < reps; r++) {
            if (cudaEventRecord(a, st) != cudaSuccess) {
                rc = probe_fail(FTMOE_ERR_CUDA, "measure_link: event record failed");
                break;
            }
            if (arm == 0) {
                if (cudaMemcpyAsync(d_dst, h_src, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) {
                    rc = probe_fail(FTMOE_ERR_CUDA, "measure_link: cudaMemcpyAsync failed");
                    break;
                }
            } else if ((rc = ftmoe_h2d_stream_copy(d_dst, h_src, bytes, st)) != FTMOE_OK) {
                break;
            }
            float ms = 0.f;
            if (cudaEventRecord(b, st) != cudaSuccess || cudaEventSynchronize(b) != cudaSuccess ||
                cudaEventElapsedTime(&ms, a, b) != cudaSuccess) {
                rc = probe_fail(FTMOE_ERR_CUDA, "measure_link: timing failed");
                break;
            }
            best[arm] = std::min(best[arm], (double)ms * 1e-3);
        }
    }
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    if (rc != FTMOE_OK) {
        cudaGetLastError();
        return rc;
    }
    *memcpy_gbps = (double)bytes / best[0] / 1e9;
    *sm_read_gbps = (double)bytes / best[1] / 1e9;
    return FTMOE_OK;
}

int ftmoe_measure_cpu_moe(int32_t format, int32_t H, int32_t I, int32_t E, const void *const *h_layer_banks,
                          const int64_t *bank_bytes, int32_t experts, int32_t threads, int32_t reps,
                          double *gbps) {
    if (!has_cpu_path(format)) return probe_fail(FTMOE_ERR_FORMAT, "measure_cpu_moe: no CPU MoE path for this format");
    if (!h_layer_banks || !bank_bytes || !gbps || E <= 0 || experts <= 0 || reps <= 0)
        return probe_fail(FTMOE_ERR_INVALID_ARG, "measure_cpu_moe: bad argument");
    const int nb = format == FTMOE_FMT_BF16 ? 2 : 6;
    int64_t per_expert = 0;
    for (int b = 0; b < nb; b++) per_expert += bank_bytes[b];
    // one token per expert, each routed to a different expert, all computed on the CPU; each
    // repetition takes the next `experts` experts of the layer (so a repetition does not find
    // the previous one's weights in the host caches while the layer has enough experts)
    std::vector<int32_t> ids(experts), slots(experts, -1);
    std::vector<uint16_t> x((size_t)experts * H, 0x3f80u);  // bf16 1.0
    std::vector<float> w(experts, 1.f), y((size_t)experts * H);
    double best = 1e30;
    for (int r = 0; r < reps; r++) {
        for (int t = 0; t < experts; t++) ids[t] = (int32_t)(((int64_t)r * experts + t) % E);
        const auto t0 = std::chrono::steady_clock::now();
        int rc = ftmoe_cpu_expert_ffn(format, H, I, experts, 1, ids.data(), slots.data(), h_layer_banks, bank_bytes,
                                      x.data(), w.data(), y.data(), threads);
        const auto t1 = std::chrono::steady_clock::now();
        if (rc != FTMOE_OK) return rc;
        best = std::min(best, std::chrono::duration<double>(t1 - t0).count());
    }
    *gbps = (double)experts * (double)per_expert / best / 1e9;
    return FTMOE_OK;
}

int ftmoe_moe_backend_decision(int32_t format, double link_gbps, double cpu_gbps, double threshold,
                               int32_t *backend, float *fetch_fraction) {
    if (!backend || !fetch_fraction) return probe_fail(FTMOE_ERR_INVALID_ARG, "backend decision: NULL output");
    if (!(threshold > 0.0)) threshold = 2.0;
    *backend = FTMOE_BACKEND_OFFLOAD;
    *fetch_fraction = 1.f;
    if (has_cpu_path(format) && link_gbps > 0.0 && cpu_gbps > threshold * link_gbps) {
        *backend = FTMOE_BACKEND_HYBRID;
        return ftmoe_hybrid_fetch_fraction(link_gbps, cpu_gbps, fetch_fraction);
    }
    return FTMOE_OK;
}

}  // extern "C"
