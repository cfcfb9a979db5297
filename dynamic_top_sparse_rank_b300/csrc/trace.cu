// Launch tracing (see trace.h and ssa_trace_begin / ssa_trace_end in ssa.h).
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "trace.h"

namespace {

struct Record {
    const char* name;
    cudaEvent_t start, stop;
};

std::atomic<bool> g_on{false};
std::mutex g_mu;
std::vector<Record> g_records;

}  // namespace

namespace ssa {

void trace_before(const char* name, cudaStream_t stream) {
    if (!g_on.load(std::memory_order_relaxed)) return;
    Record r{name, nullptr, nullptr};
    if (cudaEventCreate(&r.start) != cudaSuccess) return;
    if (cudaEventCreate(&r.stop) != cudaSuccess) {
        cudaEventDestroy(r.start);
        return;
    }
    cudaEventRecord(r.start, stream);
    std::lock_guard<std::mutex> lock(g_mu);
    g_records.push_back(r);
}

void trace_after(cudaStream_t stream) {
    if (!g_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_records.empty()) cudaEventRecord(g_records.back().stop, stream);
}

}  // namespace ssa

extern "C" {

int ssa_trace_begin(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    for (auto& r : g_records) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    g_records.clear();
    g_on.store(true);
    return 0;
}

int ssa_trace_end(ssa_trace_record* out, int max_records) {
    g_on.store(false);
    std::lock_guard<std::mutex> lock(g_mu);
    int n = 0, bad = 0;
    for (auto& r : g_records) {
        float ms = -1.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess ||
            cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
            bad = 1;
        if (out && n < max_records) {
            std::strncpy(out[n].name, r.name, sizeof(out[n].name) - 1);
            out[n].name[sizeof(out[n].name) - 1] = '\0';
            out[n].ms = ms;
        }
        ++n;
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    g_records.clear();
    return bad ? -1 : n;
}

}  // extern "C"
