// Per-launch timing of the library's own kernels: when tracing is on, every
// launch is bracketed by two CUDA events recorded on the launching stream.
#pragma once

#include <cuda_runtime.h>

namespace ssa {

void trace_before(const char* name, cudaStream_t stream);
void trace_after(cudaStream_t stream);

// Brackets one launch; a no-op (one relaxed load) while tracing is off.
struct TraceLaunch {
    cudaStream_t s;
    TraceLaunch(const char* name, cudaStream_t stream) : s(stream) { trace_before(name, stream); }
    ~TraceLaunch() { trace_after(s); }
};

}  // namespace ssa
