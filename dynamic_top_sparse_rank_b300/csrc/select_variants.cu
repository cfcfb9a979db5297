// Selection variants of the scorer's top-k (mhpq.cn/news/1098205, section
// 4.2). Boundary smoothing: after an exact top-(k+1) selection, the (k+1)-th
// key stays selected only when its score is within `delta` of the k-th one
// (the gap an fp32 subtraction of the two fp32 scores), so that near-ties at
// the boundary do not flip between runs; otherwise its slot becomes index -1
// and score -inf. (The temperature of the same section is a positive factor
// on the scores: the scale argument of the score calls.)
#ifdef SSA_HOST_EMULATION
#include "emu_device.h"   // the host stand-in of the CPU tests (tests/emu)
#else
#include "common.cuh"
#include "trace.h"
#endif

namespace ssa {

__global__ void smooth_boundary_kernel(int32_t* __restrict__ idx, float* __restrict__ score,
                                       int64_t rows, int k, float delta) {
    const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= rows) return;
    const int64_t base = row * static_cast<int64_t>(k + 1);
    if (idx[base + k] < 0) return;   // no (k+1)-th key in this row
    const float gap = __fsub_rn(score[base + k - 1], score[base + k]);
    if (!(gap < delta)) {
        idx[base + k] = -1;
        score[base + k] = -INFINITY;
    }
}

#ifndef SSA_HOST_EMULATION   // the CPU tests launch the kernel themselves
// idx / score: [rows, k + 1], sorted by score descending (the output of an
// exact top-(k+1) selection); k >= 1.
cudaError_t smooth_boundary_launch(int32_t* idx, float* score, int64_t rows, int k, float delta,
                                   cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = (rows + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    TraceLaunch tr("smooth_boundary", stream);
    smooth_boundary_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(idx, score, rows, k,
                                                                             delta);
    return cudaGetLastError();
}
#endif  // SSA_HOST_EMULATION

}  // namespace ssa
