// ssa_score_topk_noalloc: the row-wise exact score + top-k kernel, with its
// scratch in a fixed device array owned by this library instead of a
// caller-provided workspace.
//
// Who needs it: callers that are not allowed to allocate device memory on the
// path that runs this op — a plugin inside an inference engine that hands its
// ops a pre-sized memory arena and no allocator, or a latency-critical loop
// that must never call cudaMalloc (which can synchronize the device and whose
// cost is unbounded). Such a caller still passes the inputs and outputs; the
// scratch comes from the array below.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace ssa {
cudaError_t topk_rows_dispatch(const void* q_low, const void* k_low, bool bf16, int P,
                               const int64_t* row_list, int64_t rows, const int32_t* rows_dev,
                               int Tq, int Tk, int k, int causal, float scale, int32_t* idx,
                               float* score, uint32_t* ws, int64_t ws_slots, int64_t ws_stride,
                               cudaStream_t stream);
}  // namespace ssa

namespace {

// 32 MiB of scratch, held by every device that loads this library until the
// process exits. The row-wise kernel needs round_up(Tk, 64) * 4 bytes per row
// it processes at a time; it overwrites what it reads, so nothing has to be
// cleared between calls.
constexpr size_t kScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxSlots = 1024;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Host code may not use g_noalloc_scratch as an address (it names a host-side
// stand-in); the device address is looked up once per device, and again only
// if the device's context has changed since (after a cudaDeviceReset the
// module, and with it the array, is loaded anew at another address).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(f);
}

// Unique id of the calling thread's current context (0 when there is none
// or the driver cannot tell): ids are never reused within a process.
unsigned long long current_context_id() {
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

cudaError_t scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
        // the lookup made the device's context current if it was not yet
        g_scratch_ctx[dev] = ctx != 0 ? ctx : current_context_id();
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" ssa_status ssa_score_topk_noalloc(const void* q_low, const void* k_low, int dtype, int B,
                                             int H, int Tq, int Tk, int P, int k, int causal,
                                             float scale, int32_t* idx, float* score,
                                             int32_t* dev_status, void* stream) {
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0 || k < 1 || (dtype != SSA_F32 && dtype != SSA_BF16) ||
        !isfinite(scale))
        return SSA_ERR_INVALID;
    if (!(P == 16 || P == 32 || P == 64 || P == 128) || k > 2048) return SSA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * H * Tq;
    if (rows == 0) return SSA_OK;
    if (!idx || !aligned(idx, 4) || (score && !aligned(score, 4))) return SSA_ERR_INVALID;
    if (!q_low || !aligned(q_low, 16)) return SSA_ERR_INVALID;
    if (Tk > 0 && (!k_low || !aligned(k_low, 16))) return SSA_ERR_INVALID;
    // the row-wise kernel has no device-side error to report: *dev_status is
    // checked like every other call's and left unchanged
    if (dev_status && !aligned(dev_status, 4)) return SSA_ERR_INVALID;
    const int64_t stride = ((int64_t)Tk + 63) / 64 * 64;   // 32-bit keys per row slot
    const int64_t slot_bytes = stride * 4;
    if (slot_bytes > (int64_t)kScratchBytes) return SSA_ERR_UNSUPPORTED;   // Tk > 8,388,608
    int64_t slots = slot_bytes > 0 ? (int64_t)kScratchBytes / slot_bytes : kMaxSlots;
    if (slots > kMaxSlots) slots = kMaxSlots;
    if (slots > rows) slots = rows;
    void* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return SSA_ERR_CUDA;
    const float sc = scale > 0.f ? scale : (float)(1.0 / sqrt((double)P));
    cudaError_t e = ssa::topk_rows_dispatch(q_low, k_low, dtype == SSA_BF16, P, nullptr, rows,
                                            nullptr, Tq, Tk, k, causal, sc, idx, score,
                                            reinterpret_cast<uint32_t*>(scratch), slots, stride,
                                            reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
}
