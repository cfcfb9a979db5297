// Tensor-map encoding with a small per-process cache, and the one-time shared
// memory opt-in of the TMA kernels.
#include "tmap.h"

#include <mutex>

namespace ssa {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

struct Entry {
    int dev, rank;
    const void* base;
    uint64_t dims[3], strides[2];
    uint32_t box[3];
    CUtensorMap map;
    uint64_t stamp;   // 0: empty
};

constexpr int kEntries = 16;
std::mutex g_mu;
Entry g_cache[kEntries];
uint64_t g_clock = 0;

bool same(const Entry& e, int dev, const void* base, int rank, const uint64_t* dims,
          const uint64_t* strides, const uint32_t* box) {
    if (e.stamp == 0 || e.dev != dev || e.base != base || e.rank != rank) return false;
    for (int i = 0; i < rank; ++i)
        if (e.dims[i] != dims[i] || e.box[i] != box[i]) return false;
    for (int i = 0; i + 1 < rank; ++i)
        if (e.strides[i] != strides[i]) return false;
    return true;
}

}  // namespace

bool tmap_bf16_sw128(CUtensorMap* out, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box) {
    if (rank < 2 || rank > 3) return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(g_mu);
    for (Entry& e : g_cache)
        if (same(e, dev, base, rank, dims, strides, box)) {
            e.stamp = ++g_clock;
            *out = e.map;
            return true;
        }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[3], st[2];
    cuuint32_t bx[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
    CUtensorMap m;
    if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base),
           d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    Entry* victim = &g_cache[0];   // an empty slot, else the least recently used
    for (Entry& e : g_cache)
        if (e.stamp < victim->stamp) victim = &e;
    victim->dev = dev;
    victim->rank = rank;
    victim->base = base;
    for (int i = 0; i < 3; ++i) {
        victim->dims[i] = i < rank ? dims[i] : 0;
        victim->box[i] = i < rank ? box[i] : 0;
    }
    for (int i = 0; i < 2; ++i) victim->strides[i] = i + 1 < rank ? strides[i] : 0;
    victim->map = m;
    victim->stamp = ++g_clock;
    *out = m;
    return true;
}

cudaError_t set_max_dyn_smem(const void* func, int bytes) {
    struct Done {
        const void* func;
        int dev, bytes;
    };
    static Done done[64];
    static int n_done = 0;
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done[i].func == func && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && n_done < 64) done[n_done++] = {func, dev, bytes};
    return e;
}

}  // namespace ssa
