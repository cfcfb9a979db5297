// Tensor-core scorer: S = q_low . k_low^T * scale on tcgen05, one 128-query
// tile of a head against all its valid keys, 128 keys at a time. The score
// tile lives in TMEM only; an epilogue warpgroup reduces it on the fly, so the
// n x n score matrix never reaches HBM (the low-rank scorer of
// mhpq.cn/news/1098205, section 2.2; the selection of its section 3.2).
//
// The same kernel runs in three modes (the epilogue differs, the contraction
// does not, and it is deterministic, so every mode sees bit-identical scores):
//   MODE_RAW       writes the scaled scores, -inf where the key is masked
//                  (the scorer output as its own call);
//   MODE_GROUPMAX  splits each query row's valid keys into consecutive groups
//                  of g keys and writes the 16 high bits of the order key of
//                  every group's maximum score;
//   MODE_COLLECT   appends every valid key whose score reaches the row's
//                  threshold to the row's candidate list.
// The exact top-k of a row is then found from these (tile_select.cu).
//
// Block layout (192 threads): warp 0 issues TMA loads (the query tile once per
// unit, key tiles through a ring of shared-memory stages), warp 1 allocates
// TMEM and issues the MMAs (M=128 queries, N=128 keys, K=16 per instruction,
// bf16 operands K-major with the 128-byte swizzle, fp32 accumulators in one of
// two TMEM buffers), warps 2..5 are the epilogue: thread r of the warpgroup
// owns TMEM lane r, i.e. query row r of the tile, and reads its 128 scores of
// a key tile as four 32-column tcgen05.ld. Every wait on an mbarrier is
// bounded in time; a wait that runs out sets SSA_DEV_WAIT_LIMIT, stops every
// role of the block, lets copies and MMAs in flight finish and frees TMEM.
//
// Work is a list of units (head, 128-query tile) in head-major order, the
// query tiles of a head from the last (most keys under a causal mask) to the
// first; a persistent grid takes units round-robin.
#include "sm100.cuh"
#include "tile.h"

namespace ssa {

using namespace sm100;

namespace {

constexpr int kThreads = 192;
constexpr int kTBuf = 2;                      // TMEM accumulator buffers
constexpr uint32_t kTmemCols = kTBuf * kTileN;

template <int P>
struct TileCfg {
    static constexpr int KA = P / 64;                       // 128-byte K atoms per row
    static constexpr int STAGES = (P == 64) ? 4 : 2;        // key-tile ring depth
    static constexpr uint32_t QBYTES = KA * kTileM * 128;
    static constexpr uint32_t KBYTES = KA * kTileN * 128;
    static constexpr uint32_t BAR_OFF = QBYTES + STAGES * KBYTES;
    static constexpr uint32_t SMEM = BAR_OFF + 256 + 1024;  // + barriers + alignment slack
};

struct Unit {
    int bh, i0, rows, n_lo, n_hi, ntiles;
};

SSA_DEVINL Unit unit_at(const TileParams& p, int u) {
    Unit U;
    U.bh = u / p.units_per_head;
    const int qb = p.units_per_head - 1 - (u - U.bh * p.units_per_head);
    U.i0 = qb * kTileM;
    U.rows = min(kTileM, p.Tq - U.i0);
    U.n_lo = tile_valid_count(U.i0, p.Tq, p.Tk, p.causal);
    U.n_hi = tile_valid_count(U.i0 + U.rows - 1, p.Tq, p.Tk, p.causal);
    U.ntiles = (U.n_hi + kTileN - 1) / kTileN;
    return U;
}

SSA_DEVINL float max32(const float (&v)[32]) {
    float a[11];
#pragma unroll
    for (int t = 0; t < 10; ++t) a[t] = fmax3(v[3 * t], v[3 * t + 1], v[3 * t + 2]);
    a[10] = fmaxf(v[30], v[31]);
    const float b0 = fmax3(a[0], a[1], a[2]);
    const float b1 = fmax3(a[3], a[4], a[5]);
    const float b2 = fmax3(a[6], a[7], a[8]);
    const float b3 = fmaxf(a[9], a[10]);
    return fmaxf(fmax3(b0, b1, b2), b3);
}

}  // namespace

template <int P, int MODE>
__global__ void __launch_bounds__(kThreads, 2)
    tile_scores_kernel(const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ CUtensorMap kmap, const TileParams p) {
    using C = TileCfg<P>;
    constexpr int S = C::STAGES;
    constexpr uint32_t IDESC = idesc_bf16_f32(kTileM, kTileN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sq = smem;
    uint8_t* sk = smem + C::QBYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* q_full = bars;
    uint64_t* q_empty = bars + 1;
    uint64_t* k_full = bars + 2;
    uint64_t* k_empty = k_full + S;
    uint64_t* t_full = k_empty + S;
    uint64_t* t_empty = t_full + kTBuf;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(t_empty + kTBuf);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(k_full + s, 1);
            mbar_init(k_empty + s, 1);
        }
        for (int b = 0; b < kTBuf; ++b) {
            mbar_init(t_full + b, 1);
            mbar_init(t_empty + b, 128);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&kmap);
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t lim = p.wait_limit_ns;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t kc = 0, qc = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
                const Unit U = unit_at(p, u);
                if (U.ntiles == 0) continue;
                if (!mbar_wait_bounded(q_empty, (qc & 1) ^ 1, abort_flag, p.dev_status, lim)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(q_full, C::QBYTES);
#pragma unroll
                for (int a = 0; a < C::KA; ++a)
                    tma_load_2d(sq + a * 16384, &qmap, a * 64, U.bh * p.Tq + U.i0, q_full);
                ++qc;
                for (int t = 0; t < U.ntiles; ++t) {
                    const uint32_t s = kc % S;
                    if (!mbar_wait_bounded(k_empty + s, ((kc / S) & 1) ^ 1, abort_flag,
                                           p.dev_status, lim)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(k_full + s, C::KBYTES);
#pragma unroll
                    for (int a = 0; a < C::KA; ++a)
                        tma_load_2d(sk + s * C::KBYTES + a * 16384, &kmap, a * 64,
                                    U.bh * p.Tk + t * kTileN, k_full + s);
                    ++kc;
                }
            }
            // let every copy this thread started land before the block exits
            const uint32_t first = kc > (uint32_t)S ? kc - S : 0;
            for (uint32_t m = first; m < kc; ++m)
                mbar_wait_bounded(k_full + (m % S), (m / S) & 1, nullptr, p.dev_status, lim);
            if (qc > 0) mbar_wait_bounded(q_full, (qc - 1) & 1, nullptr, p.dev_status, lim);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t kc = 0, tc = 0, qc = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
                const Unit U = unit_at(p, u);
                if (U.ntiles == 0) continue;
                if (!mbar_wait_bounded(q_full, qc & 1, abort_flag, p.dev_status, lim)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sq_addr = smem_u32(sq);
                for (int t = 0; t < U.ntiles; ++t) {
                    const uint32_t s = kc % S, b = tc % kTBuf;
                    if (!mbar_wait_bounded(k_full + s, (kc / S) & 1, abort_flag, p.dev_status,
                                           lim) ||
                        !mbar_wait_bounded(t_empty + b, ((tc / kTBuf) & 1) ^ 1, abort_flag,
                                           p.dev_status, lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + b * kTileN;
                    const uint32_t sk_addr = smem_u32(sk + s * C::KBYTES);
#pragma unroll
                    for (int a = 0; a < C::KA; ++a) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = smem_desc_k_sw128(sq_addr + a * 16384 + kk * 32);
                            const uint64_t bd = smem_desc_k_sw128(sk_addr + a * 16384 + kk * 32);
                            mma_bf16(d_tmem, ad, bd, IDESC, (a | kk) != 0);
                        }
                    }
                    mma_commit(k_empty + s);
                    mma_commit(t_full + b);
                    ++kc;
                    ++tc;
                }
                if (!ok) break;
                mma_commit(q_empty);
                ++qc;
            }
            // MMAs in flight finish by themselves; wait for the last one
            if (tc > 0)
                mbar_wait_bounded(t_full + (tc - 1) % kTBuf, ((tc - 1) / kTBuf) & 1, nullptr,
                                  p.dev_status, lim);
        }
    } else {
        // ------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        uint32_t tc = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
            const Unit U = unit_at(p, u);
            const bool row_ok = r < U.rows;
            const int i = U.i0 + r;
            const int n_i = row_ok ? tile_valid_count(i, p.Tq, p.Tk, p.causal) : 0;
            const int64_t row = static_cast<int64_t>(U.bh) * p.Tq + i;
            // mode state
            int g = 0;
            bool emit = false;
            float gacc = -INFINITY;
            float tau_f = -INFINITY;
            int cnt = 0;
            if constexpr (MODE == MODE_GROUPMAX) {
                g = tile_group_size(U.n_lo, U.n_hi, p.k);
                emit = n_i > p.k;
            }
            if constexpr (MODE == MODE_COLLECT) {
                if (row_ok) {
                    const uint32_t t32 = p.tau[row];
                    tau_f = t32 == 0 ? -INFINITY : order_key_f32(t32);
                }
            }
            for (int t = 0; t < U.ntiles; ++t) {
                const uint32_t b = tc % kTBuf;
                // warp-uniform outcome: tcgen05.ld below needs the whole warp
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(t_full + b, (tc / kTBuf) & 1,
                                                              abort_flag, p.dev_status, lim));
                if (!ok) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < kTileN / 32; ++c) {
                    uint32_t raw[32];
                    tmem_ld32(t_lane + b * kTileN + c * 32, raw);
                    tmem_ld_wait();
                    const int j0 = t * kTileN + c * 32;
                    float v[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(raw[e]);
                    if constexpr (MODE == MODE_RAW) {
                        if (row_ok) {
                            float* out = p.S + row * static_cast<int64_t>(p.Tk);
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const int j = j0 + e;
                                if (j < p.Tk) out[j] = j < n_i ? v[e] * p.scale : -INFINITY;
                            }
                        }
                    } else if (j0 < n_i) {
                        if (j0 + 32 > n_i) {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (j0 + e >= n_i) v[e] = -INFINITY;
                        }
                        if constexpr (MODE == MODE_GROUPMAX) {
                            if (emit) {
                                uint16_t* gcol = p.gm + static_cast<int64_t>(u) * p.G_stride *
                                                            kTileM + r;
                                if (g >= 32) {
                                    gacc = fmaxf(gacc, max32(v));
                                    const int jend = j0 + 32;
                                    if ((jend & (g - 1)) == 0 || jend >= n_i) {
                                        gcol[static_cast<int64_t>(j0 / g) * kTileM] =
                                            static_cast<uint16_t>(f32_order_key(gacc * p.scale) >> 16);
                                        gacc = -INFINITY;
                                    }
                                } else {
                                    // in-place max tree: v[m*g] ends as the max of group m
                                    if (g >= 2) {
#pragma unroll
                                        for (int e = 0; e < 32; e += 2) v[e] = fmaxf(v[e], v[e + 1]);
                                    }
                                    if (g >= 4) {
#pragma unroll
                                        for (int e = 0; e < 32; e += 4) v[e] = fmaxf(v[e], v[e + 2]);
                                    }
                                    if (g >= 8) {
#pragma unroll
                                        for (int e = 0; e < 32; e += 8) v[e] = fmaxf(v[e], v[e + 4]);
                                    }
                                    if (g >= 16) {
#pragma unroll
                                        for (int e = 0; e < 32; e += 16) v[e] = fmaxf(v[e], v[e + 8]);
                                    }
#pragma unroll
                                    for (int e = 0; e < 32; ++e) {
                                        if ((e & (g - 1)) == 0 && j0 + e < n_i)
                                            gcol[static_cast<int64_t>((j0 + e) / g) * kTileM] =
                                                static_cast<uint16_t>(f32_order_key(v[e] * p.scale) >> 16);
                                    }
                                }
                            }
                        }
                        if constexpr (MODE == MODE_COLLECT) {
                            if (max32(v) * p.scale >= tau_f) {
                                uint64_t* crow = p.cand + row * static_cast<int64_t>(p.cap);
#pragma unroll
                                for (int e = 0; e < 32; ++e) {
                                    const float s = v[e] * p.scale;
                                    if (j0 + e < n_i && s >= tau_f) {
                                        if (cnt < p.cap)
                                            crow[cnt] = sel_key(f32_order_key(s),
                                                                static_cast<uint32_t>(j0 + e));
                                        ++cnt;
                                    }
                                }
                            }
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(t_empty + b);
                ++tc;
            }
            if (!ok) break;
            if constexpr (MODE == MODE_COLLECT) {
                if (row_ok) p.cnt[row] = cnt;
            }
            if constexpr (MODE == MODE_RAW) {
                // columns past the unit's last key tile are masked for every row
                if (row_ok) {
                    float* out = p.S + row * static_cast<int64_t>(p.Tk);
                    for (int j = U.ntiles * kTileN; j < p.Tk; ++j) out[j] = -INFINITY;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side

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

// 2-D map over rows of P bf16 elements: box = 64 elements x 128 rows, 128-byte
// swizzle (the shared-memory layout the MMA descriptors describe).
bool make_map(CUtensorMap* m, const void* base, int64_t nrows, int P) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(P), static_cast<cuuint64_t>(nrows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(P) * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int P, int MODE>
cudaError_t launch_mode(const CUtensorMap& qm, const CUtensorMap& km, const TileParams& p,
                        int grid, cudaStream_t stream) {
    using C = TileCfg<P>;
    auto kern = tile_scores_kernel<P, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, C::SMEM, stream>>>(qm, km, p);
    return cudaGetLastError();
}

}  // namespace

int tile_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

cudaError_t tile_scores_launch(const void* q_low, const void* k_low, int P, int mode,
                               TileParams p, cudaStream_t stream) {
    CUtensorMap qm, km;
    if (!make_map(&qm, q_low, static_cast<int64_t>(p.BH) * p.Tq, P) ||
        !make_map(&km, k_low, static_cast<int64_t>(p.BH) * p.Tk, P))
        return cudaErrorInvalidValue;
    p.units_per_head = (p.Tq + kTileM - 1) / kTileM;
    p.num_units = p.BH * p.units_per_head;
    if (p.num_units == 0) return cudaSuccess;
    if (p.wait_limit_ns == 0) p.wait_limit_ns = 1000000000ull;   // 1 s
    const int sms = tile_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = p.num_units < 2 * sms ? p.num_units : 2 * sms;
#define SSA_TILE_CASE(PP, MM) \
    if (P == PP && mode == MM) return launch_mode<PP, MM>(qm, km, p, grid, stream);
    SSA_TILE_CASE(64, MODE_RAW)
    SSA_TILE_CASE(64, MODE_GROUPMAX)
    SSA_TILE_CASE(64, MODE_COLLECT)
    SSA_TILE_CASE(128, MODE_RAW)
    SSA_TILE_CASE(128, MODE_GROUPMAX)
    SSA_TILE_CASE(128, MODE_COLLECT)
#undef SSA_TILE_CASE
    return cudaErrorInvalidValue;
}

}  // namespace ssa
