// Low-rank projection of the scorer on the tensor cores: out = x W^T, the
// bias-free linear maps q_low = q_proj(query), k_low = k_proj(key) from
// d_model to d_proj of the lightweight scorer (mhpq.cn/news/1098205, section
// 2.2). x is [rows, d_model] (rows = batch * heads * seq_len), W is
// [d_proj, d_model] (a linear layer's weight), out is [rows, d_proj]; bf16
// operands, fp32 accumulation, the result rounded once to bf16.
//
// One CTA per 128-row tile, two per SM. Warp 0 streams 64-column slices of
// the row tile and of W through a 4-stage TMA ring (128-byte swizzle); warp 1
// allocates TMEM and issues tcgen05.mma (M=128, N=d_proj, K=16) into one fp32
// accumulator; warps 2-5 (one row per thread) read it back, round to bf16 and
// store the row. The kernel reads x once (HBM-bound: 2*d_model bytes per row
// against 4*d_proj FLOP per byte pair); W is re-read by every CTA from L2.
// Every mbarrier wait is bounded in time.
#include "sm100.cuh"
#include "tmap.h"
#include "trace.h"

namespace ssa {

using namespace sm100;

namespace {

constexpr int kPM = 128;              // rows per CTA
constexpr int kPK = 64;               // d_model columns per stage (one 128-byte row)
constexpr int kPStages = 4;
constexpr int kPThreads = 192;
constexpr uint64_t kPDefaultWaitNs = 1000000000ull;

template <int P>
struct ProjCfg {
    static constexpr uint32_t ABYTES = kPM * kPK * 2;    // 16 KB
    static constexpr uint32_t BBYTES = P * kPK * 2;      // 8 or 16 KB
    static constexpr uint32_t STAGE = ABYTES + BBYTES;
    static constexpr uint32_t BAR_OFF = kPStages * STAGE;
    static constexpr uint32_t SMEM = BAR_OFF + 128 + 1024;
    static constexpr uint32_t TMEM_COLS = P < 32 ? 32 : P;
};

struct ProjParams {
    int64_t rows;
    int d_model;
    __nv_bfloat16* out;
    int32_t* dev_status;
    uint64_t wait_limit_ns;
};

}  // namespace

template <int P>
__global__ void __launch_bounds__(kPThreads, 2)
    lowrank_project_kernel(const __grid_constant__ CUtensorMap xmap,
                           const __grid_constant__ CUtensorMap wmap, const ProjParams p) {
    using C = ProjCfg<P>;
    constexpr uint32_t IDESC = idesc_bf16_f32(kPM, P);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* full = bars;                       // [kPStages]
    uint64_t* empty = bars + kPStages;           // [kPStages]
    uint64_t* acc_full = bars + 2 * kPStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kPM;
    const int nk = p.d_model / kPK;
    const uint64_t lim = p.wait_limit_ns ? p.wait_limit_ns : kPDefaultWaitNs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&xmap);
        prefetch_tensormap(&wmap);
    }
    if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA
        if (lane == 0) {
            int issued = 0;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % kPStages;
                if (!mbar_wait_bounded(empty + s, ((kb / kPStages) & 1) ^ 1, abort_flag, p.dev_status,
                                       lim))
                    break;
                uint8_t* st = smem + s * C::STAGE;
                mbar_arrive_expect_tx(full + s, C::STAGE);
                tma_load_2d(st, &xmap, kb * kPK, static_cast<int>(m0), full + s);
                tma_load_2d(st + C::ABYTES, &wmap, kb * kPK, 0, full + s);
                ++issued;
            }
            // the copies land before the block may exit
            const int first = issued > kPStages ? issued - kPStages : 0;
            for (int kb = first; kb < issued; ++kb)
                mbar_wait_bounded(full + kb % kPStages, (kb / kPStages) & 1, nullptr, p.dev_status, lim);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA
        if (lane == 0) {
            int done = 0;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % kPStages;
                if (!mbar_wait_bounded(full + s, (kb / kPStages) & 1, abort_flag, p.dev_status, lim))
                    break;
                tc_fence_after();
                const uint8_t* st = smem + s * C::STAGE;
                const uint64_t adesc = smem_desc_k_sw128(smem_u32(st));
                const uint64_t bdesc = smem_desc_k_sw128(smem_u32(st + C::ABYTES));
#pragma unroll
                for (int kk = 0; kk < kPK / 16; ++kk)
                    mma_bf16(tmem_base, adesc + ((kk * 32) >> 4), bdesc + ((kk * 32) >> 4), IDESC,
                             (kb | kk) != 0);
                mma_commit(empty + s);
                ++done;
            }
            // every MMA of this thread (also after a stop) is tracked by acc_full
            mma_commit(acc_full);
            mbar_wait_bounded(acc_full, 0, nullptr, p.dev_status, lim);
            if (done < nk && !*abort_flag) {
                *abort_flag = 1;
                report(p.dev_status, SSA_DEV_WAIT_LIMIT);
            }
        }
    } else {
        // ------------------------------------------------ rows out
        const int quarter = warp & 3;   // TMEM lane quarter of this warp
        const int r = quarter * 32 + lane;
        const int64_t row = m0 + r;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        const bool ok =
            __all_sync(0xffffffffu, mbar_wait_bounded(acc_full, 0, abort_flag, p.dev_status, lim));
        if (ok && !*abort_flag) {
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < P / 32; ++c) {
                uint32_t raw[32];
                tmem_ld32(t_lane + c * 32, raw);
                tmem_ld_wait();
                reg_fence(raw);
                if (row < p.rows) {
                    uint4* dst = reinterpret_cast<uint4*>(p.out + row * P + c * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t w[4];
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const int e = q * 8 + h * 2;
                            const __nv_bfloat162 b2 =
                                __floats2bfloat162_rn(__uint_as_float(raw[e]), __uint_as_float(raw[e + 1]));
                            w[h] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side

namespace {

template <int P>
cudaError_t launch_project(const CUtensorMap& xm, const CUtensorMap& wm, const ProjParams& p,
                           unsigned grid, cudaStream_t stream) {
    using C = ProjCfg<P>;
    auto kern = lowrank_project_kernel<P>;
    cudaError_t e = set_max_dyn_smem(reinterpret_cast<const void*>(kern), static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    TraceLaunch tr("lowrank_project", stream);
    kern<<<grid, kPThreads, C::SMEM, stream>>>(xm, wm, p);
    return cudaGetLastError();
}

}  // namespace

// x [rows, d_model], W [P, d_model], out [rows, P], all bf16 and 16-byte
// aligned; P in {64, 128}; d_model a positive multiple of 64 (the caller
// checks).
cudaError_t lowrank_project_launch(const void* x, const void* W, int64_t rows, int d_model, int P,
                                   void* out, int32_t* dev_status, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = (rows + kPM - 1) / kPM;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    CUtensorMap xm, wm;
    const uint64_t xdims[2] = {static_cast<uint64_t>(d_model), static_cast<uint64_t>(rows)};
    const uint64_t wdims[2] = {static_cast<uint64_t>(d_model), static_cast<uint64_t>(P)};
    const uint64_t strides[1] = {static_cast<uint64_t>(d_model) * 2};
    const uint32_t xbox[2] = {kPK, kPM};
    const uint32_t wbox[2] = {kPK, static_cast<uint32_t>(P)};
    if (!tmap_bf16_sw128(&xm, x, 2, xdims, strides, xbox) ||
        !tmap_bf16_sw128(&wm, W, 2, wdims, strides, wbox))
        return cudaErrorInvalidValue;
    ProjParams p;
    p.rows = rows;
    p.d_model = d_model;
    p.out = reinterpret_cast<__nv_bfloat16*>(out);
    p.dev_status = dev_status;
    p.wait_limit_ns = 0;
    if (P == 64) return launch_project<64>(xm, wm, p, static_cast<unsigned>(blocks), stream);
    if (P == 128) return launch_project<128>(xm, wm, p, static_cast<unsigned>(blocks), stream);
    return cudaErrorInvalidValue;
}

}  // namespace ssa
