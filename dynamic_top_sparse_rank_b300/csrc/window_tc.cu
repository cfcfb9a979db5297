// Sliding-window attention on the tensor cores: softmax(q.k^T * scale) v over
// the keys j with i - w_left <= j <= i + w_right (clipped to the sequence) of
// every query i (the local band of "注意力机制优化", section 2.2, and the band
// mask of the dense formulation; each row's softmax and weighted sum as in
// mhpq.cn/news/1098205, section 3.2), computed as dense tiles of the band.
//
// One CTA per (head, 128-query tile). The tile's band spans at most three
// 128-key tiles (the host sends wider bands, other head sizes and fp32 to the
// gather kernel), so everything fits on chip at once and the softmax needs no
// running rescale:
//   warp 0  TMA: the query tile, the band's key tiles and value tiles (3-D
//           maps [head][row][64], 128-byte swizzle; rows outside the sequence
//           read as zeros);
//   warp 1  allocates TMEM and issues the MMAs: S = Q K^T, one 128x128 fp32
//           accumulator per key tile (columns 0..383), then O = P V (M=128,
//           N=64, K=16 steps; V is read MN-major straight from its TMA
//           layout) into columns 384..447, one key tile of P at a time;
//   warps 2-5  one query row per thread: the band mask and the row maximum
//           (first pass over S), then per key tile p = exp2((s - max) *
//           scale * log2 e) in fp32, written to shared memory in the layout
//           the second MMA reads (K-major, 128-byte swizzle) as two bf16
//           parts, hi = bf16(p) and lo = bf16(p - hi), so that P V = hi V +
//           lo V keeps p to about 2^-17 (one bf16 P would cost 2^-9, too much
//           for rows with few keys); the row sum is taken in fp32; after the
//           last MMA, O divided by the sum and stored in bf16 or fp32.
// The weights of a key tile go through two 64 KB buffers in turn: the first
// reuses the query and key tiles' space (free once S is in TMEM).
// Every mbarrier wait is bounded; a wait that runs out reports
// SSA_DEV_WAIT_LIMIT, stops the other roles and TMEM is freed.
#include <float.h>

#include "sm100.cuh"
#include "tmap.h"
#include "trace.h"

namespace ssa {

using namespace sm100;

namespace {

constexpr int kWM = 128;                     // query rows per CTA
constexpr int kWN = 128;                     // keys per score tile
constexpr int kWMaxTiles = 3;                // score tiles next to the output in TMEM
constexpr int kWD = 64;                      // head size of this kernel
constexpr int kWThreads = 192;
constexpr uint32_t kTileBytes = kWN * kWD * 2;                 // 128 rows of 64 bf16
constexpr uint32_t kQOff = 0;
constexpr uint32_t kKOff = kQOff + kTileBytes;
constexpr uint32_t kVOff = kKOff + kWMaxTiles * kTileBytes;
// weight buffers: [hi | lo][2 blocks of 64 keys][128 rows][128 B] = 64 KB each
constexpr uint32_t kPPart = kWM * kWN * 2;                      // one bf16 part of a key tile
constexpr uint32_t kPBuf0 = kQOff;                              // over Q and K (64 KB)
constexpr uint32_t kPBuf1 = kVOff + kWMaxTiles * kTileBytes;
constexpr uint32_t kBarOff = kPBuf1 + 2 * kPPart;
constexpr uint32_t kWSmem = kBarOff + 128 + 1024;               // + alignment slack
constexpr uint32_t kWTmemCols = 512;
constexpr uint32_t kOCol = kWMaxTiles * kWN;                   // output accumulator
constexpr uint64_t kWDefaultWaitNs = 1000000000ull;

struct WindowParams {
    int BH, T, wl, wr;
    float scale_log2;
    void* O;
    int bf16_out;
    int32_t* dev_status;
    uint64_t wait_limit_ns;
};

// First and last key tile of query tile qt (clipped to the sequence).
__host__ __device__ inline void band_tiles(int qt, int T, int wl, int wr, int* kt0, int* kt1) {
    const int ntile = (T + kWN - 1) / kWN;
    const int lo = qt * kWM - wl;
    *kt0 = lo <= 0 ? 0 : lo / kWN;
    const long long hi = static_cast<long long>(qt) * kWM + kWM - 1 + wr;
    const long long t1 = hi / kWN;
    *kt1 = t1 > ntile - 1 ? ntile - 1 : static_cast<int>(t1);
}

}  // namespace

__global__ void __launch_bounds__(kWThreads, 1)
    window_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const WindowParams p) {
    constexpr uint32_t IDESC_S = idesc_bf16_f32(kWM, kWN);
    constexpr uint32_t IDESC_O = idesc_bf16_f32_bmn(kWM, kWD);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
    uint64_t* full_qk = bars;       // query and key tiles landed
    uint64_t* full_v = bars + 1;    // value tiles landed
    uint64_t* s_full = bars + 2;    // S in TMEM
    uint64_t* o_full = bars + 3;    // O in TMEM
    uint64_t* p_full = bars + 4;    // [2] weights of a key tile in buffer b (one arrive per softmax warp)
    uint64_t* p_empty = bars + 6;   // [2] the MMAs reading buffer b are done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntq = (p.T + kWM - 1) / kWM;
    const int bh = blockIdx.x / ntq, qt = blockIdx.x - (blockIdx.x / ntq) * ntq;
    const int i0 = qt * kWM;
    int kt0, kt1;
    band_tiles(qt, p.T, p.wl, p.wr, &kt0, &kt1);
    const int nkt = kt1 - kt0 + 1;   // 1 .. kWMaxTiles (the host checks)
    const uint64_t lim = p.wait_limit_ns ? p.wait_limit_ns : kWDefaultWaitNs;

    if (threadIdx.x == 0) {
        mbar_init(full_qk, 1);
        mbar_init(full_v, 1);
        mbar_init(s_full, 1);
        mbar_init(o_full, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(p_full + b, 4);
            mbar_init(p_empty + b, 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    if (warp == 1) tmem_alloc(tmem_slot, kWTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA
        if (lane == 0) {
            mbar_arrive_expect_tx(full_qk, kTileBytes * (1 + nkt));
            tma_load_3d(smem + kQOff, &qmap, 0, i0, bh, full_qk);
            for (int t = 0; t < nkt; ++t)
                tma_load_3d(smem + kKOff + t * kTileBytes, &kmap, 0, (kt0 + t) * kWN, bh, full_qk);
            mbar_arrive_expect_tx(full_v, kTileBytes * nkt);
            for (int t = 0; t < nkt; ++t)
                tma_load_3d(smem + kVOff + t * kTileBytes, &vmap, 0, (kt0 + t) * kWN, bh, full_v);
            // the copies land before the block may exit
            mbar_wait_bounded(full_qk, 0, nullptr, p.dev_status, lim);
            mbar_wait_bounded(full_v, 0, nullptr, p.dev_status, lim);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA
        if (lane == 0) {
            bool s_issued = false, o_issued = false;
            if (mbar_wait_bounded(full_qk, 0, abort_flag, p.dev_status, lim)) {
                tc_fence_after();
                const uint64_t adesc = smem_desc_k_sw128(smem_u32(smem + kQOff));
                for (int t = 0; t < nkt; ++t) {
                    const uint64_t bdesc = smem_desc_k_sw128(smem_u32(smem + kKOff + t * kTileBytes));
#pragma unroll
                    for (int kk = 0; kk < kWD / 16; ++kk)
                        mma_bf16(tmem_base + t * kWN, adesc + ((kk * 32) >> 4), bdesc + ((kk * 32) >> 4),
                                 IDESC_S, kk != 0);
                }
                mma_commit(s_full);
                s_issued = true;
                bool ok = mbar_wait_bounded(full_v, 0, abort_flag, p.dev_status, lim);
                for (int t = 0; ok && t < nkt; ++t) {
                    const int b = t & 1;
                    if (!mbar_wait_bounded(p_full + b, (t >> 1) & 1, abort_flag, p.dev_status, lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t buf = b ? kPBuf1 : kPBuf0;
#pragma unroll
                    for (int s8 = 0; s8 < kWN / 16; ++s8) {
                        const int k16 = s8 * 16;   // key offset within the tile
                        const uint64_t bdesc_v = smem_desc_mn_sw128(
                            smem_u32(smem + kVOff + t * kTileBytes + s8 * 16 * 128), 0);
#pragma unroll
                        for (int part = 0; part < 2; ++part) {   // hi, lo
                            const uint64_t adesc_p =
                                smem_desc_k_sw128(smem_u32(smem + buf + part * kPPart +
                                                           (k16 / 64) * (kWM * 128))) +
                                (((k16 % 64) * 2) >> 4);
                            mma_bf16(tmem_base + kOCol, adesc_p, bdesc_v, IDESC_O,
                                     (t | s8 | part) != 0);
                        }
                    }
                    mma_commit(p_empty + b);
                }
                // every MMA of this thread (also after a stop) is tracked by o_full
                mma_commit(o_full);
                o_issued = true;
            }
            // MMAs in flight finish before TMEM is freed
            if (s_issued) mbar_wait_bounded(s_full, 0, nullptr, p.dev_status, lim);
            if (o_issued) mbar_wait_bounded(o_full, 0, nullptr, p.dev_status, lim);
        }
    } else {
        // ------------------------------------------------ softmax and output
        const int quarter = warp & 3;   // TMEM lane quarter of this warp
        const int r = quarter * 32 + lane;
        const int i = i0 + r;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        const int jlo = i - p.wl > 0 ? i - p.wl : 0;
        const int jhi = i + p.wr < p.T - 1 ? i + p.wr : p.T - 1;
        const int kbase = kt0 * kWN;
        bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(s_full, 0, abort_flag, p.dev_status, lim));
        if (ok) {
            tc_fence_after();
            // pass 1: the row maximum over the band
            float m = -INFINITY;
            for (int t = 0; t < nkt; ++t) {
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t raw2[2][32];
                    tmem_ld32(t_lane + t * kWN + c2 * 64, raw2[0]);
                    tmem_ld32(t_lane + t * kWN + c2 * 64 + 32, raw2[1]);
                    tmem_ld_wait();
                    reg_fence(raw2[0]);
                    reg_fence(raw2[1]);
                    const int j0 = kbase + t * kWN + c2 * 64;
#pragma unroll
                    for (int e = 0; e < 64; ++e) {
                        const int j = j0 + e;
                        if (j >= jlo && j <= jhi) m = fmaxf(m, __uint_as_float(raw2[e >> 5][e & 31]));
                    }
                }
            }
            // pass 2, key tile by key tile: the weights as hi + lo bf16 parts
            // into buffer t % 2 (once the MMAs of tile t - 2 have read it),
            // the row sum in fp32
            float sum = 0.f;
            for (int t = 0; ok && t < nkt; ++t) {
                const int b = t & 1;
                if (t >= 2)
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(p_empty + b, ((t >> 1) - 1) & 1,
                                                                  abort_flag, p.dev_status, lim));
                if (!ok) break;
                uint8_t* prow = smem + (b ? kPBuf1 : kPBuf0) + r * 128;
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t raw2[2][32];
                    tmem_ld32(t_lane + t * kWN + c2 * 64, raw2[0]);
                    tmem_ld32(t_lane + t * kWN + c2 * 64 + 32, raw2[1]);
                    tmem_ld_wait();
                    reg_fence(raw2[0]);
                    reg_fence(raw2[1]);
                    const int j0 = kbase + t * kWN + c2 * 64;
                    uint8_t* pblk = prow + c2 * (kWM * 128);   // 64-key block of the tile
#pragma unroll
                    for (int g8 = 0; g8 < 8; ++g8) {
                        uint32_t whi[4], wlo[4];
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            float pv[2];
#pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                const int e = g8 * 8 + h * 2 + q;
                                const int j = j0 + e;
                                pv[q] = (j >= jlo && j <= jhi)
                                            ? exp2f((__uint_as_float(raw2[e >> 5][e & 31]) - m) * p.scale_log2)
                                            : 0.f;
                            }
                            sum += pv[0] + pv[1];
                            const __nv_bfloat162 hi = __floats2bfloat162_rn(pv[0], pv[1]);
                            const __nv_bfloat162 lo = __floats2bfloat162_rn(pv[0] - __low2float(hi),
                                                                            pv[1] - __high2float(hi));
                            whi[h] = *reinterpret_cast<const uint32_t*>(&hi);
                            wlo[h] = *reinterpret_cast<const uint32_t*>(&lo);
                        }
                        // 16-byte chunk g8 of the row, swizzled by the row within its 8-row atom
                        const int off = (g8 ^ (r & 7)) * 16;
                        *reinterpret_cast<uint4*>(pblk + off) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
                        *reinterpret_cast<uint4*>(pblk + kPPart + off) =
                            make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
                    }
                }
                fence_proxy_async_smem();   // the MMA reads the weights through the async proxy
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full + b);
            }
            if (ok)
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(o_full, 0, abort_flag, p.dev_status, lim));
            if (ok) {
                tc_fence_after();
                uint32_t o2[2][32];
                tmem_ld32(t_lane + kOCol, o2[0]);
                tmem_ld32(t_lane + kOCol + 32, o2[1]);
                tmem_ld_wait();
                reg_fence(o2[0]);
                reg_fence(o2[1]);
                if (i < p.T) {
                    const float inv = sum > 0.f ? 1.f / sum : 0.f;
                    const int64_t off = (static_cast<int64_t>(bh) * p.T + i) * kWD;
                    if (p.bf16_out) {
                        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.O) + off);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            uint32_t w[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                const int d = c * 8 + h * 2;
                                const __nv_bfloat162 b2 = __floats2bfloat162_rn(
                                    __uint_as_float(o2[d >> 5][d & 31]) * inv,
                                    __uint_as_float(o2[(d + 1) >> 5][(d + 1) & 31]) * inv);
                                w[h] = *reinterpret_cast<const uint32_t*>(&b2);
                            }
                            dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    } else {
                        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.O) + off);
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const int d = c * 4;
                            dst[c] = make_float4(__uint_as_float(o2[d >> 5][d & 31]) * inv,
                                                 __uint_as_float(o2[(d + 1) >> 5][(d + 1) & 31]) * inv,
                                                 __uint_as_float(o2[(d + 2) >> 5][(d + 2) & 31]) * inv,
                                                 __uint_as_float(o2[(d + 3) >> 5][(d + 3) & 31]) * inv);
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kWTmemCols);
    }
}

// ---------------------------------------------------------------- host side

namespace {

// [BH][T][64] bf16, box 64 x 128 rows x 1 head, 128-byte swizzle; rows outside
// [0, T) of a head read as zeros.
bool make_map_3d(CUtensorMap* m, const void* base, int BH, int T) {
    const uint64_t dims[3] = {static_cast<uint64_t>(kWD), static_cast<uint64_t>(T),
                              static_cast<uint64_t>(BH)};
    const uint64_t strides[2] = {static_cast<uint64_t>(kWD) * 2,
                                 static_cast<uint64_t>(kWD) * 2 * static_cast<uint64_t>(T)};
    const uint32_t box[3] = {static_cast<uint32_t>(kWD), static_cast<uint32_t>(kWN), 1};
    return tmap_bf16_sw128(m, base, 3, dims, strides, box);
}

}  // namespace

// True when the tensor-core kernel covers the call: bf16 inputs, head size 64,
// and the band of every 128-query tile within three 128-key tiles.
bool window_tc_supported(bool bf16_in, int D, int T, int wl, int wr) {
    if (!bf16_in || D != kWD || T <= 0) return false;
    const int ntq = (T + kWM - 1) / kWM;
    for (int qt = 0; qt < ntq; ++qt) {
        int kt0, kt1;
        band_tiles(qt, T, wl, wr, &kt0, &kt1);
        if (kt1 - kt0 + 1 > kWMaxTiles) return false;
    }
    return true;
}

cudaError_t window_tc_launch(const void* Q, const void* K, const void* V, void* O, bool bf16_out,
                             int BH, int T, int wl, int wr, float scale, int32_t* dev_status,
                             cudaStream_t stream) {
    CUtensorMap qm, km, vm;
    if (!make_map_3d(&qm, Q, BH, T) || !make_map_3d(&km, K, BH, T) || !make_map_3d(&vm, V, BH, T))
        return cudaErrorInvalidValue;
    WindowParams p;
    p.BH = BH;
    p.T = T;
    p.wl = wl;
    p.wr = wr;
    p.scale_log2 = scale * kLog2e;
    p.O = O;
    p.bf16_out = bf16_out ? 1 : 0;
    p.dev_status = dev_status;
    p.wait_limit_ns = 0;
    const int64_t blocks = static_cast<int64_t>(BH) * ((T + kWM - 1) / kWM);
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaError_t e = set_max_dyn_smem(reinterpret_cast<const void*>(window_tc_kernel),
                                     static_cast<int>(kWSmem));
    if (e != cudaSuccess) return e;
    TraceLaunch tr("window_tc", stream);
    window_tc_kernel<<<static_cast<unsigned>(blocks), kWThreads, kWSmem, stream>>>(qm, km, vm, p);
    return cudaGetLastError();
}

}  // namespace ssa
