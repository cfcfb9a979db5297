// Sliding-window attention on the tensor cores: softmax(q.k^T * scale) v over
// the keys j with i - w_left <= j <= i + w_right (clipped to the sequence) of
// every query i (the local band of "注意力机制优化", section 2.2, and the band
// mask of the dense formulation; each row's softmax and weighted sum as in
// mhpq.cn/news/1098205, section 3.2), computed as dense tiles of the band.
//
// Work item: one (head, 128-query tile). Its band spans at most three 128-key
// tiles (the host sends wider bands and fp32 to the gather kernel). Both
// kernels are persistent, take items round-robin, keep the weights in TMEM
// (the A operand of tcgen05.mma may sit in TMEM) and run one pass over the
// key tiles with a running shift per row (the online softmax):
// p = 2^((s - M) * scale * log2 e) in fp32, written over the tile's scores
// as two bf16 parts, hi = p truncated to bf16 and lo = bf16(p - hi), so that
// P V = hi V + lo V keeps p to about 2^-16 (one bf16 P would cost 2^-9, too
// much for rows with few keys); the row sum in fp32; O divided by it at the
// end and stored in bf16 or fp32.
//
// window_tc_kernel (head size 128): one CTA per SM, 576 threads.
//   warp 0  TMA: per item the query tile, the band's key tiles and value
//           tiles (3-D maps [head][row][64-column slice], 128-byte swizzle;
//           rows outside the sequence read as zeros) into one 224 KB stage;
//   warp 1  allocates TMEM and issues the MMAs: S = Q K^T, one 128x128 fp32
//           accumulator per key tile (columns 0..383; two tiles per N=256
//           MMA), then O = P V (M=128, N=128, K=16 steps) into columns
//           384..511 with V MN-major straight from its TMA layout;
//   warps 2-17  one query row per thread, four warps per row splitting its
//           key chunks and output columns (softmax_rows); each key tile goes
//           to the MMA warp once written, so its P V runs under the next
//           tile's softmax.
// window_tc64_kernel (head size 64): two CTAs per SM, each on 256 TMEM
// columns, in 64-key steps through a ring of three score slots (see the
// notes above it).
// Every mbarrier wait is bounded; a wait that runs out reports
// SSA_DEV_WAIT_LIMIT, stops the other roles and TMEM is freed.
#include <float.h>

#include "sm100.cuh"
#include "tile.h"
#include "tmap.h"
#include "trace.h"

namespace ssa {

using namespace sm100;

namespace {

constexpr int kWM = 128;                     // query rows per item
constexpr int kWN = 128;                     // keys per score tile
constexpr int kWMaxTiles = 3;                // score tiles next to the output in TMEM
constexpr int kNW = 4;                       // softmax warps per TMEM lane quarter
constexpr int kCPW = 4 / kNW;                // 32-key chunks of a key tile per softmax warp
constexpr int kWThreads = 64 + 128 * kNW;    // TMA warp, MMA warp, softmax warps
constexpr uint32_t kSliceBytes = 128 * 128;  // 128 rows x 64 bf16 (one 128-byte swizzle slice)
constexpr uint32_t kWTmemCols = 512;
constexpr uint32_t kOCol = kWMaxTiles * kWN; // output accumulator
constexpr uint64_t kWDefaultWaitNs = 1000000000ull;

// Shared-memory layout of head size D: per stage the query tile (D/64 slices
// of 16 KB), then the keys and then the values of the three key tiles, each
// slice-major ([slice][384 rows][128 B]: the rows of consecutive key tiles are
// contiguous, so one N=256 MMA spans two key tiles and one MN-major operand
// of N=128 spans both value slices); stages, then the barriers.
template <int D>
struct WinCfg {
    static constexpr int KA = D / 64;                          // 64-column slices
    static constexpr int STAGES = 1;
    static constexpr uint32_t TILE = KA * kSliceBytes;         // one 128-row tile
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t SLICE3 = kWMaxTiles * kSliceBytes;   // one slice of the three tiles
    static constexpr uint32_t K_OFF = TILE;
    static constexpr uint32_t V_OFF = K_OFF + kWMaxTiles * TILE;
    static constexpr uint32_t STAGE = V_OFF + kWMaxTiles * TILE;
    static constexpr uint32_t BAR_OFF = STAGES * STAGE;
    static constexpr uint32_t XCH_OFF = BAR_OFF + 256;        // [3 slots][128 rows] 32-bit words
    static constexpr uint32_t SMEM = XCH_OFF + 3 * 128 * 4 + 1024;   // + alignment slack
    static_assert(kOCol + D <= kWTmemCols, "TMEM columns");
    static_assert(SMEM <= 232448, "shared memory per block");
};

struct WindowParams {
    int BH, T, wl, wr;
    int items;                   // BH * query tiles
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

struct WinItem {
    int bh, i0, kt0, nkt;
};

__device__ inline WinItem win_item(const WindowParams& p, int item) {
    const int ntq = (p.T + kWM - 1) / kWM;
    WinItem w;
    w.bh = item / ntq;
    const int qt = item - w.bh * ntq;
    w.i0 = qt * kWM;
    int kt1;
    band_tiles(qt, p.T, p.wl, p.wr, &w.kt0, &kt1);
    w.nkt = kt1 - w.kt0 + 1;   // 1 .. kWMaxTiles (the host checks)
    return w;
}

// 2^x on the special-function unit (ex2.approx, flush-to-zero: weights below
// 2^-126 of the row maximum's are zero; -inf gives 0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace

// Turns 64 keys x 64 columns of a value tile, as TMA wrote it (row = key,
// 128 bytes of 64 bf16 columns, 128-byte swizzle: 16-byte chunk c of row r at
// r * 128 + (c ^ (r & 7)) * 16), into the K-major operand of the same 8 KB
// (row = column d, its 64 keys in 128 bytes, the same swizzle), in place.
// In 8x8 blocks: block (keys 8kb.., columns 8db..) transposed is block
// (columns 8db.., keys 8kb..) of the result, which sits exactly where block
// (db, kb) of the source was; so a block and its mirror are read together
// (ldmatrix .trans) and written crosswise (stmatrix), four pairs at a time
// (the eight diagonal blocks in two batches). The P V MMAs read V^T K-major at
// 73.5 cycles per M=128, K=16 instruction against 125 for V MN-major
// (measured at N=64 and N=128).
__device__ __forceinline__ void vt_transpose_half(uint32_t base, int lane) {
    const int m = lane >> 3, i = lane & 7;   // the lane's matrix of an x4 group and its row
    auto src = [&](int kb, int db) { return base + (8 * kb + i) * 128 + ((db ^ i) << 4); };
    auto ld4 = [&](uint32_t addr, uint32_t (&r)[4]) {
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(addr)
                     : "memory");
    };
    auto st4 = [&](uint32_t addr, const uint32_t (&r)[4]) {
        asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                     "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                     : "memory");
    };
    // the 28 blocks above the diagonal, four per batch (pair index q: the
    // q-th (kb, db) with kb < db in row-major order; row kb starts at pair
    // 7 kb - kb (kb - 1) / 2), then the eight diagonal blocks; two rounds
    // (batches 0-3, then 4-6 and the diagonal), each reading every block of
    // its batches before writing any, so the loads' latencies overlap
    auto pair_block = [](int q, int& kb, int& db) {
        kb = (q >= 7) + (q >= 13) + (q >= 18) + (q >= 22) + (q >= 25) + (q >= 27);
        db = kb + 1 + q - (7 * kb - kb * (kb - 1) / 2);
    };
    {
        uint32_t a[4][4], b[4][4];
#pragma unroll
        for (int bt = 0; bt < 4; ++bt) {
            int kb, db;
            pair_block(4 * bt + m, kb, db);
            ld4(src(kb, db), a[bt]);   // lane group m: block (kb, db) of its pair
            ld4(src(db, kb), b[bt]);   // and its mirror
        }
        __syncwarp();
#pragma unroll
        for (int bt = 0; bt < 4; ++bt) {
            int kb, db;
            pair_block(4 * bt + m, kb, db);
            st4(src(db, kb), a[bt]);   // (kb, db) transposed goes where (db, kb) was
            st4(src(kb, db), b[bt]);
        }
    }
    {
        uint32_t a[3][4], b[3][4], d[2][4];
#pragma unroll
        for (int bt = 0; bt < 3; ++bt) {
            int kb, db;
            pair_block(4 * (bt + 4) + m, kb, db);
            ld4(src(kb, db), a[bt]);
            ld4(src(db, kb), b[bt]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) ld4(src(4 * h + m, 4 * h + m), d[h]);
        __syncwarp();
#pragma unroll
        for (int bt = 0; bt < 3; ++bt) {
            int kb, db;
            pair_block(4 * (bt + 4) + m, kb, db);
            st4(src(db, kb), a[bt]);
            st4(src(kb, db), b[bt]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) st4(src(4 * h + m, 4 * h + m), d[h]);
    }
    __syncwarp();
}

// The softmax warps of window_tc_kernel: kNW per TMEM lane quarter (warp w
// reads lanes 32 (w % 4) .. 32 (w % 4) + 31, one query row per thread); warp
// g of a quarter (g = (w - 2) / 4) takes kCPW 32-key chunks of every key tile
// (chunks kCPW g ..) and D / kNW output columns.
//
// One pass, key tile by key tile, with a running shift M per row (the
// online softmax): each warp takes the maximum of its chunks (a chunk inside
// every row's band of the warp from tcgen05.ld.red, a partial one masked,
// one outside every band skipped), the quarter's warps combine them through
// shared memory (atomicMax on order keys) and meet at a bounded per-quarter
// barrier before any overwrites a score, so all hold the same tile maximum
// and take the same decisions. M moves only when the tile maximum exceeds it
// by more than 2^8 in weight: then the MMAs of the earlier tiles are waited
// for and the row's O (this warp's columns) and partial sum are scaled down,
// so weights stay below 2^8 and are exact at the maximum (the first tile sets
// M to its maximum; w = 0 gives weight 1 and O = V exactly). The weights are
// written over the warp's own S columns (a chunk's 16 hi words, two keys per
// word with the lower key in the low half, in its first 16 columns, its 16
// lo words in the next 16) and each key tile is handed to the MMA warp once
// every warp has written it. At the end the partial row sums meet the same
// way (atomicAdd), and each warp writes its output columns.
//
// Shared slots: three rotating 128-row words per quarter step (step u uses
// slot u mod 3); after the barrier of step u, warp 0 of the quarter clears
// the slot of step u - 1, which all have read before arriving, and which is
// next used at step u + 2, after the others have passed step u + 1's barrier.
template <int D>
__device__ __forceinline__ void softmax_rows(const WindowParams& p, uint32_t tmem_base, int warp,
                                             int lane, uint64_t* s_full, uint64_t* o_full,
                                             uint64_t* p_full, uint64_t* pv_done, uint64_t* pair_bar,
                                             uint32_t* slots, volatile int* abort_flag,
                                             uint64_t lim) {
    const int quarter = warp & 3;   // TMEM lane quarter of this warp
    const int g = (warp - 2) >> 2;  // which part of the chunks and of the output
    const int r = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    constexpr float kRescaleLog2 = 8.f;   // weights stay below 2^8
    uint32_t u = 0;                        // pair steps taken
    uint32_t pvpar = 0;                    // bit t: phase parity of pv_done[t]
    // one step of the pair: combine (through slot u % 3, already updated by
    // the caller), meet, clear the previous step's slot; false on a stop
    auto pair_meet = [&]() -> bool {
        tc_fence_before();
        mbar_arrive(pair_bar + quarter);
        const bool ok =
            __all_sync(0xffffffffu, mbar_wait_bounded(pair_bar + quarter, u & 1, abort_flag, p.dev_status, lim));
        tc_fence_after();
        return ok;
    };
    auto step_done = [&]() {
        if (g == 0) slots[((u + 2) % 3) * 128 + r] = 0u;
        ++u;
    };
    int n = 0;
    for (int item = blockIdx.x; item < p.items; item += gridDim.x, ++n) {
        const WinItem w = win_item(p, item);
        const int i = w.i0 + r;
        const int jlo = i - p.wl > 0 ? i - p.wl : 0;
        const int jhi = i + p.wr < p.T - 1 ? i + p.wr : p.T - 1;
        // a 32-key chunk of the item, for the warp's 32 rows together: outside
        // every row's band, inside every row's band, or partial
        const int iw = w.i0 + quarter * 32;
        const int wlo = iw - p.wl > 0 ? iw - p.wl : 0;
        const int whi = iw + 31 + p.wr < p.T - 1 ? iw + 31 + p.wr : p.T - 1;
        const int flo = iw + 31 - p.wl > 0 ? iw + 31 - p.wl : 0;
        const int fhi = iw + p.wr < p.T - 1 ? iw + p.wr : p.T - 1;
        const int kbase = w.kt0 * kWN;
        auto chunk_class = [&](int ch) {   // 0 outside, 1 inside, 2 partial
            const int j0 = kbase + 32 * ch;
            if (j0 + 31 < wlo || j0 > whi) return 0;
            return (j0 >= flo && j0 + 31 <= fhi) ? 1 : 2;
        };
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(s_full, n & 1, abort_flag, p.dev_status, lim)))
            return;
        tc_fence_after();
        float M = -INFINITY;   // the row's shift
        float l = 0.f;         // this warp's partial row sum
        for (int t = 0; t < w.nkt; ++t) {
            // this warp's two chunks of the tile and their maximum
            uint32_t v[kCPW][32];
            float mx[kCPW][2];
            int cls[kCPW];
#pragma unroll
            for (int c = 0; c < kCPW; ++c) {
                const int ch = 4 * t + kCPW * g + c;
                cls[c] = chunk_class(ch);
                const uint32_t col = t_lane + 32 * ch;
                if (cls[c] == 1) {
                    mx[c][0] = tmem_ldred_max16(col, *reinterpret_cast<uint32_t(*)[16]>(&v[c][0]));
                    mx[c][1] = tmem_ldred_max16(col + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[c][16]));
                } else if (cls[c] == 2) {
                    tmem_ld32(col, v[c]);
                }
            }
            tmem_ld_wait();
            float m = -INFINITY;
#pragma unroll
            for (int c = 0; c < kCPW; ++c) {
                if (cls[c] == 0) continue;
                reg_fence(v[c]);
                if (cls[c] == 1) {
                    reg_fence_f(mx[c][0]);
                    reg_fence_f(mx[c][1]);
                    m = fmax3(m, mx[c][0], mx[c][1]);
                } else {
                    const int j0 = kbase + 32 * (4 * t + kCPW * g + c);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (j0 + e >= jlo && j0 + e <= jhi) m = fmaxf(m, __uint_as_float(v[c][e]));
                }
            }
            // the tile maximum of the row: both halves
            uint32_t* slot = slots + (u % 3) * 128;
            if (m > -INFINITY) atomicMax(slot + r, f32_order_key(m));
            if (!pair_meet()) return;
            const uint32_t mk = slot[r];
            step_done();
            const float mt = mk == 0u ? -INFINITY : order_key_f32(mk);
            // the shift: set by the first tile with a key; moved when a
            // weight would exceed 2^8
            const bool move = mt > -INFINITY && (M == -INFINITY || (mt - M) * p.scale_log2 > kRescaleLog2);
            if (__any_sync(0xffffffffu, move && M > -INFINITY)) {
                // O holds earlier tiles' sums at the old shift: wait for their
                // MMAs, then scale this warp's O columns of the moved rows
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(pv_done + (t - 1), (pvpar >> (t - 1)) & 1,
                                                              abort_flag, p.dev_status, lim)))
                    return;
                tc_fence_after();
                const float f = move && M > -INFINITY ? ex2_approx((M - mt) * p.scale_log2) : 1.f;
#pragma unroll
                for (int c16 = 0; c16 < D / kNW / 16; ++c16) {
                    const uint32_t ocol = t_lane + kOCol + (D / kNW) * g + 16 * c16;
                    uint32_t o[16];
                    tmem_ldred_max16(ocol, o);
                    tmem_ld_wait();
                    reg_fence(o);
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                    tmem_st16(ocol, o);
                }
                tmem_st_wait();
                l *= f;
            }
            if (move) M = mt;
            // the weights of the two chunks
#pragma unroll
            for (int c = 0; c < kCPW; ++c) {
                const int ch = 4 * t + kCPW * g + c;
                uint32_t whi[16], wlo[16];
                if (cls[c]) {
                    const int j0 = kbase + 32 * ch;
                    const bool mask = cls[c] == 2;
                    float s4[2] = {0.f, 0.f};
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        float pv[2];
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            const int j = j0 + 2 * q + b;
                            // (s - M) first: exactly 0 at the maximum, whose weight is 1
                            const float x = (__uint_as_float(v[c][2 * q + b]) - M) * p.scale_log2;
                            pv[b] = ex2_approx(!mask || (j >= jlo && j <= jhi) ? x : -INFINITY);
                        }
                        s4[q & 1] += pv[0] + pv[1];
                        const uint32_t b0 = __float_as_uint(pv[0]), b1 = __float_as_uint(pv[1]);
                        whi[q] = __byte_perm(b0, b1, 0x7632);   // the high halves: bf16 truncation
                        const __nv_bfloat162 lo = __floats2bfloat162_rn(
                            pv[0] - __uint_as_float(b0 & 0xFFFF0000u), pv[1] - __uint_as_float(b1 & 0xFFFF0000u));
                        wlo[q] = *reinterpret_cast<const uint32_t*>(&lo);
                    }
                    l += s4[0] + s4[1];
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) whi[q] = wlo[q] = 0u;
                }
                tmem_st16(t_lane + 32 * ch, whi);
                tmem_st16(t_lane + 32 * ch + 16, wlo);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full + t);
        }
        for (int t = 0; t < w.nkt; ++t) pvpar ^= 1u << t;   // one pv_done phase per tile of the item
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(o_full, n & 1, abort_flag, p.dev_status, lim)))
            return;
        tc_fence_after();
        // the row sum: both halves
        uint32_t* slot = slots + (u % 3) * 128;
        atomicAdd(reinterpret_cast<float*>(slot) + r, l);
        if (!pair_meet()) return;
        const float sum = __uint_as_float(slot[r]);
        step_done();
        const float inv = sum > 0.f ? 1.f / sum : 0.f;
        const int64_t off = (static_cast<int64_t>(w.bh) * p.T + i) * D;
#pragma unroll
        for (int c16 = 0; c16 < D / kNW / 16; ++c16) {
            const int col = (D / kNW) * g + 16 * c16;   // this warp's 16-column slices of O
            uint32_t o[16];
            tmem_ldred_max16(t_lane + kOCol + col, o);
            tmem_ld_wait();
            reg_fence(o);
            if (i >= p.T) continue;
            if (p.bf16_out) {
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.O) + off + col);
#pragma unroll
                for (int c8 = 0; c8 < 2; ++c8) {
                    uint32_t wv[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int d = c8 * 8 + q * 2;
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(o[d]) * inv,
                                                                        __uint_as_float(o[d + 1]) * inv);
                        wv[q] = *reinterpret_cast<const uint32_t*>(&b2);
                    }
                    dst[c8] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            } else {
                float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.O) + off + col);
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    dst[c4] = make_float4(__uint_as_float(o[4 * c4]) * inv, __uint_as_float(o[4 * c4 + 1]) * inv,
                                          __uint_as_float(o[4 * c4 + 2]) * inv,
                                          __uint_as_float(o[4 * c4 + 3]) * inv);
            }
        }
        tc_fence_before();   // the O columns are read: the next item's MMAs may write them
    }
}

template <int D>
__global__ void __launch_bounds__(kWThreads, 1)
    window_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const WindowParams p) {
    using C = WinCfg<D>;
    constexpr int KA = C::KA;
    constexpr uint32_t IDESC_S = idesc_bf16_f32(kWM, kWN);
    constexpr uint32_t IDESC_S2 = idesc_bf16_f32(kWM, 2 * kWN);
    constexpr uint32_t IDESC_O = idesc_bf16_f32_bmn(kWM, D);   // V MN-major
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* full_qk = bars;        // [stage] query and key tiles landed
    uint64_t* full_v = bars + 2;     // [stage] value tiles landed
    uint64_t* empty = bars + 4;      // [stage] the MMAs reading the stage are done
    uint64_t* s_full = bars + 6;     // S of the item in TMEM
    uint64_t* o_full = bars + 7;     // every MMA of the item done: O in TMEM
    uint64_t* p_full = bars + 8;     // [3] weights of key tile t in TMEM (one arrive per softmax warp)
    uint64_t* pair_bar = bars + 11;  // [4] the two softmax warps of a lane quarter meet
    uint64_t* pv_done = bars + 15;   // [3] the MMAs up to key tile t's P V are done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
    uint32_t* slots = reinterpret_cast<uint32_t*>(smem + C::XCH_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t lim = p.wait_limit_ns ? p.wait_limit_ns : kWDefaultWaitNs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(full_qk + s, 1);
            mbar_init(full_v + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(s_full, 1);
        mbar_init(o_full, 1);
        for (int t = 0; t < kWMaxTiles; ++t) {
            mbar_init(p_full + t, 4 * kNW);
            mbar_init(pv_done + t, 1);
        }
        for (int q = 0; q < 4; ++q) mbar_init(pair_bar + q, 32 * kNW);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    for (int x = threadIdx.x; x < 3 * 128; x += kWThreads) slots[x] = 0u;
    if (warp == 1) tmem_alloc(tmem_slot, kWTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA (lane 0)
        int n = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < p.items; item += gridDim.x, ++n) {
            const int s = n % C::STAGES;
            const uint32_t use = static_cast<uint32_t>(n / C::STAGES);
            const WinItem w = win_item(p, item);
            uint8_t* st = smem + s * C::STAGE;
            if (lane == 0) {
                if (use > 0) ok = mbar_wait_bounded(empty + s, (use - 1) & 1, abort_flag, p.dev_status, lim);
                if (ok) {
                    mbar_arrive_expect_tx(full_qk + s, C::TILE * (1 + w.nkt));
#pragma unroll
                    for (int a = 0; a < KA; ++a)
                        tma_load_3d(st + C::Q_OFF + a * kSliceBytes, &qmap, 64 * a, w.i0, w.bh, full_qk + s);
                    for (int t = 0; t < w.nkt; ++t)
#pragma unroll
                        for (int a = 0; a < KA; ++a)
                            tma_load_3d(st + C::K_OFF + a * C::SLICE3 + t * kSliceBytes, &kmap, 64 * a,
                                        (w.kt0 + t) * kWN, w.bh, full_qk + s);
                    mbar_arrive_expect_tx(full_v + s, C::TILE * w.nkt);
                    for (int t = 0; t < w.nkt; ++t)
#pragma unroll
                        for (int a = 0; a < KA; ++a)
                            tma_load_3d(st + C::V_OFF + a * C::SLICE3 + t * kSliceBytes, &vmap, 64 * a,
                                        (w.kt0 + t) * kWN, w.bh, full_v + s);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                ok = false;
                break;
            }
        }
        // the copies land before the block may exit: the last use of each stage
        if (lane == 0)
            for (int s = 0; s < C::STAGES && s < n; ++s) {
                const uint32_t last = static_cast<uint32_t>((n - 1 - s) / C::STAGES);
                mbar_wait_bounded(full_qk + s, last & 1, nullptr, p.dev_status, lim);
                mbar_wait_bounded(full_v + s, last & 1, nullptr, p.dev_status, lim);
            }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA
        if (lane == 0) {
            int n = 0, committed = 0;
            uint32_t pt = 0;   // bit t: phase parity of p_full[t]
            bool ok = true;
            for (int item = blockIdx.x; ok && item < p.items; item += gridDim.x, ++n) {
                const int s = n % C::STAGES;
                const uint32_t use = static_cast<uint32_t>(n / C::STAGES);
                const WinItem w = win_item(p, item);
                // this item's query and key tiles landed. Its S MMAs overwrite
                // the previous item's weights; tcgen05.mma instructions of one
                // thread execute in issue order, so they run after the previous
                // item's P V MMAs that read those weights, with no wait here.
                ok = mbar_wait_bounded(full_qk + s, use & 1, abort_flag, p.dev_status, lim);
                if (!ok) break;
                tc_fence_after();
                const uint8_t* st = smem + s * C::STAGE;
                // S by key-tile pairs: N=256 over tiles 0-1, N=128 for a third
                for (int t = 0; t < w.nkt; t += 2) {
                    const uint32_t idesc = t + 1 < w.nkt ? IDESC_S2 : IDESC_S;
#pragma unroll
                    for (int a = 0; a < KA; ++a) {
                        const uint64_t ad = smem_desc_k_sw128(smem_u32(st + C::Q_OFF + a * kSliceBytes));
                        const uint64_t bd =
                            smem_desc_k_sw128(smem_u32(st + C::K_OFF + a * C::SLICE3 + t * kSliceBytes));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16(tmem_base + t * kWN, ad + ((kk * 32) >> 4), bd + ((kk * 32) >> 4),
                                     idesc, (a | kk) != 0);
                    }
                }
                mma_commit(s_full);
                ok = mbar_wait_bounded(full_v + s, use & 1, abort_flag, p.dev_status, lim);
                for (int t = 0; ok && t < w.nkt; ++t) {
                    if (!mbar_wait_bounded(p_full + t, (pt >> t) & 1, abort_flag, p.dev_status, lim)) {
                        ok = false;
                        break;
                    }
                    pt ^= 1u << t;
                    tc_fence_after();
#pragma unroll
                    for (int s8 = 0; s8 < kWN / 16; ++s8) {
                        // keys 16 s8 .. 16 s8 + 15 of the tile: their hi and lo
                        // weights (see the softmax warps' layout)
                        const uint32_t hi = t * kWN + 32 * (s8 / 2) + 8 * (s8 % 2);
                        // all D columns of V in one MN-major operand, its
                        // 64-column slices SLICE3 bytes apart
                        const uint64_t bd = smem_desc_mn_sw128(
                            smem_u32(st + C::V_OFF + t * kSliceBytes + s8 * 16 * 128), C::SLICE3);
                        mma_bf16_ta(tmem_base + kOCol, tmem_base + hi, bd, IDESC_O, (t | s8) != 0);
                        mma_bf16_ta(tmem_base + kOCol, tmem_base + hi + 16, bd, IDESC_O, 1);
                    }
                    mma_commit(pv_done + t);   // for a softmax warp that rescales O
                }
                // every MMA of the item (also after a stop) is tracked by o_full
                mma_commit(o_full);
                mma_commit(empty + s);
                ++committed;
            }
            // MMAs in flight finish before TMEM is freed
            if (committed > 0)
                mbar_wait_bounded(o_full, (committed - 1) & 1, nullptr, p.dev_status, lim);
        }
    } else {
        softmax_rows<D>(p, tmem_base, warp, lane, s_full, o_full, p_full, pv_done, pair_bar, slots,
                        abort_flag, lim);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kWTmemCols);
    }
}

// ---------------------------------------------------------------- D 64: two CTAs per SM
//
// For head size 64 the item's chain of dependent steps (scores, softmax, P V
// per key tile), not any one unit, sets the pace of window_tc_kernel, and one
// item's scores fill 384 of the 512 TMEM columns. window_tc64_kernel runs two
// CTAs per SM instead, each on 256 TMEM columns and about 100 KB of shared
// memory, so that one CTA's softmax runs while the other's MMAs and loads do,
// and within a CTA the softmax of one 64-key step runs while the tensor pipe
// works on the previous one:
//   - 64-key steps h (key tile h / 2, its half h % 2): S(h) = Q K(h)^T (N=64)
//     into score slot h % 3 (columns 0..63, 64..127, 192..255), the weights
//     over it, P(h) V(h) into O (columns 128..191); S(h + 2) is issued behind
//     P(h) V(h) and takes the slot of step h - 1, whose P V ran before it
//     (tcgen05.mma instructions of one thread run in issue order);
//   - the TMA warp streams the query tile and key and value tiles through
//     a two-slot key ring and a three-slot value ring, two tiles ahead of
//     the one it turns K-major (a tile's copy latency is then off the chain);
//   - the softmax warps (eight, two per lane quarter, each one 32-key chunk
//     of every step) take the running-shift softmax step by step; a rescale
//     of O first waits for the previous step's P V (the one before it had
//     finished ahead of this step's scores).
namespace w64 {
constexpr int kThreads = 320;                   // TMA warp, MMA warp, 8 softmax warps
constexpr int kWarps = 2;                       // softmax warps per lane quarter
constexpr uint32_t kTile = kSliceBytes;         // one 128-row x 64-column bf16 tile
constexpr uint32_t Q_OFF = 0;
constexpr uint32_t kKS = 2, kVS = 3;            // key and value ring slots
constexpr uint32_t K_OFF = Q_OFF + kTile;       // [kKS] key tile ring
constexpr uint32_t V_OFF = K_OFF + kKS * kTile; // [kVS] value tile ring (turned K-major)
constexpr uint32_t BAR_OFF = V_OFF + kVS * kTile;
constexpr uint32_t XCH_OFF = BAR_OFF + 256;     // [3 slots][128 rows] 32-bit words
constexpr uint32_t SMEM = XCH_OFF + 3 * 128 * 4 + 1024;   // + alignment slack
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kOut = 128;                  // first TMEM column of O
constexpr uint32_t kSSlots = 3;                 // score slots of 64 keys (64 columns each)
// TMEM columns of score slot j: 0..63, 64..127 and, beside O, 192..255
__device__ __forceinline__ uint32_t slot_col(uint32_t j) { return j == 2 ? 192u : 64u * j; }
static_assert(2 * (SMEM + 1024) <= 233472, "two CTAs per SM");
}  // namespace w64

__device__ __forceinline__ void softmax_rows64(const WindowParams& p, uint32_t tmem_base, int warp,
                                               int lane, uint64_t* s_full, uint64_t* o_full,
                                               uint64_t* p_full, uint64_t* pv_done, uint64_t* pair_bar,
                                               uint32_t* slots, volatile int* abort_flag, uint64_t lim) {
    using namespace w64;
    const int quarter = warp & 3;   // TMEM lane quarter of this warp
    const int g = (warp - 2) >> 2;  // which 32-key chunk of each 64-key step, and half of the output
    const int r = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    constexpr float kRescaleLog2 = 8.f;   // weights stay below 2^8
    uint32_t u = 0;                        // quarter steps taken (see softmax_rows)
    uint32_t sc = 0;                       // 64-key steps consumed (score slot ring, P V count)
    auto quarter_meet = [&]() -> bool {
        tc_fence_before();
        mbar_arrive(pair_bar + quarter);
        const bool ok =
            __all_sync(0xffffffffu, mbar_wait_bounded(pair_bar + quarter, u & 1, abort_flag, p.dev_status, lim));
        tc_fence_after();
        return ok;
    };
    auto step_done = [&]() {
        if (g == 0) slots[((u + 2) % 3) * 128 + r] = 0u;
        ++u;
    };
    int n = 0;
    for (int item = blockIdx.x; item < p.items; item += gridDim.x, ++n) {
        const WinItem w = win_item(p, item);
        const int i = w.i0 + r;
        const int jlo = i - p.wl > 0 ? i - p.wl : 0;
        const int jhi = i + p.wr < p.T - 1 ? i + p.wr : p.T - 1;
        const int iw = w.i0 + quarter * 32;
        const int wlo = iw - p.wl > 0 ? iw - p.wl : 0;
        const int whi = iw + 31 + p.wr < p.T - 1 ? iw + 31 + p.wr : p.T - 1;
        const int flo = iw + 31 - p.wl > 0 ? iw + 31 - p.wl : 0;
        const int fhi = iw + p.wr < p.T - 1 ? iw + p.wr : p.T - 1;
        const int kbase = w.kt0 * kWN;
        float M = -INFINITY;   // the row's shift
        float l = 0.f;         // this warp's partial row sum
        for (int h = 0; h < 2 * w.nkt; ++h) {
            // step h: keys kbase + 64 h .. + 63 in score slot sc % 3; this warp
            // takes their 32-key chunk g (chunk 2 h + g of the item)
            const uint32_t ss = sc % kSSlots;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(s_full + ss, (sc / kSSlots) & 1, abort_flag,
                                                          p.dev_status, lim)))
                return;
            ++sc;
            tc_fence_after();
            const uint32_t col = t_lane + slot_col(ss) + 32 * g;
            const int j0 = kbase + 32 * (2 * h + g);
            // 0 outside every band of the warp, 1 inside all of them, 2 partial
            const int cls = (j0 + 31 < wlo || j0 > whi) ? 0 : (j0 >= flo && j0 + 31 <= fhi) ? 1 : 2;
            float m = -INFINITY;
            {
                uint32_t v[32];
                if (cls == 1) {
                    float m0 = tmem_ldred_max16(col, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                    float m1 = tmem_ldred_max16(col + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                    tmem_ld_wait();
                    reg_fence_f(m0);
                    reg_fence_f(m1);
                    m = fmaxf(m0, m1);
                } else if (cls == 2) {
                    tmem_ld32(col, v);
                    tmem_ld_wait();
                    reg_fence(v);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (j0 + e >= jlo && j0 + e <= jhi) m = fmaxf(m, __uint_as_float(v[e]));
                }
            }
            uint32_t* slot = slots + (u % 3) * 128;
            if (m > -INFINITY) atomicMax(slot + r, f32_order_key(m));
            if (!quarter_meet()) return;
            const uint32_t mk = slot[r];
            step_done();
            const float mt = mk == 0u ? -INFINITY : order_key_f32(mk);
            const bool move = mt > -INFINITY && (M == -INFINITY || (mt - M) * p.scale_log2 > kRescaleLog2);
            if (__any_sync(0xffffffffu, move && M > -INFINITY)) {
                // O holds the earlier steps' sums at the old shift: once the
                // previous step's P V is done (the one before it finished
                // ahead of this step's scores), scale this warp's columns of
                // the moved rows
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(pv_done, (sc - 2) & 1, abort_flag,
                                                              p.dev_status, lim)))
                    return;
                tc_fence_after();
                const float f = move && M > -INFINITY ? ex2_approx((M - mt) * p.scale_log2) : 1.f;
                const uint32_t ocol = t_lane + w64::kOut + 32 * g;
                uint32_t o[32];
                tmem_ld32(ocol, o);
                tmem_ld_wait();
                reg_fence(o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                tmem_st32(ocol, o);
                tmem_st_wait();
                l *= f;
            }
            if (move) M = mt;
            uint32_t whi[16], wlo[16];
            if (cls) {
                uint32_t v[32];
                tmem_ld32(col, v);
                tmem_ld_wait();
                reg_fence(v);
                const bool mask = cls == 2;
                float s2[2] = {0.f, 0.f};
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    float pv[2];
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        const int j = j0 + 2 * q + b;
                        const float x = (__uint_as_float(v[2 * q + b]) - M) * p.scale_log2;
                        pv[b] = ex2_approx(!mask || (j >= jlo && j <= jhi) ? x : -INFINITY);
                    }
                    s2[q & 1] += pv[0] + pv[1];
                    const uint32_t b0 = __float_as_uint(pv[0]), b1 = __float_as_uint(pv[1]);
                    whi[q] = __byte_perm(b0, b1, 0x7632);
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(
                        pv[0] - __uint_as_float(b0 & 0xFFFF0000u), pv[1] - __uint_as_float(b1 & 0xFFFF0000u));
                    wlo[q] = *reinterpret_cast<const uint32_t*>(&lo);
                }
                l += s2[0] + s2[1];
            } else {
#pragma unroll
                for (int q = 0; q < 16; ++q) whi[q] = wlo[q] = 0u;
            }
            tmem_st16(col, whi);
            tmem_st16(col + 16, wlo);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full + ss);
        }
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(o_full, n & 1, abort_flag, p.dev_status, lim)))
            return;
        tc_fence_after();
        uint32_t* slot = slots + (u % 3) * 128;
        atomicAdd(reinterpret_cast<float*>(slot) + r, l);
        if (!quarter_meet()) return;
        const float sum = __uint_as_float(slot[r]);
        step_done();
        const float inv = sum > 0.f ? 1.f / sum : 0.f;
        uint32_t o[32];
        tmem_ld32(t_lane + w64::kOut + 32 * g, o);
        tmem_ld_wait();
        reg_fence(o);
        tc_fence_before();   // the O columns are read: the next item's MMAs may write them
        if (i < p.T) {
            const int64_t off = (static_cast<int64_t>(w.bh) * p.T + i) * 64 + 32 * g;
            if (p.bf16_out) {
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.O) + off);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    uint32_t wv[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int d = c8 * 8 + q * 2;
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(o[d]) * inv,
                                                                        __uint_as_float(o[d + 1]) * inv);
                        wv[q] = *reinterpret_cast<const uint32_t*>(&b2);
                    }
                    dst[c8] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            } else {
                float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.O) + off);
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4)
                    dst[c4] = make_float4(__uint_as_float(o[4 * c4]) * inv, __uint_as_float(o[4 * c4 + 1]) * inv,
                                          __uint_as_float(o[4 * c4 + 2]) * inv,
                                          __uint_as_float(o[4 * c4 + 3]) * inv);
            }
        }
    }
}

__global__ void __launch_bounds__(w64::kThreads, 2)
    window_tc64_kernel(const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const WindowParams p) {
    using namespace w64;
    constexpr uint32_t IDESC_S = idesc_bf16_f32(kWM, 64);    // one 64-key step
    constexpr uint32_t IDESC_O = idesc_bf16_f32(kWM, 64);   // V^T K-major
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
    uint64_t* q_full = bars;         // the query tile landed
    uint64_t* q_empty = bars + 1;    // the item's S MMAs are done
    uint64_t* k_full = bars + 2;          // [kKS] key tile landed
    uint64_t* k_empty = k_full + kKS;     // [kKS] its S MMA is done
    uint64_t* v_full = k_empty + kKS;     // [kVS] value tile landed
    uint64_t* vt_full = v_full + kVS;     // [kVS] value tile turned K-major
    uint64_t* v_empty = vt_full + kVS;    // [kVS] its P V MMAs are done
    uint64_t* s_full = v_empty + kVS;     // [kSSlots] a 64-key step's scores in its slot
    uint64_t* p_full = s_full + kSSlots;  // [kSSlots] its weights (one arrive per softmax warp)
    uint64_t* pv_done = p_full + kSSlots; // a step's P V MMAs are done
    uint64_t* o_full = pv_done + 1;       // every MMA of the item done
    uint64_t* pair_bar = o_full + 1;      // [4] the two softmax warps of a lane quarter meet
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pair_bar + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint32_t* slots = reinterpret_cast<uint32_t*>(smem + XCH_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t lim = p.wait_limit_ns ? p.wait_limit_ns : kWDefaultWaitNs;
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (uint32_t s = 0; s < kKS; ++s) {
            mbar_init(k_full + s, 1);
            mbar_init(k_empty + s, 1);
        }
        for (uint32_t s = 0; s < kVS; ++s) {
            mbar_init(v_full + s, 1);
            mbar_init(vt_full + s, 1);
            mbar_init(v_empty + s, 1);
        }
        for (uint32_t s = 0; s < kSSlots; ++s) {
            mbar_init(s_full + s, 1);
            mbar_init(p_full + s, 4 * w64::kWarps);
        }
        mbar_init(pv_done, 1);
        mbar_init(o_full, 1);
        for (int q = 0; q < 4; ++q) mbar_init(pair_bar + q, 32 * w64::kWarps);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    for (int x = threadIdx.x; x < 3 * 128; x += kThreads) slots[x] = 0u;
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA (lane 0) and the
        // turning of each landed value tile K-major (whole warp). The block's
        // key tiles are numbered c = 0, 1, ... over its items in order; lane 0
        // has the copies of tiles c + 1 and c + 2 in flight while the warp
        // turns tile c, so no tile waits for its copy to be issued.
        int ld_item = blockIdx.x, ld_t = 0;   // the next tile to copy: its item and key tile
        WinItem ld_w{};
        if (ld_item < p.items) ld_w = win_item(p, ld_item);
        uint32_t nq = 0, nl = 0;              // query tiles, key and value tile pairs issued
        // lane 0: the next tile's key and value copies, after its item's query
        // tile if it is the item's first; false when a wait ran out or the
        // block stopped (what was issued is counted)
        auto issue_next = [&]() -> bool {
            if (ld_item >= p.items) return true;
            if (ld_t == 0) {
                if (nq > 0 && !mbar_wait_bounded(q_empty, (nq - 1) & 1, abort_flag, p.dev_status, lim))
                    return false;
                mbar_arrive_expect_tx(q_full, kTile);
                tma_load_3d(smem + Q_OFF, &qmap, 0, ld_w.i0, ld_w.bh, q_full);
                ++nq;
            }
            const uint32_t ks = nl % kKS, vs = nl % kVS;
            if (nl >= kKS && !mbar_wait_bounded(k_empty + ks, (nl / kKS - 1) & 1, abort_flag, p.dev_status, lim))
                return false;
            if (nl >= kVS && !mbar_wait_bounded(v_empty + vs, (nl / kVS - 1) & 1, abort_flag, p.dev_status, lim))
                return false;
            const int key0 = (ld_w.kt0 + ld_t) * kWN;
            mbar_arrive_expect_tx(k_full + ks, kTile);
            tma_load_3d(smem + K_OFF + ks * kTile, &kmap, 0, key0, ld_w.bh, k_full + ks);
            mbar_arrive_expect_tx(v_full + vs, kTile);
            tma_load_3d(smem + V_OFF + vs * kTile, &vmap, 0, key0, ld_w.bh, v_full + vs);
            ++nl;
            if (++ld_t == ld_w.nkt) {
                ld_t = 0;
                ld_item += gridDim.x;
                if (ld_item < p.items) ld_w = win_item(p, ld_item);
            }
            return true;
        };
        bool ok = true;
        if (lane == 0) ok = issue_next() && issue_next();
        ok = __shfl_sync(0xffffffffu, ok, 0);
        uint32_t vc = 0;   // value tiles turned
        for (int item = blockIdx.x; ok && item < p.items; item += gridDim.x) {
            const int nkt = win_item(p, item).nkt;
            for (int t = 0; t < nkt; ++t) {
                const uint32_t vs = vc % kVS;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(v_full + vs, (vc / kVS) & 1, abort_flag,
                                                              p.dev_status, lim))) {
                    ok = false;
                    break;
                }
                for (int h = 0; h < 2; ++h)
                    vt_transpose_half(smem_u32(smem + V_OFF + vs * kTile + h * (kTile / 2)), lane);
                fence_proxy_async_smem();   // the MMAs read the tile through the async proxy
                __syncwarp();
                if (lane == 0) mbar_arrive(vt_full + vs);
                ++vc;
                if (lane == 0) ok = issue_next();
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
        }
        // the copies land before the block may exit (slot s last held tile
        // s + kS * floor((n - 1 - s) / kS) of the n issued)
        if (lane == 0) {
            if (nq > 0) mbar_wait_bounded(q_full, (nq - 1) & 1, nullptr, p.dev_status, lim);
            for (uint32_t s = 0; s < kKS; ++s)
                if (nl > s) mbar_wait_bounded(k_full + s, ((nl - 1 - s) / kKS) & 1, nullptr, p.dev_status, lim);
            for (uint32_t s = 0; s < kVS; ++s)
                if (nl > s) mbar_wait_bounded(v_full + s, ((nl - 1 - s) / kVS) & 1, nullptr, p.dev_status, lim);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA
        // Per item, 64-key steps h = 0 .. 2 nkt - 1 (key tile h / 2, its half
        // h % 2): S(h) into score slot h % 3 (counted over the block's steps),
        // then, once its weights are written, P(h) V(h) into O. S(h + 2) is
        // issued right behind P(h) V(h), so the softmax warps work on step
        // h + 1 while the tensor pipe runs P(h) V(h): S(h + 2) takes the slot
        // of step h - 1, whose P V ran before it (tcgen05.mma instructions of
        // one thread run in issue order).
        if (lane == 0) {
            int n = 0;
            uint32_t kc = 0, vc = 0, sc = 0, pc = 0, committed = 0;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < p.items; item += gridDim.x, ++n) {
                const WinItem w = win_item(p, item);
                if (!mbar_wait_bounded(q_full, n & 1, abort_flag, p.dev_status, lim)) break;
                const uint64_t qd = smem_desc_k_sw128(smem_u32(smem + Q_OFF));
                const int H = 2 * w.nkt;
                auto issue_s = [&](int h) -> bool {
                    const uint32_t ks = kc % kKS;
                    if ((h & 1) == 0) {   // a new key tile
                        if (!mbar_wait_bounded(k_full + ks, (kc / kKS) & 1, abort_flag, p.dev_status, lim))
                            return false;
                        tc_fence_after();
                    }
                    const uint64_t kd = smem_desc_k_sw128(smem_u32(smem + K_OFF + ks * kTile + (h & 1) * (kTile / 2)));
                    const uint32_t d = tmem_base + slot_col(sc % kSSlots);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(d, qd + ((kk * 32) >> 4), kd + ((kk * 32) >> 4), IDESC_S, kk != 0);
                    if (h & 1) {
                        mma_commit(k_empty + ks);
                        ++kc;
                    }
                    if (h == H - 1) mma_commit(q_empty);
                    mma_commit(s_full + sc % kSSlots);
                    ++sc;
                    return true;
                };
                ok = issue_s(0) && issue_s(1);
                for (int h = 0; ok && h < H; ++h) {
                    const uint32_t ps = pc % kSSlots, vs = vc % kVS;
                    ok = mbar_wait_bounded(p_full + ps, (pc / kSSlots) & 1, abort_flag, p.dev_status, lim);
                    if (ok && (h & 1) == 0)
                        ok = mbar_wait_bounded(vt_full + vs, (vc / kVS) & 1, abort_flag, p.dev_status, lim);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t pcol = slot_col(ps);
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4) {
                        // keys 16 s4 .. 16 s4 + 15 of the step: their hi and lo
                        // weights (chunk s4 / 2: hi words in its first 16
                        // columns, lo in the next 16) and a 32-byte K slice of
                        // V^T's 64-key half h % 2
                        const uint32_t hi = pcol + 32 * (s4 / 2) + 8 * (s4 % 2);
                        const uint64_t bd =
                            smem_desc_k_sw128(smem_u32(smem + V_OFF + vs * kTile + (h & 1) * (kTile / 2))) +
                            ((s4 * 32) >> 4);
                        mma_bf16_ta(tmem_base + w64::kOut, tmem_base + hi, bd, IDESC_O, (h | s4) != 0);
                        mma_bf16_ta(tmem_base + w64::kOut, tmem_base + hi + 16, bd, IDESC_O, 1);
                    }
                    mma_commit(pv_done);
                    if (h & 1) {
                        mma_commit(v_empty + vs);
                        ++vc;
                    }
                    ++pc;
                    if (h + 2 < H) ok = issue_s(h + 2);
                }
                // every MMA of the item (also after a stop) is tracked by o_full
                mma_commit(o_full);
                ++committed;
            }
            if (committed > 0) mbar_wait_bounded(o_full, (committed - 1) & 1, nullptr, p.dev_status, lim);
        }
    } else {
        softmax_rows64(p, tmem_base, warp, lane, s_full, o_full, p_full, pv_done, pair_bar, slots, abort_flag,
                       lim);
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

// [BH][T][D] bf16, box 64 columns x 128 rows x 1 head, 128-byte swizzle (a
// D = 128 tile is two boxes, at columns 0 and 64); rows outside [0, T) of a
// head read as zeros.
bool make_map_3d(CUtensorMap* m, const void* base, int BH, int T, int D) {
    const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(T),
                              static_cast<uint64_t>(BH)};
    const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2,
                                 static_cast<uint64_t>(D) * 2 * static_cast<uint64_t>(T)};
    const uint32_t box[3] = {64u, static_cast<uint32_t>(kWN), 1};
    return tmap_bf16_sw128(m, base, 3, dims, strides, box);
}

template <int D>
cudaError_t window_tc_run(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                          const WindowParams& p, cudaStream_t stream) {
    static_assert(D == 128, "head size 64 runs window_tc64_kernel");
    const int sms = tile_sm_count();
    const int grid = p.items < sms ? p.items : sms;
    cudaError_t e = set_max_dyn_smem(reinterpret_cast<const void*>(window_tc_kernel<D>),
                                     static_cast<int>(WinCfg<D>::SMEM));
    if (e != cudaSuccess) return e;
    TraceLaunch tr("window_tc", stream);
    window_tc_kernel<D><<<grid, kWThreads, WinCfg<D>::SMEM, stream>>>(qm, km, vm, p);
    return cudaGetLastError();
}

}  // namespace

// True when the tensor-core kernel covers the call: bf16 inputs, head size 64
// or 128, and the band of every 128-query tile within three 128-key tiles.
bool window_tc_supported(bool bf16_in, int D, int T, int wl, int wr) {
    if (!bf16_in || (D != 64 && D != 128) || T <= 0) return false;
    const int ntq = (T + kWM - 1) / kWM;
    for (int qt = 0; qt < ntq; ++qt) {
        int kt0, kt1;
        band_tiles(qt, T, wl, wr, &kt0, &kt1);
        if (kt1 - kt0 + 1 > kWMaxTiles) return false;
    }
    return true;
}

cudaError_t window_tc_launch(const void* Q, const void* K, const void* V, void* O, bool bf16_out,
                             int BH, int T, int D, int wl, int wr, float scale,
                             int32_t* dev_status, cudaStream_t stream) {
    if (D != 64 && D != 128) return cudaErrorInvalidValue;
    const int64_t items = static_cast<int64_t>(BH) * ((T + kWM - 1) / kWM);
    if (items == 0) return cudaSuccess;
    if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    CUtensorMap qm, km, vm;
    if (!make_map_3d(&qm, Q, BH, T, D) || !make_map_3d(&km, K, BH, T, D) ||
        !make_map_3d(&vm, V, BH, T, D))
        return cudaErrorInvalidValue;
    WindowParams p;
    p.BH = BH;
    p.T = T;
    p.wl = wl;
    p.wr = wr;
    p.items = static_cast<int>(items);
    p.scale_log2 = scale * kLog2e;
    p.O = O;
    p.bf16_out = bf16_out ? 1 : 0;
    p.dev_status = dev_status;
    p.wait_limit_ns = 0;
    if (D == 128) return window_tc_run<128>(qm, km, vm, p, stream);
    // D 64: two CTAs per SM, each on its own items
    const int64_t grid = std::min<int64_t>(items, 2 * static_cast<int64_t>(tile_sm_count()));
    cudaError_t e = set_max_dyn_smem(reinterpret_cast<const void*>(window_tc64_kernel),
                                     static_cast<int>(w64::SMEM));
    if (e != cudaSuccess) return e;
    TraceLaunch tr("window_tc", stream);
    window_tc64_kernel<<<static_cast<unsigned>(grid), w64::kThreads, w64::SMEM, stream>>>(qm, km, vm, p);
    return cudaGetLastError();
}

}  // namespace ssa
