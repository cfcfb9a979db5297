// Tensor-core scorer: S = q_low . k_low^T * scale on tcgen05, one 256-query
// unit of a head against all its valid keys, 128 keys at a time. The scores
// live in TMEM only; the epilogue warps reduce them on the fly, so the n x n
// score matrix never reaches HBM (the low-rank scorer of mhpq.cn/news/1098205,
// section 2.2; the selection of its section 3.2).
//
// The same kernel runs in three modes (the epilogue differs, the contraction
// does not, and it is deterministic, so every mode sees bit-identical scores):
//   MODE_RAW       writes the scaled scores, -inf where the key is masked
//                  (the scorer output as its own call);
//   MODE_GROUPMAX  splits each query row's valid keys into groups of g keys
//                  (layout in tile.h) and writes the 16 high bits of the order
//                  key of every group's maximum score;
//   MODE_COLLECT   appends every valid key whose score reaches the row's
//                  threshold to the row's candidate lists, as (raw score
//                  bits, key index) pairs.
// The exact top-k of a row is then found from these (tile_select.cu).
//
// Block layout (608 threads, one block per SM): warp 0 issues TMA loads (the
// two 128-row query tiles of a unit, key tiles through a ring of shared-memory
// stages), warp 1 allocates all 512 TMEM columns and issues the MMAs: every
// 128-key tile is multiplied with both query tiles (M=128, N=128, K=16 per
// instruction, bf16 operands K-major with the 128-byte swizzle, fp32
// accumulators), so one 16 KB key tile feeds 512 tensor-core cycles and the
// load ring hides the full latency of freeing and refilling a stage. Tile t of
// a unit goes to TMEM buffer t % 2, which holds one accumulator per query
// tile. Warps 2..17 are the epilogue, four groups of four warps, one per
// (buffer, query tile): warp w of a group reads TMEM lane quarter w%4 (one
// query row per thread), all 128 columns as four 32-column tcgen05.ld, frees
// the buffer and works on the scores in registers. Warp 18 waits, for every
// tile, until its key stage has landed and its TMEM buffer is free, and hands
// the tile to the MMA warp through a named barrier: a thread that issues MMAs
// and then polls an mbarrier itself waits behind the shared-memory operand
// reads of its MMAs in flight, which leaves the tensor pipe idle for several
// hundred cycles per poll, while a named barrier costs a few tens. Every wait
// on an mbarrier is bounded in time; a wait that runs out sets SSA_DEV_WAIT_LIMIT, stops
// every role of the block, lets copies and MMAs in flight finish and frees
// TMEM.
//
// Work is a list of units (head, 256-query block) in head-major order, the
// query blocks of a head from the last (most keys under a causal mask) to the
// first; a persistent grid takes units round-robin.
#include <float.h>

#include "sm100.cuh"
#include "tile.h"
#include "tmap.h"
#include "trace.h"

namespace ssa {

using namespace sm100;

namespace {

constexpr int kEpiWarps = 16;
constexpr int kWaiterWarp = 2 + kEpiWarps;
constexpr int kThreads = 32 * (kWaiterWarp + 1);
constexpr uint32_t kHandoffBar = 1;          // named barrier: waiter warp + MMA warp
constexpr int kTBuf = kTileGroups;            // TMEM tile buffers (two accumulators each)
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kDefaultWaitNs = 1000000000ull;

// Candidate queue of one epilogue warp (MODE_COLLECT), a ring of 64 entries:
// each entry is a 16-key half-chunk holding at least one candidate (its 16 raw
// scores, its first key, the lane = row that owns it); the warp drains 32
// entries at a time, one per lane, so the per-candidate work runs on full
// warps. Fewer than 32 entries wait before a step and a step adds at most 32,
// so the ring never holds more than 63 and a drain never moves entries. The
// scores are stored slot-major, float4 slot i of entry q at [i][q], so that
// lanes touching consecutive entries touch consecutive 16-byte words (no bank
// conflicts).
constexpr int kQueue = 64;                                   // entries, power of two
constexpr int kSub = 16;                                     // keys per entry
constexpr uint32_t kQueueWarpBytes = kQueue * kSub * 4 + kQueue * 4 + 2 * 32 * 4;

// The rare part of a candidate-queue drain (see the drain in
// tile_scores_kernel), run after a drain in which some row's list reached its
// capacity. Out of line: the drain is inlined at nine places, and keeping this
// code out of them keeps the common path as fast as without it.
//  - The drain's slots came from a shared-memory atomic, in no particular
//    order. For each row whose list is now over its capacity, the lanes that
//    hold its entries (not adjacent in general) add up their candidate counts
//    in lane order through the drained entries' key words (free by now) and
//    store the drain's candidates again, in ring order, into the same slots.
//  - A candidate past the capacity that scores above the row's bound (order
//    key > tau) flags the row; one exactly at the bound is dropped.
//  - A row whose list is full moves its test to the first raw score whose
//    scaled order key exceeds the bound (tau's low 16 bits are zero, so
//    tau + 1 does not wrap; a row without a bound never fills past its keys).
// Returns the lane's test. qb is the warp's queue (ring, key words, counts,
// flags); packed holds the drain's ring position q_head mod 64 (bits 0..15),
// its entry count n (16..23) and the TMEM buffer tb (24..31), few arguments
// being what keeps the call site cheap; bits are this lane's candidates.
__device__ __noinline__ float drain_fixup(uint8_t* qb, const uint32_t* tau, uint64_t* cand,
                                          int64_t row0, uint32_t packed, uint32_t bits, int capc,
                                          float t_hot, float scale) {
    const int q_head = static_cast<int>(packed & 0xFFFFu), n = static_cast<int>((packed >> 16) & 0xFFu);
    const int tb = static_cast<int>(packed >> 24);
    const int lane = threadIdx.x & 31;
    const bool act = lane < n;
    float4* qv = reinterpret_cast<float4*>(qb);
    uint32_t* qm = reinterpret_cast<uint32_t*>(qb + kQueue * kSub * 4);
    int* qcnt = reinterpret_cast<int*>(qb + kQueue * (kSub * 4 + 4));
    int* qovf = qcnt + 32;
    const uint32_t qmeta = act ? qm[(q_head + lane) & (kQueue - 1)] : 0u;
    const int owner = static_cast<int>(qmeta & 31u);
    const int qi = (q_head + lane) & (kQueue - 1);
    const int nb = __popc(bits);
    const uint32_t peers = __match_any_sync(0xffffffffu, act ? owner : 32 + lane);
    __syncwarp();   // every plain store and count is in, every key word read
    if (act) qm[qi] = static_cast<uint32_t>(nb);
    __syncwarp();
    int before = 0, total = 0;
    for (uint32_t m = peers; m; m &= m - 1) {
        const int l = __ffs(m) - 1;
        const int c = static_cast<int>(qm[(q_head + l) & (kQueue - 1)]);
        total += c;
        if (l < lane) before += c;
    }
    const int end = act ? qcnt[owner] : 0;
    if (act && nb > 0 && end > capc) {
        // the row's list is over its capacity: this drain's candidates again,
        // in ring order, and a check of those past the capacity
        int sl = end - total + before;
        const uint32_t tau_own = tau[row0 + owner];
        uint64_t* dst = cand + ((row0 + owner) * kTBuf + tb) * static_cast<int64_t>(capc);
        const uint32_t jb = (qmeta >> 5) * kSub;
        bool above = false;
        for (uint32_t b = bits; b; b &= b - 1, ++sl) {
            const int e = __ffs(b) - 1;
            const float x = reinterpret_cast<const float*>(qv + (e >> 2) * kQueue + qi)[e & 3];
            if (sl < capc)
                dst[sl] = (static_cast<uint64_t>(__float_as_uint(x)) << 32) | (jb + static_cast<uint32_t>(e));
            else if (f32_order_key(x * scale) > tau_own)
                above = true;
        }
        if (above) qovf[owner] = 1;
    }
    __syncwarp();
    if (qcnt[lane] >= capc) {
        const uint32_t t32 = tau[row0 + lane];
        t_hot = t32 == 0 ? -FLT_MAX : tile_raw_threshold(order_key_f32(t32 + 1u), scale);
    }
    return t_hot;
}

template <int P, int MODE>
struct TileCfg {
    static constexpr int KA = P / 64;                       // 128-byte K atoms per row
    static constexpr bool QUEUE = MODE == MODE_COLLECT;
    static constexpr int STAGES = (P == 64) ? (QUEUE ? 5 : 8) : (QUEUE ? 2 : 4);   // key ring
    static constexpr int QSLOTS = (P == 64) ? 2 : 1;        // query-unit slots
    static constexpr uint32_t QHALF = KA * kTileM * 128;    // one 128-row query tile
    static constexpr uint32_t QBYTES = 2 * QHALF;           // a unit's two query tiles
    static constexpr uint32_t KBYTES = KA * kTileN * 128;
    static constexpr uint32_t K_OFF = QSLOTS * QBYTES;
    static constexpr uint32_t BAR_OFF = K_OFF + STAGES * KBYTES;
    static constexpr uint32_t QUEUE_OFF = BAR_OFF + 512;
    static constexpr uint32_t SMEM =
        QUEUE_OFF + (QUEUE ? kEpiWarps * kQueueWarpBytes : 0) + 1024;   // + alignment slack
};

struct Unit {
    int bh, i0, rows, n_lo, n_hi, ntiles;
};

// The k-th unit of this CTA (kNoUnit past the last, -2 for an empty slot).
// Causal units shrink from the last query block to the first, so with enough
// units each work item pairs the unit qb of a head with the unit
// units_per_head-1-qb of the same head (every pair then holds about the same
// number of key tiles) and the pairs go round-robin over the persistent grid:
// the slowest CTA has about 1% more work than the mean instead of 8-15%, and
// the CTAs still work on one or two heads at a time (their k_low stays in
// L2). With fewer than two units per CTA, units go round-robin one by one.
constexpr int kNoUnit = -1;
SSA_DEVINL int cta_unit(const TileParams& p, int k) {
    if (!p.pair_units) {
        const int u = blockIdx.x + k * gridDim.x;
        return u < p.num_units ? u : kNoUnit;
    }
    const int P = (p.units_per_head + 1) >> 1;   // pairs per head
    const int pi = blockIdx.x + (k >> 1) * gridDim.x;
    if (pi >= p.BH * P) return kNoUnit;
    const int bh = pi / P, j = pi - (pi / P) * P;
    const int l = (k & 1) ? p.units_per_head - 1 - j : j;
    if ((k & 1) && l == j) return -2;
    return bh * p.units_per_head + l;
}

SSA_DEVINL Unit unit_at(const TileParams& p, int u) {
    Unit U;
    U.bh = u / p.units_per_head;
    const int qb = p.units_per_head - 1 - (u - U.bh * p.units_per_head);
    U.i0 = qb * kUnitM;
    U.rows = min(kUnitM, p.Tq - U.i0);
    U.n_lo = tile_valid_count(U.i0, p.Tq, p.Tk, p.causal);
    U.n_hi = tile_valid_count(U.i0 + U.rows - 1, p.Tq, p.Tk, p.causal);
    U.ntiles = (U.n_hi + kTileN - 1) / kTileN;
    return U;
}

SSA_DEVINL float max8(const float* v) {
    return fmaxf(fmax3(v[0], v[1], v[2]), fmax3(v[3], v[4], fmaxf(v[5], fmaxf(v[6], v[7]))));
}

// Maximum of 16 scores: an fmax3 tree (8 instructions).
SSA_DEVINL float max16(const float* v) {
    const float a = fmax3(v[0], v[1], v[2]), b = fmax3(v[3], v[4], v[5]);
    const float c = fmax3(v[6], v[7], v[8]), d = fmax3(v[9], v[10], v[11]);
    const float e = fmax3(v[12], v[13], v[14]);
    return fmaxf(fmax3(a, b, c), fmax3(d, e, v[15]));
}

// Maximum of the G consecutive scores at w (G a power of two <= 16).
template <int G>
SSA_DEVINL float max_of(const float* w) {
    if constexpr (G == 1) return w[0];
    else if constexpr (G == 2) return fmaxf(w[0], w[1]);
    else if constexpr (G == 4) return fmax3(w[0], w[1], fmaxf(w[2], w[3]));
    else if constexpr (G == 8) return max8(w);
    else return fmaxf(max8(w), max8(w + 8));
}

// Group maxima of a 32-key chunk starting at key j0 (a multiple of 32) for a
// group size G < 32: the chunk holds 32/G whole groups, group (j0+e)/G for
// e = 0, G, 2G, ...; each group with a valid key writes the 16 high bits of
// the order key of its scaled maximum (masked keys were set to -inf).
template <int G>
SSA_DEVINL void small_groups(const float (&v)[32], int j0, int n_i, uint16_t* gcol, float scale) {
#pragma unroll
    for (int e = 0; e < 32; e += G)
        if (j0 + e < n_i)
            gcol[static_cast<int64_t>((j0 + e) / G) * kUnitM] =
                static_cast<uint16_t>(f32_order_key(max_of<G>(v + e) * scale) >> 16);
}

// As small_groups for any group size g in {1, 2, 4} (rows of fewer than 8k
// keys only): one running maximum, written at the last key of each group.
SSA_DEVINL void tiny_groups(const float (&v)[32], int j0, int n_i, uint16_t* gcol, float scale,
                            int g) {
    float run = -INFINITY;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        run = (e & (g - 1)) == 0 ? v[e] : fmaxf(run, v[e]);
        if ((e & (g - 1)) == g - 1 && j0 + e - (g - 1) < n_i)
            gcol[static_cast<int64_t>((j0 + e) / g) * kUnitM] =
                static_cast<uint16_t>(f32_order_key(run * scale) >> 16);
    }
}

// Bit e of the result is set iff v[e] >= t (e < 8): one set + one funnel
// shift per element, no branches.
SSA_DEVINL uint32_t ge_mask8(const float* v, float t) {
    uint32_t m = 0;
#pragma unroll
    for (int e = 7; e >= 0; --e) {
        uint32_t d;
        asm("set.ge.u32.f32 %0, %1, %2;" : "=r"(d) : "f"(v[e]), "f"(t));
        m = __funnelshift_l(d, m, 1);   // (m << 1) | (d >> 31)
    }
    return m;
}

}  // namespace

template <int P, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    tile_scores_kernel(const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ CUtensorMap kmap, const TileParams p) {
    using C = TileCfg<P, MODE>;
    constexpr int S = C::STAGES;
    constexpr uint32_t IDESC = idesc_bf16_f32(kTileM, kTileN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sq = smem;                                   // query-unit slots
    uint8_t* sk = smem + C::K_OFF;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* q_full = bars;                              // [QSLOTS]
    uint64_t* q_empty = bars + 2;                         // [QSLOTS]
    uint64_t* k_full = bars + 4;                          // [S]
    uint64_t* k_empty = k_full + S;                       // [S]
    uint64_t* t_full = k_empty + S;                       // [kTBuf]
    uint64_t* t_empty = t_full + kTBuf;                   // [kTBuf]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(t_empty + kTBuf);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::QSLOTS; ++i) {
            mbar_init(q_full + i, 1);
            mbar_init(q_empty + i, 1);
        }
        for (int s = 0; s < S; ++s) {
            mbar_init(k_full + s, 1);
            mbar_init(k_empty + s, 1);
        }
        for (int b = 0; b < kTBuf; ++b) {
            mbar_init(t_full + b, 1);
            mbar_init(t_empty + b, kEpiWarps / kTBuf);   // one arrive per epilogue warp
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
    const uint64_t lim = p.wait_limit_ns ? p.wait_limit_ns : kDefaultWaitNs;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t kc = 0, qc = 0;
            bool ok = true;
            for (int wk = 0; ok; ++wk) {
                const int u = cta_unit(p, wk);
                if (u == kNoUnit) break;
                if (u < 0) continue;   // the second half of an unpaired middle unit
                const Unit U = unit_at(p, u);
                if (U.ntiles == 0) continue;
                const uint32_t qs = qc % C::QSLOTS, quse = qc / C::QSLOTS;
                if (!mbar_wait_bounded(q_empty + qs, (quse & 1) ^ 1, abort_flag, p.dev_status,
                                       lim)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(q_full + qs, C::QBYTES);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int a = 0; a < C::KA; ++a)
                        tma_load_2d(sq + qs * C::QBYTES + h * C::QHALF + a * 16384, &qmap, a * 64,
                                    U.bh * p.Tq + U.i0 + h * kTileM, q_full + qs);
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
            const uint32_t qfirst = qc > (uint32_t)C::QSLOTS ? qc - C::QSLOTS : 0;
            for (uint32_t m = qfirst; m < qc; ++m)
                mbar_wait_bounded(q_full + (m % C::QSLOTS), (m / C::QSLOTS) & 1, nullptr,
                                  p.dev_status, lim);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // The whole warp runs the loop (the handoff barrier counts whole
        // warps); lane 0 issues. The waiter warp has checked every barrier
        // the tile needs before the handoff; its OR carries "stop".
        uint32_t kc = 0, qc = 0;
        uint32_t tpar = 0;                     // bit b: phase parity of TMEM buffer b
        int last_b = -1;
        bool ok = true;
        // descriptors of the first K slice of stage 0 and of query slot 0;
        // other stages, slots and K slices only move the start address
        const uint64_t bdesc0 = smem_desc_k_sw128(smem_u32(sk));
        const uint64_t adesc0 = smem_desc_k_sw128(smem_u32(sq));
        for (int wk = 0; ok; ++wk) {
            const int u = cta_unit(p, wk);
            if (u == kNoUnit) break;
            if (u < 0) continue;   // the second half of an unpaired middle unit
            const Unit U = unit_at(p, u);
            if (U.ntiles == 0) continue;
            const uint32_t qs = qc % C::QSLOTS;
            const uint64_t adesc = adesc0 + ((qs * C::QBYTES) >> 4);
            for (int t = 0; t < U.ntiles; ++t) {
                const uint32_t s = kc % S, b = t & (kTBuf - 1);
                if (bar_red_or(kHandoffBar, 64, false)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t bdesc = bdesc0 + ((s * C::KBYTES) >> 4);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t d_tmem = tmem_base + (2 * b + h) * kTileN;
#pragma unroll
                        for (int a = 0; a < C::KA; ++a) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint64_t off = (a * 16384 + kk * 32) >> 4;
                                mma_bf16(d_tmem, adesc + ((h * C::QHALF) >> 4) + off, bdesc + off,
                                         IDESC, (a | kk) != 0);
                            }
                        }
                    }
                    mma_commit(k_empty + s);
                    mma_commit(t_full + b);
                }
                __syncwarp();
                tpar ^= 1u << b;
                last_b = static_cast<int>(b);
                ++kc;
            }
            if (!ok) break;
            if (lane == 0) mma_commit(q_empty + qs);
            __syncwarp();
            ++qc;
        }
        // MMAs in flight finish by themselves; wait for the last one
        if (lane == 0 && last_b >= 0)
            mbar_wait_bounded(t_full + last_b, ((tpar >> last_b) & 1) ^ 1, nullptr, p.dev_status,
                              lim);
        __syncwarp();
    } else if (warp == kWaiterWarp) {
        // ------------------------------------------------ MMA handoff
        // Same unit and tile sequence as the MMA warp, one handoff per tile:
        // lane 0 waits for the unit's query tiles (first tile of a unit), the
        // tile's key stage and its TMEM buffer. A failed wait (time limit or
        // abort) is handed over as "stop" and both warps leave their loops.
        uint32_t kc = 0, qc = 0;
        uint32_t tpar = 0;
        bool ok = true;
        for (int wk = 0; ok; ++wk) {
            const int u = cta_unit(p, wk);
            if (u == kNoUnit) break;
            if (u < 0) continue;   // the second half of an unpaired middle unit
            const Unit U = unit_at(p, u);
            if (U.ntiles == 0) continue;
            const uint32_t qs = qc % C::QSLOTS, quse = qc / C::QSLOTS;
            bool good = true;
            if (lane == 0) good = mbar_wait_bounded(q_full + qs, quse & 1, abort_flag, p.dev_status, lim);
            for (int t = 0; t < U.ntiles; ++t) {
                const uint32_t s = kc % S, b = t & (kTBuf - 1);
                const uint32_t par = (tpar >> b) & 1;
                if (lane == 0)
                    good = good &&
                           mbar_wait_bounded(k_full + s, (kc / S) & 1, abort_flag, p.dev_status, lim) &&
                           mbar_wait_bounded(t_empty + b, par ^ 1, abort_flag, p.dev_status, lim);
                good = __shfl_sync(0xffffffffu, good, 0);
                if (bar_red_or(kHandoffBar, 64, !good)) {
                    ok = false;
                    break;
                }
                tpar ^= 1u << b;
                ++kc;
            }
            if (!ok) break;
            ++qc;
        }
    } else {
        // ------------------------------------------------ epilogue
        const int quarter = warp & 3;          // TMEM lane quarter of this warp
        const int grp4 = (warp - 2) >> 2;      // epilogue warp group
        const int tb = grp4 >> 1;              // TMEM tile buffer = tile % 2
        const int half = grp4 & 1;             // query tile (accumulator) of the unit
        const int r = half * kTileM + quarter * 32 + lane;   // query row within the unit
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                static_cast<uint32_t>((2 * tb + half) * kTileN);
        const int capc = p.cap / kTBuf;        // this buffer's candidate list of the row
        uint32_t tpar = 0;                     // phase parity of TMEM buffer tb
        bool ok = true;
        // MODE_COLLECT queue of this warp and the candidate count of each row
        float4* qv = nullptr;                  // [kSub/4][kQueue] raw scores
        uint32_t* qm = nullptr;                // [kQueue] (first key / kSub) << 5 | owning lane
        int* qcnt = nullptr;                   // [32] candidates appended per row
        int* qovf = nullptr;                   // [32] a key above the bound found no slot
        int q_head = 0, q_tail = 0;            // warp-uniform ring positions (unwrapped)
        int64_t row0 = 0;                      // global row of lane 0
        float t_hot = -FLT_MAX;                // raw-score bound of this thread's row
                                               // (above the bound once its list is full)
        if constexpr (MODE == MODE_COLLECT) {
            uint8_t* qb = smem + C::QUEUE_OFF + (warp - 2) * kQueueWarpBytes;
            qv = reinterpret_cast<float4*>(qb);
            qm = reinterpret_cast<uint32_t*>(qb + kQueue * kSub * 4);
            qcnt = reinterpret_cast<int*>(qb + kQueue * (kSub * 4 + 4));
            qovf = qcnt + 32;
            qcnt[lane] = 0;
            qovf[lane] = 0;
            __syncwarp();
        }
        // Drain the `n` (<= 32) ring entries from q_head on, entry l by lane l: its
        // candidates (scores >= the owning row's bound) are appended to that
        // row's list; a shared-memory count per row hands out the slots.
        //
        // A full list. Ring entries of a row sit in key order, and the list of
        // (row, buffer) takes that buffer's tiles in ascending key order, so a
        // list that keeps its first cap/2 candidates in key order holds
        // cap/2 >= k keys that all score >= the bound and precede every later
        // key. A later key that scores exactly at the bound is beaten by all
        // of them (equal or higher score, lower index) and cannot be in the
        // row's top k: it is dropped, and from then on the row's test moves
        // to the first raw score above the bound, for queueing and draining
        // alike. A later key above the bound that finds no slot flags the
        // row, which the row-wise kernel then redoes. Slots from the
        // shared-memory atomic come in no particular order within a drain;
        // drain_fixup puts a drain that takes a list past its capacity back
        // in ring order.
        auto drain = [&](int n) {
            const bool act = lane < n;
            const int qi = (q_head + lane) & (kQueue - 1);
            const uint32_t meta = act ? qm[qi] : 0u;
            const int owner = static_cast<int>(meta & 31u);
            const float t_own = __shfl_sync(0xffffffffu, t_hot, owner);
            uint32_t bits = 0;
            if (act) {
                const float4 a = qv[qi], b = qv[kQueue + qi], c4 = qv[2 * kQueue + qi],
                             d4 = qv[3 * kQueue + qi];
                const float w0[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                const float w1[8] = {c4.x, c4.y, c4.z, c4.w, d4.x, d4.y, d4.z, d4.w};
                bits = ge_mask8(w0, t_own) | (ge_mask8(w1, t_own) << 8);
            }
            const uint32_t bits0 = bits;
            int slot = 0;
            if (bits) {
                slot = atomicAdd(qcnt + owner, __popc(bits));
                uint64_t* dst = p.cand + ((row0 + owner) * kTBuf + tb) * static_cast<int64_t>(capc);
                const uint32_t jb = (meta >> 5) * kSub;
                while (bits) {
                    const int e = __ffs(bits) - 1;
                    bits &= bits - 1;
                    if (slot < capc)
                        dst[slot] = (static_cast<uint64_t>(__float_as_uint(
                                         reinterpret_cast<const float*>(qv + (e >> 2) * kQueue + qi)[e & 3]))
                                     << 32) |
                                    (jb + static_cast<uint32_t>(e));
                    ++slot;
                }
            }
            if (__any_sync(0xffffffffu, bits0 != 0 && slot >= capc))   // a list filled
                t_hot = drain_fixup(reinterpret_cast<uint8_t*>(qv), p.tau, p.cand, row0,
                                    static_cast<uint32_t>(q_head & (kQueue - 1)) | (static_cast<uint32_t>(n) << 16) |
                                        (static_cast<uint32_t>(tb) << 24),
                                    bits0, capc, t_hot, p.scale);
            q_head += n;
            __syncwarp();
        };
        for (int wk = 0; ok; ++wk) {
            const int u = cta_unit(p, wk);
            if (u == kNoUnit) break;
            if (u < 0) continue;   // the second half of an unpaired middle unit
            const Unit U = unit_at(p, u);
            const bool row_ok = r < U.rows;
            const int i = U.i0 + r;
            const int n_i = row_ok ? tile_valid_count(i, p.Tq, p.Tk, p.causal) : 0;
            const int64_t row = static_cast<int64_t>(U.bh) * p.Tq + i;
            // mode state
            int g = 0, m_shift = 0, g_shift = 0;   // g and m = g/32 are powers of two
            float gacc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            t_hot = -FLT_MAX;
            uint16_t* gcol = nullptr;
            if constexpr (MODE == MODE_GROUPMAX) {
                g = tile_group_size(U.n_lo, U.n_hi, p.k);
                g_shift = g > 0 ? __ffs(g) - 1 : 0;
                m_shift = g >= 32 ? g_shift - 5 : 0;
                if (n_i <= p.k) g = 0;   // this row selects all its keys: no groups
                gcol = p.gm + static_cast<int64_t>(u) * p.G_stride * kUnitM + r;
            }
            if constexpr (MODE == MODE_COLLECT) {
                if (row_ok) {
                    const uint32_t t32 = p.tau[row];
                    t_hot = tile_raw_threshold(t32 == 0 ? -INFINITY : order_key_f32(t32), p.scale);
                }
            }
            row0 = row - lane;
            for (int t = tb; t < U.ntiles; t += kTBuf) {
                // warp-uniform outcome: tcgen05.ld below needs the whole warp
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(t_full + tb, tpar, abort_flag,
                                                              p.dev_status, lim));
                if (!ok) break;
                tpar ^= 1;
                tc_fence_after();
                // four 16-column loads in flight per wait, each with the
                // maximum of its 16 scores reduced on the way out of TMEM
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                  uint32_t raw[4][16];
                  float mx[4];
#pragma unroll
                  for (int h4 = 0; h4 < 4; ++h4)
                      mx[h4] = tmem_ldred_max16(t_lane + c2 * 64 + 16 * h4, raw[h4]);
                  tmem_ld_wait();
#pragma unroll
                  for (int h4 = 0; h4 < 4; ++h4) {
                      reg_fence(raw[h4]);
                      reg_fence_f(mx[h4]);
                  }
                  if (c2 == 1) {
                      tc_fence_before();
                      __syncwarp();
                      if (lane == 0) mbar_arrive(t_empty + tb);   // the buffer is free again
                  }
                  if constexpr (MODE == MODE_COLLECT) {
                      // every score >= the row's bound is a candidate: the 16-key
                      // half-chunks holding one are queued and drained 32 at a
                      // time. The four tests of the two chunks come first (they
                      // are independent), then the appends.
                      const int jp = t * kTileN + c2 * 64;   // first key of the pair
                      float v[64];
#pragma unroll
                      for (int e = 0; e < 16; ++e) {
#pragma unroll
                          for (int h4 = 0; h4 < 4; ++h4) v[16 * h4 + e] = __uint_as_float(raw[h4][e]);
                      }
                      // mask the keys past the row's last one: only in the chunks
                      // where a row of this warp ends or has ended (a warp-uniform
                      // branch); there the maxima come from the masked registers
                      if (__any_sync(0xffffffffu, jp + 64 > n_i)) {
                          if (jp + 64 > n_i) {
#pragma unroll
                              for (int e = 0; e < 64; ++e)
                                  if (jp + e >= n_i) v[e] = -INFINITY;
#pragma unroll
                              for (int hs = 0; hs < 4; ++hs) mx[hs] = max16(v + 16 * hs);
                          }
                      }
                      uint32_t B[4];
                      bool hot[4];
#pragma unroll
                      for (int hs = 0; hs < 4; ++hs) hot[hs] = mx[hs] >= t_hot;   // masked keys are -inf
#pragma unroll
                      for (int hs = 0; hs < 4; ++hs) B[hs] = __ballot_sync(0xffffffffu, hot[hs]);
                      const uint32_t below = (1u << lane) - 1;
                      const int tot = __popc(B[0]) + __popc(B[1]) + __popc(B[2]) + __popc(B[3]);
                      if (q_tail - q_head + tot <= kQueue) {
                          // the usual case: every entry of the four half-chunks
                          // fits the ring, so they go in without a drain between
                          // (a row's entries still sit in key order); then the
                          // ring drains down to fewer than 32
                          int qb = q_tail;
#pragma unroll
                          for (int hs = 0; hs < 4; ++hs) {
                              const float* w = v + 16 * hs;
                              if (hot[hs]) {
                                  const int q = (qb + __popc(B[hs] & below)) & (kQueue - 1);
                                  qv[q] = make_float4(w[0], w[1], w[2], w[3]);
                                  qv[kQueue + q] = make_float4(w[4], w[5], w[6], w[7]);
                                  qv[2 * kQueue + q] = make_float4(w[8], w[9], w[10], w[11]);
                                  qv[3 * kQueue + q] = make_float4(w[12], w[13], w[14], w[15]);
                                  qm[q] = (static_cast<uint32_t>((jp + 16 * hs) / kSub) << 5) |
                                          static_cast<uint32_t>(lane);
                              }
                              qb += __popc(B[hs]);
                          }
                          q_tail = qb;
                          if (q_tail - q_head >= 32) {
                              __syncwarp();   // the queued entries are visible to every lane
                              drain(32);
                              if (q_tail - q_head >= 32) drain(32);
                          }
                      } else {
#pragma unroll
                          for (int hs = 0; hs < 4; ++hs) {
                              if (B[hs]) {
                                  if (hot[hs]) {
                                      const float* w = v + 16 * hs;
                                      const int q = (q_tail + __popc(B[hs] & below)) & (kQueue - 1);
                                      qv[q] = make_float4(w[0], w[1], w[2], w[3]);
                                      qv[kQueue + q] = make_float4(w[4], w[5], w[6], w[7]);
                                      qv[2 * kQueue + q] = make_float4(w[8], w[9], w[10], w[11]);
                                      qv[3 * kQueue + q] = make_float4(w[12], w[13], w[14], w[15]);
                                      qm[q] = (static_cast<uint32_t>((jp + 16 * hs) / kSub) << 5) |
                                              static_cast<uint32_t>(lane);
                                  }
                                  q_tail += __popc(B[hs]);
                                  if (q_tail - q_head >= 32) {
                                      __syncwarp();
                                      drain(32);
                                  }
                              }
                          }
                      }
                  } else {
#pragma unroll
                  for (int c1 = 0; c1 < 2; ++c1) {
                    const int c = 2 * c2 + c1;
                    const int j0 = t * kTileN + c * 32;
                    float v[32];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        v[e] = __uint_as_float(raw[2 * c1][e]);
                        v[16 + e] = __uint_as_float(raw[2 * c1 + 1][e]);
                    }
                    if constexpr (MODE == MODE_RAW) {
                        if (row_ok) {
                            float* out = p.S + row * static_cast<int64_t>(p.Tk);
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const int j = j0 + e;
                                if (j < p.Tk) out[j] = j < n_i ? v[e] * p.scale : -INFINITY;
                            }
                        }
                    } else {
                        const bool live = j0 < n_i;   // this row has keys in the chunk
                        // the 16-key maxima from TMEM hold for whole halves;
                        // in the chunk where the row ends they come from the
                        // masked registers
                        float m0 = mx[2 * c1], m1 = mx[2 * c1 + 1];
                        if (live && j0 + 32 > n_i) {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (j0 + e >= n_i) v[e] = -INFINITY;
                            m0 = max16(v);
                            m1 = max16(v + 16);
                        }
                        if constexpr (MODE == MODE_GROUPMAX) {
                            if (live && g >= 32) {
                                gacc[c] = fmax3(gacc[c], m0, m1);
                                // last tile of the group, or the row has no key in this
                                // chunk of this buffer's next tile
                                const int lt = t / kTBuf;
                                if (((lt + 1) & ((1 << m_shift) - 1)) == 0 ||
                                    (t + kTBuf) * kTileN + c * 32 >= n_i) {
                                    const int grp = ((lt >> m_shift) * kTBuf + tb) * 4 + c;
                                    gcol[static_cast<int64_t>(grp) * kUnitM] =
                                        static_cast<uint16_t>(f32_order_key(gacc[c] * p.scale) >> 16);
                                    gacc[c] = -INFINITY;
                                }
                            } else if (live && g == 16) {
                                gcol[static_cast<int64_t>(j0 / 16) * kUnitM] =
                                    static_cast<uint16_t>(f32_order_key(m0 * p.scale) >> 16);
                                if (j0 + 16 < n_i)
                                    gcol[static_cast<int64_t>(j0 / 16 + 1) * kUnitM] =
                                        static_cast<uint16_t>(f32_order_key(m1 * p.scale) >> 16);
                            } else if (live && g == 8) {
                                small_groups<8>(v, j0, n_i, gcol, p.scale);
                            } else if (live && g > 0) {
                                tiny_groups(v, j0, n_i, gcol, p.scale, g);
                            }
                        }
                    }
                  }
                  }
                }
            }
            if (!ok) break;
            if constexpr (MODE == MODE_COLLECT) {
                __syncwarp();
                if (q_tail > q_head) drain(q_tail - q_head);
                q_head = q_tail = 0;
                // a flagged row reads as one over its capacity: redone row-wise
                if (row_ok) p.cnt[row * kTBuf + tb] = qovf[lane] ? capc + 1 : min(qcnt[lane], capc);
                qcnt[lane] = 0;
                qovf[lane] = 0;
                __syncwarp();
            }
            if constexpr (MODE == MODE_RAW) {
                // columns past the unit's last key tile are masked for every row
                if (row_ok) {
                    float* out = p.S + row * static_cast<int64_t>(p.Tk);
                    for (int j = U.ntiles * kTileN + tb; j < p.Tk; j += kTBuf) out[j] = -INFINITY;
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

// 2-D map over rows of P bf16 elements: box = 64 elements x 128 rows, 128-byte
// swizzle (the shared-memory layout the MMA descriptors describe).
bool make_map(CUtensorMap* m, const void* base, int64_t nrows, int P) {
    const uint64_t dims[2] = {static_cast<uint64_t>(P), static_cast<uint64_t>(nrows)};
    const uint64_t strides[1] = {static_cast<uint64_t>(P) * 2};
    const uint32_t box[2] = {64, 128};
    return tmap_bf16_sw128(m, base, 2, dims, strides, box);
}

template <int P, int MODE>
cudaError_t launch_mode(const CUtensorMap& qm, const CUtensorMap& km, const TileParams& p,
                        int grid, cudaStream_t stream) {
    using C = TileCfg<P, MODE>;
    auto kern = tile_scores_kernel<P, MODE>;
    cudaError_t e = set_max_dyn_smem(reinterpret_cast<const void*>(kern), static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    TraceLaunch tr(MODE == MODE_RAW ? "tile_scores.raw"
                   : MODE == MODE_GROUPMAX ? "tile_scores.groupmax" : "tile_scores.collect",
                   stream);
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
    p.units_per_head = (p.Tq + kUnitM - 1) / kUnitM;
    p.num_units = p.BH * p.units_per_head;
    if (p.num_units == 0) return cudaSuccess;
    const int sms = tile_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    p.pair_units = p.num_units >= 2 * sms;
    const int items = p.pair_units ? p.BH * ((p.units_per_head + 1) / 2) : p.num_units;
    const int grid = items < sms ? items : sms;
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
