// Exact top-k from the tensor-core score passes (mhpq.cn/news/1098205,
// section 3.2: torch.topk over the scores, top_k = min(top_k, seq_len),
// masked keys never selected; ties to the lower key index, output sorted by
// score descending).
//
// Why the two score passes give the exact answer. Split the valid keys of a
// row into G >= k disjoint groups and let tau be the k-th largest of the G
// group maxima. The k groups with the largest maxima hold k distinct keys
// whose scores are all >= tau, so the k-th largest score of the row is >= tau
// and every key of the top k has a score >= tau. Rounding the group maxima
// down to the 16 high bits of their order key keeps this true. So:
//   pass 1 (tile kernel, MODE_GROUPMAX) writes the rounded group maxima;
//   group_select_kernel finds tau per row (a 2 x 8-bit radix select);
//   pass 2 (tile kernel, MODE_COLLECT) keeps every valid key with score >= tau;
//   cand_sort_kernel selects the k_eff largest candidates (radix select) and
//   sorts them by (score desc, index asc).
// With G between 2k and 4k, about k + k^2/(2G) <= 1.25k keys pass the bound.
// Once a list is full the candidate pass drops later keys that score exactly
// at the bound (each is beaten by the cap/2 >= k earlier keys of that list),
// so heavy ties at the bound do not overflow it; a row where a key above the
// bound found no slot is put on an overflow list and redone by the row-wise
// kernel.
#ifdef SSA_HOST_EMULATION
#include "emu_device.h"   // the host stand-in of the CPU tests (tests/emu)
#include "tile.h"
#else
#include "common.cuh"
#include "tile.h"
#include "tmap.h"
#include "trace.h"
#endif

namespace ssa {

// ---------------------------------------------------------------- tau
//
// One block per 128-row half of a unit. Histograms live in shared memory as
// [bin][row pair] words holding two 16-bit counters (a row has < 65536
// groups). Thread t works on rows 8(t % 16) .. 8(t % 16) + 7 and reads the
// eight rows' maxima of one group in a 128-bit load (16 threads read one
// group's 256 bytes), groups t / 16, t / 16 + 16, ...; eight loads in flight
// per thread.
constexpr int kSelThreads = 256;
constexpr int kSelUnroll = 8;
constexpr int kSelPairs = kTileM / 2;
constexpr int kSelOcts = kTileM / 8;
constexpr int kSelGStep = kSelThreads / kSelOcts;

__global__ void __launch_bounds__(kSelThreads) group_select_kernel(
    const uint16_t* __restrict__ gm, uint32_t* __restrict__ tau, int BH, int Tq, int Tk, int k,
    int causal, int G_stride) {
#ifdef SSA_HOST_EMULATION
    static uint32_t hist[256 * kSelPairs];
#else
    extern __shared__ uint32_t hist[];   // 256 * kSelPairs words
#endif
    __shared__ int n_row[kTileM], g_row[kTileM];   // valid keys, groups with a valid key
    __shared__ uint32_t sel_hi[kTileM], need[kTileM];
    const int units_per_head = (Tq + kUnitM - 1) / kUnitM;
    const int num_items = BH * units_per_head * 2;   // (unit, 128-row half)
    const int tid = threadIdx.x;
    const int qd = tid % kSelOcts;                   // rows 8qd .. 8qd+7
    for (int w = blockIdx.x; w < num_items; w += gridDim.x) {
        const int u = w >> 1, h = w & 1;
        const int bh = u / units_per_head;
        const int qb = units_per_head - 1 - (u - bh * units_per_head);
        const int i0u = qb * kUnitM;
        const int rows_u = min(kUnitM, Tq - i0u);
        const int rows = min(kTileM, rows_u - h * kTileM);
        if (rows <= 0) continue;
        // the group size and layout belong to the whole 256-row unit
        const int n_lo = tile_valid_count(i0u, Tq, Tk, causal);
        const int n_hi = tile_valid_count(i0u + rows_u - 1, Tq, Tk, causal);
        const int g = tile_group_size(n_lo, n_hi, k);
        const int i0 = i0u + h * kTileM;
        uint32_t* tau_u = tau + static_cast<int64_t>(bh) * Tq + i0;
        if (g == 0) {   // no row has more than k valid keys: select everything
            if (tid < rows) tau_u[tid] = 0;
            continue;
        }
        const int G_u = tile_groups_in_unit(n_hi, g);
        // row pair pr of this half: 32-bit words of the [group][256 rows] array
        const uint4* gu = reinterpret_cast<const uint4*>(
                              gm + static_cast<int64_t>(u) * G_stride * kUnitM + h * kTileM) + qd;
        if (tid < kTileM) {
            const int nr = tid < rows ? tile_valid_count(i0 + tid, Tq, Tk, causal) : 0;
            n_row[tid] = nr;
            g_row[tid] = nr > k ? tile_groups_of_row(nr, g, G_u) : 0;
        }
        for (int x = tid; x < 256 * kSelPairs; x += kSelThreads) hist[x] = 0;
        __syncthreads();
        int Gr[8];
        int Gm = 0;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            Gr[r] = g_row[8 * qd + r];
            Gm = max(Gm, Gr[r]);
        }
        // pass 1: high byte of every group maximum of the rows
        for (int g0 = tid / kSelOcts; g0 < Gm; g0 += kSelGStep * kSelUnroll) {
            uint4 v[kSelUnroll];
#pragma unroll
            for (int q = 0; q < kSelUnroll; ++q) {
                const int grp = g0 + q * kSelGStep;
                v[q] = grp < Gm ? gu[static_cast<int64_t>(grp) * (kUnitM / 8)] : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < kSelUnroll; ++q) {
                const int grp = g0 + q * kSelGStep;
                const uint32_t w4[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if (grp < Gr[r])
                        atomicAdd(&hist[((w4[r >> 1] >> (16 * (r & 1) + 8)) & 0xFFu) * kSelPairs + 4 * qd + (r >> 1)],
                                  1u << (16 * (r & 1)));
            }
        }
        __syncthreads();
        if (tid < kTileM) {
            uint32_t hi = 0, nd = 0;
            if (n_row[tid] > k) {
                uint32_t cum = 0;
                for (int b = 255; b >= 0; --b) {
                    const uint32_t cb = (hist[b * kSelPairs + (tid >> 1)] >> ((tid & 1) * 16)) & 0xFFFFu;
                    if (cum + cb >= static_cast<uint32_t>(k)) {
                        hi = b;
                        nd = k - cum;
                        break;
                    }
                    cum += cb;
                }
            }
            sel_hi[tid] = hi;
            need[tid] = nd;
        }
        __syncthreads();
        for (int x = tid; x < 256 * kSelPairs; x += kSelThreads) hist[x] = 0;
        __syncthreads();
        // pass 2: low byte of the group maxima in the selected high-byte bin
        {
            uint32_t hsr[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) hsr[r] = sel_hi[8 * qd + r];
            for (int g0 = tid / kSelOcts; g0 < Gm; g0 += kSelGStep * kSelUnroll) {
                uint4 v[kSelUnroll];
#pragma unroll
                for (int q = 0; q < kSelUnroll; ++q) {
                    const int grp = g0 + q * kSelGStep;
                    v[q] = grp < Gm ? gu[static_cast<int64_t>(grp) * (kUnitM / 8)] : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int q = 0; q < kSelUnroll; ++q) {
                    const int grp = g0 + q * kSelGStep;
                    const uint32_t w4[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const uint32_t x = (w4[r >> 1] >> (16 * (r & 1))) & 0xFFFFu;
                        if (grp < Gr[r] && (x >> 8) == hsr[r])
                            atomicAdd(&hist[(x & 0xFFu) * kSelPairs + 4 * qd + (r >> 1)], 1u << (16 * (r & 1)));
                    }
                }
            }
        }
        __syncthreads();
        if (tid < rows) {
            uint32_t t32 = 0;
            if (n_row[tid] > k) {
                uint32_t cum = 0, lo = 0;
                for (int b = 255; b >= 0; --b) {
                    const uint32_t cb = (hist[b * kSelPairs + (tid >> 1)] >> ((tid & 1) * 16)) & 0xFFFFu;
                    if (cum + cb >= need[tid]) {
                        lo = b;
                        break;
                    }
                    cum += cb;
                }
                t32 = ((sel_hi[tid] << 8) | lo) << 16;
            }
            tau_u[tid] = t32;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- sort
//
// One warp per row. The candidate pass stores (raw score bits, index) pairs;
// the row's answer is its k_eff largest composite keys (order key of
// raw * scale, then the smaller index) in descending order.
//  1. Radix select (MSB first, 8-bit digits) over the 32-bit score order keys
//     held in registers finds the k_eff-th largest score T: a digit all
//     candidates share is skipped without a histogram (found from the OR and
//     AND of all keys), and the search stops as soon as the remaining rank
//     fills a whole bin.
//  2. The candidates above T, and of those equal to T the ones with the
//     smallest indices (rank by index among the ties, which sit in a short
//     shared-memory list), are compacted into shared memory as composite keys
//     (the index is read back from the candidate list) and sorted descending
//     by a bitonic network in registers (strides below E inside a lane, the
//     others across lanes by shuffles). With more ties at T than the list
//     holds, a radix select over their indices picks the winners instead.
// Keys live in registers batch-major: register b of lane l holds element
// 32*b + l.
constexpr int kSortWarps = 8;
constexpr int kMaxTies = 256;

template <int E, int STRIDE>
SSA_DEVINL void bitonic_stage_in_lane(uint64_t (&x)[E], int lane, int size) {
#pragma unroll
    for (int r = 0; r < E; ++r) {
        if ((r & STRIDE) == 0) {
            const int e = lane * E + r;
            const bool desc = (e & size) == 0;
            const uint64_t a = x[r], b = x[r + STRIDE];
            if ((a < b) == desc) {
                x[r] = b;
                x[r + STRIDE] = a;
            }
        }
    }
}

// All in-lane stages of a merge of `size` elements (strides E/2 .. 1).
template <int E>
SSA_DEVINL void bitonic_in_lane_tail(uint64_t (&x)[E], int lane, int size) {
    if constexpr (E >= 16) bitonic_stage_in_lane<E, 8>(x, lane, size);
    if constexpr (E >= 8) bitonic_stage_in_lane<E, 4>(x, lane, size);
    if constexpr (E >= 4) bitonic_stage_in_lane<E, 2>(x, lane, size);
    if constexpr (E >= 2) bitonic_stage_in_lane<E, 1>(x, lane, size);
}

// Sorts the 32*E keys of a warp in descending order (bitonic network).
// Merges up to E elements run inside each lane (unrolled); for larger merges
// the cross-lane strides (>= E, by shuffles) run as a loop and the in-lane
// tail is shared, which keeps the code small enough for the instruction cache.
template <int E>
SSA_DEVINL void warp_bitonic_desc(uint64_t (&x)[E], int lane) {
    constexpr int N = 32 * E;
    if constexpr (E >= 2) {
        bitonic_stage_in_lane<E, 1>(x, lane, 2);
    }
    if constexpr (E >= 4) {
        bitonic_stage_in_lane<E, 2>(x, lane, 4);
        bitonic_stage_in_lane<E, 1>(x, lane, 4);
    }
    if constexpr (E >= 8) {
        bitonic_stage_in_lane<E, 4>(x, lane, 8);
        bitonic_stage_in_lane<E, 2>(x, lane, 8);
        bitonic_stage_in_lane<E, 1>(x, lane, 8);
    }
    if constexpr (E >= 16) {
        bitonic_stage_in_lane<E, 8>(x, lane, 16);
        bitonic_stage_in_lane<E, 4>(x, lane, 16);
        bitonic_stage_in_lane<E, 2>(x, lane, 16);
        bitonic_stage_in_lane<E, 1>(x, lane, 16);
    }
#pragma unroll 1
    for (int size = 2 * E; size <= N; size <<= 1) {
#pragma unroll 1
        for (int stride = size >> 1; stride >= E; stride >>= 1) {
            const int lx = stride / E;
            const bool lower = (lane & lx) == 0;
            const bool desc = ((lane * E) & size) == 0;   // the same for all r of the lane
            const bool take_max = lower == desc;
#pragma unroll
            for (int r = 0; r < E; ++r) {
                const uint64_t y = __shfl_xor_sync(0xffffffffu, x[r], lx);
                const bool y_big = y > x[r];
                x[r] = (take_max == y_big) ? y : x[r];
            }
        }
        bitonic_in_lane_tail<E>(x, lane, size);
    }
}

template <int NB, int E>   // NB batches of 32 candidates; E = winners per lane (32E >= k)
__global__ void __launch_bounds__(kSortWarps * 32, 4) cand_sort_kernel(
    const uint64_t* __restrict__ cand, const int32_t* __restrict__ cnt, int64_t rows, int Tq,
    int Tk, int k, int causal, float scale, int32_t* __restrict__ idx_out,
    float* __restrict__ score_out, int64_t* __restrict__ ovf_list,
    int32_t* __restrict__ ovf_count, int32_t* dev_status) {
    constexpr int CAP = 32 * NB;      // two lists of CAP/2
    constexpr int CAPC = CAP / 2;
    constexpr int W = 32 * E;         // sorted winners
    __shared__ uint32_t bins_all[kSortWarps][256];   // histogram, then the list of ties
    __shared__ uint64_t win_all[kSortWarps][W];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const uint32_t below = (1u << lane) - 1;
    uint32_t* bins = bins_all[wid];
    uint64_t* win = win_all[wid];
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kSortWarps + wid;
    if (row >= rows) return;
    const int i = static_cast<int>(row % Tq);
    const int n = tile_valid_count(i, Tq, Tk, causal);
    const int keff = min(k, n);
    const int c0 = n > 0 ? cnt[row * 2] : 0, c1 = n > 0 ? cnt[row * 2 + 1] : 0;
    if (c0 > CAPC || c1 > CAPC) {   // redone by the row-wise kernel (informational status)
        if (lane == 0) {
            ovf_list[atomicAdd(ovf_count, 1)] = row;
            report(dev_status, SSA_DEV_OVERFLOW);
        }
        return;
    }
    const int c = c0 + c1;
    const uint64_t* src = cand + row * CAP;
    // element e of the row: list 0 holds e < c0, list 1 the rest
    auto elem = [&](int e) -> uint64_t { return e < c0 ? src[e] : src[CAPC + e - c0]; };
    uint32_t ok[NB];   // score order keys; 0 (below every real key) for no element
    uint32_t kor = 0, kand = ~0u;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const int e = 32 * b + lane;
        ok[b] = 0;
        if (e < c) {
            ok[b] = f32_order_key(__uint_as_float(static_cast<uint32_t>(elem(e) >> 32)) * scale);
            kor |= ok[b];
            kand &= ok[b];
        }
    }
    // 1. radix select of the keff-th largest score key T
    uint32_t thr = 0;        // winners: keys >= thr (all of them) ...
    bool partial = false;    // ... or keys > thr plus `need` of the keys == thr
    uint32_t need = static_cast<uint32_t>(keff);
    if (keff > 0 && keff < c) {
        const uint32_t vary = __reduce_or_sync(0xffffffffu, kor) ^ __reduce_and_sync(0xffffffffu, kand);
        const uint32_t same = __reduce_and_sync(0xffffffffu, kand);
        uint32_t prefix = 0, pmask = 0, inbin = static_cast<uint32_t>(c);
        bool whole = false;
        for (int d = 3; d >= 0; --d) {
            const int sh = 8 * d;
            const uint32_t dm = 0xFFu << sh;
            if ((vary & dm) == 0) {   // every candidate has this digit
                prefix |= same & dm;
                pmask |= dm;
                continue;
            }
            for (int t = lane; t < 256; t += 32) bins[t] = 0;
            __syncwarp();
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (32 * b >= c) break;
                if (32 * b + lane < c && (ok[b] & pmask) == prefix) atomicAdd(&bins[(ok[b] >> sh) & 0xFFu], 1u);
            }
            __syncwarp();
            // bin holding the need-th largest: lane l owns bins 255-8l .. 248-8l
            uint32_t cb[8], tot = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                cb[q] = bins[255 - 8 * lane - q];
                tot += cb[q];
            }
            uint32_t incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t excl = incl - tot;
            uint32_t sel = 0, above = 0, cnt_sel = 0;
            const bool mine = excl < need && need <= incl;
            if (mine) {
                uint32_t a = excl;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (a + cb[q] >= need) {
                        sel = 255 - 8 * lane - q;
                        above = a;
                        cnt_sel = cb[q];
                        break;
                    }
                    a += cb[q];
                }
            }
            const unsigned who = __ballot_sync(0xffffffffu, mine);
            const int src_lane = __ffs(who) - 1;
            sel = __shfl_sync(0xffffffffu, sel, src_lane);
            above = __shfl_sync(0xffffffffu, above, src_lane);
            inbin = __shfl_sync(0xffffffffu, cnt_sel, src_lane);
            __syncwarp();
            prefix |= sel << sh;
            pmask |= dm;
            need -= above;
            if (inbin == need) {   // the whole bin is selected: keys >= its lowest key
                whole = true;
                break;
            }
        }
        thr = prefix;   // digits below the last fixed one are zero
        // every digit fixed and only part of the keys equal to T selected
        partial = !whole && need < inbin;
    }
    // 2. compact the winners into shared memory (swizzled: the sort's lane
    //    pl reads its register pr at pl*E + (pr ^ (pl % E)), free of bank
    //    conflicts); the ties at T go to a list first
    int base = 0, nties = 0;
    uint32_t* ties = bins;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        if (32 * b >= c) break;
        const int e = 32 * b + lane;
        const bool valid = e < c;
        const bool up = valid && (partial ? ok[b] > thr : ok[b] >= thr);
        const bool tie = partial && valid && ok[b] == thr;
        const unsigned mu = __ballot_sync(0xffffffffu, up);
        const unsigned mt = __ballot_sync(0xffffffffu, tie);
        if (up || tie) {
            const uint32_t j = static_cast<uint32_t>(elem(e));
            if (up) {
                const int pos = base + __popc(mu & below);
                const int pl = pos / E, pr = pos % E;
                if (pos < W) win[pl * E + (pr ^ (pl % E))] = sel_key(ok[b], j);
            } else {
                const int tp = nties + __popc(mt & below);
                if (tp < kMaxTies) ties[tp] = j;
            }
        }
        base += __popc(mu);
        nties += __popc(mt);
    }
    if (partial && nties > kMaxTies) {
        // More ties at T than the short list holds (heavy ties, e.g. equal
        // scores): the `need` smallest indices among them by a radix select
        // over the index bits, most significant digit first, digits that all
        // ties share skipped; the winners are then the ties with an index <= J.
        // (the candidates are read again rather than kept in registers, which
        // keeps this rare path from costing the common one registers)
        auto tie_index = [&](int e, uint32_t& j) -> bool {
            if (e >= c) return false;
            const uint64_t v = elem(e);
            j = static_cast<uint32_t>(v);
            return f32_order_key(__uint_as_float(static_cast<uint32_t>(v >> 32)) * scale) == thr;
        };
        uint32_t jor = 0, jand = ~0u;
        for (int e = lane; e < c; e += 32) {
            uint32_t j;
            if (tie_index(e, j)) {
                jor |= j;
                jand &= j;
            }
        }
        jand = __reduce_and_sync(0xffffffffu, jand);
        const uint32_t jvary = __reduce_or_sync(0xffffffffu, jor) ^ jand;
        uint32_t jpre = 0, jmask = 0, rem = need;
        for (int d = 3; d >= 0; --d) {
            const int sh = 8 * d;
            const uint32_t dm = 0xFFu << sh;
            if ((jvary & dm) == 0) {
                jpre |= jand & dm;
                jmask |= dm;
                continue;
            }
            for (int t = lane; t < 256; t += 32) bins[t] = 0;
            __syncwarp();
            for (int e = lane; e < c; e += 32) {
                uint32_t j;
                if (tie_index(e, j) && (j & jmask) == jpre) atomicAdd(&bins[(j >> sh) & 0xFFu], 1u);
            }
            __syncwarp();
            // the smallest digit whose running count reaches rem: lane l owns
            // bins 8l .. 8l+7
            uint32_t cb[8], tot = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                cb[q] = bins[8 * lane + q];
                tot += cb[q];
            }
            uint32_t incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t excl = incl - tot;
            uint32_t sel = 0, lower = 0, cnt_sel = 0;
            const bool mine = excl < rem && rem <= incl;
            if (mine) {
                uint32_t a = excl;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (a + cb[q] >= rem) {
                        sel = 8 * lane + q;
                        lower = a;
                        cnt_sel = cb[q];
                        break;
                    }
                    a += cb[q];
                }
            }
            const int src_lane = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
            sel = __shfl_sync(0xffffffffu, sel, src_lane);
            lower = __shfl_sync(0xffffffffu, lower, src_lane);
            cnt_sel = __shfl_sync(0xffffffffu, cnt_sel, src_lane);
            __syncwarp();
            jpre |= sel << sh;
            jmask |= dm;
            rem -= lower;
            if (cnt_sel == rem) break;   // the whole bin wins: any lower digits
        }
        const uint32_t J = jpre | ~jmask;
        for (int e0 = 0; e0 < c; e0 += 32) {
            uint32_t j = 0;
            const bool w = tie_index(e0 + lane, j) && j <= J;
            const unsigned mw = __ballot_sync(0xffffffffu, w);
            if (w) {
                const int pos = base + __popc(mw & below);
                const int pl = pos / E, pr = pos % E;
                if (pos < W) win[pl * E + (pr ^ (pl % E))] = sel_key(thr, j);
            }
            base += __popc(mw);
        }
    } else if (partial) {
        __syncwarp();
        // a tie wins iff fewer than `need` ties have a smaller index
        for (int q0 = 0; q0 < nties; q0 += 32) {
            const int q = q0 + lane;
            bool w = false;
            uint32_t j = 0;
            if (q < nties) {
                j = ties[q];
                uint32_t rank = 0;
                for (int r = 0; r < nties; ++r) rank += ties[r] < j;
                w = rank < need;
            }
            const unsigned mw = __ballot_sync(0xffffffffu, w);
            if (w) {
                const int pos = base + __popc(mw & below);
                const int pl = pos / E, pr = pos % E;
                if (pos < W) win[pl * E + (pr ^ (pl % E))] = sel_key(thr, j);
            }
            base += __popc(mw);
        }
    }
    __syncwarp();
    uint64_t y[E];
#pragma unroll
    for (int r = 0; r < E; ++r) {
        const int e = lane * E + r;
        y[r] = e < keff ? win[lane * E + (r ^ (lane % E))] : 0ull;   // swizzled: no bank conflicts
    }
    warp_bitonic_desc<E>(y, lane);
    int32_t* io = idx_out + row * k;
    float* so = score_out ? score_out + row * k : nullptr;
    const int e0 = lane * E;   // this lane's E consecutive outputs
    bool vec = false;
    if constexpr (E % 4 == 0)
        vec = e0 + E <= k && (reinterpret_cast<uintptr_t>(io + e0) & 15) == 0 &&
              (so == nullptr || (reinterpret_cast<uintptr_t>(so + e0) & 15) == 0);
    if (vec) {   // 16-byte stores: a quarter of the store requests
#pragma unroll
        for (int r4 = 0; r4 < E; r4 += 4) {
            int32_t iv[4];
            float sv[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const bool in = e0 + r4 + t < keff;
                iv[t] = in ? static_cast<int32_t>(sel_key_index(y[r4 + t])) : -1;
                sv[t] = in ? order_key_f32(sel_key_okey(y[r4 + t])) : -INFINITY;
            }
            *reinterpret_cast<int4*>(io + e0 + r4) = make_int4(iv[0], iv[1], iv[2], iv[3]);
            if (so) *reinterpret_cast<float4*>(so + e0 + r4) = make_float4(sv[0], sv[1], sv[2], sv[3]);
        }
    } else {
#pragma unroll
        for (int r = 0; r < E; ++r) {
            const int e = e0 + r;
            if (e < k) {
                if (e < keff) {
                    io[e] = static_cast<int32_t>(sel_key_index(y[r]));
                    if (so) so[e] = order_key_f32(sel_key_okey(y[r]));
                } else {
                    io[e] = -1;
                    if (so) so[e] = -INFINITY;
                }
            }
        }
    }
}

#ifndef SSA_HOST_EMULATION   // the CPU tests launch the kernels themselves
cudaError_t tile_select_launch(const uint16_t* gm, uint32_t* tau, int BH, int Tq, int Tk, int k,
                               int causal, cudaStream_t stream) {
    const int items = 2 * BH * ((Tq + kUnitM - 1) / kUnitM);
    if (items == 0) return cudaSuccess;
    const int sms = tile_sm_count();
    const int grid = items < 3 * sms ? items : 3 * sms;
    constexpr int kHistBytes = 256 * kSelPairs * 4;
    cudaError_t e = set_max_dyn_smem(reinterpret_cast<const void*>(group_select_kernel), kHistBytes);
    if (e != cudaSuccess) return e;
    TraceLaunch tr("group_select", stream);
    group_select_kernel<<<grid, kSelThreads, kHistBytes, stream>>>(gm, tau, BH, Tq, Tk, k, causal,
                                                                   tile_group_stride(k));
    return cudaGetLastError();
}

cudaError_t tile_sort_launch(const uint64_t* cand, const int32_t* cnt, int64_t rows, int Tq,
                             int Tk, int k, int causal, float scale, int32_t* idx, float* score,
                             int64_t* ovf_list, int32_t* ovf_count, int32_t* dev_status,
                             cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = (rows + kSortWarps - 1) / kSortWarps;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int cap = tile_cand_cap(k);   // 2 * pow2ceil(k), at least 64
    TraceLaunch tr("cand_sort", stream);
#define SSA_SORT_CASE(NB)                                                                      \
    if (cap == 32 * NB) {                                                                      \
        cand_sort_kernel<NB, NB / 2><<<static_cast<unsigned>(blocks), kSortWarps * 32, 0,      \
                                       stream>>>(cand, cnt, rows, Tq, Tk, k, causal, scale,    \
                                                 idx, score, ovf_list, ovf_count, dev_status); \
        return cudaGetLastError();                                                             \
    }
    SSA_SORT_CASE(2)
    SSA_SORT_CASE(4)
    SSA_SORT_CASE(8)
    SSA_SORT_CASE(16)
    SSA_SORT_CASE(32)
#undef SSA_SORT_CASE
    return cudaErrorInvalidValue;
}
#endif  // SSA_HOST_EMULATION

}  // namespace ssa
