// Row-wise exact score + top-k: one CTA per query row.
//
// Scores S_j = fp32(q_low . k_low_j) * scale of every valid key are written as
// order-preserving 32-bit keys into the row's workspace slot; an MSB-first
// radix select (four 8-bit digits) finds the exact k-th largest key value v;
// the row's selection is every key above v plus, in ascending index order, as
// many keys equal to v as are still needed (the lower index wins a tie); a
// bitonic sort on the composite key (score, ~index) orders the selection.
// (mhpq.cn/news/1098205, section 2.2 scorer and section 3.2 torch.topk with
// top_k = min(top_k, seq_len) and masked keys never selected.)
//
// This kernel serves the decode shape (few query rows, long key rows), the
// rows the fused tensor-core path hands back, and any shape without a fused
// path. The dot products use the same lane layout as the gather kernel: L
// lanes share one 16-byte-sliced key row, a transpose-reduction leaves one
// score per lane.
#ifdef SSA_HOST_EMULATION
#include "emu_device.h"   // the host stand-in of the CPU tests (tests/emu)
#else
#include "common.cuh"
#include "trace.h"
#endif

namespace ssa {

constexpr int TOPK_THREADS = 512;
constexpr int TOPK_WARPS = TOPK_THREADS / 32;
constexpr int TOPK_KMAX = 2048;

template <int L>
SSA_DEVINL float transpose_reduce_t(float (&part)[L], int lane) {
#pragma unroll
    for (int o = L / 2; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int m = 0; m < o; ++m) {
            float send = upper ? part[m] : part[m + o];
            float keep = upper ? part[m + o] : part[m];
            part[m] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return part[0];
}

// Warp-aggregated shared-memory histogram increment.
SSA_DEVINL void hist_add(uint32_t* hist, uint32_t bin, bool active) {
    const unsigned act = __ballot_sync(0xffffffffu, active);
    if (!active) return;
    const unsigned peers = __match_any_sync(act, bin);
    const int leader = __ffs(peers) - 1;
    if ((threadIdx.x & 31) == leader) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

struct SelectState {
    uint32_t prefix;    // digits fixed so far (in the high bits)
    uint32_t need;      // selected keys still needed at or below the prefix
    int shift;          // bit position of the next digit
    int done;           // 1: every key >= thresh is selected, no tie handling
    uint32_t thresh;    // selection threshold key (valid once done or shift < 0)
};

// One warp finds the digit whose bin contains the need-th largest key.
// hist[256] holds this pass's counts.
SSA_DEVINL void pick_digit(const uint32_t* hist, SelectState* st) {
    const int lane = threadIdx.x & 31;
    // lane l owns bins 255-8l .. 248-8l (descending)
    uint32_t c[8];
    uint32_t tot = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        c[b] = hist[255 - 8 * lane - b];
        tot += c[b];
    }
    // exclusive prefix over lanes (counts of all higher bins)
    uint32_t incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const uint32_t excl = incl - tot;
    const uint32_t need = st->need;
    const bool mine = excl < need && need <= incl;
    if (mine) {
        uint32_t above = excl;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            if (above + c[b] >= need) {
                const uint32_t digit = 255 - 8 * lane - b;
                const uint32_t in_bin = c[b];
                const uint32_t need_in = need - above;
                const uint32_t prefix = st->prefix | (digit << st->shift);
                st->prefix = prefix;
                st->need = need_in;
                if (in_bin == need_in) {     // the whole bin is selected
                    st->done = 1;
                    st->thresh = prefix;
                } else if (st->shift == 0) { // exact value found
                    st->done = 0;
                    st->thresh = prefix;
                }
                st->shift -= 8;
                break;
            }
            above += c[b];
        }
    }
}

template <bool BF16, int P>
struct ScoreGeom {
    static constexpr int ESIZE = BF16 ? 2 : 4;
    static constexpr int R = P * ESIZE;
    static constexpr int L = R / 16;
    static constexpr int G = 32 / L;
    static constexpr int E = 16 / ESIZE;
};

template <bool BF16, int P>
__global__ void __launch_bounds__(TOPK_THREADS) topk_rows_kernel(
    const void* __restrict__ q_low, const void* __restrict__ k_low, const int64_t* __restrict__ row_list,
    int64_t rows, const int32_t* __restrict__ rows_dev, int Tq, int Tk, int k, int causal,
    float scale, int32_t* __restrict__ idx_out, float* __restrict__ score_out,
    uint32_t* __restrict__ ws, int64_t ws_stride) {
    using Gm = ScoreGeom<BF16, P>;
    constexpr int L = Gm::L, G = Gm::G, E = Gm::E, R = Gm::R;
    __shared__ uint32_t hist[256];
    __shared__ uint64_t sel[TOPK_KMAX];
    __shared__ SelectState st;
    __shared__ uint32_t n_sel;
    __shared__ uint32_t warp_cnt[TOPK_WARPS];
    __shared__ uint32_t tie_base;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane / L, s = lane % L;
    uint32_t* wrow = ws + (int64_t)blockIdx.x * ws_stride;
    if (rows_dev) rows = *rows_dev;   // row count known only on the device

    for (int64_t rr = blockIdx.x; rr < rows; rr += gridDim.x) {
        const int64_t row = row_list ? row_list[rr] : rr;
        const int64_t bh = row / Tq;
        const int i = (int)(row - bh * Tq);
        int nv = Tk;
        if (causal) {
            const int64_t last = (int64_t)i + (Tk - Tq);
            nv = last < 0 ? 0 : (last + 1 < (int64_t)Tk ? (int)(last + 1) : Tk);
        }
        const int keff = min(nv, k);

        float q[E];
        Vec16<BF16>::to_f32(ldg16(reinterpret_cast<const char*>(q_low) + row * R + s * 16), q);
        const char* Kb = reinterpret_cast<const char*>(k_low) + bh * (int64_t)Tk * R + s * 16;

        if (tid < 256) hist[tid] = 0;
        if (tid == 0) {
            st.prefix = 0;
            st.need = (uint32_t)keff;
            st.shift = 24;
            st.done = 0;
            st.thresh = 0;
            n_sel = 0;
            if (nv <= k) {   // every valid key is selected
                st.done = 1;
                st.thresh = 0;
                st.shift = -8;
            }
        }
        __syncthreads();
        const bool need_select = !(nv <= k);

        // ---- scores (+ histogram of the top digit)
        for (int c0 = warp * 32; c0 < nv; c0 += TOPK_WARPS * 32) {
            float part[L];
            uint4 kv[L];
#pragma unroll
            for (int r = 0; r < L; ++r) {
                int j = c0 + r * G + g;
                j = j < nv ? j : 0;
                kv[r] = ldg16(Kb + (int64_t)j * R);
            }
#pragma unroll
            for (int r = 0; r < L; ++r) {
                float kf[E];
                Vec16<BF16>::to_f32(kv[r], kf);
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) a = fmaf(q[e], kf[e], a);
                part[r] = a;
            }
            const float dot = transpose_reduce_t<L>(part, lane);
            const int j = c0 + s * G + g;
            const uint32_t key = f32_order_key(dot * scale);
            const bool valid = j < nv;
            if (valid) wrow[j] = key;
            if (need_select) hist_add(hist, key >> 24, valid);
        }
        __syncthreads();

        // ---- radix select over the remaining digits
        if (need_select) {
            for (int pass = 0; pass < 4; ++pass) {
                if (warp == 0) pick_digit(hist, &st);
                __syncthreads();
                if (st.done || st.shift < 0) break;
                if (tid < 256) hist[tid] = 0;
                __syncthreads();
                const int sh = st.shift;
                const uint32_t pre = st.prefix >> (sh + 8);
                for (int j0 = 0; j0 < nv; j0 += TOPK_THREADS) {
                    const int j = j0 + tid;
                    uint32_t key = j < nv ? wrow[j] : 0u;
                    const bool match = j < nv && (key >> (sh + 8)) == pre;
                    hist_add(hist, (key >> sh) & 0xFFu, match);
                }
                __syncthreads();
            }
        }
        __syncthreads();

        // ---- collect: keys above the threshold (or >= it when done)
        const uint32_t thr = st.thresh;
        const bool inclusive = st.done != 0;
        for (int j0 = 0; j0 < nv; j0 += TOPK_THREADS) {
            const int j = j0 + tid;
            const uint32_t key = j < nv ? wrow[j] : 0u;
            const bool take = j < nv && (inclusive ? key >= thr : key > thr);
            const unsigned b = __ballot_sync(0xffffffffu, take);
            uint32_t base = 0;
            if (lane == 0 && b) base = atomicAdd(&n_sel, (uint32_t)__popc(b));
            base = __shfl_sync(0xffffffffu, base, 0);
            const uint32_t slot = base + __popc(b & ((1u << lane) - 1));
            if (take && slot < (uint32_t)TOPK_KMAX) sel[slot] = sel_key(key, (uint32_t)j);
        }
        __syncthreads();
        // ---- ties at the exact k-th value: lowest indices first
        if (!inclusive) {
            const uint32_t need_eq = (uint32_t)keff - n_sel;
            if (tid == 0) tie_base = 0;
            __syncthreads();
            for (int j0 = 0; j0 < nv; j0 += TOPK_THREADS) {
                if (tie_base >= need_eq) break;   // uniform: read after a barrier
                const int j = j0 + tid;
                const bool eq = j < nv && wrow[j] == thr;
                const unsigned b = __ballot_sync(0xffffffffu, eq);
                if (lane == 0) warp_cnt[warp] = __popc(b);
                __syncthreads();
                uint32_t before = tie_base;
                for (int w = 0; w < warp; ++w) before += warp_cnt[w];
                const uint32_t rank = before + __popc(b & ((1u << lane) - 1));
                const uint32_t total_base = n_sel;
                if (eq && rank < need_eq && total_base + rank < (uint32_t)TOPK_KMAX)
                    sel[total_base + rank] = sel_key(thr, (uint32_t)j);
                __syncthreads();
                if (tid == 0) {
                    uint32_t t = 0;
                    for (int w = 0; w < TOPK_WARPS; ++w) t += warp_cnt[w];
                    tie_base += t;
                }
                __syncthreads();
            }
            __syncthreads();
        }

        // ---- sort the keff selected keys, descending
        int n2 = 1;
        while (n2 < keff) n2 <<= 1;
        for (int t = keff + tid; t < n2; t += TOPK_THREADS) sel[t] = 0ull;
        __syncthreads();
        for (int size = 2; size <= n2; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int t = tid; t < (n2 >> 1); t += TOPK_THREADS) {
                    const int lo = 2 * t - (t & (stride - 1));
                    const int hi = lo + stride;
                    const bool desc = (lo & size) == 0;
                    const uint64_t a = sel[lo], b2 = sel[hi];
                    if ((a < b2) == desc) {
                        sel[lo] = b2;
                        sel[hi] = a;
                    }
                }
                __syncthreads();
            }
        }

        // ---- write
        int32_t* io = idx_out + row * (int64_t)k;
        float* so = score_out ? score_out + row * (int64_t)k : nullptr;
        for (int t = tid; t < k; t += TOPK_THREADS) {
            if (t < keff) {
                const uint64_t key = sel[t];
                io[t] = (int32_t)sel_key_index(key);
                if (so) so[t] = order_key_f32(sel_key_okey(key));
            } else {
                io[t] = -1;
                if (so) so[t] = -INFINITY;
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------ long rows
//
// Rows with many keys and few rows to spread them over (decode: one query
// per head against a long key cache) run split into chunks of kChunkKeys
// keys, one CTA per (row, chunk), so that every SM streams k_low at once:
//   topk_chunk_kernel  scores its chunk into shared memory and selects the
//                      chunk's exact top-min(k, n) (same radix select and tie
//                      rule as the row kernel), written unordered as
//                      composite keys (score order key, ~index);
//   topk_merge_kernel  gathers the chunks' selections of a row, finds the
//                      k_eff largest by a radix select over the distinct
//                      composite keys and sorts those (bitonic, descending).
// A key of the row's top k has fewer than k keys ahead of it in the row,
// hence fewer than k in its chunk: it is in its chunk's selection, so the
// merge of the chunk selections holds the row's whole top k.
constexpr int kChunkKeys = 8192;
constexpr int kChunkThreads = 256;
constexpr int kChunkWarps = kChunkThreads / 32;
constexpr int kMergeMax = 4096;     // candidates a row's merge holds
constexpr int kMergeThreads = 512;

template <bool BF16, int P>
__global__ void __launch_bounds__(kChunkThreads, 4) topk_chunk_kernel(
    const void* __restrict__ q_low, const void* __restrict__ k_low, int nchunks, int Tq, int Tk,
    int k, int causal, float scale, uint64_t* __restrict__ cand, int32_t* __restrict__ cnt) {
    using Gm = ScoreGeom<BF16, P>;
    constexpr int L = Gm::L, G = Gm::G, E = Gm::E, R = Gm::R;
    __shared__ uint32_t skey[kChunkKeys];
    __shared__ uint32_t hist[256];
    __shared__ SelectState st;
    __shared__ uint32_t n_sel;
    __shared__ uint32_t warp_cnt[kChunkWarps];
    __shared__ uint32_t tie_base;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane / L, s = lane % L;
    const int64_t row = static_cast<int64_t>(blockIdx.x) / nchunks;
    const int c = static_cast<int>(static_cast<int64_t>(blockIdx.x) - row * nchunks);
    const int64_t bh = row / Tq;
    const int i = static_cast<int>(row - bh * Tq);
    int nv = Tk;
    if (causal) {
        const int64_t last = static_cast<int64_t>(i) + (Tk - Tq);
        nv = last < 0 ? 0 : (last + 1 < static_cast<int64_t>(Tk) ? static_cast<int>(last + 1) : Tk);
    }
    const int j_lo = c * kChunkKeys;
    const int n = max(0, min(kChunkKeys, nv - j_lo));   // this chunk's valid keys
    const int kcap = min(k, kChunkKeys);                // slots of a chunk's selection
    const int kc = min(k, n);
    uint64_t* out = cand + static_cast<int64_t>(blockIdx.x) * kcap;
    if (tid == 0) cnt[blockIdx.x] = kc;
    if (n == 0) return;

    float q[E];
    Vec16<BF16>::to_f32(ldg16(reinterpret_cast<const char*>(q_low) + row * R + s * 16), q);
    const char* Kb = reinterpret_cast<const char*>(k_low) + (bh * static_cast<int64_t>(Tk) + j_lo) * R +
                     s * 16;
    const bool need_select = n > kc;
    if (tid < 256) hist[tid] = 0;
    if (tid == 0) {
        st.prefix = 0;
        st.need = static_cast<uint32_t>(kc);
        st.shift = 24;
        st.done = need_select ? 0 : 1;
        st.thresh = 0;
        n_sel = 0;
    }
    __syncthreads();

    // ---- scores of the chunk (+ histogram of the top digit)
    for (int c0 = warp * 32; c0 < n; c0 += kChunkWarps * 32) {
        float part[L];
        uint4 kv[L];
#pragma unroll
        for (int r = 0; r < L; ++r) {
            int j = c0 + r * G + g;
            j = j < n ? j : 0;
            kv[r] = ldg16(Kb + static_cast<int64_t>(j) * R);
        }
#pragma unroll
        for (int r = 0; r < L; ++r) {
            float kf[E];
            Vec16<BF16>::to_f32(kv[r], kf);
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) a = fmaf(q[e], kf[e], a);
            part[r] = a;
        }
        const float dot = transpose_reduce_t<L>(part, lane);
        const int j = c0 + s * G + g;
        const uint32_t key = f32_order_key(dot * scale);
        const bool valid = j < n;
        if (valid) skey[j] = key;
        if (need_select) hist_add(hist, key >> 24, valid);
    }
    __syncthreads();

    // ---- radix select over the remaining digits (keys in shared memory)
    if (need_select) {
        for (int pass = 0; pass < 4; ++pass) {
            if (warp == 0) pick_digit(hist, &st);
            __syncthreads();
            if (st.done || st.shift < 0) break;
            if (tid < 256) hist[tid] = 0;
            __syncthreads();
            const int sh = st.shift;
            const uint32_t pre = st.prefix >> (sh + 8);
            for (int j0 = 0; j0 < n; j0 += kChunkThreads) {
                const int j = j0 + tid;
                const uint32_t key = j < n ? skey[j] : 0u;
                const bool match = j < n && (key >> (sh + 8)) == pre;
                hist_add(hist, (key >> sh) & 0xFFu, match);
            }
            __syncthreads();
        }
    }
    __syncthreads();

    // ---- keys above the threshold (or >= it when the whole bin is taken)
    const uint32_t thr = st.thresh;
    const bool inclusive = st.done != 0;
    for (int j0 = 0; j0 < n; j0 += kChunkThreads) {
        const int j = j0 + tid;
        const uint32_t key = j < n ? skey[j] : 0u;
        const bool take = j < n && (inclusive ? key >= thr : key > thr);
        const unsigned b = __ballot_sync(0xffffffffu, take);
        uint32_t base = 0;
        if (lane == 0 && b) base = atomicAdd(&n_sel, static_cast<uint32_t>(__popc(b)));
        base = __shfl_sync(0xffffffffu, base, 0);
        const uint32_t slot = base + __popc(b & ((1u << lane) - 1));
        if (take && slot < static_cast<uint32_t>(kcap))
            out[slot] = sel_key(key, static_cast<uint32_t>(j_lo + j));
    }
    __syncthreads();
    // ---- ties at the exact kc-th value: lowest indices first
    if (!inclusive) {
        const uint32_t need_eq = static_cast<uint32_t>(kc) - n_sel;
        if (tid == 0) tie_base = 0;
        __syncthreads();
        for (int j0 = 0; j0 < n; j0 += kChunkThreads) {
            if (tie_base >= need_eq) break;   // uniform: read after a barrier
            const int j = j0 + tid;
            const bool eq = j < n && skey[j] == thr;
            const unsigned b = __ballot_sync(0xffffffffu, eq);
            if (lane == 0) warp_cnt[warp] = __popc(b);
            __syncthreads();
            uint32_t before = tie_base;
            for (int w = 0; w < warp; ++w) before += warp_cnt[w];
            const uint32_t rank = before + __popc(b & ((1u << lane) - 1));
            const uint32_t total_base = n_sel;
            if (eq && rank < need_eq && total_base + rank < static_cast<uint32_t>(kcap))
                out[total_base + rank] = sel_key(thr, static_cast<uint32_t>(j_lo + j));
            __syncthreads();
            if (tid == 0) {
                uint32_t t = 0;
                for (int w = 0; w < kChunkWarps; ++w) t += warp_cnt[w];
                tie_base += t;
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(
    const uint64_t* __restrict__ cand, const int32_t* __restrict__ cnt, int nchunks, int Tq,
    int Tk, int k, int causal, int32_t* __restrict__ idx_out, float* __restrict__ score_out) {
    constexpr int KPT = kMergeMax / kMergeThreads;   // candidates per thread
    __shared__ uint64_t buf[kMergeMax];   // the candidates, then the winners
    __shared__ uint32_t hist[256];
    __shared__ int off[65];
    __shared__ uint64_t s_prefix;
    __shared__ int s_need, s_done;
    __shared__ uint32_t n_win;
    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t row = blockIdx.x;
    const int i = static_cast<int>(row % Tq);
    int nv = Tk;
    if (causal) {
        const int64_t last = static_cast<int64_t>(i) + (Tk - Tq);
        nv = last < 0 ? 0 : (last + 1 < static_cast<int64_t>(Tk) ? static_cast<int>(last + 1) : Tk);
    }
    const int keff = min(k, nv);
    const int kcap = min(k, kChunkKeys);
    if (tid == 0) {   // where each chunk's selection goes (nchunks <= 64)
        int o = 0;
        for (int c = 0; c < nchunks; ++c) {
            off[c] = o;
            o += cnt[row * nchunks + c];
        }
        off[nchunks] = o;
        s_prefix = 0;
        s_need = keff;
        s_done = 0;
        n_win = 0;
    }
    __syncthreads();
    const int total = off[nchunks];   // <= nchunks * kcap <= kMergeMax, >= keff
    for (int c = 0; c < nchunks; ++c) {
        const uint64_t* src = cand + (row * nchunks + c) * static_cast<int64_t>(kcap);
        const int m = off[c + 1] - off[c];
        for (int t = tid; t < m; t += kMergeThreads) buf[off[c] + t] = src[t];
    }
    __syncthreads();
    uint64_t mine[KPT];   // candidate t0*kMergeThreads + tid of the row, 0 past the last
#pragma unroll
    for (int r = 0; r < KPT; ++r) {
        const int t = r * kMergeThreads + tid;
        mine[r] = t < total ? buf[t] : 0ull;
    }
    __syncthreads();   // every thread holds its candidates before buf is reused
    // The composite keys are distinct (they hold the index), so the keff-th
    // largest is unique: a radix select over its 8-bit digits, most
    // significant first, stops as soon as the remaining rank fills a bin;
    // the winners are then every key at or above the prefix found.
    if (keff < total) {
        for (int sh = 56; sh >= 0; sh -= 8) {
            if (tid < 256) hist[tid] = 0;
            __syncthreads();
            const uint64_t pre = s_prefix;
#pragma unroll
            for (int r = 0; r < KPT; ++r) {
                const int t = r * kMergeThreads + tid;
                const uint64_t key = mine[r];
                const bool match = t < total && (sh == 56 || (key >> (sh + 8)) == (pre >> (sh + 8)));
                hist_add(hist, static_cast<uint32_t>((key >> sh) & 0xFFu), match);
            }
            __syncthreads();
            if (tid < 32) {   // the bin holding the need-th largest: lane l owns bins 255-8l ..
                uint32_t c8[8], tot = 0;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    c8[q] = hist[255 - 8 * lane - q];
                    tot += c8[q];
                }
                uint32_t incl = tot;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const uint32_t need = static_cast<uint32_t>(s_need);
                uint32_t above = incl - tot;
                if (above < need && need <= incl) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        if (above + c8[q] >= need) {
                            const uint32_t d = 255u - 8u * lane - q;
                            s_prefix = pre | (static_cast<uint64_t>(d) << sh);
                            s_need = static_cast<int>(need - above);
                            s_done = c8[q] == need - above;   // the whole bin is taken
                            break;
                        }
                        above += c8[q];
                    }
                }
            }
            __syncthreads();
            if (s_done) break;
        }
    }
    // winners: every key at or above the prefix (exactly keff of them),
    // compacted to the front of buf (the candidates are in registers now)
    const uint64_t thr = keff < total ? s_prefix : 0ull;
    uint64_t* win = buf;
#pragma unroll
    for (int r = 0; r < KPT; ++r) {
        const int t = r * kMergeThreads + tid;
        const bool take = t < total && mine[r] >= thr;
        const unsigned b = __ballot_sync(0xffffffffu, take);
        uint32_t base = 0;
        if (lane == 0 && b) base = atomicAdd(&n_win, static_cast<uint32_t>(__popc(b)));
        base = __shfl_sync(0xffffffffu, base, 0);
        const uint32_t slot = base + __popc(b & ((1u << lane) - 1));
        if (take && slot < static_cast<uint32_t>(TOPK_KMAX)) win[slot] = mine[r];
    }
    __syncthreads();
    // sort the winners descending (bitonic over the next power of two)
    int n2 = 1;
    while (n2 < keff) n2 <<= 1;
    for (int t = keff + tid; t < n2; t += kMergeThreads) win[t] = 0ull;   // below every key
    __syncthreads();
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = tid; t < (n2 >> 1); t += kMergeThreads) {
                const int lo = 2 * t - (t & (stride - 1));
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const uint64_t a = win[lo], b = win[hi];
                if ((a < b) == desc) {
                    win[lo] = b;
                    win[hi] = a;
                }
            }
            __syncthreads();
        }
    }
    int32_t* io = idx_out + row * static_cast<int64_t>(k);
    float* so = score_out ? score_out + row * static_cast<int64_t>(k) : nullptr;
    for (int t = tid; t < k; t += kMergeThreads) {
        if (t < keff) {
            const uint64_t key = win[t];
            io[t] = static_cast<int32_t>(sel_key_index(key));
            if (so) so[t] = order_key_f32(sel_key_okey(key));
        } else {
            io[t] = -1;
            if (so) so[t] = -INFINITY;
        }
    }
}

// Chunks per row of Tk keys, or 0 when the chunked path does not apply
// (short rows, or more candidates than a row's merge holds).
inline int topk_chunk_count(int Tk, int k) {
    if (Tk < 2 * kChunkKeys) return 0;
    const int nchunks = (Tk + kChunkKeys - 1) / kChunkKeys;
    const int kcap = k < kChunkKeys ? k : kChunkKeys;
    if (nchunks > 64 || static_cast<int64_t>(nchunks) * kcap > kMergeMax) return 0;
    return nchunks;
}

#ifndef SSA_HOST_EMULATION   // the CPU tests launch the kernel themselves
// rows_dev != NULL: the number of rows of row_list is read on the device
// (at most `rows`), so a list built by an earlier kernel needs no host sync.
cudaError_t topk_rows_dispatch(const void* q_low, const void* k_low, bool bf16, int P,
                               const int64_t* row_list, int64_t rows, const int32_t* rows_dev,
                               int Tq, int Tk, int k, int causal, float scale, int32_t* idx,
                               float* score, uint32_t* ws, int64_t ws_slots, int64_t ws_stride,
                               cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const int64_t grid = rows < ws_slots ? rows : ws_slots;
    TraceLaunch tr("topk_rows", stream);
#define SSA_TOPK_CASE(BF, PP)                                                                \
    if (bf16 == BF && P == PP) {                                                             \
        topk_rows_kernel<BF, PP><<<(unsigned)grid, TOPK_THREADS, 0, stream>>>(              \
            q_low, k_low, row_list, rows, rows_dev, Tq, Tk, k, causal, scale, idx, score, ws,  \
            ws_stride);                                                                      \
        return cudaGetLastError();                                                           \
    }
    SSA_TOPK_CASE(true, 16)
    SSA_TOPK_CASE(true, 32)
    SSA_TOPK_CASE(true, 64)
    SSA_TOPK_CASE(true, 128)
    SSA_TOPK_CASE(false, 16)
    SSA_TOPK_CASE(false, 32)
    SSA_TOPK_CASE(false, 64)
    SSA_TOPK_CASE(false, 128)
#undef SSA_TOPK_CASE
    return cudaErrorInvalidValue;
}

int topk_chunks_for(int Tk, int k) { return topk_chunk_count(Tk, k); }

size_t topk_chunks_workspace(int64_t rows, int Tk, int k) {
    const int nchunks = topk_chunk_count(Tk, k);
    if (nchunks == 0) return 0;
    const int64_t kcap = k < kChunkKeys ? k : kChunkKeys;
    const size_t cand = static_cast<size_t>(rows * nchunks * kcap * 8 + 255) / 256 * 256;
    const size_t cnt = static_cast<size_t>(rows * nchunks * 4 + 255) / 256 * 256;
    return cand + cnt;
}

// Every row of B*H*Tq (no row list) through the chunked long-row path; the
// workspace holds topk_chunks_workspace(rows, Tk, k) bytes.
cudaError_t topk_chunks_dispatch(const void* q_low, const void* k_low, bool bf16, int P,
                                 int64_t rows, int Tq, int Tk, int k, int causal, float scale,
                                 int32_t* idx, float* score, void* ws, cudaStream_t stream) {
    const int nchunks = topk_chunk_count(Tk, k);
    if (rows <= 0 || nchunks == 0) return cudaErrorInvalidValue;
    const int64_t blocks = rows * nchunks;
    if (blocks > 0x7fffffffLL || rows > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int64_t kcap = k < kChunkKeys ? k : kChunkKeys;
    uint64_t* cand = reinterpret_cast<uint64_t*>(ws);
    int32_t* cnt = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ws) +
                                              (rows * nchunks * kcap * 8 + 255) / 256 * 256);
    {
        TraceLaunch tr("topk_chunks", stream);
#define SSA_CHUNK_CASE(BF, PP)                                                                   \
        if (bf16 == BF && P == PP) {                                                             \
            topk_chunk_kernel<BF, PP><<<(unsigned)blocks, kChunkThreads, 0, stream>>>(            \
                q_low, k_low, nchunks, Tq, Tk, k, causal, scale, cand, cnt);                     \
        } else
        SSA_CHUNK_CASE(true, 16) SSA_CHUNK_CASE(true, 32) SSA_CHUNK_CASE(true, 64)
        SSA_CHUNK_CASE(true, 128) SSA_CHUNK_CASE(false, 16) SSA_CHUNK_CASE(false, 32)
        SSA_CHUNK_CASE(false, 64) SSA_CHUNK_CASE(false, 128) return cudaErrorInvalidValue;
#undef SSA_CHUNK_CASE
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    TraceLaunch tr("topk_merge", stream);
    topk_merge_kernel<<<(unsigned)rows, kMergeThreads, 0, stream>>>(cand, cnt, nchunks, Tq, Tk, k,
                                                                    causal, idx, score);
    return cudaGetLastError();
}
#endif  // SSA_HOST_EMULATION

}  // namespace ssa
