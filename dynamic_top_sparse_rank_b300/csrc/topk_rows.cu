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
#endif  // SSA_HOST_EMULATION

}  // namespace ssa
