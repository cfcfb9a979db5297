// Backward of the sparse attention and of the low-rank scorer under the
// straight-through estimator (mhpq.cn/news/1098205, section 2.3): the forward
// keeps its hard top-k; the selected (query, key) pairs pass the exact
// gradients of the attention over those keys, keys a row did not select get
// nothing from it, and the score of every selected pair receives the gradient
// of that pair's attention logit.
//
// Row i with selected keys j_t, logits l_t = scale * Q_i . K_{j_t},
// p = softmax(l), dp_t = dO_i . V_{j_t}, delta = sum_t p_t dp_t:
//   dS[i][t] = p_t (dp_t - delta)
//   dQ_i     = scale * sum_t dS[i][t] K_{j_t}
//   dK_j     = scale * sum_{(i,t): j_t = j} dS[i][t] Q_i
//   dV_j     =         sum_{(i,t): j_t = j} p_t dO_i
// and for the scorer S = sigma * q_low . k_low:
//   dq_low_i = sigma * sum_t dS[i][t] k_low_{j_t}
//   dk_low_j = sigma * sum_{(i,t): j_t = j} dS[i][t] q_low_i
//
// Query side (one warp per query row, the lane layout of the forward gather
// kernel): one pass over the index list gathers K_j and V_j once, keeps the
// running max m and, rescaled like the forward's online softmax, the sums
// s = sum e^(l-m), w = sum e^(l-m) dp, A = sum e^(l-m) (dp - c) K_j and
// B = sum e^(l-m) K_j; it parks l_t and dp_t in the row's dS and p slots.
// Then delta = w / s and dQ_i = scale (A - (delta - c) B) / s without a
// second gather, and a pass over the row's own slots turns (l_t, dp_t) into
// p_t and dS[i][t]. The shift c is the dp of the row's first selected key, a
// stand-in for delta within the spread of the dp: without it A and delta B
// nearly cancel when the row's dp are close to one another (value rows
// alike), and dQ would keep only the bits the cancellation leaves.
//
// Key side: the index lists are transposed per key/value head into key-major
// lists of pair ids (h_g * Tq + i) * k + t, h_g the query head within the
// group that shares the key/value head (a counting sort: count, scan per
// key/value head, fill). One warp per key then sums over the rows that chose
// it, gathering Q_i and dO_i (q_low_i for the scorer). No atomics on the
// gradients; the order of a key's list, and so the fp32 rounding of its sums,
// depends on the fill's atomics. With a scorer shared by several query heads,
// their dS are summed per index head first.
//
// Compiled with SSA_HOST_EMULATION (and a host stand-in for common.cuh), the
// same kernels and C entry points build as plain C++ whose launches run every
// thread on the host. The CPU tests use that build to check the kernels'
// indexing, lane layout and arithmetic against the oracle. libssa.so never
// contains it.
#ifdef SSA_HOST_EMULATION
#include "emu_device.h"   // the host stand-in of the CPU tests (tests/emu)
#else
#include "common.cuh"
#include "trace.h"
#endif

namespace ssa {

namespace {

template <bool BF16_IN, int D>
struct BwdGeom {
    static constexpr int ESIZE = BF16_IN ? 2 : 4;
    static constexpr int R = D * ESIZE;   // bytes per row
    static constexpr int L = R / 16;      // lanes per row
    static constexpr int G = 32 / L;      // rows per warp load
    static constexpr int E = 16 / ESIZE;  // elements per lane slice
    static_assert(L >= 1 && L <= 32 && (32 % L) == 0, "row must be 16..512 bytes, power of two");
};

template <int L>
SSA_DEVINL float transpose_reduce_b(float (&part)[L], int lane) {
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

SSA_DEVINL float warp_max_b(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

SSA_DEVINL float warp_sum_b(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int E>
SSA_DEVINL void store_f32(float* dst, const float* v) {
#pragma unroll
    for (int e = 0; e < E; e += 4)
        *reinterpret_cast<float4*>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
}

// Sum of acc over the G lane groups that hold the same slice s (lanes s,
// s + L, s + 2L, ...); every lane ends with the total.
template <int L, int E>
SSA_DEVINL void reduce_groups(float (&acc)[E]) {
#pragma unroll
    for (int o = L; o < 32; o <<= 1) {
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
    }
}

}  // namespace

// Head grouping: H query heads; query head h reads key/value head h / gk and
// index list head h / gi (gk = H / H_kv, gi = H / H_idx; both 1 in the plain
// layout, where every head has its own).
struct BwdHeads {
    int H, gk, gi;
};

// ------------------------------------------------------------- query side

// One warp per query row (rows of [B, H, Tq]). dS and prob are [rows, k] fp32;
// on return slot t of row i holds dS[i][t] and p_t (0 in padded or skipped
// slots).
template <bool BF16_IN, int D>
__global__ void __launch_bounds__(256, 2) attn_bwd_query_kernel(
    const void* __restrict__ Q, const void* __restrict__ K, const void* __restrict__ V,
    const void* __restrict__ dO, const int32_t* __restrict__ idx, int64_t rows, int Tq, int Tk,
    int k, float scale, const BwdHeads hd, float* __restrict__ dQ, float* dS, float* prob,
    int32_t* dev_status) {
    using Gm = BwdGeom<BF16_IN, D>;
    constexpr int L = Gm::L, G = Gm::G, E = Gm::E, R = Gm::R;
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int g = lane / L, s = lane % L;
    const int64_t bh = row / Tq;
    const int i_row = (int)(row - bh * Tq);
    const int64_t b = bh / hd.H;
    const int h = (int)(bh - b * hd.H);
    const int64_t bkv = b * (hd.H / hd.gk) + h / hd.gk;                       // key/value head
    const int64_t irow_id = (b * (hd.H / hd.gi) + h / hd.gi) * Tq + i_row;    // index list row
    const char* Kb = reinterpret_cast<const char*>(K) + bkv * (int64_t)Tk * R + s * 16;
    const char* Vb = reinterpret_cast<const char*>(V) + bkv * (int64_t)Tk * R + s * 16;
    const float scale_log2 = scale * kLog2e;

    float q[E], go[E];
    Vec16<BF16_IN>::to_f32(ldg16(reinterpret_cast<const char*>(Q) + row * R + s * 16), q);
    Vec16<BF16_IN>::to_f32(ldg16(reinterpret_cast<const char*>(dO) + row * R + s * 16), go);

    float A[E], Bk[E];
#pragma unroll
    for (int e = 0; e < E; ++e) A[e] = Bk[e] = 0.f;
    float m = -INFINITY, lsum = 0.f, wsum = 0.f;   // m in log2 units
    float cshift = 0.f;                             // see the header: set at the first selected key
    bool have_c = false;
    const int n_entries = Tk > 0 ? k : 0;
    const int32_t* irow = idx + irow_id * (int64_t)k;
    float* dsr = dS + row * (int64_t)k;
    float* pr = prob + row * (int64_t)k;

    for (int t0 = 0; t0 < n_entries; t0 += 32) {
        const int t = t0 + lane;
        const int j = t < n_entries ? __ldg(irow + t) : -1;
        if (t < n_entries && (j < -1 || j >= Tk)) report(dev_status, SSA_DEV_BAD_INDEX);
        const bool ok = (j >= 0) && (j < Tk);
        const int jj = ok ? j : 0;

        float pl[L], pd[L];
        {
            uint4 kv[L];
#pragma unroll
            for (int r = 0; r < L; ++r) {
                const int jc = __shfl_sync(0xffffffffu, jj, r * G + g);
                kv[r] = ldg16(Kb + (int64_t)jc * R);
            }
#pragma unroll
            for (int r = 0; r < L; ++r) {
                float kf[E];
                Vec16<BF16_IN>::to_f32(kv[r], kf);
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) a = fmaf(q[e], kf[e], a);
                pl[r] = a;
            }
        }
        {
            uint4 vv[L];
#pragma unroll
            for (int r = 0; r < L; ++r) {
                const int jc = __shfl_sync(0xffffffffu, jj, r * G + g);
                vv[r] = ldg16(Vb + (int64_t)jc * R);
            }
#pragma unroll
            for (int r = 0; r < L; ++r) {
                float vf[E];
                Vec16<BF16_IN>::to_f32(vv[r], vf);
                float b = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) b = fmaf(go[e], vf[e], b);
                pd[r] = b;
            }
        }
        // lane (g, s) now owns slot s*G + g of the chunk
        const float dot = transpose_reduce_b<L>(pl, lane);
        const float dp_raw = transpose_reduce_b<L>(pd, lane);
        const int slot = s * G + g;
        const bool ok_mine = __shfl_sync(0xffffffffu, ok, slot);
        const float lg = ok_mine ? dot * scale_log2 : -INFINITY;
        const float dp = ok_mine ? dp_raw : 0.f;
        const float mn = fmaxf(m, warp_max_b(lg));
        const float msafe = (mn == -INFINITY) ? 0.f : mn;
        const float alpha = exp2f(m - msafe);
        const float ew = exp2f(lg - msafe);   // 0 for skipped slots
        lsum = lsum * alpha + ew;
        wsum = wsum * alpha + ew * dp;
        m = mn;
        if (!have_c) {   // warp-uniform: the dp of the first slot with a key
            const unsigned live = __ballot_sync(0xffffffffu, ok_mine);
            if (live) {
                cshift = __shfl_sync(0xffffffffu, dp, __ffs(live) - 1);
                have_c = true;
            }
        }
        if (t0 + slot < n_entries) {   // park l (log2 units) and dp in the row's slots
            dsr[t0 + slot] = lg;
            pr[t0 + slot] = dp;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
            A[e] *= alpha;
            Bk[e] *= alpha;
        }
        // the chunk's key rows again (L1 hits: this warp read them above)
        // rather than held in registers through the reductions
#pragma unroll
        for (int r = 0; r < L; ++r) {
            // slot r*G + g sits in lane (g, r)
            const float er = __shfl_sync(0xffffffffu, ew, g * L + r);
            const float edr = __shfl_sync(0xffffffffu, ew * (dp - cshift), g * L + r);
            const int jc = __shfl_sync(0xffffffffu, jj, r * G + g);
            float kf[E];
            Vec16<BF16_IN>::to_f32(ldg16(Kb + (int64_t)jc * R), kf);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                A[e] = fmaf(edr, kf[e], A[e]);
                Bk[e] = fmaf(er, kf[e], Bk[e]);
            }
        }
    }
    reduce_groups<L, E>(A);
    reduce_groups<L, E>(Bk);
    lsum = warp_sum_b(lsum);
    wsum = warp_sum_b(wsum);
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const float delta = wsum * inv;
    if (g == 0) {
        float out[E];
#pragma unroll
        for (int e = 0; e < E; ++e) out[e] = scale * (A[e] - (delta - cshift) * Bk[e]) * inv;
        store_f32<E>(dQ + row * (int64_t)D + s * E, out);
    }
    __syncwarp();   // the parked values were written by other lanes
    const float msafe = (m == -INFINITY) ? 0.f : m;
    for (int t = lane; t < k; t += 32) {
        float p = 0.f, d = 0.f;
        if (t < n_entries) {
            const float lg = dsr[t];
            if (lg != -INFINITY) {
                p = exp2f(lg - msafe) * inv;
                d = p * (pr[t] - delta);
            }
        }
        dsr[t] = d;
        pr[t] = p;
    }
}

// ------------------------------------------------------- key-major lists

// Slot e of the query rows [B, H, Tq, k]: the key it names (from its index
// list row), its key/value head and its pair id within that head's lists,
// ((h % gk) * Tq + i) * k + t.
struct PairSlot {
    int j;
    int64_t bkv;
    int32_t pid;
};

SSA_DEVINL PairSlot pair_slot(const int32_t* idx, int64_t e, int Tq, int k, const BwdHeads& hd) {
    const int64_t row = e / k;
    const int t = (int)(e - row * k);
    const int64_t bh = row / Tq;
    const int i = (int)(row - bh * Tq);
    const int64_t b = bh / hd.H;
    const int h = (int)(bh - b * hd.H);
    PairSlot ps;
    ps.j = __ldg(idx + ((b * (hd.H / hd.gi) + h / hd.gi) * Tq + i) * k + t);
    ps.bkv = b * (hd.H / hd.gk) + h / hd.gk;
    ps.pid = (int32_t)(((int64_t)(h % hd.gk) * Tq + i) * k + t);
    return ps;
}

// cnt[bkv*Tk + j] += number of query-head slots of key/value head bkv that
// name key j (entries = B*H*Tq*k slots).
__global__ void pair_count_kernel(const int32_t* __restrict__ idx, int64_t entries, int Tq, int Tk,
                                  int k, const BwdHeads hd, int32_t* __restrict__ cnt,
                                  int32_t* dev_status) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < entries;
         e += (int64_t)gridDim.x * blockDim.x) {
        const PairSlot ps = pair_slot(idx, e, Tq, k, hd);
        if (ps.j == -1) continue;
        if (ps.j < -1 || ps.j >= Tk) {
            report(dev_status, SSA_DEV_BAD_INDEX);
            continue;
        }
        atomicAdd(cnt + ps.bkv * Tk + ps.j, 1);
    }
}

// Per key/value head (one block each): off[bkv*(Tk+1) + j] = sum of cnt over
// keys < j of the head (so off[.. + Tk] is the head's pair count); cnt
// becomes the fill cursor (= off).
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads) pair_scan_kernel(int32_t* __restrict__ cnt,
                                                                 int32_t* __restrict__ off,
                                                                 int Tk) {
    __shared__ int32_t part[kScanThreads];
    const int64_t bkv = blockIdx.x;
    int32_t* c = cnt + bkv * Tk;
    int32_t* o = off + bkv * (int64_t)(Tk + 1);
    const int per = (Tk + kScanThreads - 1) / kScanThreads;
    const int lo = min(Tk, (int)threadIdx.x * per), hi = min(Tk, lo + per);
    int32_t local = 0;
    for (int j = lo; j < hi; ++j) local += c[j];
    part[threadIdx.x] = local;
    __syncthreads();
    // Hillis-Steele inclusive scan of the per-thread sums
    for (int d = 1; d < kScanThreads; d <<= 1) {
        const int32_t v = threadIdx.x >= d ? part[threadIdx.x - d] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    int32_t run = part[threadIdx.x] - local;   // exclusive
    for (int j = lo; j < hi; ++j) {
        const int32_t cj = c[j];
        o[j] = run;
        c[j] = run;
        run += cj;
    }
    if (threadIdx.x == kScanThreads - 1) o[Tk] = part[kScanThreads - 1];
}

// list[bkv*gk*Tq*k + pos] = the pair id of every usable slot of key/value
// head bkv, grouped by key (pos from the key's cursor).
__global__ void pair_fill_kernel(const int32_t* __restrict__ idx, int64_t entries, int Tq, int Tk,
                                 int k, const BwdHeads hd, int32_t* __restrict__ cursor,
                                 int32_t* __restrict__ list) {
    const int64_t per_kv = (int64_t)hd.gk * Tq * k;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < entries;
         e += (int64_t)gridDim.x * blockDim.x) {
        const PairSlot ps = pair_slot(idx, e, Tq, k, hd);
        if (ps.j < 0 || ps.j >= Tk) continue;
        const int32_t pos = atomicAdd(cursor + ps.bkv * Tk + ps.j, 1);
        list[ps.bkv * per_kv + pos] = ps.pid;
    }
}

// ---------------------------------------------------------------- key side

// One warp per key (bkv, j) of the key/value heads: for every pair id
// pid = (h_g * Tq + i) * k + t of its list (query head h = hkv * gk + h_g of
// the same batch), acc1 += w1[slot] * X1[qrow] and acc2 += w2[slot] *
// X2[qrow], with qrow = (b * H + h) * Tq + i a row of the [B, H, Tq, D]
// arrays X1/X2 and slot = qrow * k + t one of the [B, H, Tq, k] weights.
// out1 = f1 * acc1, out2 = acc2 (fp32 [B, H / gk, Tk, D]). TWO == false: only
// the first sum (the scorer's dk_low).
template <bool BF16_IN, int D, bool TWO>
__global__ void __launch_bounds__(256) pair_key_kernel(
    const void* __restrict__ X1, const void* __restrict__ X2, const float* __restrict__ w1,
    const float* __restrict__ w2, const int32_t* __restrict__ off, const int32_t* __restrict__ list,
    int64_t keys, int Tq, int Tk, int k, const BwdHeads hd, float f1, float* __restrict__ out1,
    float* __restrict__ out2) {
    using Gm = BwdGeom<BF16_IN, D>;
    constexpr int L = Gm::L, G = Gm::G, E = Gm::E, R = Gm::R;
    const int lane = threadIdx.x & 31;
    const int64_t key = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (key >= keys) return;
    const int g = lane / L, s = lane % L;
    const int64_t bkv = key / Tk;
    const int j = (int)(key - bkv * Tk);
    const int Hkv = hd.H / hd.gk;
    const int64_t b = bkv / Hkv;
    const int hkv = (int)(bkv - b * Hkv);
    const int64_t per_q = (int64_t)Tq * k;               // pair ids of one query head
    const int32_t* o = off + bkv * (int64_t)(Tk + 1);
    const int32_t beg = o[j], end = o[j + 1];
    const int32_t* lst = list + bkv * (int64_t)hd.gk * per_q;
    const int64_t row0 = (b * hd.H + (int64_t)hkv * hd.gk) * Tq;   // first query row of the group
    const char* X1b = reinterpret_cast<const char*>(X1) + s * 16;
    const char* X2b = TWO ? reinterpret_cast<const char*>(X2) + s * 16 : nullptr;

    float a1[E], a2[E];
#pragma unroll
    for (int e = 0; e < E; ++e) a1[e] = a2[e] = 0.f;
    for (int c0 = beg; c0 < end; c0 += 32) {
        const int n = min(32, end - c0);
        int64_t qrow = row0;   // this lane's pair: its query row (row0 for lanes past n)
        float x1 = 0.f, x2 = 0.f;
        if (lane < n) {
            const int32_t pid = __ldg(lst + c0 + lane);
            const int64_t qi = pid / k;                   // h_g * Tq + i
            qrow = row0 + qi;
            const int64_t slot = qrow * k + (pid - qi * k);
            x1 = __ldg(w1 + slot);
            if constexpr (TWO) x2 = __ldg(w2 + slot);
        }
#pragma unroll
        for (int r = 0; r < L; ++r) {
            const int sl = r * G + g;   // pair slot handled by this lane group in round r
            const int64_t ic = __shfl_sync(0xffffffffu, qrow, sl);
            const float c1 = __shfl_sync(0xffffffffu, x1, sl);
            const float c2 = __shfl_sync(0xffffffffu, x2, sl);
            if (sl < n) {
                float v1[E];
                Vec16<BF16_IN>::to_f32(ldg16(X1b + (int64_t)ic * R), v1);
#pragma unroll
                for (int e = 0; e < E; ++e) a1[e] = fmaf(c1, v1[e], a1[e]);
                if constexpr (TWO) {
                    float v2[E];
                    Vec16<BF16_IN>::to_f32(ldg16(X2b + (int64_t)ic * R), v2);
#pragma unroll
                    for (int e = 0; e < E; ++e) a2[e] = fmaf(c2, v2[e], a2[e]);
                }
            }
        }
    }
    reduce_groups<L, E>(a1);
    if constexpr (TWO) reduce_groups<L, E>(a2);
    if (g == 0) {
#pragma unroll
        for (int e = 0; e < E; ++e) a1[e] *= f1;
        store_f32<E>(out1 + key * D + s * E, a1);
        if constexpr (TWO) store_f32<E>(out2 + key * D + s * E, a2);
    }
}

// ------------------------------------------------------ scorer query side

// dq_low_i = sigma * sum_t dS[i][t] k_low_{j_t}: one warp per query row.
template <bool BF16_IN, int P>
__global__ void __launch_bounds__(256) scorer_bwd_query_kernel(
    const void* __restrict__ k_low, const int32_t* __restrict__ idx, const float* __restrict__ dS,
    int64_t rows, int Tq, int Tk, int k, float sigma, float* __restrict__ dq,
    int32_t* dev_status) {
    using Gm = BwdGeom<BF16_IN, P>;
    constexpr int L = Gm::L, G = Gm::G, E = Gm::E, R = Gm::R;
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int g = lane / L, s = lane % L;
    const int64_t bh = row / Tq;
    const char* Kb = reinterpret_cast<const char*>(k_low) + bh * (int64_t)Tk * R + s * 16;
    const int32_t* irow = idx + row * (int64_t)k;
    const float* drow = dS + row * (int64_t)k;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    const int n_entries = Tk > 0 ? k : 0;
    for (int t0 = 0; t0 < n_entries; t0 += 32) {
        const int t = t0 + lane;
        const int j = t < n_entries ? __ldg(irow + t) : -1;
        if (t < n_entries && (j < -1 || j >= Tk)) report(dev_status, SSA_DEV_BAD_INDEX);
        const bool ok = (j >= 0) && (j < Tk);
        const float w = ok ? __ldg(drow + t) : 0.f;
        const int jj = ok ? j : 0;
#pragma unroll
        for (int r = 0; r < L; ++r) {
            const int sl = r * G + g;
            const int jc = __shfl_sync(0xffffffffu, jj, sl);
            const float wc = __shfl_sync(0xffffffffu, w, sl);
            float kf[E];
            Vec16<BF16_IN>::to_f32(ldg16(Kb + (int64_t)jc * R), kf);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(wc, kf[e], acc[e]);
        }
    }
    reduce_groups<L, E>(acc);
    if (g == 0) {
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] *= sigma;
        store_f32<E>(dq + row * (int64_t)P + s * E, acc);
    }
}

// ----------------------------------------------------------------- launch

// Under SSA_HOST_EMULATION (the CPU tests) a launch runs the kernel's threads
// on the host; otherwise it is a plain launch on `stream`.
#ifdef SSA_HOST_EMULATION
#define SSA_LAUNCH(kfn, grid, block, stream, ...) \
    emu_launch((grid), (block), [&] { kfn(__VA_ARGS__); })
#else
#define SSA_LAUNCH(kfn, grid, block, stream, ...) \
    kfn<<<(grid), (block), 0, (stream)>>>(__VA_ARGS__)
#endif

namespace {

constexpr int kBwdWarps = 8;   // warps per block of the warp-per-row/key kernels

// Blocks for one warp per item; -1 past the grid limit.
int64_t warp_blocks(int64_t items) {
    const int64_t b = (items + kBwdWarps - 1) / kBwdWarps;
    return b > 0x7fffffffLL ? -1 : b;
}

// Grid of the grid-stride kernels over the index lists.
unsigned stride_grid(int64_t n) {
    const int64_t b = (n + 255) / 256;
    return (unsigned)(b < 148 * 16 ? (b > 0 ? b : 1) : 148 * 16);
}

// Key-major lists of the usable slots of every key/value head: off
// [B*Hkv, Tk+1] and list [B*Hkv, gk*Tq*k] (pair ids), with cnt [B*Hkv, Tk] as
// scratch (Hkv = H / gk key/value heads).
cudaError_t pair_lists_build(const int32_t* idx, int B, int Tq, int Tk, int k, const BwdHeads& hd,
                             int32_t* cnt, int32_t* off, int32_t* list, int32_t* dev_status,
                             cudaStream_t stream) {
    const int64_t entries = (int64_t)B * hd.H * Tq * k;
    const int64_t key_heads = (int64_t)B * (hd.H / hd.gk);
    cudaError_t e = cudaMemsetAsync(cnt, 0, sizeof(int32_t) * (size_t)(key_heads * Tk), stream);
    if (e != cudaSuccess) return e;
    {
        TraceLaunch tr("pair_lists.count", stream);
        auto* kc = &pair_count_kernel;
        SSA_LAUNCH(kc, stride_grid(entries), 256, stream, idx, entries, Tq, Tk, k, hd, cnt,
                   dev_status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {
        TraceLaunch tr("pair_lists.scan", stream);
        auto* ks = &pair_scan_kernel;
        SSA_LAUNCH(ks, (unsigned)key_heads, kScanThreads, stream, cnt, off, Tk);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    TraceLaunch tr("pair_lists.fill", stream);
    auto* kf = &pair_fill_kernel;
    SSA_LAUNCH(kf, stride_grid(entries), 256, stream, idx, entries, Tq, Tk, k, hd, cnt, list);
    return cudaGetLastError();
}

// dS summed over the gi query heads that share each index head:
// out[B, H/gi, Tq, k] from dS[B, H, Tq, k].
__global__ void pair_grad_group_sum_kernel(const float* __restrict__ dS, int64_t n_out,
                                           int64_t per_head, int gi, float* __restrict__ out) {
    for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < n_out;
         o += (int64_t)gridDim.x * blockDim.x) {
        const int64_t bhi = o / per_head, rem = o - bhi * per_head;
        float acc = 0.f;
        for (int gg = 0; gg < gi; ++gg) acc += __ldg(dS + (bhi * gi + gg) * per_head + rem);
        out[o] = acc;
    }
}

template <bool BF, int DD>
cudaError_t attn_bwd_t(const void* Q, const void* K, const void* V, const void* dO,
                       const int32_t* idx, int B, int Tq, int Tk, int k, const BwdHeads& hd,
                       float scale, float* dQ, float* dK, float* dV, float* dS, float* prob,
                       int32_t* cnt, int32_t* off, int32_t* list, int32_t* dev_status,
                       cudaStream_t stream) {
    const int64_t rows = (int64_t)B * hd.H * Tq, keys = (int64_t)B * (hd.H / hd.gk) * Tk;
    const int64_t qb = warp_blocks(rows), kb = warp_blocks(keys);
    if (qb < 0 || kb < 0) return cudaErrorInvalidConfiguration;
    cudaError_t e;
    if (qb > 0) {
        TraceLaunch tr("attn_bwd.query", stream);
        auto* kq = &attn_bwd_query_kernel<BF, DD>;
        SSA_LAUNCH(kq, (unsigned)qb, kBwdWarps * 32, stream, Q, K, V, dO, idx, rows, Tq, Tk, k,
                   scale, hd, dQ, dS, prob, dev_status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (kb == 0) return cudaSuccess;
    if ((e = pair_lists_build(idx, B, Tq, Tk, k, hd, cnt, off, list, dev_status, stream)) !=
        cudaSuccess)
        return e;
    TraceLaunch tr("attn_bwd.key", stream);
    auto* kk = &pair_key_kernel<BF, DD, true>;
    SSA_LAUNCH(kk, (unsigned)kb, kBwdWarps * 32, stream, Q, dO, dS, prob, off, list, keys, Tq, Tk,
               k, hd, scale, dK, dV);
    return cudaGetLastError();
}

// The scorer's backward on H_idx scorer heads (idx, q_low, k_low) from the
// pair gradients of H = gi * H_idx query heads: those are first summed over
// each index head's query heads (into dS_sum), then every scorer head is a
// plain head of its own.
template <bool BF, int PP>
cudaError_t scorer_bwd_t(const void* q_low, const void* k_low, const int32_t* idx,
                         const float* dS, int B, int H_idx, int gi, int Tq, int Tk, int k,
                         float sigma, float* dq_low, float* dk_low, float* dS_sum, int32_t* cnt,
                         int32_t* off, int32_t* list, bool lists_ready, int32_t* dev_status,
                         cudaStream_t stream) {
    const int64_t rows = (int64_t)B * H_idx * Tq, keys = (int64_t)B * H_idx * Tk;
    const int64_t qb = warp_blocks(rows), kb = warp_blocks(keys);
    if (qb < 0 || kb < 0) return cudaErrorInvalidConfiguration;
    cudaError_t e;
    const float* g = dS;
    if (gi > 1 && rows > 0) {
        TraceLaunch tr("scorer_bwd.group_sum", stream);
        auto* ksum = &pair_grad_group_sum_kernel;
        SSA_LAUNCH(ksum, stride_grid(rows * k), 256, stream, dS, rows * k, (int64_t)Tq * k, gi,
                   dS_sum);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        g = dS_sum;
    }
    if (qb > 0) {
        TraceLaunch tr("scorer_bwd.query", stream);
        auto* kq = &scorer_bwd_query_kernel<BF, PP>;
        SSA_LAUNCH(kq, (unsigned)qb, kBwdWarps * 32, stream, k_low, idx, g, rows, Tq, Tk, k,
                   sigma, dq_low, dev_status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (kb == 0) return cudaSuccess;
    const BwdHeads plain{H_idx, 1, 1};
    if (!lists_ready &&
        (e = pair_lists_build(idx, B, Tq, Tk, k, plain, cnt, off, list, dev_status, stream)) !=
            cudaSuccess)
        return e;
    TraceLaunch tr("scorer_bwd.key", stream);
    auto* kk = &pair_key_kernel<BF, PP, false>;
    const void* no_x = nullptr;
    const float* no_w = nullptr;
    float* no_out = nullptr;
    SSA_LAUNCH(kk, (unsigned)kb, kBwdWarps * 32, stream, q_low, no_x, g, no_w, off, list, keys,
               Tq, Tk, k, plain, sigma, dk_low, no_out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t attn_bwd_launch(const void* Q, const void* K, const void* V, const void* dO,
                            bool bf16, int D, const int32_t* idx, int B, int H, int H_kv,
                            int H_idx, int Tq, int Tk, int k, float scale, float* dQ, float* dK,
                            float* dV, float* dS, float* prob, int32_t* cnt, int32_t* off,
                            int32_t* list, int32_t* dev_status, cudaStream_t stream) {
    const BwdHeads hd{H, H / H_kv, H / H_idx};
#define SSA_BWD_CASE(BF, DD)                                                                  \
    if (bf16 == BF && D == DD)                                                                \
        return attn_bwd_t<BF, DD>(Q, K, V, dO, idx, B, Tq, Tk, k, hd, scale, dQ, dK, dV, dS,   \
                                  prob, cnt, off, list, dev_status, stream);
    SSA_BWD_CASE(true, 64)
    SSA_BWD_CASE(true, 128)
    SSA_BWD_CASE(false, 64)
    SSA_BWD_CASE(false, 128)
#undef SSA_BWD_CASE
    return cudaErrorInvalidValue;
}

cudaError_t scorer_bwd_launch(const void* q_low, const void* k_low, bool bf16, int P,
                              const int32_t* idx, const float* dS, int B, int H, int H_idx,
                              int Tq, int Tk, int k, float sigma, float* dq_low, float* dk_low,
                              float* dS_sum, int32_t* cnt, int32_t* off, int32_t* list,
                              bool lists_ready, int32_t* dev_status, cudaStream_t stream) {
    const int gi = H / H_idx;
#define SSA_SBWD_CASE(BF, PP)                                                                 \
    if (bf16 == BF && P == PP)                                                                \
        return scorer_bwd_t<BF, PP>(q_low, k_low, idx, dS, B, H_idx, gi, Tq, Tk, k, sigma,     \
                                    dq_low, dk_low, dS_sum, cnt, off, list, lists_ready,       \
                                    dev_status, stream);
    SSA_SBWD_CASE(true, 16)
    SSA_SBWD_CASE(true, 32)
    SSA_SBWD_CASE(true, 64)
    SSA_SBWD_CASE(true, 128)
    SSA_SBWD_CASE(false, 16)
    SSA_SBWD_CASE(false, 32)
    SSA_SBWD_CASE(false, 64)
    SSA_SBWD_CASE(false, 128)
#undef SSA_SBWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace ssa

// ------------------------------------------------------------------ C ABI

namespace ssa {
namespace {

int64_t up256(int64_t x) { return (x + 255) / 256 * 256; }

struct BwdWorkspace {
    int64_t cnt, off, list, extra, total;
};

// cnt [KH*Tk] | off [KH*(Tk+1)] | list [slots] | extra [extra_floats] fp32,
// KH key heads and `slots` query-head slots (B*H*Tq*k).
BwdWorkspace bwd_workspace(int64_t KH, int64_t Tk, int64_t slots, int64_t extra_floats) {
    BwdWorkspace w;
    int64_t o = 0;
    w.cnt = o;
    o += up256(KH * Tk * 4);
    w.off = o;
    o += up256(KH * (Tk + 1) * 4);
    w.list = o;
    o += up256(slots * 4);
    w.extra = o;
    o += up256(extra_floats * 4);
    w.total = o > 0 ? o : 256;
    return w;
}

bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool heads_ok(int H, int Hs) { return H >= 1 && Hs >= 1 && H % Hs == 0; }

}  // namespace
}  // namespace ssa

extern "C" {

size_t ssa_sparse_attn_grouped_bwd_workspace_size(int B, int H, int H_kv, int Tq, int Tk, int k) {
    if (B < 0 || Tq < 0 || Tk < 0 || k < 1 || !ssa::heads_ok(H, H_kv)) return 0;
    const int64_t slots = (int64_t)B * H * Tq * k;
    return (size_t)ssa::bwd_workspace((int64_t)B * H_kv, Tk, slots, slots).total;
}

size_t ssa_sparse_attn_bwd_workspace_size(int B, int H, int Tq, int Tk, int k) {
    if (H < 0) return 0;
    return H == 0 ? ssa_sparse_attn_grouped_bwd_workspace_size(B, 1, 1, 0, Tk, k)
                  : ssa_sparse_attn_grouped_bwd_workspace_size(B, H, H, Tq, Tk, k);
}

size_t ssa_scorer_grouped_bwd_workspace_size(int B, int H, int H_idx, int Tq, int Tk, int k) {
    if (B < 0 || Tq < 0 || Tk < 0 || k < 1 || !ssa::heads_ok(H, H_idx)) return 0;
    const int64_t slots = (int64_t)B * H_idx * Tq * k;
    return (size_t)ssa::bwd_workspace((int64_t)B * H_idx, Tk, slots, H > H_idx ? slots : 0).total;
}

size_t ssa_scorer_bwd_workspace_size(int B, int H, int Tq, int Tk, int k) {
    if (H < 0) return 0;
    return H == 0 ? ssa_scorer_grouped_bwd_workspace_size(B, 1, 1, 0, Tk, k)
                  : ssa_scorer_grouped_bwd_workspace_size(B, H, H, Tq, Tk, k);
}

ssa_status ssa_sparse_attn_grouped_bwd(const void* Q, const void* K, const void* V,
                                       const void* dO, int dtype, int B, int H, int H_kv, int Tq,
                                       int Tk, int D, const int32_t* idx, int H_idx, int k,
                                       float scale, float* dQ, float* dK, float* dV, float* dS,
                                       float* prob, void* workspace, size_t workspace_bytes,
                                       int32_t* dev_status, void* stream) {
    if (B < 0 || Tq < 0 || Tk < 0 || k < 1 || (dtype != SSA_F32 && dtype != SSA_BF16) ||
        !isfinite(scale) || !ssa::heads_ok(H, H_kv) || !ssa::heads_ok(H, H_idx))
        return SSA_ERR_INVALID;
    if (!(D == 64 || D == 128)) return SSA_ERR_UNSUPPORTED;
    // pair ids are 32-bit per key/value head
    if ((int64_t)(H / H_kv) * Tq * k > INT32_MAX) return SSA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * H * Tq, keys = (int64_t)B * H_kv * Tk;
    if (rows == 0 && keys == 0) return SSA_OK;
    if ((int64_t)B * H > INT32_MAX) return SSA_ERR_UNSUPPORTED;
    // query-side buffers are needed when there are query rows, key-side ones
    // when there are keys; every pointer given must be aligned
    if (rows > 0 && (!Q || !dO || !idx || !dQ || !dS)) return SSA_ERR_INVALID;
    if (keys > 0 && (!K || !V || !dK || !dV)) return SSA_ERR_INVALID;
    if (!ssa::al(Q, 16) || !ssa::al(K, 16) || !ssa::al(V, 16) || !ssa::al(dO, 16) ||
        !ssa::al(dQ, 16) || !ssa::al(dK, 16) || !ssa::al(dV, 16) || !ssa::al(dS, 4) ||
        !ssa::al(idx, 4) || !ssa::al(prob, 4) || !ssa::al(dev_status, 4))
        return SSA_ERR_INVALID;
    const int64_t slots = rows * k;
    const ssa::BwdWorkspace w = ssa::bwd_workspace((int64_t)B * H_kv, Tk, slots, slots);
    if (!workspace || !ssa::al(workspace, 256) || workspace_bytes < (size_t)w.total)
        return SSA_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    float* pr = prob ? prob : reinterpret_cast<float*>(ws + w.extra);
    const float sc = scale > 0.f ? scale : (float)(1.0 / sqrt((double)D));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 0) {   // no query rows: every key's gradient is zero
        cudaError_t e = cudaMemsetAsync(dK, 0, sizeof(float) * (size_t)(keys * D), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dV, 0, sizeof(float) * (size_t)(keys * D), s);
        return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
    }
    const cudaError_t e = ssa::attn_bwd_launch(
        Q, K, V, dO, dtype == SSA_BF16, D, idx, B, H, H_kv, H_idx, Tq, Tk, k, sc, dQ, dK, dV, dS,
        pr, reinterpret_cast<int32_t*>(ws + w.cnt), reinterpret_cast<int32_t*>(ws + w.off),
        reinterpret_cast<int32_t*>(ws + w.list), dev_status, s);
    return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
}

ssa_status ssa_sparse_attn_bwd(const void* Q, const void* K, const void* V, const void* dO,
                               int dtype, int B, int H, int Tq, int Tk, int D, const int32_t* idx,
                               int k, float scale, float* dQ, float* dK, float* dV, float* dS,
                               float* prob, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream) {
    if (H < 0) return SSA_ERR_INVALID;
    if (H == 0) {   // no heads: nothing to do once the other arguments are valid
        if (B < 0 || Tq < 0 || Tk < 0 || k < 1 || (dtype != SSA_F32 && dtype != SSA_BF16) ||
            !isfinite(scale))
            return SSA_ERR_INVALID;
        return (D == 64 || D == 128) ? SSA_OK : SSA_ERR_UNSUPPORTED;
    }
    return ssa_sparse_attn_grouped_bwd(Q, K, V, dO, dtype, B, H, H, Tq, Tk, D, idx, H, k, scale,
                                       dQ, dK, dV, dS, prob, workspace, workspace_bytes,
                                       dev_status, stream);
}

ssa_status ssa_scorer_grouped_bwd(const void* q_low, const void* k_low, int dtype, int B, int H,
                                  int H_idx, int Tq, int Tk, int P, const int32_t* idx, int k,
                                  const float* dS, float scale, float* dq_low, float* dk_low,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                  void* stream) {
    if (B < 0 || Tq < 0 || Tk < 0 || k < 1 || (dtype != SSA_F32 && dtype != SSA_BF16) ||
        !isfinite(scale) || !ssa::heads_ok(H, H_idx))
        return SSA_ERR_INVALID;
    if (!(P == 16 || P == 32 || P == 64 || P == 128)) return SSA_ERR_UNSUPPORTED;
    if ((int64_t)Tq * k > INT32_MAX) return SSA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * H_idx * Tq, keys = (int64_t)B * H_idx * Tk;
    if (rows == 0 && keys == 0) return SSA_OK;
    if ((int64_t)B * H > INT32_MAX) return SSA_ERR_UNSUPPORTED;
    if (rows > 0 && (!q_low || !idx || !dS || !dq_low)) return SSA_ERR_INVALID;
    if (keys > 0 && (!k_low || !dk_low)) return SSA_ERR_INVALID;
    if (!ssa::al(q_low, 16) || !ssa::al(k_low, 16) || !ssa::al(dq_low, 16) ||
        !ssa::al(dk_low, 16) || !ssa::al(dS, 4) || !ssa::al(idx, 4) || !ssa::al(dev_status, 4))
        return SSA_ERR_INVALID;
    const int64_t slots = rows * k;
    const ssa::BwdWorkspace w =
        ssa::bwd_workspace((int64_t)B * H_idx, Tk, slots, H > H_idx ? slots : 0);
    if (!workspace || !ssa::al(workspace, 256) || workspace_bytes < (size_t)w.total)
        return SSA_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    const float sg = scale > 0.f ? scale : (float)(1.0 / sqrt((double)P));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 0) {
        const cudaError_t e = cudaMemsetAsync(dk_low, 0, sizeof(float) * (size_t)(keys * P), s);
        return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
    }
    const cudaError_t e = ssa::scorer_bwd_launch(
        q_low, k_low, dtype == SSA_BF16, P, idx, dS, B, H, H_idx, Tq, Tk, k, sg, dq_low, dk_low,
        reinterpret_cast<float*>(ws + w.extra), reinterpret_cast<int32_t*>(ws + w.cnt),
        reinterpret_cast<int32_t*>(ws + w.off), reinterpret_cast<int32_t*>(ws + w.list), false,
        dev_status, s);
    return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
}

ssa_status ssa_scorer_bwd(const void* q_low, const void* k_low, int dtype, int B, int H, int Tq,
                          int Tk, int P, const int32_t* idx, int k, const float* dS, float scale,
                          float* dq_low, float* dk_low, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream) {
    if (H < 0) return SSA_ERR_INVALID;
    if (H == 0) {
        if (B < 0 || Tq < 0 || Tk < 0 || k < 1 || (dtype != SSA_F32 && dtype != SSA_BF16) ||
            !isfinite(scale))
            return SSA_ERR_INVALID;
        return (P == 16 || P == 32 || P == 64 || P == 128) ? SSA_OK : SSA_ERR_UNSUPPORTED;
    }
    return ssa_scorer_grouped_bwd(q_low, k_low, dtype, B, H, H, Tq, Tk, P, idx, k, dS, scale,
                                  dq_low, dk_low, workspace, workspace_bytes, dev_status, stream);
}

size_t ssa_sparse_attn_scorer_bwd_workspace_size(int B, int H, int Tq, int Tk, int k) {
    return ssa_sparse_attn_bwd_workspace_size(B, H, Tq, Tk, k);
}

// Both backward calls in one: the key-major lists of the index lists, which
// the attention's key side and the scorer's key side both walk, are built
// once.
ssa_status ssa_sparse_attn_scorer_bwd(const void* Q, const void* K, const void* V, const void* dO,
                                      const void* q_low, const void* k_low, int dtype, int B,
                                      int H, int Tq, int Tk, int D, int P, const int32_t* idx,
                                      int k, float scale, float scorer_scale, float* dQ,
                                      float* dK, float* dV, float* dS, float* prob,
                                      float* dq_low, float* dk_low, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status,
                                      void* stream) {
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0 || k < 1 || (dtype != SSA_F32 && dtype != SSA_BF16) ||
        !isfinite(scale) || !isfinite(scorer_scale))
        return SSA_ERR_INVALID;
    if (!(D == 64 || D == 128) || !(P == 16 || P == 32 || P == 64 || P == 128))
        return SSA_ERR_UNSUPPORTED;
    if ((int64_t)Tq * k > INT32_MAX || (int64_t)B * H > INT32_MAX) return SSA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * H * Tq, keys = (int64_t)B * H * Tk;
    if (rows == 0 && keys == 0) return SSA_OK;
    if (rows > 0 && (!Q || !dO || !idx || !dQ || !dS || !q_low || !dq_low)) return SSA_ERR_INVALID;
    if (keys > 0 && (!K || !V || !dK || !dV || !k_low || !dk_low)) return SSA_ERR_INVALID;
    if (!ssa::al(Q, 16) || !ssa::al(K, 16) || !ssa::al(V, 16) || !ssa::al(dO, 16) ||
        !ssa::al(q_low, 16) || !ssa::al(k_low, 16) || !ssa::al(dQ, 16) || !ssa::al(dK, 16) ||
        !ssa::al(dV, 16) || !ssa::al(dq_low, 16) || !ssa::al(dk_low, 16) || !ssa::al(dS, 4) ||
        !ssa::al(idx, 4) || !ssa::al(prob, 4) || !ssa::al(dev_status, 4))
        return SSA_ERR_INVALID;
    const int64_t slots = rows * k;
    const ssa::BwdWorkspace w = ssa::bwd_workspace((int64_t)B * H, Tk, slots, slots);
    if (!workspace || !ssa::al(workspace, 256) || workspace_bytes < (size_t)w.total)
        return SSA_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    float* pr = prob ? prob : reinterpret_cast<float*>(ws + w.extra);
    const float sc = scale > 0.f ? scale : (float)(1.0 / sqrt((double)D));
    const float sg = scorer_scale > 0.f ? scorer_scale : (float)(1.0 / sqrt((double)P));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 0) {   // no query rows: every key's gradient is zero
        cudaError_t e = cudaMemsetAsync(dK, 0, sizeof(float) * (size_t)(keys * D), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dV, 0, sizeof(float) * (size_t)(keys * D), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dk_low, 0, sizeof(float) * (size_t)(keys * P), s);
        return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
    }
    int32_t* cnt = reinterpret_cast<int32_t*>(ws + w.cnt);
    int32_t* off = reinterpret_cast<int32_t*>(ws + w.off);
    int32_t* list = reinterpret_cast<int32_t*>(ws + w.list);
    cudaError_t e = ssa::attn_bwd_launch(Q, K, V, dO, dtype == SSA_BF16, D, idx, B, H, H, H, Tq,
                                         Tk, k, sc, dQ, dK, dV, dS, pr, cnt, off, list,
                                         dev_status, s);
    // the attention's key side built the lists (there are keys whenever there
    // are query rows); the scorer's key side walks the same ones
    if (e == cudaSuccess)
        e = ssa::scorer_bwd_launch(q_low, k_low, dtype == SSA_BF16, P, idx, dS, B, H, H, Tq, Tk, k,
                                   sg, dq_low, dk_low, nullptr, cnt, off, list, keys > 0,
                                   dev_status, s);
    return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
}

}  // extern "C"
