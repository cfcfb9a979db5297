// Gather attention: one warp per query row, online softmax in fp32.
//
// ssa_sparse_attn: the keys of a row are the entries of its index list
// (mhpq.cn/news/1098205, section 3.2: gather the selected K and V, softmax of
// the scaled logits, weighted sum of V). The running max / running sum form of
// the softmax follows "Attention机制优化：原理、挑战与工程实践", section 2.3.1,
// with every intermediate in fp32 (its section 4.2).
//
// Layout of the work inside a warp. A key row of D elements is R = D*esize
// bytes, read as 16-byte vectors by L = R/16 lanes; the warp holds G = 32/L
// key rows per load instruction, so every load is a fully coalesced run of
// whole rows. Keys are processed in chunks of 32 index entries:
//   1. lane l loads entry t0+l of the index list (one coalesced 128-byte read);
//   2. in round r (r < L) lane (g, s) (g = lane/L, s = lane%L) multiplies its
//      16-byte slice of key row r*G+g with its slice of q;
//   3. a transpose-reduction over the L lanes of a group leaves the full logit
//      of chunk slot s*G+g in lane (g, s) after L-1 shuffles, so the 32 logits
//      of the chunk sit one per lane;
//   4. the chunk max and the rescale factor update the running max; each lane
//      keeps a partial running sum;
//   5. in round r lane (g, s) adds p(slot r*G+g) times its slice of the value
//      row to its accumulator; the G groups are summed at the end.
// Padding entries (-1) and the tail of the last chunk are masked with a -inf
// logit (their loads read row 0 of the head, which is always valid memory).
#ifdef SSA_HOST_EMULATION
#include "emu_device.h"   // the host stand-in of the CPU tests (tests/emu)
#else
#include "common.cuh"
#include "trace.h"
#endif

namespace ssa {

template <bool BF16_IN, int D>
struct RowGeom {
    static constexpr int ESIZE = BF16_IN ? 2 : 4;
    static constexpr int R = D * ESIZE;   // bytes per key row
    static constexpr int L = R / 16;      // lanes per key row
    static constexpr int G = 32 / L;      // key rows per warp load
    static constexpr int E = 16 / ESIZE;  // elements per lane slice
    static_assert(L >= 1 && L <= 32 && (32 % L) == 0, "row must be 16..512 bytes, power of two");
};

// Sum of part[0..L) across the L lanes of each lane group; lane s of the group
// ends with the total of entry s in part[0].
template <int L>
SSA_DEVINL float transpose_reduce(float (&part)[L], int lane) {
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

SSA_DEVINL float warp_max(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

SSA_DEVINL float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// acc + sum of the products of the 8 bf16 pairs of two 16-byte slices, each
// product and sum in fp32 (fma.rn.f32.bf16: the bf16 operands need no
// conversion instruction).
#ifdef SSA_HOST_EMULATION
SSA_DEVINL float dot8_bf16(const uint4& a, const uint4& b, float acc) {
    float fa[8], fb[8];   // bf16 -> fp32 is exact, so one fused multiply-add per pair
    bf16x8_to_f32(a, fa);
    bf16x8_to_f32(b, fb);
    for (int e = 0; e < 8; ++e) acc = fmaf(fa[e], fb[e], acc);
    return acc;
}
#else
SSA_DEVINL float dot8_bf16(const uint4& a, const uint4& b, float acc) {
    asm("{\n\t.reg .b16 a0, a1, a2, a3, a4, a5, a6, a7, b0, b1, b2, b3, b4, b5, b6, b7;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t mov.b32 {a2, a3}, %2;\n\t"
        "mov.b32 {a4, a5}, %3;\n\t mov.b32 {a6, a7}, %4;\n\t"
        "mov.b32 {b0, b1}, %5;\n\t mov.b32 {b2, b3}, %6;\n\t"
        "mov.b32 {b4, b5}, %7;\n\t mov.b32 {b6, b7}, %8;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n\t fma.rn.f32.bf16 %0, a1, b1, %0;\n\t"
        "fma.rn.f32.bf16 %0, a2, b2, %0;\n\t fma.rn.f32.bf16 %0, a3, b3, %0;\n\t"
        "fma.rn.f32.bf16 %0, a4, b4, %0;\n\t fma.rn.f32.bf16 %0, a5, b5, %0;\n\t"
        "fma.rn.f32.bf16 %0, a6, b6, %0;\n\t fma.rn.f32.bf16 %0, a7, b7, %0;\n\t}"
        : "+f"(acc)
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w));
    return acc;
}
#endif

template <bool BF16_OUT, int E>
SSA_DEVINL void store_out(void* O, int64_t elem_off, const float* v) {
    if constexpr (BF16_OUT) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(O) + elem_off;
        if constexpr (E == 8) {
            uint4 w;
            uint32_t* wp = &w.x;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                wp[i] = *reinterpret_cast<uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(o) = w;
        } else {
            uint2 w;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(v[2], v[3]);
            w.x = *reinterpret_cast<uint32_t*>(&h0);
            w.y = *reinterpret_cast<uint32_t*>(&h1);
            *reinterpret_cast<uint2*>(o) = w;
        }
    } else {
        float* o = reinterpret_cast<float*>(O) + elem_off;
#pragma unroll
        for (int i = 0; i < E; i += 4)
            *reinterpret_cast<float4*>(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
}

// BAND == false: keys from idx[row, 0..k).  BAND == true: keys
// max(0, i - wl) .. min(Tk - 1, i + wr) (window attention, Tq == Tk).
//
// Grouped heads (hm.grouped): query head h of H reads key/value head
// h / (H / H_kv) and index list h / (H / H_idx) (grouped-query and
// multi-query attention, and a scorer shared by all heads whose index list is
// broadcast, the layout of mhpq.cn/news/1098205, section 3.2). With
// hm.head_inner (key/value heads shared by groups of query heads) the warps
// walk rows in (batch, key/value head, query, head of the group) order: one
// key/value head at a time, so its K and V stay in L2 (at 128K, one head's K
// and V are 64 MB, two are more than L2), and the heads of a group, which
// share the index list when H_idx <= H_kv, gather the same rows side by side.
template <bool BF16_IN, int D, bool BF16_OUT, bool BAND>
__global__ void __launch_bounds__(256, 3) attn_rows_kernel(
    const void* __restrict__ Q, const void* __restrict__ K, const void* __restrict__ V,
    const int32_t* __restrict__ idx, void* __restrict__ O, int64_t rows, int Tq, int Tk, int k,
    int wl, int wr, float scale_log2, int32_t* dev_status, const HeadMap hm) {
    using Gm = RowGeom<BF16_IN, D>;
    constexpr int L = Gm::L, G = Gm::G, E = Gm::E, R = Gm::R;
    const int lane = threadIdx.x & 31;
    const int64_t wrow = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (wrow >= rows) return;
    const int g = lane / L, s = lane % L;
    int64_t row, bh, irow_id;   // query/output row, key/value head, index row
    int i;
    if (hm.grouped) {
        const int64_t per_b = (int64_t)Tq * hm.H;
        const int64_t b = wrow / per_b;
        const int64_t rem = wrow - b * per_b;
        int h;
        if (hm.head_inner) {
            const int gsz = hm.H / hm.H_kv;                  // query heads per key/value head
            const int64_t per_kv = (int64_t)Tq * gsz;
            const int kvh = (int)(rem / per_kv);
            const int64_t rem2 = rem - kvh * per_kv;
            i = (int)(rem2 / gsz);
            h = kvh * gsz + (int)(rem2 - (int64_t)i * gsz);
        } else {
            h = (int)(rem / Tq);
            i = (int)(rem - (int64_t)h * Tq);
        }
        row = (b * hm.H + h) * Tq + i;
        bh = b * hm.H_kv + h / (hm.H / hm.H_kv);
        irow_id = (b * hm.H_idx + h / (hm.H / hm.H_idx)) * Tq + i;
    } else {
        row = wrow;
        bh = row / Tq;
        i = (int)(row - bh * Tq);
        irow_id = row;
    }
    const char* Kb = reinterpret_cast<const char*>(K) + bh * (int64_t)Tk * R + s * 16;
    const char* Vb = reinterpret_cast<const char*>(V) + bh * (int64_t)Tk * R + s * 16;

    // bf16 inputs: q stays packed and the scale goes onto the dot product;
    // f32 inputs: q is pre-scaled
    const uint4 q16 = ldg16(reinterpret_cast<const char*>(Q) + row * R + s * 16);
    float q[E];
    Vec16<BF16_IN>::to_f32(q16, q);
#pragma unroll
    for (int e = 0; e < E; ++e) q[e] *= scale_log2;

    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float m = -INFINITY, lsum = 0.f;

    int n_entries, band_lo = 0;
    if constexpr (BAND) {
        band_lo = max(0, i - wl);
        const int band_hi = min(Tk - 1, i + wr);
        n_entries = max(0, band_hi - band_lo + 1);
    } else {
        n_entries = Tk > 0 ? k : 0;   // no key at all: every row outputs zeros
    }
    const int32_t* irow = BAND ? nullptr : idx + irow_id * (int64_t)k;

    for (int t0 = 0; t0 < n_entries; t0 += 32) {
        const int t = t0 + lane;
        int j;
        if constexpr (BAND) {
            j = t < n_entries ? band_lo + t : -1;
        } else {
            j = t < n_entries ? __ldg(irow + t) : -1;
            if (t < n_entries && (j < -1 || j >= Tk)) report(dev_status, SSA_DEV_BAD_INDEX);
        }
        const bool ok = (j >= 0) && (j < Tk);
        const int jj = ok ? j : 0;

        float part[L];
        {
            uint4 kv[L];
#pragma unroll
            for (int r = 0; r < L; ++r) {
                const int jc = __shfl_sync(0xffffffffu, jj, r * G + g);
                kv[r] = ldg16(Kb + (int64_t)jc * R);
            }
#pragma unroll
            for (int r = 0; r < L; ++r) {
                if constexpr (BF16_IN) {
                    part[r] = dot8_bf16(q16, kv[r], 0.f);
                } else {
                    float kf[E];
                    Vec16<BF16_IN>::to_f32(kv[r], kf);
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) a = fmaf(q[e], kf[e], a);
                    part[r] = a;
                }
            }
        }
        uint4 vv[L];
#pragma unroll
        for (int r = 0; r < L; ++r) {
            const int jc = __shfl_sync(0xffffffffu, jj, r * G + g);
            vv[r] = ldg16(Vb + (int64_t)jc * R);
        }
        float dot = transpose_reduce<L>(part, lane);
        if constexpr (BF16_IN) dot *= scale_log2;
        const bool ok_mine = __shfl_sync(0xffffffffu, ok, s * G + g);
        const float lg = ok_mine ? dot : -INFINITY;
        const float mn = fmaxf(m, warp_max(lg));
        const float msafe = (mn == -INFINITY) ? 0.f : mn;
        const float alpha = exp2f(m - msafe);
        const float p = exp2f(lg - msafe);
        lsum = lsum * alpha + p;
        m = mn;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] *= alpha;
#pragma unroll
        for (int r = 0; r < L; ++r) {
            const float pr = __shfl_sync(0xffffffffu, p, g * L + r);
            float vf[E];
            Vec16<BF16_IN>::to_f32(vv[r], vf);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(pr, vf[e], acc[e]);
        }
    }
#pragma unroll
    for (int o = L; o < 32; o <<= 1) {
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
    }
    lsum = warp_sum(lsum);
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    if (g == 0) {
        float out[E];
#pragma unroll
        for (int e = 0; e < E; ++e) out[e] = acc[e] * inv;
        store_out<BF16_OUT, E>(O, row * (int64_t)D + s * E, out);
    }
}

#ifndef SSA_HOST_EMULATION   // the CPU tests launch the kernel themselves
template <bool BF16_IN, int D, bool BF16_OUT, bool BAND>
static cudaError_t launch_attn_rows(const void* Q, const void* K, const void* V, const int32_t* idx,
                                    void* O, int64_t rows, int Tq, int Tk, int k, int wl, int wr,
                                    float scale, int32_t* dev_status, const HeadMap& hm,
                                    cudaStream_t stream) {
    constexpr int WARPS = 8;
    const int64_t blocks = (rows + WARPS - 1) / WARPS;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    TraceLaunch tr(BAND ? "attn_rows.window" : "attn_rows.sparse", stream);
    attn_rows_kernel<BF16_IN, D, BF16_OUT, BAND><<<(unsigned)blocks, WARPS * 32, 0, stream>>>(
        Q, K, V, idx, O, rows, Tq, Tk, k, wl, wr, scale * kLog2e, dev_status, hm);
    return cudaGetLastError();
}

template <bool BAND>
cudaError_t attn_rows_dispatch(const void* Q, const void* K, const void* V, bool bf16_in, int D,
                               const int32_t* idx, void* O, bool bf16_out, int64_t rows, int Tq,
                               int Tk, int k, int wl, int wr, float scale, int32_t* dev_status,
                               const HeadMap& hm, cudaStream_t stream) {
#define SSA_ATTN_CASE(BI, DD, BO)                                                               \
    if (bf16_in == BI && D == DD && bf16_out == BO)                                             \
        return launch_attn_rows<BI, DD, BO, BAND>(Q, K, V, idx, O, rows, Tq, Tk, k, wl, wr, scale, \
                                                  dev_status, hm, stream);
    SSA_ATTN_CASE(true, 64, true)
    SSA_ATTN_CASE(true, 64, false)
    SSA_ATTN_CASE(true, 128, true)
    SSA_ATTN_CASE(true, 128, false)
    SSA_ATTN_CASE(false, 64, true)
    SSA_ATTN_CASE(false, 64, false)
    SSA_ATTN_CASE(false, 128, true)
    SSA_ATTN_CASE(false, 128, false)
#undef SSA_ATTN_CASE
    return cudaErrorInvalidValue;
}

template cudaError_t attn_rows_dispatch<false>(const void*, const void*, const void*, bool, int,
                                               const int32_t*, void*, bool, int64_t, int, int, int,
                                               int, int, float, int32_t*, const HeadMap&,
                                               cudaStream_t);
template cudaError_t attn_rows_dispatch<true>(const void*, const void*, const void*, bool, int,
                                              const int32_t*, void*, bool, int64_t, int, int, int,
                                              int, int, float, int32_t*, const HeadMap&,
                                              cudaStream_t);
#endif  // SSA_HOST_EMULATION

}  // namespace ssa
