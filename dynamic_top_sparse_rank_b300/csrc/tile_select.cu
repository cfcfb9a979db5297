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
//   cand_sort_kernel sorts a row's candidates by (score desc, index asc) and
//   writes the first k_eff.
// With G between 2k and 4k, about k + k^2/(2G) <= 1.25k keys pass the bound.
// A row with more candidates than its list holds (heavy ties at the k-th
// score) is put on an overflow list and redone by the row-wise kernel.
#include "common.cuh"
#include "tile.h"
#include "trace.h"

namespace ssa {

// ---------------------------------------------------------------- tau
//
// One block per 128-row half of a unit. Histograms live in shared memory as
// [bin][row pair] words holding two 16-bit counters (a row has < 65536
// groups). Thread t reads row t % 128 of group after group (a warp reads 64
// contiguous bytes per load), eight loads in flight per thread.
constexpr int kSelThreads = 256;
constexpr int kSelUnroll = 8;

__global__ void __launch_bounds__(kSelThreads) group_select_kernel(
    const uint16_t* __restrict__ gm, uint32_t* __restrict__ tau, int BH, int Tq, int Tk, int k,
    int causal, int G_stride) {
    extern __shared__ uint32_t hist[];   // 256 * (kTileM / 2) words
    __shared__ int n_row[kTileM];
    __shared__ uint32_t sel_hi[kTileM], need[kTileM];
    const int units_per_head = (Tq + kUnitM - 1) / kUnitM;
    const int num_items = BH * units_per_head * 2;   // (unit, 128-row half)
    const int tid = threadIdx.x;
    const int r = tid % kTileM;
    const int gstep = kSelThreads / kTileM;
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
        const uint16_t* gu = gm + static_cast<int64_t>(u) * G_stride * kUnitM + h * kTileM;
        if (tid < kTileM) n_row[tid] = tid < rows ? tile_valid_count(i0 + tid, Tq, Tk, causal) : 0;
        for (int x = tid; x < 256 * (kTileM / 2); x += kSelThreads) hist[x] = 0;
        __syncthreads();
        const int n_r = n_row[r];
        const bool active = n_r > k;
        const int word = r >> 1;
        const uint32_t one = 1u << ((r & 1) * 16);
        // pass 1: high byte of every group maximum of the row
        if (active) {
            for (int g0 = tid / kTileM; g0 < G_u; g0 += gstep * kSelUnroll) {
                uint32_t v[kSelUnroll];
#pragma unroll
                for (int q = 0; q < kSelUnroll; ++q) {
                    const int grp = g0 + q * gstep;
                    v[q] = (grp < G_u && tile_group_first_key(grp, g) < n_r)
                               ? static_cast<uint32_t>(gu[static_cast<int64_t>(grp) * kUnitM + r])
                               : 0x10000u;
                }
#pragma unroll
                for (int q = 0; q < kSelUnroll; ++q)
                    if (v[q] < 0x10000u) atomicAdd(&hist[(v[q] >> 8) * (kTileM / 2) + word], one);
            }
        }
        __syncthreads();
        if (tid < kTileM) {
            uint32_t hi = 0, nd = 0;
            if (n_row[tid] > k) {
                uint32_t cum = 0;
                for (int b = 255; b >= 0; --b) {
                    const uint32_t cb =
                        (hist[b * (kTileM / 2) + (tid >> 1)] >> ((tid & 1) * 16)) & 0xFFFFu;
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
        for (int x = tid; x < 256 * (kTileM / 2); x += kSelThreads) hist[x] = 0;
        __syncthreads();
        // pass 2: low byte of the group maxima in the selected high-byte bin
        if (active) {
            const uint32_t hsel = sel_hi[r];
            for (int g0 = tid / kTileM; g0 < G_u; g0 += gstep * kSelUnroll) {
                uint32_t v[kSelUnroll];
#pragma unroll
                for (int q = 0; q < kSelUnroll; ++q) {
                    const int grp = g0 + q * gstep;
                    v[q] = (grp < G_u && tile_group_first_key(grp, g) < n_r)
                               ? static_cast<uint32_t>(gu[static_cast<int64_t>(grp) * kUnitM + r])
                               : 0x10000u;
                }
#pragma unroll
                for (int q = 0; q < kSelUnroll; ++q)
                    if ((v[q] >> 8) == hsel)
                        atomicAdd(&hist[(v[q] & 0xFFu) * (kTileM / 2) + word], one);
            }
        }
        __syncthreads();
        if (tid < rows) {
            uint32_t t32 = 0;
            if (n_row[tid] > k) {
                uint32_t cum = 0, lo = 0;
                for (int b = 255; b >= 0; --b) {
                    const uint32_t cb =
                        (hist[b * (kTileM / 2) + (tid >> 1)] >> ((tid & 1) * 16)) & 0xFFFFu;
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
// One warp per row: the row's candidates (composite keys, see sel_key) are
// loaded lane-major (lane l holds elements l*E .. l*E+E-1), sorted descending
// by a bitonic network (strides below E inside a lane, the others across
// lanes by shuffles), and the first k_eff written out.
template <int E>
SSA_DEVINL void warp_bitonic_desc(uint64_t (&x)[E], int lane) {
    constexpr int N = 32 * E;
#pragma unroll
    for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride >= E) {
                const int lx = stride / E;
#pragma unroll
                for (int r = 0; r < E; ++r) {
                    const int e = lane * E + r;
                    const uint64_t y = __shfl_xor_sync(0xffffffffu, x[r], lx);
                    const bool lower = (e & stride) == 0;
                    const bool desc = (e & size) == 0;
                    const bool take_max = lower == desc;
                    const bool y_big = y > x[r];
                    x[r] = (take_max == y_big) ? y : x[r];
                }
            } else {
#pragma unroll
                for (int r = 0; r < E; ++r) {
                    if ((r & stride) == 0) {
                        const int e = lane * E + r;
                        const bool desc = (e & size) == 0;
                        const uint64_t a = x[r], b = x[r + stride];
                        if ((a < b) == desc) {
                            x[r] = b;
                            x[r + stride] = a;
                        }
                    }
                }
            }
        }
    }
}

template <int E>
__global__ void __launch_bounds__(256) cand_sort_kernel(
    const uint64_t* __restrict__ cand, const int32_t* __restrict__ cnt, int64_t rows, int Tq,
    int Tk, int k, int causal, int32_t* __restrict__ idx_out, float* __restrict__ score_out,
    int64_t* __restrict__ ovf_list, int32_t* __restrict__ ovf_count) {
    constexpr int CAP = 32 * E;       // two lists of CAP/2 = 16E; lane l reads list l/16
    constexpr int CAPC = CAP / 2;
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int i = static_cast<int>(row % Tq);
    const int n = tile_valid_count(i, Tq, Tk, causal);
    const int keff = min(k, n);
    int c_list = 0;
    if (n > 0 && lane < 2) c_list = cnt[row * 2 + lane];
    const bool overflow = __any_sync(0xffffffffu, c_list > CAPC);
    if (overflow) {
        if (lane == 0) ovf_list[atomicAdd(ovf_count, 1)] = row;
        return;
    }
    const int my_cnt = __shfl_sync(0xffffffffu, c_list, lane >> 4);
    const int off = (lane & 15) * E;   // offset of this lane's elements in its list
    uint64_t x[E];
    const uint64_t* src = cand + row * CAP + (lane >> 4) * CAPC + off;
#pragma unroll
    for (int r = 0; r < E; r += 2) {
        if (off + r + 1 < my_cnt) {
            const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(src + r);
            x[r] = v.x;
            x[r + 1] = v.y;
        } else {
            x[r] = off + r < my_cnt ? src[r] : 0ull;
            x[r + 1] = 0ull;
        }
    }
    warp_bitonic_desc<E>(x, lane);
    int32_t* io = idx_out + row * k;
    float* so = score_out ? score_out + row * k : nullptr;
#pragma unroll
    for (int r = 0; r < E; ++r) {
        const int e = lane * E + r;
        if (e < k) {
            if (e < keff) {
                io[e] = static_cast<int32_t>(sel_key_index(x[r]));
                if (so) so[e] = order_key_f32(sel_key_okey(x[r]));
            } else {
                io[e] = -1;
                if (so) so[e] = -INFINITY;
            }
        }
    }
}

cudaError_t tile_select_launch(const uint16_t* gm, uint32_t* tau, int BH, int Tq, int Tk, int k,
                               int causal, cudaStream_t stream) {
    const int items = 2 * BH * ((Tq + kUnitM - 1) / kUnitM);
    if (items == 0) return cudaSuccess;
    const int sms = tile_sm_count();
    const int grid = items < 3 * sms ? items : 3 * sms;
    constexpr int kHistBytes = 256 * (kTileM / 2) * 4;
    cudaError_t e = cudaFuncSetAttribute(group_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kHistBytes);
    if (e != cudaSuccess) return e;
    TraceLaunch tr("group_select", stream);
    group_select_kernel<<<grid, kSelThreads, kHistBytes, stream>>>(gm, tau, BH, Tq, Tk, k, causal,
                                                                   tile_group_stride(k));
    return cudaGetLastError();
}

cudaError_t tile_sort_launch(const uint64_t* cand, const int32_t* cnt, int64_t rows, int Tq,
                             int Tk, int k, int causal, int32_t* idx, float* score,
                             int64_t* ovf_list, int32_t* ovf_count, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int cap = tile_cand_cap(k);
    TraceLaunch tr("cand_sort", stream);
#define SSA_SORT_CASE(EE)                                                                      \
    if (cap == 32 * EE) {                                                                      \
        cand_sort_kernel<EE><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(               \
            cand, cnt, rows, Tq, Tk, k, causal, idx, score, ovf_list, ovf_count);              \
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

}  // namespace ssa
