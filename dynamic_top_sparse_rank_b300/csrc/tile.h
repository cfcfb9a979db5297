// Definitions shared by the tensor-core score+top-k path (host and device):
// tile sizes, the per-row valid key count, the group size rule, the launch
// parameters of the tile kernel and the workspace layout of the whole path.
#pragma once

#ifndef SSA_HOST_EMULATION
#include <cuda_runtime.h>
#endif
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

namespace ssa {

constexpr int kTileM = 128;   // query rows per accumulator (TMEM lanes)
constexpr int kUnitM = 256;   // query rows per unit: two accumulators share every key tile
constexpr int kTileN = 128;   // keys per MMA tile (TMEM columns per accumulator)

enum TileMode { MODE_RAW = 0, MODE_GROUPMAX = 1, MODE_COLLECT = 2 };

// Number of keys query i may select: all Tk, or under the bottom-right causal
// mask the keys j <= i + (Tk - Tq).
__host__ __device__ __forceinline__ int tile_valid_count(int i, int Tq, int Tk, int causal) {
    if (!causal) return Tk;
    const int64_t last = static_cast<int64_t>(i) + (Tk - Tq);
    if (last < 0) return 0;
    return last + 1 < Tk ? static_cast<int>(last + 1) : Tk;
}

// Group size g of a unit whose rows have between n_lo and n_hi valid keys.
// A row with n > k valid keys is split into at least min(n, 2k) groups (more
// than k, which the exact bound needs; about 2k or more keeps the k-th largest
// group maximum a tight lower bound on the k-th largest score), and g is a
// power of two. 0 when no row of the unit has more than k valid keys (every
// valid key is then selected).
__host__ __device__ __forceinline__ int tile_group_size(int n_lo, int n_hi, int k) {
    if (n_hi <= k) return 0;
    const int n_ref = n_lo > k + 1 ? n_lo : k + 1;
    const int q = n_ref / (2 * k);
    int g = 1;
    while (g * 2 <= q) g *= 2;
    return g;
}

// Layout of the groups of a row (both the score kernel and the selection use
// it). g < 32: group grp holds the consecutive keys [grp*g, grp*g + g).
// g >= 32 (m = g/32): the key tiles of a unit alternate between kTileGroups
// TMEM buffers, each drained by its own epilogue warps (tile t by buffer
// t % 2); group grp = 4*(2*T + b) + c holds the 32-key chunk c of the m tiles
// T*m .. T*m + m - 1 among those of buffer b, i.e. of tiles 2*(T*m + i) + b,
// i < m. Every warp then forms its groups alone. Groups need not be
// contiguous: any partition of the valid keys into G >= k groups gives a
// valid bound.
constexpr int kTileGroups = 2;

__host__ __device__ __forceinline__ int tile_group_first_key(int grp, int g) {
    if (g < 32) return grp * g;
    const int m = g / 32;
    const int T = grp / (4 * kTileGroups), b = (grp / 4) % kTileGroups, c = grp % 4;
    return (T * m * kTileGroups + b) * 128 + c * 32;
}

// Number of groups of a row with n valid keys among the first `limit` group
// indices: the first keys increase with the index, so the groups holding a
// valid key are exactly 0 .. count-1 (binary search for g >= 32).
__host__ __device__ __forceinline__ int tile_groups_of_row(int n, int g, int limit) {
    if (n <= 0) return 0;
    if (g < 32) {
        const int c = (n + g - 1) / g;
        return c < limit ? c : limit;
    }
    int lo = 0, hi = limit;   // first index in [lo, hi] whose first key is >= n
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (tile_group_first_key(mid, g) < n)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

// Number of group indices a unit uses (rows have up to n_hi valid keys).
__host__ __device__ __forceinline__ int tile_groups_in_unit(int n_hi, int g) {
    if (g < 32) return (n_hi + g - 1) / g;
    const int m = g / 32;
    const int tiles = (n_hi + 127) / 128;
    const int per_buffer = (tiles + kTileGroups - 1) / kTileGroups;   // tiles of buffer 0
    return 4 * kTileGroups * ((per_buffer + m - 1) / m);
}

// Groups per unit that the group-maximum array reserves: a unit's rows have
// n_hi <= n_ref + 255 valid keys and g > n_ref / (4k), so a unit uses fewer
// than 4k + 256 / g + 28 indices.
__host__ __device__ __forceinline__ int tile_group_stride(int k) { return 4 * k + 288; }

// Candidate capacity per row: twice the next power of two >= k, split in two
// equal lists (one per TMEM tile buffer and its epilogue warps). The bound from the
// group maxima leaves about 1.25 k candidates; a row that fills one of its
// lists (heavy ties at its k-th score) is recomputed by the row-wise kernel.
__host__ __device__ __forceinline__ int tile_cand_cap(int k) {
    int c = 32;
    while (c < k) c *= 2;
    return 2 * c;
}

// Bits of a float and the order-preserving map of the finite floats onto
// uint32 used by the threshold search below (-0 and +0 get adjacent keys).
__host__ __device__ __forceinline__ uint32_t tile_f32_bits(float f) {
#ifdef __CUDA_ARCH__
    return __float_as_uint(f);
#else
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
#endif
}

__host__ __device__ __forceinline__ float tile_bits_f32(uint32_t u) {
#ifdef __CUDA_ARCH__
    return __uint_as_float(u);
#else
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
#endif
}

// Threshold on the unscaled dot products: the smallest float x with
// fl(x * scale) >= t (scale > 0). fl(x * scale) is non-decreasing in x, so
// `raw >= x` decides `fl(raw * scale) >= t` exactly without a multiply per
// score. t = -inf gives -FLT_MAX: every finite score qualifies, a masked
// (-inf) one does not; +inf when no finite score reaches t. The answer is
// found by bisection over the ordered finite floats (31 steps, once per row),
// not by stepping from t / scale: when the products are subnormal many
// consecutive x give the same product and the boundary can lie many ulps
// below the quotient.
__host__ __device__ __forceinline__ float tile_raw_threshold(float t, float scale) {
    if (t == -INFINITY) return -FLT_MAX;
    if (!(FLT_MAX * scale >= t)) return INFINITY;
    if (-FLT_MAX * scale >= t) return -FLT_MAX;
    // ordered keys: negative floats map to ~bits, non-negative ones to
    // bits | 2^31; lo fails the test, hi passes it
    uint32_t lo = ~tile_f32_bits(-FLT_MAX), hi = tile_f32_bits(FLT_MAX) | 0x80000000u;
    while (hi - lo > 1) {
        const uint32_t mid = lo + (hi - lo) / 2;
        const float x = tile_bits_f32((mid & 0x80000000u) ? (mid & 0x7FFFFFFFu) : ~mid);
        if (x * scale >= t)
            hi = mid;
        else
            lo = mid;
    }
    return tile_bits_f32((hi & 0x80000000u) ? (hi & 0x7FFFFFFFu) : ~hi);
}

struct TileParams {
    int BH, Tq, Tk, k, causal;
    float scale;
    int units_per_head, num_units;   // filled by the launcher
    int pair_units;                  // launcher: work items are unit pairs (see tile_scores.cu)
    float* S;                        // MODE_RAW: [BH, Tq, Tk]
    uint16_t* gm;                    // MODE_GROUPMAX: [units, G_stride, 256]
    int G_stride;
    const uint32_t* tau;             // MODE_COLLECT: [BH*Tq] order-key thresholds
    uint64_t* cand;                  // MODE_COLLECT: [BH*Tq, 2, cap/2] (raw score bits << 32) | index
    int32_t* cnt;                    // MODE_COLLECT: [BH*Tq, 2] candidates found
    int cap;                         // per row; half per TMEM tile buffer
    int32_t* dev_status;
    uint64_t wait_limit_ns;          // 0: one second
};

cudaError_t tile_scores_launch(const void* q_low, const void* k_low, int P, int mode,
                               TileParams p, cudaStream_t stream);
int tile_sm_count();

// Workspace of the tile path, carved from the caller's buffer (offsets in
// bytes, each 256-byte aligned).
struct TileWorkspace {
    size_t ovf_count, tau, cnt, ovf_list, gm, cand, rowwise, total;
    int64_t rowwise_slots, rowwise_stride;
};

inline TileWorkspace tile_workspace(int64_t BH, int Tq, int Tk, int k) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    TileWorkspace w;
    const int64_t rows = BH * Tq;
    const int64_t units = BH * ((Tq + kUnitM - 1) / kUnitM);
    size_t o = 0;
    w.ovf_count = o; o += 256;
    w.tau = o; o += up(rows * 4);
    w.cnt = o; o += up(rows * 8);
    w.ovf_list = o; o += up(rows * 8);
    w.gm = o; o += up(static_cast<size_t>(units) * tile_group_stride(k) * kUnitM * 2);
    w.cand = o; o += up(static_cast<size_t>(rows) * tile_cand_cap(k) * 8);
    w.rowwise_slots = rows < 256 ? rows : 256;
    w.rowwise_stride = (static_cast<int64_t>(Tk) + 63) / 64 * 64;
    w.rowwise = o; o += up(static_cast<size_t>(w.rowwise_slots) * w.rowwise_stride * 4);
    w.total = o;
    return w;
}

}  // namespace ssa
