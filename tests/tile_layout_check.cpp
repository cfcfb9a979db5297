// Host-side check of the group layout the tensor-core top-k relies on
// (dynamic_top_sparse_rank_b300/csrc/tile.h), built with g++ by
// tests/test_tile_layout.py. The exactness argument needs, for every row with
// more than k valid keys, a partition of its valid keys into more than k groups
// (the rule gives at least min(n, 2k)); the selection needs the groups holding a valid
// key to be exactly 0 .. count-1; the group-maximum array needs every group
// index a unit writes to stay below the reserved stride. The key -> group map
// is re-derived here from the score kernel's tile order (tile t of a unit goes
// to TMEM buffer t % 2; chunk c of 32 keys; m = g / 32 consecutive tiles of a
// buffer form a group), independently of tile_group_first_key. It also checks
// the candidate threshold on the unscaled dot products (tile_raw_threshold):
// for a bound t and scale s, a raw score x must pass `x >= threshold` exactly
// when fl(x * s) >= t, or the candidate pass would drop a key of the top-k.
// Host float arithmetic is IEEE single precision here, as the kernel's is
// (no fast-math, no flush to zero).
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

#include "tile.h"

using namespace ssa;

static int fails = 0;
#define CHECK(cond, ...)                      \
    do {                                      \
        if (!(cond)) {                        \
            if (fails < 20) {                 \
                std::printf("FAIL: ");        \
                std::printf(__VA_ARGS__);     \
                std::printf("\n");            \
            }                                 \
            ++fails;                          \
        }                                     \
    } while (0)

static int group_of_key(int j, int g) {
    if (g < 32) return j / g;
    const int m = g / 32;
    const int t = j / 128, b = t % 2, lt = t / 2, c = (j % 128) / 32;
    return ((lt / m) * 2 + b) * 4 + c;
}

int main() {
    // 1. layout: first keys increase, each key's group has it at or after the
    //    group's first key, and the first key is the smallest key of its group
    for (int g : {1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024}) {
        const int nmax = 1 << 17;
        std::vector<int> minkey(nmax + 1, -1);
        int maxgrp = -1;
        for (int j = 0; j < nmax; ++j) {
            const int grp = group_of_key(j, g);
            CHECK(grp >= 0 && grp <= nmax, "g %d key %d group %d", g, j, grp);
            if (minkey[grp] < 0) minkey[grp] = j;
            if (grp > maxgrp) maxgrp = grp;
            CHECK(tile_group_first_key(grp, g) <= j, "g %d key %d before its group's first key", g, j);
        }
        int prev = -1;
        for (int grp = 0; grp <= maxgrp; ++grp) {
            const int fk = tile_group_first_key(grp, g);
            CHECK(fk > prev, "g %d group %d first key %d not increasing", g, grp, fk);
            prev = fk;
            if (minkey[grp] >= 0)
                CHECK(minkey[grp] == fk, "g %d group %d first key %d, smallest key %d", g, grp, fk,
                      minkey[grp]);
        }
        // 2. the groups with a valid key are 0 .. tile_groups_of_row - 1
        for (int n = 1; n <= nmax; n = n < 4096 ? n + 1 : n + 997) {
            int count = 0;
            for (int grp = 0; grp <= maxgrp; ++grp)
                if (tile_group_first_key(grp, g) < n) ++count;
            CHECK(tile_groups_of_row(n, g, maxgrp + 1) == count, "g %d n %d count", g, n);
        }
    }
    // 3. the shapes of the workloads and of the parity tests: every unit's
    //    group indices stay below the stride; a row of n > k keys gets at
    //    least min(n, 2k) groups
    struct Shape {
        int Tq, Tk, k, causal;
    };
    const Shape shapes[] = {{131072, 131072, 512, 1}, {32768, 32768, 256, 1}, {4096, 4096, 64, 1},
                            {1000, 1000, 64, 1},       {1000, 5000, 100, 0},   {300, 700, 31, 0},
                            {5000, 1000, 64, 1},       {64, 64, 1, 1},         {129, 129, 128, 1},
                            {600, 600, 64, 1},         {131072, 131072, 32, 1}, {2048, 65536, 512, 0}};
    for (const Shape& s : shapes) {
        const int units = (s.Tq + kUnitM - 1) / kUnitM;
        for (int u = 0; u < units; ++u) {
            const int i0 = u * kUnitM, rows = (s.Tq - i0) < kUnitM ? (s.Tq - i0) : kUnitM;
            const int n_lo = tile_valid_count(i0, s.Tq, s.Tk, s.causal);
            const int n_hi = tile_valid_count(i0 + rows - 1, s.Tq, s.Tk, s.causal);
            const int g = tile_group_size(n_lo, n_hi, s.k);
            if (g == 0) {
                CHECK(n_hi <= s.k, "Tq %d unit %d: no groups but %d keys > k", s.Tq, u, n_hi);
                continue;
            }
            const int G_u = tile_groups_in_unit(n_hi, g);
            CHECK(G_u <= tile_group_stride(s.k), "Tq %d k %d unit %d: %d groups > stride %d", s.Tq,
                  s.k, u, G_u, tile_group_stride(s.k));
            // every key of every row maps below G_u
            CHECK(group_of_key(n_hi - 1, g) < G_u, "Tq %d unit %d: last key's group %d >= %d", s.Tq,
                  u, group_of_key(n_hi - 1, g), G_u);
            for (int r = 0; r < rows; ++r) {
                const int n = tile_valid_count(i0 + r, s.Tq, s.Tk, s.causal);
                if (n <= s.k) continue;
                const int G = tile_groups_of_row(n, g, G_u);
                const int want = n < 2 * s.k ? n : 2 * s.k;   // g = 1 at most gives n groups
                CHECK(G >= want && G > s.k, "Tq %d k %d row %d: %d keys, %d groups < min(n, 2k)",
                      s.Tq, s.k, i0 + r, n, G);
            }
        }
    }
    // 4. candidate capacity: each TMEM buffer's list holds at least k
    for (int k = 1; k <= 2048; ++k) CHECK(tile_cand_cap(k) / 2 >= k, "k %d cap %d", k, tile_cand_cap(k));
    // 5. the raw threshold is the exact boundary of {x finite : fl(x * s) >= t}
    {
        auto passes = [](float x, float t, float s) { return x * s >= t; };
        auto check_one = [&](float t, float s) {
            const float x = tile_raw_threshold(t, s);
            CHECK(x != -INFINITY && !std::isnan(x), "t %a s %a: threshold %a", t, s, x);
            if (x == INFINITY) {   // no finite score reaches t
                CHECK(!passes(FLT_MAX, t, s), "t %a s %a: +inf threshold but FLT_MAX passes", t, s);
                return;
            }
            CHECK(passes(x, t, s), "t %a s %a: threshold %a fails", t, s, x);
            if (x > -FLT_MAX) {
                const float below = std::nextafter(x, -INFINITY);
                CHECK(!passes(below, t, s), "t %a s %a: %a below the threshold %a passes", t, s,
                      below, x);
            }
        };
        auto from_bits = [](uint32_t u) {
            float f;
            std::memcpy(&f, &u, 4);
            return f;
        };
        std::vector<float> scales = {0.25f, 1.0f / std::sqrt(32.0f), 0.125f, 1.0f / std::sqrt(128.0f),
                                     1.0f, 1.25f, 10.0f, 0.01f, 3.0f, 1e-30f, 1e30f, FLT_MIN,
                                     1e-40f, 0.1f * 0.125f, 1.0f / 0.1f * 0.125f};
        uint64_t lcg = 0x9E3779B97F4A7C15ull;
        auto next32 = [&]() {
            lcg = lcg * 6364136223846793005ull + 1442695040888963407ull;
            return static_cast<uint32_t>(lcg >> 32);
        };
        for (int i = 0; i < 200; ++i)   // log-uniform in [2^-100, 2^100)
            scales.push_back(std::ldexp(1.0f + (next32() >> 9) * 0x1p-23f,
                                        static_cast<int>(next32() % 200) - 100));
        // every bound the selection can produce: an order key truncated to its
        // high 16 bits, decoded back to a float (finite ones only)
        for (uint32_t k16 = 1; k16 < 65536; ++k16) {
            const uint32_t key = k16 << 16;
            const uint32_t u = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
            const float t = from_bits(u);
            if (!std::isfinite(t)) continue;
            for (float s : scales) check_one(t, s);
        }
        check_one(-INFINITY, 0.125f);
        CHECK(tile_raw_threshold(-INFINITY, 0.125f) == -FLT_MAX, "t -inf must give -FLT_MAX");
        // arbitrary finite bounds, subnormals included
        for (int i = 0; i < 2000000; ++i) {
            const float t = from_bits(next32());
            if (!std::isfinite(t)) continue;
            check_one(t, scales[next32() % scales.size()]);
        }
    }
    if (fails) {
        std::printf("FAILED %d\n", fails);
        return 1;
    }
    std::printf("OK\n");
    return 0;
}
