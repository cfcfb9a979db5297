// The selection stages of the tensor-core top-k (tile_select.cu: the bound
// from the group maxima, the candidate sort) built for the host: see
// emu_device.h in this directory. The launches mirror the library's: 256
// threads per block; for the bound at most 3 x 148 blocks over the
// (unit, half) items; for the sort one warp per row, the template chosen by
// the candidate capacity. Compiled by tests/emu/tile_check.py.
#define SSA_HOST_EMULATION 1
#include "tile_select.cu"

extern "C" int emu_group_select(const uint16_t* gm, uint32_t* tau, int BH, int Tq, int Tk, int k,
                                int causal) {
    const int items = 2 * BH * ((Tq + ssa::kUnitM - 1) / ssa::kUnitM);
    if (items == 0) return 0;
    const unsigned grid = (unsigned)std::min(items, 3 * 148);
    emu_launch(grid, ssa::kSelThreads, [&] {
        ssa::group_select_kernel(gm, tau, BH, Tq, Tk, k, causal, ssa::tile_group_stride(k));
    });
    return 0;
}

extern "C" int emu_cand_sort(const uint64_t* cand, const int32_t* cnt, int64_t rows, int Tq,
                             int Tk, int k, int causal, float scale, int32_t* idx, float* score,
                             int64_t* ovf_list, int32_t* ovf_count, int32_t* dev_status) {
    const unsigned blocks = (unsigned)((rows + ssa::kSortWarps - 1) / ssa::kSortWarps);
    const int cap = ssa::tile_cand_cap(k);
#define C(NB)                                                                                   \
    if (cap == 32 * NB) {                                                                       \
        emu_launch(blocks, ssa::kSortWarps * 32, [&] {                                          \
            ssa::cand_sort_kernel<NB, NB / 2>(cand, cnt, rows, Tq, Tk, k, causal, scale, idx,   \
                                              score, ovf_list, ovf_count, dev_status);          \
        });                                                                                     \
        return 0;                                                                               \
    }
    C(2) C(4) C(8) C(16) C(32)
#undef C
    return 1;
}

extern "C" int emu_tile_cand_cap(int k) { return ssa::tile_cand_cap(k); }
extern "C" int emu_tile_group_stride(int k) { return ssa::tile_group_stride(k); }
