// The forward's CUDA-core kernels (row-wise top-k and its long-row chunks, gather and window
// attention, boundary smoothing) built for the host: see emu_device.h in this
// directory. The launches mirror the library's: one 512-thread block per
// row-wise top-k row (a grid of min(rows, slots) blocks), one warp per
// attention row in 256-thread blocks, 256 rows per smoothing block. Compiled
// by tests/emu/fwd_check.py.
#define SSA_HOST_EMULATION 1
#include "attn_rows.cu"
#include "select_variants.cu"
#include "topk_rows.cu"

extern "C" int emu_topk_rows(const void* q_low, const void* k_low, int bf16, int P,
                             const int64_t* row_list, int64_t rows, int Tq, int Tk, int k,
                             int causal, float scale, int32_t* idx, float* score, uint32_t* ws,
                             int64_t ws_slots, int64_t ws_stride) {
    const unsigned grid = (unsigned)std::min<int64_t>(rows, ws_slots);
#define C(BF, PP)                                                                          \
    if (bf16 == BF && P == PP) {                                                           \
        emu_launch(grid, ssa::TOPK_THREADS, [&] {                                          \
            ssa::topk_rows_kernel<BF, PP>(q_low, k_low, row_list, rows, nullptr, Tq, Tk, k, \
                                          causal, scale, idx, score, ws, ws_stride);       \
        });                                                                                \
        return 0;                                                                          \
    }
    C(1, 16) C(1, 32) C(1, 64) C(1, 128) C(0, 16) C(0, 32) C(0, 64) C(0, 128)
#undef C
    return 1;
}

// The long-row path: one 256-thread block per (row, key chunk), then one
// 512-thread block per row for the merge, as the library launches them.
extern "C" int emu_topk_chunks(const void* q_low, const void* k_low, int bf16, int P, int64_t rows,
                               int Tq, int Tk, int k, int causal, float scale, int32_t* idx,
                               float* score, uint64_t* cand, int32_t* cnt) {
    const int nchunks = ssa::topk_chunk_count(Tk, k);
    if (nchunks == 0) return 2;
    const unsigned blocks = (unsigned)(rows * nchunks);
#define C(BF, PP)                                                                             \
    if (bf16 == BF && P == PP) {                                                              \
        emu_launch(blocks, ssa::kChunkThreads, [&] {                                          \
            ssa::topk_chunk_kernel<BF, PP>(q_low, k_low, nchunks, Tq, Tk, k, causal, scale,   \
                                           cand, cnt);                                        \
        });                                                                                   \
    } else
    C(1, 16) C(1, 32) C(1, 64) C(1, 128) C(0, 16) C(0, 32) C(0, 64) C(0, 128) return 1;
#undef C
    emu_launch((unsigned)rows, ssa::kMergeThreads, [&] {
        ssa::topk_merge_kernel(cand, cnt, nchunks, Tq, Tk, k, causal, idx, score);
    });
    return 0;
}

extern "C" int emu_topk_chunk_count(int Tk, int k) { return ssa::topk_chunk_count(Tk, k); }

extern "C" int emu_attn_rows(const void* Q, const void* K, const void* V, int bf16_in, int D,
                             const int32_t* idx, void* O, int bf16_out, int64_t rows, int Tq,
                             int Tk, int k, int wl, int wr, float scale, int32_t* dev_status,
                             int H, int H_kv, int H_idx, int grouped, int head_inner, int band) {
    const ssa::HeadMap hm{H, H_kv, H_idx, grouped, head_inner};
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    const float sl2 = scale * ssa::kLog2e;
#define C(BI, DD, BO, BA)                                                                     \
    if (bf16_in == BI && D == DD && bf16_out == BO && band == BA) {                           \
        emu_launch(blocks, 256, [&] {                                                         \
            ssa::attn_rows_kernel<BI, DD, BO, BA>(Q, K, V, idx, O, rows, Tq, Tk, k, wl, wr, sl2, \
                                                  dev_status, hm);                            \
        });                                                                                   \
        return 0;                                                                             \
    }
    C(1, 64, 1, 0) C(1, 64, 0, 0) C(1, 128, 1, 0) C(1, 128, 0, 0)
    C(0, 64, 1, 0) C(0, 64, 0, 0) C(0, 128, 1, 0) C(0, 128, 0, 0)
    C(1, 64, 1, 1) C(1, 64, 0, 1) C(1, 128, 1, 1) C(1, 128, 0, 1)
    C(0, 64, 1, 1) C(0, 64, 0, 1) C(0, 128, 1, 1) C(0, 128, 0, 1)
#undef C
    return 1;
}

extern "C" int emu_smooth(int32_t* idx, float* score, int64_t rows, int k, float delta) {
    emu_launch((unsigned)((rows + 255) / 256), 256,
               [&] { ssa::smooth_boundary_kernel(idx, score, rows, k, delta); });
    return 0;
}
