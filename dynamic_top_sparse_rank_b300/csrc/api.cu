// The C ABI of libssa.so: argument checks, workspace sizing, dispatch.
// Every call validates on the host and launches nothing on a bad argument.
#include <math.h>

#include "common.cuh"
#include "tile.h"

namespace ssa {
cudaError_t topk_rows_dispatch(const void* q_low, const void* k_low, bool bf16, int P,
                               const int64_t* row_list, int64_t rows, const int32_t* rows_dev,
                               int Tq, int Tk, int k, int causal, float scale, int32_t* idx,
                               float* score, uint32_t* ws, int64_t ws_slots, int64_t ws_stride,
                               cudaStream_t stream);
int topk_chunks_for(int Tk, int k);
size_t topk_chunks_workspace(int64_t rows, int Tk, int k);
cudaError_t topk_chunks_dispatch(const void* q_low, const void* k_low, bool bf16, int P,
                                 int64_t rows, int Tq, int Tk, int k, int causal, float scale,
                                 int32_t* idx, float* score, void* ws, cudaStream_t stream);
cudaError_t tile_select_launch(const uint16_t* gm, uint32_t* tau, int BH, int Tq, int Tk, int k,
                               int causal, cudaStream_t stream);
cudaError_t tile_sort_launch(const uint64_t* cand, const int32_t* cnt, int64_t rows, int Tq,
                             int Tk, int k, int causal, float scale, int32_t* idx, float* score,
                             int64_t* ovf_list, int32_t* ovf_count, int32_t* dev_status,
                             cudaStream_t stream);
cudaError_t lowrank_project_launch(const void* x, const void* W, int64_t rows, int d_model, int P,
                                   void* out, int32_t* dev_status, cudaStream_t stream);
bool window_tc_supported(bool bf16_in, int D, int T, int wl, int wr);
cudaError_t smooth_boundary_launch(int32_t* idx, float* score, int64_t rows, int k, float delta,
                                   cudaStream_t stream);
cudaError_t window_tc_launch(const void* Q, const void* K, const void* V, void* O, bool bf16_out,
                             int BH, int T, int D, int wl, int wr, float scale,
                             int32_t* dev_status, cudaStream_t stream);
template <bool BAND>
cudaError_t attn_rows_dispatch(const void* Q, const void* K, const void* V, bool bf16_in, int D,
                               const int32_t* idx, void* O, bool bf16_out, int64_t rows, int Tq,
                               int Tk, int k, int wl, int wr, float scale, int32_t* dev_status,
                               const HeadMap& hm, cudaStream_t stream);
}  // namespace ssa

namespace {

constexpr int kMaxK = 2048;
constexpr int64_t kRowSlots = 1024;   // row-wise top-k: concurrent rows with a workspace slot

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool dtype_ok(int d) { return d == SSA_F32 || d == SSA_BF16; }
bool p_ok(int P) { return P == 16 || P == 32 || P == 64 || P == 128; }
bool d_ok(int D) { return D == 64 || D == 128; }
// A scale is a finite factor (<= 0 selects the default); NaN and inf are rejected.
bool scale_ok(float s) { return isfinite(s); }
int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Row-wise path: one slot of Tk 32-bit keys per concurrently processed row.
int64_t rowwise_slots(int64_t rows) { return rows < kRowSlots ? rows : kRowSlots; }
int64_t rowwise_stride(int Tk) { return round_up((int64_t)Tk, 64); }

// The tensor-core path serves bf16 scorer inputs with d_proj 64 or 128 and
// k <= 512 when there are enough query rows per head to fill 128-row tiles,
// and at most 2^31 - 1 rows of q_low and of k_low (its TMA coordinates,
// head * T + row, are 32-bit); everything else (decode, fp32, other d_proj,
// larger k) runs row-wise.
bool use_tile_path(int dtype, int B, int H, int P, int Tq, int Tk, int k) {
    return dtype == SSA_BF16 && (P == 64 || P == 128) && k <= 512 && Tq >= 64 && Tk > 0 &&
           (int64_t)B * H * Tq <= INT32_MAX && (int64_t)B * H * Tk <= INT32_MAX;
}

// Rows that the row-wise path takes split into key chunks (one CTA per row
// and chunk): long rows (decode: one query per head against a long key
// cache), when there are too few of them for one CTA per row to fill the GPU
// and the chunks' selections fit a row's merge.
bool use_chunked_rows(int64_t rows, int Tk, int k) {
    return rows <= 4 * kRowSlots && ssa::topk_chunks_for(Tk, k) > 0;
}

}  // namespace

extern "C" {

int ssa_version(void) { return (0 << 16) | 1; }

const char* ssa_status_string(int status) {
    switch (status) {
        case SSA_OK: return "ok";
        case SSA_ERR_INVALID: return "invalid argument (null or misaligned pointer, bad size or dtype)";
        case SSA_ERR_UNSUPPORTED: return "unsupported size (P in {16,32,64,128}, D in {64,128}, k <= 2048)";
        case SSA_ERR_CUDA: return "CUDA launch or runtime error";
        case SSA_ERR_TIMEOUT: return "a bounded device-side wait ran out";
        case SSA_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

ssa_status ssa_device_status(const int32_t* dev_status, int32_t* bits, void* stream) {
    if (!dev_status || !aligned(dev_status, 4)) return SSA_ERR_INVALID;
    int32_t h = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&h, dev_status, sizeof h, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return SSA_ERR_CUDA;
    if (bits) *bits = h;
    if (h & SSA_DEV_WAIT_LIMIT) return SSA_ERR_TIMEOUT;
    if (h & SSA_DEV_BAD_INDEX) return SSA_ERR_INVALID;
    return SSA_OK;
}

static size_t path_workspace_bytes(int dtype, int B, int H, int Tq, int Tk, int P, int k) {
    const int64_t rows = (int64_t)B * H * Tq;
    if (rows == 0 || Tk == 0) return 256;
    if (use_tile_path(dtype, B, H, P, Tq, Tk, k))
        return ssa::tile_workspace((int64_t)B * H, Tq, Tk, k).total;
    if (use_chunked_rows(rows, Tk, k)) return ssa::topk_chunks_workspace(rows, Tk, k);
    return (size_t)round_up(rowwise_slots(rows) * rowwise_stride(Tk) * 4, 256);
}

size_t ssa_score_topk_workspace_size(int B, int H, int Tq, int Tk, int P, int k, int causal) {
    (void)causal;
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0 || !p_ok(P) || k < 1 || k > kMaxK) return 0;
    // the larger of the two paths' needs, so the size does not depend on dtype
    const size_t a = path_workspace_bytes(SSA_BF16, B, H, Tq, Tk, P, k);
    const size_t b = path_workspace_bytes(SSA_F32, B, H, Tq, Tk, P, k);
    return a > b ? a : b;
}

ssa_status ssa_score_topk(const void* q_low, const void* k_low, int dtype, int B, int H, int Tq,
                          int Tk, int P, int k, int causal, float scale, int32_t* idx,
                          float* score, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream) {
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0 || !dtype_ok(dtype) || k < 1 || !scale_ok(scale))
        return SSA_ERR_INVALID;
    if (!p_ok(P) || k > kMaxK) return SSA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * H * Tq;
    if (rows == 0) return SSA_OK;
    if (!idx || !aligned(idx, 4) || (score && !aligned(score, 4))) return SSA_ERR_INVALID;
    if (!q_low || !aligned(q_low, 16)) return SSA_ERR_INVALID;
    if (Tk > 0 && (!k_low || !aligned(k_low, 16))) return SSA_ERR_INVALID;
    if (dev_status && !aligned(dev_status, 4)) return SSA_ERR_INVALID;
    const size_t need = path_workspace_bytes(dtype, B, H, Tq, Tk, P, k);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return SSA_ERR_WORKSPACE;
    const float sc = scale > 0.f ? scale : (float)(1.0 / sqrt((double)P));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!use_tile_path(dtype, B, H, P, Tq, Tk, k)) {
        if (use_chunked_rows(rows, Tk, k)) {
            cudaError_t e = ssa::topk_chunks_dispatch(q_low, k_low, dtype == SSA_BF16, P, rows, Tq,
                                                      Tk, k, causal, sc, idx, score, workspace, s);
            return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
        }
        // Tk == 0: every row is empty; the row kernel writes the padding.
        cudaError_t e = ssa::topk_rows_dispatch(q_low, k_low, dtype == SSA_BF16, P, nullptr, rows,
                                                nullptr, Tq, Tk, k, causal, sc, idx, score,
                                                reinterpret_cast<uint32_t*>(workspace),
                                                rowwise_slots(rows), rowwise_stride(Tk), s);
        return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
    }
    // tensor-core path: group maxima -> per-row bound -> candidates -> sort,
    // rows whose candidates overflow redone row-wise
    const int BH = B * H;
    const ssa::TileWorkspace w = ssa::tile_workspace(BH, Tq, Tk, k);
    char* ws = reinterpret_cast<char*>(workspace);
    int32_t* ovf_count = reinterpret_cast<int32_t*>(ws + w.ovf_count);
    uint32_t* tau = reinterpret_cast<uint32_t*>(ws + w.tau);
    int32_t* cnt = reinterpret_cast<int32_t*>(ws + w.cnt);
    int64_t* ovf_list = reinterpret_cast<int64_t*>(ws + w.ovf_list);
    uint16_t* gm = reinterpret_cast<uint16_t*>(ws + w.gm);
    uint64_t* cand = reinterpret_cast<uint64_t*>(ws + w.cand);
    ssa::TileParams p = {};
    p.BH = BH;
    p.Tq = Tq;
    p.Tk = Tk;
    p.k = k;
    p.causal = causal ? 1 : 0;
    p.scale = sc;
    p.gm = gm;
    p.G_stride = ssa::tile_group_stride(k);
    p.tau = tau;
    p.cand = cand;
    p.cnt = cnt;
    p.cap = ssa::tile_cand_cap(k);
    p.dev_status = dev_status;
    cudaError_t e = cudaMemsetAsync(ovf_count, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = ssa::tile_scores_launch(q_low, k_low, P, ssa::MODE_GROUPMAX, p, s);
    if (e == cudaSuccess) e = ssa::tile_select_launch(gm, tau, BH, Tq, Tk, k, p.causal, s);
    if (e == cudaSuccess) e = ssa::tile_scores_launch(q_low, k_low, P, ssa::MODE_COLLECT, p, s);
    if (e == cudaSuccess)
        e = ssa::tile_sort_launch(cand, cnt, rows, Tq, Tk, k, p.causal, sc, idx, score,
                                  ovf_list, ovf_count, dev_status, s);
    if (e == cudaSuccess)
        e = ssa::topk_rows_dispatch(q_low, k_low, true, P, ovf_list, rows, ovf_count, Tq, Tk, k,
                                    p.causal, sc, idx, score,
                                    reinterpret_cast<uint32_t*>(ws + w.rowwise), w.rowwise_slots,
                                    w.rowwise_stride, s);
    return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
}

ssa_status ssa_lowrank_scores(const void* q_low, const void* k_low, int dtype, int B, int H,
                              int Tq, int Tk, int P, int causal, float scale, float* S,
                              int32_t* dev_status, void* stream) {
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0 || !dtype_ok(dtype) || !scale_ok(scale))
        return SSA_ERR_INVALID;
    if (!p_ok(P)) return SSA_ERR_UNSUPPORTED;
    if (dtype != SSA_BF16 || !(P == 64 || P == 128)) return SSA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * H * Tq;
    if (rows == 0 || Tk == 0) return SSA_OK;
    if (rows > INT32_MAX || (int64_t)B * H * Tk > INT32_MAX) return SSA_ERR_UNSUPPORTED;
    if (!S || !aligned(S, 4) || !q_low || !k_low || !aligned(q_low, 16) || !aligned(k_low, 16))
        return SSA_ERR_INVALID;
    if (dev_status && !aligned(dev_status, 4)) return SSA_ERR_INVALID;
    ssa::TileParams p = {};
    p.BH = B * H;
    p.Tq = Tq;
    p.Tk = Tk;
    p.k = 1;
    p.causal = causal ? 1 : 0;
    p.scale = scale > 0.f ? scale : (float)(1.0 / sqrt((double)P));
    p.S = S;
    p.dev_status = dev_status;
    cudaError_t e = ssa::tile_scores_launch(q_low, k_low, P, ssa::MODE_RAW, p,
                                            reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
}

size_t ssa_score_topk_smooth_workspace_size(int B, int H, int Tq, int Tk, int P, int k,
                                            int causal) {
    if (k < 1 || k >= kMaxK) return 0;   // the selection runs with k + 1 <= kMaxK
    const size_t a = ssa_score_topk_workspace_size(B, H, Tq, Tk, P, k + 1, causal);
    if (a == 0) return 0;
    const int64_t rows = (int64_t)B * H * Tq;
    return (size_t)round_up((int64_t)a, 256) + (size_t)round_up(rows * (k + 1) * 4, 256);
}

ssa_status ssa_score_topk_smooth(const void* q_low, const void* k_low, int dtype, int B, int H,
                                 int Tq, int Tk, int P, int k, int causal, float scale,
                                 float delta, int32_t* idx, float* score, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0 || !dtype_ok(dtype) || k < 1 || !scale_ok(scale) ||
        isnan(delta))
        return SSA_ERR_INVALID;
    if (!p_ok(P) || k >= kMaxK) return SSA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * H * Tq;
    if (rows == 0) return SSA_OK;
    const size_t a = ssa_score_topk_workspace_size(B, H, Tq, Tk, P, k + 1, causal);
    const size_t need = ssa_score_topk_smooth_workspace_size(B, H, Tq, Tk, P, k, causal);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return SSA_ERR_WORKSPACE;
    // scores of the k+1 selection: the caller's, else scratch after the selection's workspace
    float* sc = score ? score
                      : reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                 round_up((int64_t)a, 256));
    const ssa_status st = ssa_score_topk(q_low, k_low, dtype, B, H, Tq, Tk, P, k + 1, causal,
                                         scale, idx, sc, workspace, a, dev_status, stream);
    if (st != SSA_OK) return st;
    cudaError_t e = ssa::smooth_boundary_launch(idx, sc, rows, k, delta,
                                                reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
}

ssa_status ssa_lowrank_project(const void* x, const void* W, int dtype, int64_t rows, int d_model,
                               int P, void* out, int32_t* dev_status, void* stream) {
    if (rows < 0 || d_model <= 0 || !dtype_ok(dtype)) return SSA_ERR_INVALID;
    if (dtype != SSA_BF16 || !(P == 64 || P == 128) || d_model % 64 != 0) return SSA_ERR_UNSUPPORTED;
    if (rows > INT32_MAX) return SSA_ERR_UNSUPPORTED;   // 32-bit TMA row coordinates
    if (rows == 0) return SSA_OK;
    if (!x || !W || !out || !aligned(x, 16) || !aligned(W, 16) || !aligned(out, 16))
        return SSA_ERR_INVALID;
    if (dev_status && !aligned(dev_status, 4)) return SSA_ERR_INVALID;
    cudaError_t e = ssa::lowrank_project_launch(x, W, rows, d_model, P, out, dev_status,
                                                reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
}

ssa_status ssa_sparse_attn(const void* Q, const void* K, const void* V, int dtype, int B, int H,
                           int Tq, int Tk, int D, const int32_t* idx, int k, float scale, void* O,
                           int out_dtype, int32_t* dev_status, void* stream) {
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0 || k < 1 || !dtype_ok(dtype) || !dtype_ok(out_dtype) ||
        !scale_ok(scale))
        return SSA_ERR_INVALID;
    if (!d_ok(D)) return SSA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * H * Tq;
    if (rows == 0) return SSA_OK;
    if (!Q || !K || !V || !idx || !O) return SSA_ERR_INVALID;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(idx, 4))
        return SSA_ERR_INVALID;
    if (dev_status && !aligned(dev_status, 4)) return SSA_ERR_INVALID;
    const float sc = scale > 0.f ? scale : (float)(1.0 / sqrt((double)D));
    cudaError_t e = ssa::attn_rows_dispatch<false>(Q, K, V, dtype == SSA_BF16, D, idx, O,
                                                   out_dtype == SSA_BF16, rows, Tq, Tk, k, 0, 0,
                                                   sc, dev_status, ssa::HeadMap{1, 1, 1, 0, 0},
                                                   reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
}

ssa_status ssa_sparse_attn_grouped(const void* Q, const void* K, const void* V, int dtype, int B,
                                   int H, int H_kv, int Tq, int Tk, int D, const int32_t* idx,
                                   int H_idx, int k, float scale, void* O, int out_dtype,
                                   int32_t* dev_status, void* stream) {
    if (B < 0 || H < 1 || H_kv < 1 || H_idx < 1 || Tq < 0 || Tk < 0 || k < 1 || !dtype_ok(dtype) ||
        !dtype_ok(out_dtype) || H % H_kv != 0 || H % H_idx != 0 || !scale_ok(scale))
        return SSA_ERR_INVALID;
    if (!d_ok(D)) return SSA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * H * Tq;
    if (rows == 0) return SSA_OK;
    if (!Q || !K || !V || !idx || !O) return SSA_ERR_INVALID;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(idx, 4))
        return SSA_ERR_INVALID;
    if (dev_status && !aligned(dev_status, 4)) return SSA_ERR_INVALID;
    const float sc = scale > 0.f ? scale : (float)(1.0 / sqrt((double)D));
    ssa::HeadMap hm{H, H_kv, H_idx, 1, H_kv < H ? 1 : 0};
    cudaError_t e = ssa::attn_rows_dispatch<false>(Q, K, V, dtype == SSA_BF16, D, idx, O,
                                                   out_dtype == SSA_BF16, rows, Tq, Tk, k, 0, 0,
                                                   sc, dev_status, hm,
                                                   reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
}

ssa_status ssa_window_attn(const void* Q, const void* K, const void* V, int dtype, int B, int H,
                           int T, int D, int w_left, int w_right, float scale, void* O,
                           int out_dtype, int32_t* dev_status, void* stream) {
    if (B < 0 || H < 0 || T < 0 || w_left < 0 || w_right < 0 || !dtype_ok(dtype) ||
        !dtype_ok(out_dtype) || !scale_ok(scale))
        return SSA_ERR_INVALID;
    if (!d_ok(D)) return SSA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * H * T;
    if (rows == 0) return SSA_OK;
    if (!Q || !K || !V || !O) return SSA_ERR_INVALID;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16))
        return SSA_ERR_INVALID;
    if (dev_status && !aligned(dev_status, 4)) return SSA_ERR_INVALID;
    const float sc = scale > 0.f ? scale : (float)(1.0 / sqrt((double)D));
    // a radius beyond the sequence changes nothing; clamping keeps i + w in int range
    if (w_left > T) w_left = T;
    if (w_right > T) w_right = T;
    cudaError_t e;
    if (ssa::window_tc_supported(dtype == SSA_BF16, D, T, w_left, w_right)) {
        // dense band tiles on the tensor cores
        e = ssa::window_tc_launch(Q, K, V, O, out_dtype == SSA_BF16, B * H, T, D, w_left, w_right,
                                  sc, dev_status, reinterpret_cast<cudaStream_t>(stream));
    } else {
        e = ssa::attn_rows_dispatch<true>(Q, K, V, dtype == SSA_BF16, D, nullptr, O,
                                          out_dtype == SSA_BF16, rows, T, T, 1, w_left, w_right,
                                          sc, dev_status, ssa::HeadMap{1, 1, 1, 0, 0},
                                          reinterpret_cast<cudaStream_t>(stream));
    }
    return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA;
}

}  // extern "C"
