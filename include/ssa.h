/*
 * ssa.h — C ABI of the dynamic top-k sparse attention library (libssa.so).
 *
 * The library computes the forward pass of dynamic top-k sparse attention on
 * one NVIDIA B300 (sm_103a), in three calls:
 *
 *   ssa_score_topk   low-rank scorer S = q_low . k_low^T * d_proj^-0.5 fused
 *                    with an exact per-query top-k key selection
 *                    (mhpq.cn/news/1098205, sections 2.2 and 3.2);
 *   ssa_sparse_attn  softmax(q . K_sel^T / sqrt(d)) . V_sel over the selected
 *                    keys only (same page, section 3.2; scaled dot-product
 *                    attention as in "Attention机制优化：原理、挑战与工程实践",
 *                    section 1.1, with the online softmax of its section 2.3.1);
 *   ssa_window_attn  sliding-window attention, keys |i - j| <= w clipped at
 *                    the sequence ends (nxmr.cn/news/163144, section 2.2).
 *
 * Conventions shared by every call
 *  - Pointers named as device pointers must point to device memory of the
 *    current CUDA device; the caller owns every buffer. The library allocates
 *    no device memory in these calls: scratch space is the caller's
 *    `workspace`.
 *  - Layouts are dense row-major: [B, H, T, d] means element (b, h, t, e) sits
 *    at ((b*H + h)*T + t)*d + e. Every device pointer must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *    asynchronous on that stream and return after the launch.
 *  - Host-detectable errors (null pointers, unsupported sizes, misalignment,
 *    a workspace that is too small, a NaN or infinite `scale` or a NaN
 *    `delta`) return a status synchronously and launch nothing. A failed
 *    launch returns SSA_ERR_CUDA.
 *  - Errors found on the device (an index out of range, a bounded wait that
 *    ran out) never trap: the kernel ORs a bit into *dev_status (an int32 in
 *    device memory, may be NULL) and carries on or returns. The caller clears
 *    *dev_status and reads it back when it wants to know, directly or through
 *    ssa_device_status, which turns a wait that ran out into SSA_ERR_TIMEOUT.
 *  - Nothing is thrown across the ABI.
 */
#ifndef SSA_H_
#define SSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes of every call. */
typedef enum {
    SSA_OK = 0,
    SSA_ERR_INVALID = 1,     /* null pointer, negative size, bad enum value, misaligned pointer */
    SSA_ERR_UNSUPPORTED = 2, /* a size outside the supported set (see each call) */
    SSA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    SSA_ERR_TIMEOUT = 4,     /* a bounded device-side wait ran out (from ssa_device_status) */
    SSA_ERR_WORKSPACE = 5    /* workspace NULL or smaller than the size query returned */
} ssa_status;

/* Element types of tensors at the ABI. */
typedef enum {
    SSA_F32 = 0,  /* IEEE binary32 */
    SSA_BF16 = 1  /* bfloat16 (upper 16 bits of a binary32) */
} ssa_dtype;

/* Bits ORed into *dev_status by kernels. */
#define SSA_DEV_BAD_INDEX 0x1   /* an index list entry outside [-1, Tk); the entry is skipped */
#define SSA_DEV_WAIT_LIMIT 0x2  /* a bounded device-side wait ran out; the tile is abandoned */
#define SSA_DEV_OVERFLOW 0x4    /* a row's candidate list overflowed (a key above the bound found it
                                   full); the row was redone exactly by the row-wise kernel */

/*
 * ssa_device_status — turns the device-side error bits into a status.
 *
 * Boundary plumbing, with no counterpart on the pages: the host end of the
 * error rule above.
 *
 * Waits for the work queued on `stream` so far, reads *dev_status (the int32
 * the calls above OR their device-side bits into) and returns:
 *   SSA_ERR_TIMEOUT  if SSA_DEV_WAIT_LIMIT is set (a bounded wait of a
 *                    tensor-core kernel ran out; that kernel's outputs are
 *                    incomplete),
 *   SSA_ERR_INVALID  else if SSA_DEV_BAD_INDEX is set (an index list held an
 *                    entry outside [-1, Tk); it was skipped),
 *   SSA_OK           otherwise (SSA_DEV_OVERFLOW alone is informational: the
 *                    rows were redone exactly).
 * The raw bits are written to *bits when bits is not NULL. *dev_status is
 * not cleared. A failed CUDA call returns SSA_ERR_CUDA; a NULL or misaligned
 * dev_status returns SSA_ERR_INVALID.
 *
 *   dev_status  device int32, 4-byte aligned
 *   bits        host int32 or NULL
 *   stream      cudaStream_t the calls ran on (synchronized)
 */
ssa_status ssa_device_status(const int32_t* dev_status, int32_t* bits, void* stream);

/* Library version, (major << 16) | minor. */
int ssa_version(void);

/* Static text for a status code (never NULL). */
const char* ssa_status_string(int status);

/*
 * Bytes of device workspace ssa_score_topk needs for these sizes (0 if the
 * sizes are unsupported). Depends only on the arguments.
 */
size_t ssa_score_topk_workspace_size(int B, int H, int Tq, int Tk, int P, int k, int causal);

/*
 * ssa_score_topk — low-rank scorer fused with exact per-query top-k.
 *
 * Source: mhpq.cn/news/1098205, section 2.2 (scores = q_low . k_low^T scaled by
 * d_proj^-0.5) and section 3.2 (torch.topk over the scores; top_k =
 * min(top_k, seq_len); masked positions get -inf before selection so they are
 * never selected).
 *
 * For every query row (b, h, i), with the valid key set
 *   valid(i) = [0, Tk)                                    if causal == 0,
 *   valid(i) = { j : 0 <= j <= i + (Tk - Tq), j < Tk }    if causal != 0
 *              (bottom-right alignment: the last query sees every key),
 * the score of key j is s_j = fp32(sum_p q_low[b,h,i,p] * k_low[b,h,j,p]) *
 * scale, products and sums in fp32 (bf16 inputs are exact in fp32; integer
 * valued inputs give exact scores). For bf16 inputs with P in {64, 128},
 * k <= 512, Tq >= 64 and B*H*Tq, B*H*Tk below 2^31 the sum runs on the tensor cores with fp32
 * accumulation in the hardware's order (the scores ssa_lowrank_scores
 * returns); otherwise as a sequential fp32 sum. The selection is exact for
 * the scores so computed. The call writes the k_eff = min(k,
 * |valid(i)|) valid keys with the largest scores, ordered by score
 * descending, equal scores by key index ascending (the lower index wins a tie).
 * Slots k_eff..k-1 hold index -1 and score -inf.
 *
 *   q_low     device, [B, H, Tq, P], dtype `dtype`
 *   k_low     device, [B, H, Tk, P], dtype `dtype`
 *   dtype     SSA_F32 or SSA_BF16
 *   P         d_proj, one of 16, 32, 64, 128
 *   k         1 <= k <= 2048
 *   scale     score scale; <= 0 selects fp32(1 / sqrt(P))
 *   idx       device, int32 [B, H, Tq, k], written
 *   score     device, float [B, H, Tq, k], written; may be NULL
 *   workspace device scratch of at least ssa_score_topk_workspace_size(...)
 *             bytes, 256-byte aligned (its contents on entry do not matter;
 *             it is overwritten)
 *   dev_status device int32 or NULL (see conventions)
 *   stream    cudaStream_t
 *
 * Returns SSA_OK, SSA_ERR_INVALID, SSA_ERR_UNSUPPORTED, SSA_ERR_WORKSPACE or
 * SSA_ERR_CUDA. B*H*Tq == 0 is valid and launches nothing.
 */
ssa_status ssa_score_topk(const void* q_low, const void* k_low, int dtype, int B, int H, int Tq,
                          int Tk, int P, int k, int causal, float scale, int32_t* idx,
                          float* score, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream);

/*
 * ssa_score_topk_smooth — the top-k with boundary smoothing.
 *
 * Source: mhpq.cn/news/1098205, section 4.2: when the k-th and the (k+1)-th
 * scores differ by less than a threshold, both are selected, so that k varies
 * a little and near-ties at the boundary do not flip between runs. (The
 * temperature of the same section, scores / T, is the `scale` argument:
 * scale = d_proj^-0.5 / T; a positive factor leaves the ordering unchanged.)
 *
 * Runs the exact selection of ssa_score_topk with k + 1 (same scores, order
 * and tie rule; the tensor-core path while k + 1 <= 512), then keeps slot k
 * (the (k+1)-th key) only if it holds a key and fp32(score[k-1] - score[k]) <
 * delta; otherwise slot k becomes index -1 / score -inf. delta <= 0 gives the
 * plain top-k in the first k slots.
 *
 *   idx       device, int32 [B, H, Tq, k + 1], written
 *   score     device, float [B, H, Tq, k + 1], written; may be NULL
 *   workspace at least ssa_score_topk_smooth_workspace_size(...) bytes,
 *             256-byte aligned
 *   other arguments as ssa_score_topk; 1 <= k <= 2047.
 *
 * The index lists feed ssa_sparse_attn with k + 1 entries per row (-1
 * entries are skipped).
 */
size_t ssa_score_topk_smooth_workspace_size(int B, int H, int Tq, int Tk, int P, int k, int causal);
ssa_status ssa_score_topk_smooth(const void* q_low, const void* k_low, int dtype, int B, int H,
                                 int Tq, int Tk, int P, int k, int causal, float scale,
                                 float delta, int32_t* idx, float* score, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * ssa_lowrank_scores — the low-rank scorer alone, materialised.
 *
 * Source: mhpq.cn/news/1098205, section 2.2 (scores = q_low . k_low^T scaled
 * by d_proj^-0.5, a [b, h, n, n] tensor) with the masking of section 3.2,
 * note 3 (masked positions hold -inf).
 *
 * S[b,h,i,j] = fp32(sum_p q_low[b,h,i,p] * k_low[b,h,j,p]) * scale for j in
 * valid(i) (as defined for ssa_score_topk), -inf otherwise. The contraction
 * runs on the tensor cores with fp32 accumulation; it is the same contraction
 * ssa_score_topk uses, so for bf16 inputs S holds exactly the scores that call
 * ranks (integer-valued inputs give exact scores).
 *
 *   q_low     device, [B, H, Tq, P], bf16
 *   k_low     device, [B, H, Tk, P], bf16
 *   P         64 or 128 (other d_proj or fp32 inputs: SSA_ERR_UNSUPPORTED)
 *   scale     <= 0 selects fp32(1 / sqrt(P))
 *   S         device, float [B, H, Tq, Tk], written (B*H*Tq*Tk*4 bytes:
 *             meant for inspection and small problems)
 *   dev_status device int32 or NULL
 *
 * Returns SSA_OK, SSA_ERR_INVALID, SSA_ERR_UNSUPPORTED or SSA_ERR_CUDA.
 */
ssa_status ssa_lowrank_scores(const void* q_low, const void* k_low, int dtype, int B, int H,
                              int Tq, int Tk, int P, int causal, float scale, float* S,
                              int32_t* dev_status, void* stream);

/*
 * ssa_lowrank_project — the scorer's low-rank projection on the tensor cores.
 *
 * Source: mhpq.cn/news/1098205, section 2.2: the lightweight scorer maps the
 * query and the key of every head from d_model to d_proj with bias-free
 * linear layers, q_low = q_proj(query), k_low = k_proj(key); this call is one
 * such map, run once for the queries and once for the keys.
 *
 *   out[r, p] = bf16( sum_c x[r, c] * W[p, c] )   for r < rows, p < P,
 *
 * products and sums in fp32 on the tensor cores (the hardware's summation
 * order), rounded once to bf16 (round to nearest even). Integer-valued inputs
 * whose sums stay below 2^24 in magnitude give the exact sum.
 *
 *   x        device, bf16 [rows, d_model] (for a [B, H, T, d_model] input,
 *            rows = B*H*T), 16-byte aligned
 *   W        device, bf16 [P, d_model] (a linear layer's weight), 16-byte aligned
 *   dtype    SSA_BF16 (SSA_F32 returns SSA_ERR_UNSUPPORTED)
 *   rows     0 <= rows <= 2^31 - 1 (larger: SSA_ERR_UNSUPPORTED)
 *   d_model  a positive multiple of 64
 *   P        64 or 128
 *   out      device, bf16 [rows, P], written, 16-byte aligned (feeds
 *            ssa_score_topk as q_low or k_low)
 *   dev_status device int32 or NULL (see conventions)
 *   stream   cudaStream_t
 *
 * Returns SSA_OK, SSA_ERR_INVALID, SSA_ERR_UNSUPPORTED or SSA_ERR_CUDA.
 * rows == 0 is valid and launches nothing.
 */
ssa_status ssa_lowrank_project(const void* x, const void* W, int dtype, int64_t rows, int d_model,
                               int P, void* out, int32_t* dev_status, void* stream);

/*
 * ssa_sparse_attn — attention over the selected keys only.
 *
 * Source: mhpq.cn/news/1098205, section 3.2 (gather the selected K and V,
 * logits = q . k * head_dim^-0.5, softmax, weighted sum of V); the softmax is
 * the online (running max and sum) form of "Attention机制优化：原理、挑战与工程
 * 实践", section 2.3.1, kept in fp32 as its section 4.2 advises.
 *
 * For every query row (b, h, i):
 *   O[b,h,i,:] = sum_t softmax_t(Q[b,h,i,:] . K[b,h,idx_t,:] * scale) V[b,h,idx_t,:]
 * over the entries idx_t = idx[b,h,i,t], t < k, with idx_t != -1. Repeated
 * entries count once per occurrence. Entries outside [-1, Tk) set
 * SSA_DEV_BAD_INDEX in *dev_status and are skipped. A row with no usable
 * entry outputs zeros. Arithmetic is fp32 (inputs converted exactly).
 *
 *   Q         device, [B, H, Tq, D], dtype `dtype`
 *   K, V      device, [B, H, Tk, D], dtype `dtype`
 *   D         head_dim, 64 or 128
 *   idx       device, int32 [B, H, Tq, k] (as written by ssa_score_topk)
 *   k         >= 1
 *   scale     logit scale; <= 0 selects 1 / sqrt(D)
 *   O         device, [B, H, Tq, D], dtype `out_dtype`, written
 *             (bf16 output is rounded to nearest even)
 */
ssa_status ssa_sparse_attn(const void* Q, const void* K, const void* V, int dtype, int B, int H,
                           int Tq, int Tk, int D, const int32_t* idx, int k, float scale, void* O,
                           int out_dtype, int32_t* dev_status, void* stream);

/*
 * ssa_sparse_attn_grouped — ssa_sparse_attn with heads that share keys,
 * values or index lists.
 *
 * Source: mhpq.cn/news/1098205, section 3.2: the scorer may be shared by all
 * heads ([batch, seq_len, d_proj]) and its index list broadcast to every head;
 * "Attention机制优化：原理、挑战与工程实践" (bjdmk.com.cn), sections 3.1-3.2:
 * grouped-query and multi-query attention, where groups of query heads read
 * one key/value head.
 *
 * Query head h (of H) attends, for its row i, the keys listed in index row
 * (b, h / (H / H_idx), i) using key/value head h / (H / H_kv); otherwise the
 * arithmetic is that of ssa_sparse_attn (same scale, padding and error rules).
 *
 *   Q, O     [B, H, Tq, D]; K, V [B, H_kv, Tk, D]; idx int32 [B, H_idx, Tq, k]
 *   H_kv, H_idx  >= 1, each dividing H (H_kv = H_idx = H gives ssa_sparse_attn)
 *
 * When groups of query heads share a key/value head, rows run one key/value
 * head at a time (its K and V stay in L2), query by query, with the heads of
 * the group side by side. Returns as ssa_sparse_attn; H % H_kv or H % H_idx != 0 is
 * SSA_ERR_INVALID.
 */
ssa_status ssa_sparse_attn_grouped(const void* Q, const void* K, const void* V, int dtype, int B,
                                   int H, int H_kv, int Tq, int Tk, int D, const int32_t* idx,
                                   int H_idx, int k, float scale, void* O, int out_dtype,
                                   int32_t* dev_status, void* stream);

/*
 * ssa_window_attn — sliding-window (local band) attention.
 *
 * Source: nxmr.cn/news/163144, section 2.2 (each token attends the positions
 * within radius w of itself, all others get -inf before the softmax), which
 * is also the boolean mask of "Attention机制改进：稀疏注意力应用", section
 * 性能收益与硬件适配. It is the fixed-index special case of ssa_sparse_attn:
 *   O[b,h,i,:] = softmax over j in [max(0, i - w_left), min(T - 1, i + w_right)]
 *                of Q[b,h,i,:] . K[b,h,j,:] * scale, applied to V[b,h,j,:].
 *
 *   Q, K, V   device, [B, H, T, D], dtype `dtype`
 *   D         64 or 128
 *   w_left, w_right   >= 0 (the symmetric window of radius w is w, w)
 *   scale     <= 0 selects 1 / sqrt(D)
 *   O         device, [B, H, T, D], dtype `out_dtype`, written
 */
ssa_status ssa_window_attn(const void* Q, const void* K, const void* V, int dtype, int B, int H,
                           int T, int D, int w_left, int w_right, float scale, void* O,
                           int out_dtype, int32_t* dev_status, void* stream);

/*
 * ssa_score_topk_noalloc — ssa_score_topk for callers that cannot allocate.
 *
 * The pages have no counterpart to this call: it exists for users of this
 * library that may not allocate device memory where they run the op — a plugin
 * inside an inference engine that hands its ops a pre-sized memory arena and
 * no allocator, or a latency-critical loop that must never call cudaMalloc
 * (it can synchronize the device and its cost is unbounded). Such a caller
 * passes inputs and outputs as for ssa_score_topk, but no workspace.
 *
 * It computes exactly what ssa_score_topk computes (same arguments, same
 * results), always with the row-wise kernel, whose scratch lives in one fixed
 * 32 MiB device array inside this library (every device that loads the
 * library holds it until the process exits). The kernel needs
 * round_up(Tk, 64) * 4 bytes of it per query row in flight, so Tk may be at
 * most 8,388,608; larger Tk returns SSA_ERR_UNSUPPORTED and launches nothing.
 * The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture. If the device's context is replaced (cudaDeviceReset), the next
 * call looks the address up again in the new context. All calls share the
 * one array and it keeps the last call's contents (the kernel overwrites
 * every scratch word before reading it, so nothing needs clearing); calls
 * whose kernels overlap on the GPU (different streams, no ordering between
 * them) race on it and must be serialized by the caller.
 *
 * dev_status is checked (4-byte aligned or NULL) like every other call's, but
 * the row-wise kernel has no device-side error condition, so this call never
 * writes it.
 */
ssa_status ssa_score_topk_noalloc(const void* q_low, const void* k_low, int dtype, int B, int H,
                                  int Tq, int Tk, int P, int k, int causal, float scale,
                                  int32_t* idx, float* score, int32_t* dev_status, void* stream);

/*
 * ssa_sparse_attn_bwd — gradients of ssa_sparse_attn under the straight-through
 * estimator.
 *
 * Source: mhpq.cn/news/1098205, section 2.3: the forward keeps a hard top-k;
 * in the backward the selected positions pass their gradients normally and
 * the others get none, and the scorer's gradient arrives through the attention
 * weights of the selected positions. Read as: dQ, dK, dV are the exact
 * gradients of the forward with the index lists held fixed, and the score of
 * each selected pair receives the gradient of that pair's attention logit,
 *   dS[b,h,i,t] = p_t (dO_i . V_{j_t} - sum_u p_u dO_i . V_{j_u}),
 * with p the row's softmax weights; 0 in slots holding -1.
 *
 *   Q, dO      device, [B, H, Tq, D]; K, V device, [B, H, Tk, D]; all `dtype`
 *   idx        device, int32 [B, H, Tq, k], as for ssa_sparse_attn (-1 skipped,
 *              repeats counted per entry, other out-of-range entries skipped
 *              and reported with SSA_DEV_BAD_INDEX)
 *   scale      logit scale of the forward; <= 0 selects 1 / sqrt(D)
 *   dQ         device, float [B, H, Tq, D], written
 *   dK, dV     device, float [B, H, Tk, D], written (zero for keys no row chose)
 *   dS         device, float [B, H, Tq, k], written
 *   prob       device, float [B, H, Tq, k], written with p, or NULL
 *   workspace  at least ssa_sparse_attn_bwd_workspace_size(B, H, Tq, Tk, k)
 *              bytes, 256-byte aligned
 *
 * D in {64, 128}; Tq * k <= 2^31 - 1 (larger: SSA_ERR_UNSUPPORTED). Query-side
 * pointers (Q, dO, idx, dQ, dS) may be NULL when B*H*Tq == 0 and key-side ones
 * (K, V, dK, dV) when B*H*Tk == 0. Fp32 sums: dK, dV gather each key's pairs
 * in an order that varies from run to run, so their last bits may too.
 * Returns SSA_OK, SSA_ERR_INVALID, SSA_ERR_UNSUPPORTED, SSA_ERR_WORKSPACE or
 * SSA_ERR_CUDA.
 */
size_t ssa_sparse_attn_bwd_workspace_size(int B, int H, int Tq, int Tk, int k);
ssa_status ssa_sparse_attn_bwd(const void* Q, const void* K, const void* V, const void* dO,
                               int dtype, int B, int H, int Tq, int Tk, int D, const int32_t* idx,
                               int k, float scale, float* dQ, float* dK, float* dV, float* dS,
                               float* prob, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream);

/*
 * ssa_sparse_attn_grouped_bwd — ssa_sparse_attn_bwd for the layouts of
 * ssa_sparse_attn_grouped: query head h (of H) reads key/value head
 * h / (H / H_kv) and index head h / (H / H_idx) (mhpq.cn/news/1098205,
 * section 3.2, a scorer shared by all heads; "Attention机制优化：原理、挑战与
 * 工程实践" (bjdmk.com.cn), sections 3.1-3.2, grouped-query attention).
 * Each query head's gradients are those of ssa_sparse_attn_bwd on its own
 * operands. A shared key/value head's dK and dV sum over the query heads
 * that read it.
 *
 *   Q, dO, dQ [B, H, Tq, D]; K, V, dK, dV [B, H_kv, Tk, D]
 *   idx [B, H_idx, Tq, k]; dS, prob [B, H, Tq, k] (per query head)
 *   H_kv, H_idx >= 1, each dividing H; (H / H_kv) * Tq * k <= 2^31 - 1
 *   workspace: ssa_sparse_attn_grouped_bwd_workspace_size(B, H, H_kv, Tq, Tk, k)
 *
 * Other rules as ssa_sparse_attn_bwd. H_kv = H_idx = H is ssa_sparse_attn_bwd.
 */
size_t ssa_sparse_attn_grouped_bwd_workspace_size(int B, int H, int H_kv, int Tq, int Tk, int k);
ssa_status ssa_sparse_attn_grouped_bwd(const void* Q, const void* K, const void* V,
                                       const void* dO, int dtype, int B, int H, int H_kv, int Tq,
                                       int Tk, int D, const int32_t* idx, int H_idx, int k,
                                       float scale, float* dQ, float* dK, float* dV, float* dS,
                                       float* prob, void* workspace, size_t workspace_bytes,
                                       int32_t* dev_status, void* stream);

/*
 * ssa_scorer_bwd — the scorer's gradients under the same estimator.
 *
 * Source: mhpq.cn/news/1098205, sections 2.2 (S = q_low . k_low^T * scale) and
 * 2.3. With dS from ssa_sparse_attn_bwd:
 *   dq_low[b,h,i] = scale * sum_t dS[b,h,i,t] k_low[b,h,j_t]
 *   dk_low[b,h,j] = scale * sum over (i, t) with j_t = j of dS[b,h,i,t] q_low[b,h,i]
 *
 *   q_low [B,H,Tq,P], k_low [B,H,Tk,P] device, `dtype`; idx int32 and dS float
 *   [B,H,Tq,k]; dq_low [B,H,Tq,P] and dk_low [B,H,Tk,P] float, written.
 *   scale <= 0 selects fp32(1 / sqrt(P)). P in {16, 32, 64, 128};
 *   Tq * k <= 2^31 - 1. workspace: ssa_scorer_bwd_workspace_size(...) bytes,
 *   256-byte aligned. Same NULL, status and error rules as
 *   ssa_sparse_attn_bwd.
 */
size_t ssa_scorer_bwd_workspace_size(int B, int H, int Tq, int Tk, int k);
ssa_status ssa_scorer_bwd(const void* q_low, const void* k_low, int dtype, int B, int H, int Tq,
                          int Tk, int P, const int32_t* idx, int k, const float* dS, float scale,
                          float* dq_low, float* dk_low, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream);

/*
 * ssa_sparse_attn_scorer_bwd — ssa_sparse_attn_bwd and ssa_scorer_bwd in one
 * call, for the plain layout (every head its own keys, values and scorer).
 *
 * Source: mhpq.cn/news/1098205, sections 2.2 and 2.3, as for the two calls.
 * The gradients are exactly those of ssa_sparse_attn_bwd followed by
 * ssa_scorer_bwd on the dS it produced (same arguments, same rules); the key
 * sides of both walk the key-major lists of the index lists, which this call
 * builds once instead of twice.
 *
 *   Q, dO, dQ [B, H, Tq, D]; K, V, dK, dV [B, H, Tk, D]; idx, dS, prob
 *   [B, H, Tq, k]; q_low, dq_low [B, H, Tq, P]; k_low, dk_low [B, H, Tk, P]
 *   scale         attention logit scale (<= 0: 1 / sqrt(D))
 *   scorer_scale  scorer scale (<= 0: fp32(1 / sqrt(P)))
 *   workspace     ssa_sparse_attn_scorer_bwd_workspace_size(B, H, Tq, Tk, k)
 *                 bytes, 256-byte aligned
 *
 * D in {64, 128}, P in {16, 32, 64, 128}, Tq * k <= 2^31 - 1. Returns as
 * ssa_sparse_attn_bwd.
 */
size_t ssa_sparse_attn_scorer_bwd_workspace_size(int B, int H, int Tq, int Tk, int k);
ssa_status ssa_sparse_attn_scorer_bwd(const void* Q, const void* K, const void* V, const void* dO,
                                      const void* q_low, const void* k_low, int dtype, int B,
                                      int H, int Tq, int Tk, int D, int P, const int32_t* idx,
                                      int k, float scale, float scorer_scale, float* dQ,
                                      float* dK, float* dV, float* dS, float* prob,
                                      float* dq_low, float* dk_low, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status,
                                      void* stream);

/*
 * ssa_scorer_grouped_bwd — the scorer's gradients when H query heads share
 * H_idx scorer heads (H_idx = 1: the shared scorer of mhpq.cn/news/1098205,
 * section 3.2). The score of a pair in index head hi feeds the logits of
 * every query head that reads hi. Its gradient is therefore the sum of their
 * dS, and then the ssa_scorer_bwd formulas apply per scorer head.
 *
 *   q_low [B, H_idx, Tq, P], k_low [B, H_idx, Tk, P], idx [B, H_idx, Tq, k]
 *   dS [B, H, Tq, k] (from ssa_sparse_attn_grouped_bwd); H_idx divides H
 *   dq_low [B, H_idx, Tq, P], dk_low [B, H_idx, Tk, P] float, written
 *   workspace: ssa_scorer_grouped_bwd_workspace_size(B, H, H_idx, Tq, Tk, k)
 *
 * Other rules as ssa_scorer_bwd. H_idx = H is ssa_scorer_bwd.
 */
size_t ssa_scorer_grouped_bwd_workspace_size(int B, int H, int H_idx, int Tq, int Tk, int k);
ssa_status ssa_scorer_grouped_bwd(const void* q_low, const void* k_low, int dtype, int B, int H,
                                  int H_idx, int Tq, int Tk, int P, const int32_t* idx, int k,
                                  const float* dS, float scale, float* dq_low, float* dk_low,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                  void* stream);

/*
 * ssa_selftest_wait_limit — exercises the bounded device waits.
 *
 * The tensor-core kernels wait on mbarriers for their TMA copies and MMAs.
 * Each wait gives up after a time limit, sets SSA_DEV_WAIT_LIMIT in
 * *dev_status and lets the kernel return, so that a copy or MMA that never
 * completes leaves an error status and a usable context, not a hung GPU.
 * This call launches one block that takes that path on purpose: it waits on
 * an mbarrier that nothing completes until limit_ns has passed.
 *
 *   dev_status  device int32 (required); SSA_DEV_WAIT_LIMIT is ORed into it
 *   limit_ns    1 .. 1e9 (one second)
 *
 * Returns SSA_OK (launched), SSA_ERR_INVALID or SSA_ERR_CUDA.
 */
ssa_status ssa_selftest_wait_limit(int32_t* dev_status, uint64_t limit_ns, void* stream);

/*
 * Launch tracing. Between ssa_trace_begin() and ssa_trace_end(), every kernel
 * this library launches is bracketed by two CUDA events recorded on the
 * launching stream (the tracing itself launches nothing and allocates no
 * device memory). ssa_trace_end() waits for the recorded events, copies up to
 * max_records (kernel name, milliseconds) pairs in launch order into `out`
 * (may be NULL), stops tracing and returns the number of launches recorded,
 * or -1 if a CUDA event call failed. Meant for profiling: tracing adds two
 * event records per launch.
 */
typedef struct {
    char name[56];
    float ms;
} ssa_trace_record;

int ssa_trace_begin(void);
int ssa_trace_end(ssa_trace_record* out, int max_records);

#ifdef __cplusplus
}
#endif

#endif /* SSA_H_ */
