/*
 * kd_topk_kl.h - fused, chunked top-K KL distillation loss on one B300 (sm_103a).
 *
 * What it computes.  "Making Knowledge Distillation Cheap Enough to Run at
 * Scale" (aipuls.nl summary, section "Summary", second paragraph) describes a
 * teacher whose top-100 logits per token position are cached offline, and a
 * student trained with a KL-divergence loss that runs as a fused, chunked
 * kernel which never forms the full sequence-by-vocabulary matrix and keeps
 * its working memory bounded by one chunk.  The agent-gateway.com news piece
 * ("Hugging Face and Multiverse Computing cut KD memory costs", paragraphs on
 * the second bottleneck) restates the chunked, fused evaluation.  The pages
 * give no formula; this library fixes the following definition:
 *
 *   z      = h W^T                       student logits, T x V (never stored)
 *   lse_t  = log sum_v exp(z_tv / tau)   full-vocabulary log-normaliser
 *   p_tk   = softmax_k(teacher_logits_tk / tau)   renormalised over the K cached entries
 *   row_kl_t = valid_t ? sum_k p_tk (log p_tk - (z_t,idx_tk / tau - lse_t)) : 0
 *   loss   = sum_t row_kl_t / N_valid    (0 when N_valid = 0)
 *   G_tv   = g (valid_t / N_valid) (exp(z_tv/tau - lse_t) - sum_{k: idx_tk = v} p_tk) / tau
 *   dh     = G W,  dW = G^T h
 *
 * The direction KL(teacher || student) and the mean over valid tokens follow
 * the dense sketch in the asibiont.com rewrite ("A Concrete Implementation
 * Sketch").  No tau^2 factor.  Duplicate indices in a row count once per slot.
 *
 * Conventions shared by every entry point:
 *  - Pointers marked "device" are CUDA device pointers on the current device;
 *    the library never allocates, frees or copies to the host.  The caller
 *    owns every buffer, including the workspace `ws`.
 *  - Row-major, contiguous, 16-byte aligned arrays:
 *      h              bf16 [T x d]
 *      W              bf16 [V x d]   (nn.Linear weight layout)
 *      teacher_idx    int32 [T x K]  values in [0, V)
 *      teacher_logits fp32 [T x K]
 *      valid          uint8 [T]      nonzero = row takes part in the loss
 *  - Limits: T >= 1, V >= 1 with V % 8 == 0, d >= 64 with d % 64 == 0,
 *    1 <= K <= min(V, 32767), tau > 0 and finite, chunk >= 1.  T, V, d, K
 *    and chunk must each fit in 31 bits.
 *  - Host-side errors (bad arguments, workspace too small, launch failures)
 *    are returned synchronously as a kd_status and nothing is launched for
 *    argument errors.
 *  - Device-side errors are asynchronous: the kernels write the first error
 *    (KD_ERR_INDEX_RANGE for a teacher index outside [0, V), KD_ERR_TIMEOUT
 *    if an internal pipeline wait exceeds its bound) into *dev_status, which
 *    each call first resets to 0 on `stream`.  Read it after synchronising the
 *    stream.  Outputs are unspecified when it is nonzero.  The kernels never
 *    trap.
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default).
 *  - kd_topk_kl_forward, kd_topk_kl_backward and kd_topk_kl_forward_backward
 *    only enqueue stream-ordered work and never synchronise the host, so a
 *    sequence of them can be captured in a CUDA graph and replayed, once each
 *    kernel involved has run on the device (its first use sets a function
 *    attribute, which is done outside capture).
 */
#ifndef KD_TOPK_KL_H_
#define KD_TOPK_KL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */

typedef enum kd_status {
  KD_OK = 0,
  KD_ERR_INVALID_ARG = 1,  /* null pointer, bad size, tau <= 0, misalignment */
  KD_ERR_UNSUPPORTED = 2,  /* no sm_103a device, or shape outside the limits above */
  KD_ERR_WORKSPACE = 3,    /* ws_bytes smaller than kd_topk_kl_workspace_size() */
  KD_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
  KD_ERR_INDEX_RANGE = 5,  /* device: a teacher index is outside [0, V) */
  KD_ERR_TIMEOUT = 6,      /* device: a bounded pipeline wait ran out */
  KD_ERR_SCRATCH_LIMIT = 7, /* kd_topk_kl_forward_noalloc: shape too big for its scratch */
  KD_ERR_INTERNAL = 8,      /* device: an internal bound proved false (a library bug) */
  KD_ERR_NONFINITE = 9      /* device (kd_teacher_topk): a row's logits are not all finite */
} kd_status;

/*
 * Workspace bytes for kd_topk_kl_forward (*fwd_bytes) and
 * kd_topk_kl_backward (*bwd_bytes) at this shape.  Either output pointer may
 * be NULL.  The forward workspace holds the per-row sorted teacher entries and
 * one fp32 log-sum-exp partial per (row, 256-column vocabulary tile); the
 * backward workspace holds the sorted entries and one bf16 gradient chunk of
 * chunk x V elements (the only buffer whose size depends on V times a row
 * count: the "memory bounded by a single chunk" of the aipuls.nl summary).
 * Host-only; returns KD_ERR_INVALID_ARG / KD_ERR_UNSUPPORTED on bad shapes.
 */
int kd_topk_kl_workspace_size(int64_t T, int64_t V, int64_t d, int32_t K, int64_t chunk,
                              size_t* fwd_bytes, size_t* bwd_bytes);

/*
 * Number of kernels kd_topk_kl_forward / kd_topk_kl_backward enqueue at this
 * shape (the status/counter resets are cudaMemsetAsync calls and are not
 * counted).  Host-only; either output pointer may be NULL.
 */
int kd_topk_kl_launch_count(int64_t T, int64_t V, int64_t d, int32_t K, int64_t chunk,
                            int32_t* fwd_launches, int32_t* bwd_launches);

/*
 * Forward: loss, per-row lse, per-row KL (aipuls.nl "Summary": the KL between
 * the cached teacher top-K and the student, evaluated tile by tile without a
 * T x V buffer).
 *
 * Inputs  (device): h, W, teacher_idx, teacher_logits, valid as above.
 * Outputs (device): loss     fp32 scalar
 *                   lse      fp32 [T]   log sum_v exp(z_tv / tau), every row;
 *                            or NULL for a loss-only (evaluation) forward
 *                   row_kl   fp32 [T]   or NULL; 0 for invalid rows
 *                   gathered_idx int32 [T x K] or NULL: for every (t, k), the
 *                            vocabulary column whose logit the kernel read
 *                            for slot k (diagnostic; equals teacher_idx).
 * `chunk` is accepted for symmetry with the backward and is not used here:
 * the forward holds no chunk-sized buffer.
 * ws/ws_bytes: caller-owned device scratch, at least *fwd_bytes.
 */
int kd_topk_kl_forward(const void* h, const void* W, const int32_t* teacher_idx,
                       const float* teacher_logits, const uint8_t* valid, int64_t T, int64_t V,
                       int64_t d, int32_t K, float tau, int64_t chunk, float* loss, float* lse,
                       float* row_kl, int32_t* gathered_idx, void* ws, size_t ws_bytes,
                       int32_t* dev_status, struct CUstream_st* stream);

/*
 * Backward: dh = G W and dW = G^T h for the loss above scaled by grad_loss.
 * Rows are processed in chunks of `chunk` rows: for each chunk the logit tiles
 * are recomputed, G is written as bf16 into the chunk buffer in `ws`, and two
 * tensor-core contractions produce that chunk's rows of dh and add its
 * contribution to dW (the first chunk overwrites dW).
 *
 * lse: device fp32 [T] as produced by kd_topk_kl_forward for the same inputs.
 * Outputs (device): dh fp32 [T x d] (overwritten; rows of invalid tokens are
 * exactly 0), dW fp32 [V x d] (overwritten).
 * ws/ws_bytes: caller-owned device scratch, at least *bwd_bytes.  It need not
 * hold anything from the forward.
 */
int kd_topk_kl_backward(const void* h, const void* W, const int32_t* teacher_idx,
                        const float* teacher_logits, const uint8_t* valid, int64_t T, int64_t V,
                        int64_t d, int32_t K, float tau, int64_t chunk, const float* lse,
                        float grad_loss, float* dh, float* dW, void* ws, size_t ws_bytes,
                        int32_t* dev_status, struct CUstream_st* stream);

/*
 * Forward and backward in one call, for a training step (the aipuls.nl
 * "Summary" describes the loss as the student's training objective, computed
 * chunk by chunk with memory bounded by one chunk), in a single sweep that
 * computes each row's logits once instead of twice.  Rows are taken in the
 * order valid rows, then invalid rows; per chunk of `chunk` rows of that order
 * each valid row gets an offset o (the student's logit at the teacher's
 * highest cached entry), and the logit GEMM forms the lse partials and the
 * gather and also stores every valid row's logits as bf16 values
 * exp((z - o) / tau) into the chunk's G buffer (chunk x V x 2 bytes, as in
 * kd_topk_kl_backward).  With the chunk's lse, G = s exp(o / tau - lse) times
 * those values away from the cached columns, which a small pass rewrites; the
 * dh contraction applies the per-row factor to its output and the dW
 * contraction takes it inside h_c^T (rounded to bf16).  A chunk in which some
 * row's largest logit lies more than 64 ln 2 tau above its offset (the stored
 * values would leave the range those steps can carry) has its G recomputed
 * from the lse by the backward's logit GEMM instead; that launch returns at
 * once for the other chunks.  No T x V buffer exists at any time.
 *
 * Results: loss, lse and row_kl equal kd_topk_kl_forward's bit for bit; dh and
 * dW equal kd_topk_kl_backward's to within bf16 rounding (G is rounded once on
 * either route, at a different scale, and dW's h_c^T once more here).
 *
 * grad_loss: d(objective)/d(loss), as in kd_topk_kl_backward.
 * flags: 0, KD_ACCUMULATE_DW, KD_VALID_ROWS_ONLY or both.  With
 *   KD_ACCUMULATE_DW, dW += G^T h instead of dW = G^T h (gradient accumulation
 *   over micro-batches); dh is always overwritten.  With KD_VALID_ROWS_ONLY the
 *   logits of rows with valid = 0 are not formed at all (they add nothing to
 *   the loss or the gradients): their lse is written as NaN and their row_kl
 *   as 0; everything else is as without the flag, bit for bit.
 * Outputs (device): loss, lse (required), row_kl (or NULL), dh, dW.
 * ws/ws_bytes: at least *bytes of kd_topk_kl_forward_backward_workspace_size.
 */
#define KD_ACCUMULATE_DW 1u
#define KD_VALID_ROWS_ONLY 2u
/*
 * Workspace bytes (*bytes) and number of kernel launches (*launches, the
 * status/counter resets and the dh zeroing are cudaMemsetAsync calls and are
 * not counted) of kd_topk_kl_forward_backward at this shape; either pointer
 * may be NULL.  About 2 chunk V bytes plus O(T K) tables and the backward's
 * chunk buffers.
 * Host-only; KD_ERR_INVALID_ARG / KD_ERR_UNSUPPORTED on bad shapes.
 */
int kd_topk_kl_forward_backward_workspace_size(int64_t T, int64_t V, int64_t d, int32_t K,
                                               int64_t chunk, size_t* bytes, int32_t* launches);
int kd_topk_kl_forward_backward(const void* h, const void* W, const int32_t* teacher_idx,
                                const float* teacher_logits, const uint8_t* valid, int64_t T,
                                int64_t V, int64_t d, int32_t K, float tau, int64_t chunk,
                                float grad_loss, uint32_t flags, float* loss, float* lse,
                                float* row_kl, float* dh, float* dW, void* ws, size_t ws_bytes,
                                int32_t* dev_status, struct CUstream_st* stream);

/*
 * Residual-mass variant.  The pages cache only the teacher's top-100 logits per
 * position (aipuls.nl summary, section "Summary") and leave open what happens
 * to the probability mass outside them.  kd_topk_kl_forward renormalises the
 * teacher over the K entries; this variant instead takes the teacher's
 * full-vocabulary log-normaliser at temperature tau, cached beside the top-K,
 *
 *   teacher_lse_t = log sum_v exp(teacher_logit_tv / tau)   (fp32 [T], device),
 *
 * and compares teacher and student over K + 1 outcomes: the K cached entries
 * and "everything else".
 *
 *   P_tk = exp(teacher_logits_tk / tau - teacher_lse_t),  R_t = 1 - sum_k P_tk
 *   q_tk = exp(z_t,idx_tk / tau - lse_t),                 Q_t = 1 - sum_k q_tk
 *   row_kl_t = sum_k P_tk (log P_tk - log q_tk) + R_t (log R_t - log Q_t)
 *              (the last term is 0 when R_t = 0; R_t is clamped at 0)
 *   G_tv = s_t / tau (q_tv (1 - R_t/Q_t) + (R_t/Q_t) c_tv q_tv - sum_{k: idx_tk = v} P_tk)
 *   with s_t = grad_loss valid_t / N_valid and c_tv the number of slots holding v.
 *
 * The forward also writes outside_mass_t = Q_t (fp32 [T], device, or NULL);
 * the backward needs it (with lse) from the forward.  Q_t is not formed as
 * 1 - sum_k q_tk, which loses every digit in fp32 once the student puts
 * nearly all its mass on the cached entries (the well-distilled regime): the
 * forward sums the columns outside the cache on their own (their log-sum-exp
 * Lu_t), so Q_t = exp(Lu_t - lse_t) to fp32 relative precision (a row that
 * repeats an index subtracts that slot's extra q).  Other arguments, outputs,
 * workspace sizes and errors as kd_topk_kl_forward / _backward.  A row whose
 * student puts all its mass on the cached entries (Q_t = 0) while R_t > 0 has
 * an infinite loss, as the definition says.
 */
int kd_topk_kl_forward_residual(const void* h, const void* W, const int32_t* teacher_idx,
                                const float* teacher_logits, const float* teacher_lse,
                                const uint8_t* valid, int64_t T, int64_t V, int64_t d, int32_t K,
                                float tau, int64_t chunk, float* loss, float* lse, float* row_kl,
                                float* outside_mass, void* ws, size_t ws_bytes,
                                int32_t* dev_status, struct CUstream_st* stream);
int kd_topk_kl_backward_residual(const void* h, const void* W, const int32_t* teacher_idx,
                                 const float* teacher_logits, const float* teacher_lse,
                                 const uint8_t* valid, int64_t T, int64_t V, int64_t d, int32_t K,
                                 float tau, int64_t chunk, const float* lse,
                                 const float* outside_mass, float grad_loss, float* dh, float* dW,
                                 void* ws, size_t ws_bytes, int32_t* dev_status,
                                 struct CUstream_st* stream);
/*
 * The residual-mass variant's training step in one call, as
 * kd_topk_kl_forward_backward for the main loss: the same single sweep, with
 * the lse partials over the columns outside the cache, and the per-row factor
 * of the stored values times g = 1 - R/Q (every uncached column's gradient is
 * s q (1 - R/Q)); the cached columns are rewritten as s (q (1 + (c - 1) R/Q) - P)
 * divided by that factor.  A chunk with a row where |1 - R/Q| < 2^-16 (R close
 * to Q) has its G recomputed from the lse, like a chunk whose stored values
 * would leave range.  outside_mass (fp32 [T], device) is required and written
 * as kd_topk_kl_forward_residual writes it.  Results: loss, lse, row_kl and
 * outside_mass equal kd_topk_kl_forward_residual's bit for bit; dh and dW equal
 * kd_topk_kl_backward_residual's to within bf16 rounding.  Flags, workspace
 * (kd_topk_kl_forward_backward_workspace_size) and errors as
 * kd_topk_kl_forward_backward.
 */
int kd_topk_kl_forward_backward_residual(const void* h, const void* W, const int32_t* teacher_idx,
                                         const float* teacher_logits, const float* teacher_lse,
                                         const uint8_t* valid, int64_t T, int64_t V, int64_t d,
                                         int32_t K, float tau, int64_t chunk, float grad_loss,
                                         uint32_t flags, float* loss, float* lse, float* row_kl,
                                         float* outside_mass, float* dh, float* dW, void* ws,
                                         size_t ws_bytes, int32_t* dev_status,
                                         struct CUstream_st* stream);

/*
 * Teacher-side top-K cache producer (aipuls.nl summary, section "Summary": the
 * teacher runs once and its top-100 logits per position are cached offline).
 * From the teacher's final hidden states h (bf16 [T x d]) and LM-head weight W
 * (bf16 [V x d]) it writes, per row t, without forming the T x V logits:
 *
 *   topk_idx    int32 [T x K]  the K vocabulary indices of the largest
 *                              z_tv = h_t . W_v, ordered by z descending, equal
 *                              z by the lower index first (the result is unique)
 *   topk_logits fp32  [T x K]  those z_tv (raw logits, fp32 accumulation)
 *   full_lse    fp32  [T]      log sum_v exp(z_tv / tau), or NULL: the
 *                              teacher_lse that kd_topk_kl_forward_residual takes
 *
 * One tensor-core logit GEMM per chunk of `chunk` rows records each
 * 256-column tile's largest logit and lse partials and stores the chunk's fp32
 * logits in the workspace; a per-row threshold (the K-th largest tile maximum)
 * bounds the candidates to at most (K - 1) * 256 + 1 per row, a scan of the
 * stored logits collects them, and an exact selection orders the K largest.
 * The workspace holds one chunk's logits and candidates:
 * kd_teacher_topk_workspace_size(...) ~ chunk * (4 V + 8 min(V, (K - 1) * 256 + 1))
 * bytes (3.3 GB + 0.8 GB at chunk = 4096, V = 201088, K = 100); a smaller chunk
 * bounds it.  Limits and errors as kd_topk_kl_forward (KD_ERR_INTERNAL in
 * *dev_status would mean a candidate bound was exceeded, which the
 * construction rules out).  A row whose logits include NaN or +inf (from
 * non-finite or overflowing h or W), or whose full-vocabulary normaliser is
 * not finite, has no defined top-K: the call sets KD_ERR_NONFINITE and writes
 * that row as topk_idx = -1, topk_logits = NaN, full_lse = NaN; the other rows
 * are unaffected.  Deterministic.
 */
int kd_teacher_topk_workspace_size(int64_t T, int64_t V, int64_t d, int32_t K, int64_t chunk,
                                   size_t* bytes);
int kd_teacher_topk(const void* h, const void* W, int64_t T, int64_t V, int64_t d, int32_t K,
                    float tau, int64_t chunk, int32_t* topk_idx, float* topk_logits,
                    float* full_lse, void* ws, size_t ws_bytes, int32_t* dev_status,
                    struct CUstream_st* stream);

/*
 * Teacher-entropy token filter, the producer of the valid mask (asibiont.com
 * rewrite, section "Distillation Token Filtering": score each token by the
 * entropy of the teacher's distribution and keep, per batch, a fixed
 * percentage of the tokens with the highest entropy).
 *
 *   p_tk = softmax_k(teacher_logits_tk / tau) over the K cached entries
 *   H_t  = -sum_k p_tk log p_tk                      (natural log)
 *   N_in = number of rows with valid_in != 0
 *   n_keep = ceil(N_in * keep_num / keep_den)        (exact integer arithmetic)
 *   valid_out[t] = 1 for the n_keep rows with valid_in != 0 and the largest
 *                  H_t (equal H_t: the lower row first), else 0.
 *
 * Inputs (device): teacher_logits fp32 [T x K] (finite), valid_in uint8 [T].
 * Outputs (device): valid_out uint8 [T]; entropy fp32 [T] or NULL.
 * Limits: T >= 1, K >= 1, tau > 0, 0 <= keep_num <= keep_den, keep_den >= 1.
 * ws/ws_bytes: caller-owned device scratch, 256-byte aligned, at least
 * kd_entropy_filter_workspace_size(T).  *dev_status is reset to 0 (the filter
 * raises no device error).  Deterministic: the result depends only on the
 * inputs.
 */
int kd_entropy_filter_workspace_size(int64_t T, size_t* bytes);
int kd_entropy_filter(const float* teacher_logits, const uint8_t* valid_in, int64_t T, int32_t K,
                      float tau, int32_t keep_num, int32_t keep_den, uint8_t* valid_out,
                      float* entropy, void* ws, size_t ws_bytes, int32_t* dev_status,
                      struct CUstream_st* stream);

/* Static, NUL-terminated description of a kd_status value (never NULL). */
const char* kd_topk_kl_status_string(int status);

/*
 * Diagnostic of the contraction step alone: C = A B^T on the same tcgen05
 * tensor-core pipeline that produces the logit tiles z = h W^T above, with an
 * fp32 store epilogue instead of the loss.  C fp32 [M x N] row-major.
 * a_mn = 0: A is bf16 [M x Kd] row-major (K-major); a_mn = 1: A is given as
 * bf16 [Kd x M] row-major (M contiguous).  Likewise b_mn for B ([N x Kd] or
 * [Kd x N]).  Limits: M, N, Kd >= 1 and multiples of 8 (a contraction tail
 * shorter than 64 is zero-filled by TMA).  Device pointers; stream as above.
 */
int kd_gemm_bf16_diag(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t Kd,
                      int32_t a_mn, int32_t b_mn, int32_t* dev_status,
                      struct CUstream_st* stream);

/*
 * The same diagnostic product on the CTA-pair pipeline that the logit GEMMs
 * use: clusters of two CTAs, each 256 x BN tile computed by tcgen05.mma with
 * cta_group::2 (each CTA holds 128 rows of A and BN/2 rows of B in its shared
 * memory and 128 rows of the accumulator in its tensor memory).  Both operands
 * K-major: A bf16 [M x Kd], B bf16 [N x Kd]; C fp32 [M x N].  Limits as
 * kd_gemm_bf16_diag.
 */
int kd_gemm_bf16_diag_pair(const void* A, const void* B, float* C, int64_t M, int64_t N,
                           int64_t Kd, int32_t* dev_status, struct CUstream_st* stream);

/*
 * Self-test of the failure detection every pipeline wait relies on (the pages
 * describe no failure handling; this checks the library's own bound).  One
 * thread waits on an mbarrier that nothing arrives on, through the same
 * bounded wait the contraction kernels use; after limit_ns (1 ns .. 1 s) the
 * wait gives up and the kernel writes KD_ERR_TIMEOUT to *dev_status (device
 * int32, reset to 0 first) and returns, leaving the context usable.
 */
int kd_pipeline_wait_selftest(uint64_t limit_ns, int32_t* dev_status, struct CUstream_st* stream);

/*
 * Forward without any allocation, for callers that cannot call cudaMalloc:
 * for example code that runs inside another framework's memory manager, which
 * owns the whole device pool and forbids side allocations, or a host runtime
 * that allows no device allocation after start-up (cudaMalloc can also
 * synchronise the device, which some callers must avoid).  The pages have no
 * counterpart to this entry point; it exists for those callers only.
 *
 * Same inputs, outputs and results as kd_topk_kl_forward, but the workspace
 * is a fixed 32 MiB array built into the library (no ws / ws_bytes and no
 * chunk argument).  Shapes whose forward workspace (kd_topk_kl_workspace_size
 * *fwd_bytes) exceeds 32 MiB are rejected with KD_ERR_SCRATCH_LIMIT before
 * anything is launched; at V = 201088, K = 100 that admits up to about 7300 rows.
 * The library calls no cudaMalloc, cudaFree or other allocating routine here.
 *
 * - Every GPU that loads the library holds the 32 MiB array until the process
 *   exits.  The array belongs to the library's device module, and CUDA
 *   reserves it when it loads that module on a device.  With lazy module
 *   loading (CUDA's default) that happens on the first use of any of the
 *   library's kernels or of the array on that device, which may be this
 *   entry's first call: that load reserves the array and the kernel images,
 *   and may synchronise.  A caller that must not see either during its steady
 *   state makes one warm-up call (this entry or any other library call) on
 *   each device at start-up.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make that
 *   first call before any stream capture.
 * - All calls share the one array per device, and it keeps the last call's
 *   contents.  Calls whose work overlaps on the GPU (different streams, or
 *   several host threads) race on it; serialise them.
 */
int kd_topk_kl_forward_noalloc(const void* h, const void* W, const int32_t* teacher_idx,
                               const float* teacher_logits, const uint8_t* valid, int64_t T,
                               int64_t V, int64_t d, int32_t K, float tau, float* loss, float* lse,
                               float* row_kl, int32_t* gathered_idx, int32_t* dev_status,
                               struct CUstream_st* stream);

/*
 * Diagnostic launch timing, for measurement only (the pages describe no such
 * facility).  Contraction kernels are identified by these ids:
 *   KD_KERNEL_LOGITS_FWD  forward logit tiles with the lse / gather epilogue
 *   KD_KERNEL_LOGITS_BWD  backward logit recompute with the gradient epilogue
 *   KD_KERNEL_DH          dh = G W (computed as dh^T = W^T G^T)
 *   KD_KERNEL_DW          dW = G^T h (computed as dW^T = h^T G)
 *   KD_KERNEL_TOPK_PASS1  teacher top-K producer: logits, tile maxima, lse partials
 *   KD_KERNEL_TOPK_SCAN   teacher top-K producer: candidate scan of the stored
 *                         logits (a SIMT kernel, timed the same way)
 *   KD_KERNEL_SWEEP_FIX   single sweep (kd_topk_kl_forward_backward): the pass
 *                         that writes G's cached columns into the stored values
 *                         (a SIMT kernel); that entry's logit GEMM is timed as
 *                         KD_KERNEL_LOGITS_FWD and its recompute of a flagged
 *                         chunk's G as KD_KERNEL_LOGITS_BWD
 *
 * kd_timing_start(capacity): creates 2 x capacity CUDA events on the current
 *   device (no device memory is allocated) and starts recording: from then on
 *   every launch of an id above that the entry points make (the contractions
 *   of the loss entries and of kd_teacher_topk, the producer's candidate scan
 *   and the single sweep's cached-column pass), from any host thread, is
 *   bracketed by an event pair recorded on its stream, until `capacity`
 *   launches have been recorded.  Restarting discards earlier records.
 * kd_timing_stop(): stops recording; the records stay readable.
 * kd_timing_query(kernel, *launches, *total_ms): waits for the recorded
 *   launches of that kernel id and returns their count and summed duration.
 * kd_timing_release(): stops recording and destroys the events.
 * One recorder per process; the calls are serialised internally.
 */
enum {
  KD_KERNEL_LOGITS_FWD = 0,
  KD_KERNEL_LOGITS_BWD = 1,
  KD_KERNEL_DH = 3,
  KD_KERNEL_DW = 4,
  KD_KERNEL_TOPK_PASS1 = 5,
  KD_KERNEL_TOPK_SCAN = 6,
  KD_KERNEL_SWEEP_FIX = 7
};
int kd_timing_start(int32_t capacity);
int kd_timing_stop(void);
int kd_timing_query(int32_t kernel, int32_t* launches, double* total_ms);
int kd_timing_release(void);

#ifdef __cplusplus
}
#endif

#endif /* KD_TOPK_KL_H_ */
