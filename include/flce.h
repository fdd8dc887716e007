/*
 * flce.h - C ABI of the language-model loss head for GB300 (sm_103a).
 *
 * Two operations, each split into a forward and a backward call:
 *
 *   ce_logits_*  masked cross-entropy over GIVEN logits [N, V]; the backward can
 *                write the gradient into the logits storage (in place).
 *                Defined by Automodel PR #2996 "feat(loss): chunked masked CE,
 *                packing-mask preservation, scoped MoE AC", first commit message
 *                (forward: per-row fp32 logsumexp and label-logit gather summed
 *                into a scalar, only the logits and labels kept; backward:
 *                softmax recomputed per chunk, gradient optionally written into
 *                the logits storage) and its inplace_grad follow-up commit.
 *
 *   flce_*       fused linear cross-entropy: logits = H W^T (+ bias) are formed
 *                tile by tile and never stored.  Defined by Liger-Kernel issue
 *                #533 "Gradient checkpointing for grad_weight in LFCE" (feature
 *                pitch: the chunked logits, grad_W accumulated with an addmm of
 *                dlogits^T H at beta = 1, and the fully recomputed variant in the
 *                follow-up comments, whose backward recomputes the logits) and
 *                Liger-Kernel issue #941 "[Question] No gain in VRAM usage with
 *                LigerFusedLinearCrossEntropyLoss" (input [B*T, D], weight
 *                [V, D] in the tied-embedding layout, optional bias).
 *
 * Notation: N tokens (rows), V vocabulary, D hidden size; y_i the label of row
 * i; valid_i = (y_i != ignore_index); n_valid = sum_i valid_i;
 * lse_i = log sum_j exp(z_ij); loss_i = valid_i * (lse_i - z_{i,y_i}).
 *
 * Reduction.  S = sum_i loss_i.  The loss is S * scale with
 *   scale = 1 / num_label_tokens   if num_label_tokens >= 0 is given,
 *         = 1                      for FLCE_SUM,
 *         = 1 / n_valid            for FLCE_MEAN,
 * and scale = 0 whenever that divisor is 0 (all rows ignored under MEAN, or
 * num_label_tokens == 0): the loss and every gradient are then 0.
 * The backward gradient is dz_ij = valid_i (exp(z_ij - lse_i) - [j == y_i]) g scale
 * with g = *grad_loss.
 *
 * Memory.  Every pointer is a DEVICE pointer unless stated otherwise; the
 * caller allocates every buffer (inputs, outputs, workspace) and keeps
 * ownership.  The library never allocates or frees device memory, never
 * synchronises, and enqueues all its work on the caller's `stream`.
 * Matrices are row-major with unit stride along the last dimension.
 *
 * Errors.  Every entry point returns a flce_status_t.  Errors that the host can
 * see (null pointers, bad sizes, bad alignment, too small a workspace) are
 * returned before anything is enqueued.  Errors only the device can see (a
 * label outside [0, V) that is not ignore_index; a bounded wait that gave up;
 * in the debug build, an index check that failed) are written to the device
 * word *status with "first error wins" semantics:
 * the library never clears *status, so a nonzero value stays until the caller
 * resets it.  Rows whose label is out of range contribute nothing to the loss,
 * n_valid or the gradients.  No kernel traps or asserts.
 *
 * Determinism.  No floating-point atomics are used: two identical calls give
 * bitwise-identical results.
 */
#ifndef FLCE_H
#define FLCE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FLCE_API __attribute__((visibility("default")))
#else
#define FLCE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* flce_stream_t;

typedef enum {
  FLCE_OK = 0,
  FLCE_EINVAL = -1,      /* null pointer, bad enum value, bad flag           */
  FLCE_ESHAPE = -2,      /* a size is out of range or inconsistent           */
  FLCE_EDTYPE = -3,      /* unsupported dtype                                */
  FLCE_EALIGN = -4,      /* a pointer or row stride breaks an alignment rule */
  FLCE_ELABEL = -5,      /* (device) label outside [0,V) and != ignore_index */
  FLCE_EWORKSPACE = -6,  /* workspace pointer null or too small              */
  FLCE_ECUDA = -7,       /* a CUDA runtime/driver call failed                */
  FLCE_ENOSUP = -8,      /* valid request this library does not support      */
  FLCE_ETIMEOUT = -9,    /* (device) a bounded wait inside a kernel gave up  */
  FLCE_EBOUNDS = -10     /* (device, checked builds) an index left its range  */
} flce_status_t;

typedef enum { FLCE_BF16 = 0, FLCE_F32 = 1 } flce_dtype_t;
typedef enum { FLCE_SUM = 0, FLCE_MEAN = 1 } flce_reduction_t;

/* Human-readable name of a status code (static storage; never NULL). */
FLCE_API const char* flce_status_string(int status);

/* Description of the last CUDA runtime/driver failure behind an FLCE_ECUDA
 * returned on the calling thread (thread-local storage; never NULL). */
FLCE_API const char* flce_last_cuda_error(void);

/* ------------------------------------------------------------------------ */
/* Cross-entropy on given logits                                            */
/* ------------------------------------------------------------------------ */

/* Bytes of device workspace ce_logits_fwd needs for N rows (4 bytes per row,
 * rounded up to 256).  Returns 0 for N <= 0. */
FLCE_API size_t ce_logits_workspace_bytes(int64_t N, int64_t V);

/* Forward.  logits: [N, ld] of dtype dt, row i at logits + i*ld elements, the
 * first V columns used (ld >= V).  labels: [N] int64.  Outputs:
 *   loss      [1] f32   the reduced loss (see "Reduction")
 *   n_valid   [1] i64   number of rows with a valid label (exact)
 *   lse       [N] f32   per-row log-sum-exp (saved for the backward; written
 *                       for every row, ignored ones included)
 *   loss_rows [N] f32   optional (may be NULL): loss_i, 0 on ignored rows
 *   label_logit [N] f32 optional (may be NULL): z_{i,y_i} widened to fp32
 *                       exactly, NaN on ignored rows
 * ws/ws_bytes: workspace of at least ce_logits_workspace_bytes(N, V) bytes,
 * 16-byte aligned.  status: device word, see "Errors".
 * N == 0 is valid (loss 0, n_valid 0).  Requires 1 <= V < 2^31, ld >= V. */
FLCE_API int ce_logits_fwd(const void* logits, int dt, int64_t N, int64_t V, int64_t ld,
                  const int64_t* labels, int64_t ignore_index, int reduction,
                  int64_t num_label_tokens, float* loss, int64_t* n_valid, float* lse,
                  float* loss_rows, float* label_logit, void* ws, size_t ws_bytes,
                  int32_t* status, flce_stream_t stream);

/* 1 when this library was built with device-side index checks
 * (FLCE_DEVICE_CHECKS=1: the debug build that stands in for a memory checker;
 * an index outside its tensor or buffer records FLCE_EBOUNDS in the status
 * word and the access is skipped, never a trap), 0 for the ordinary build.
 * The source pages have no counterpart. */
FLCE_API int flce_device_checks(void);

/* Self-test of the device-side index check: one thread checks an index equal
 * to the length of a range (one past its end) and performs no access either
 * way.  In a checked build *status becomes FLCE_EBOUNDS; in the ordinary
 * build the check is compiled out and *status is left unchanged. */
FLCE_API int flce_bounds_selftest(int32_t* status, flce_stream_t stream);

/* Self-test of the failure path: launches one warp that waits, with the same
 * bounded mbarrier wait every kernel of this library uses, on a barrier that
 * nothing arrives on.  After limit_ns (at most 2 s) the wait gives up and
 * FLCE_ETIMEOUT is written to *status (a larger limit returns FLCE_ESHAPE
 * and launches nothing); the kernel returns normally and the
 * context stays usable.  The source pages have no counterpart. */
FLCE_API int flce_wait_selftest(int32_t* status, uint64_t limit_ns, flce_stream_t stream);

/* Label masking for packed sequences: labels and doc_ids are [B, T] int64
 * (device, row-major); doc_ids holds 1, 2, ... for the packed documents of a
 * row and 0 for padding (the indexed packing mask of Automodel PR #2996,
 * "fix(models): preserve indexed packing masks").  In place, labels[b, t]
 * becomes ignore_index where doc_ids[b, t] == 0 or where position t is the
 * last of its document (the next token belongs to another document, or the
 * row ends); other labels are left as they are. */
FLCE_API int flce_mask_packed_labels(int64_t* labels, const int64_t* doc_ids, int64_t B,
                                     int64_t T, int64_t ignore_index, flce_stream_t stream);

/* Largest N ce_logits_fwd_noalloc accepts. */
#define CE_LOGITS_NOALLOC_MAX_ROWS (1 << 20)

/* ce_logits_fwd without a workspace argument, for callers that cannot
 * allocate device memory: for example a runtime that hands all device memory
 * to its own pool at start-up and forbids further cudaMalloc, or a
 * latency-critical loop where the device-wide synchronisation a cudaMalloc or
 * cudaFree can cause is not acceptable.  The source pages have no counterpart;
 * it is an addition of this library.
 *
 * Same arguments and results as ce_logits_fwd, without ws/ws_bytes and the
 * optional loss_rows/label_logit outputs.  The caller still allocates and
 * passes every input and output.  The per-row scratch lives in a static
 * device array of CE_LOGITS_NOALLOC_MAX_ROWS floats (4 MiB) that every GPU
 * which loads the library holds until the process exits; N above that
 * maximum returns FLCE_ESHAPE and enqueues nothing.  No cudaMalloc, cudaFree
 * or other allocating call is made.
 *
 * The first call on each device looks up the device address of the scratch
 * array (cudaGetSymbolAddress, with that device current) and caches it with
 * the id of the current context; make that first call before any stream
 * capture on the device.  After a cudaDeviceReset (a new primary context) the
 * next call looks the address up again, in the new context: make that call
 * before any stream capture as well.
 *
 * All calls share the one array and it keeps the last call's contents (none
 * of which has to be cleared: each call writes every row it later reads).
 * Calls whose work overlaps on the GPU (on different streams, or from
 * different threads without ordering) race on the array and give wrong
 * results: order them on one stream or with events. */
FLCE_API int ce_logits_fwd_noalloc(const void* logits, int dt, int64_t N, int64_t V, int64_t ld,
                  const int64_t* labels, int64_t ignore_index, int reduction,
                  int64_t num_label_tokens, float* loss, int64_t* n_valid, float* lse,
                  int32_t* status, flce_stream_t stream);

/* Backward.  Reads logits, labels, lse (from ce_logits_fwd), n_valid (from
 * ce_logits_fwd; only read for FLCE_MEAN without num_label_tokens) and
 * grad_loss ([1] f32 device: the incoming gradient g of the loss), and writes
 * grad_logits [N, ld_grad] of dtype dt (first V columns of each row).
 * inplace_grad != 0: grad_logits must equal logits and ld_grad == ld; the
 * logits are overwritten by their gradient (Automodel PR #2996, inplace_grad).
 * inplace_grad == 0: grad_logits must not overlap the logits.
 *
 * lse may be NULL: the backward that keeps only the logits and the labels
 * from the forward (Automodel PR #2996, the memory bullet: nothing but the
 * inputs is saved).  Each row's lse is then formed again inside the kernel.
 * A row of at most 8 x 64 KiB (V <= 262144 bf16, 131072 f32; one 16-byte
 * block less when rows start inside a block) is split over a thread-block
 * cluster that holds it in shared memory, so the logits are still read once,
 * provided the gradient rows start at the same offsets within their 16-byte
 * blocks as the logits rows (in place, or both buffers aligned alike); longer
 * rows, and gradient buffers at other offsets, read the logits twice.  The
 * result equals the saved-lse backward up to the rounding of the recomputed
 * lse (fp32, a few ulp). */
FLCE_API int ce_logits_bwd(const void* logits, int dt, int64_t N, int64_t V, int64_t ld,
                  const int64_t* labels, int64_t ignore_index, int reduction,
                  int64_t num_label_tokens, const float* lse, const int64_t* n_valid,
                  const float* grad_loss, int inplace_grad, void* grad_logits,
                  int64_t ld_grad, int32_t* status, flce_stream_t stream);

/* Bytes of device workspace ce_logits_fwd_bwd needs for N rows.  Returns 0
 * for N <= 0. */
FLCE_API size_t ce_logits_fwd_bwd_workspace_bytes(int64_t N, int64_t V);

/* Forward and backward in one call: the loss (as ce_logits_fwd) and the
 * gradient of the logits (as ce_logits_bwd) when the incoming gradient is
 * known before the loss, typically g = 1 for a loss that is the last node.
 * The eager-gradient counterpart of flce_fwd_bwd for given logits: the
 * gradient is formed while the loss is computed and handed out later, as
 * Liger's fused linear cross-entropy does with its weight gradient
 * (Liger-Kernel issue #533, "Gradient checkpointing for grad_weight in
 * LFCE"); the pages define no such call for given logits.
 *
 * Arguments as ce_logits_fwd and ce_logits_bwd.  grad_loss ([1] f32 device)
 * may be NULL, meaning g = 1 (scale later with flce_grad_scale).  lse ([N] f32)
 * may be NULL; when given it holds the lse of every row with a valid label
 * (other rows: unspecified).  inplace_grad, grad_logits, ld_grad: as in
 * ce_logits_bwd; in place, the logits are overwritten by their gradient.
 * ws: ce_logits_fwd_bwd_workspace_bytes(N, V) bytes, 16-byte aligned.
 *
 * Rows of at most 8 x 64 KiB whose gradient rows start at the same offsets
 * within their 16-byte blocks as the logits rows (in place, or both buffers
 * aligned alike) are read once: a thread-block cluster holds each row in
 * shared memory, forms its lse and loss and writes its gradient (rows with an
 * ignored label are not read).  Other rows run the forward and then the
 * backward (two reads). */
FLCE_API int ce_logits_fwd_bwd(const void* logits, int dt, int64_t N, int64_t V, int64_t ld,
                  const int64_t* labels, int64_t ignore_index, int reduction,
                  int64_t num_label_tokens, const float* grad_loss, float* loss,
                  int64_t* n_valid, float* lse, int inplace_grad, void* grad_logits,
                  int64_t ld_grad, void* ws, size_t ws_bytes, int32_t* status,
                  flce_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Fused linear cross-entropy                                               */
/* ------------------------------------------------------------------------ */

/* Bytes of device workspace for flce_fwd and flce_bwd with these sizes.
 * `chunk` says how the backward splits its work: chunk > 0, row chunks of
 * that many rows (a multiple of 128 unless it covers all N); chunk < 0
 * (bf16 only), slices of -chunk vocabulary columns (a multiple of 256) over
 * all rows at once; chunk == 0, the library default (flce_default_chunk).
 * The same workspace serves both calls.  With the default, the workspace
 * stays within one [2048, V] fp32 tile (2048 * V * 4 bytes) for bf16 inputs:
 * Automodel PR #2996 ("Motivation") bounds the fp32 transient of its chunked
 * loss by chunk_size * V * 4 bytes, and the chunk of that bound is fixed here
 * at 2048 rows. */
FLCE_API size_t flce_workspace_bytes(int dt, int64_t N, int64_t D, int64_t V, int64_t chunk);

/* Row chunk the backward uses when chunk == 0 is passed (0 for invalid
 * sizes).  Row chunks read and write the fp32 grad_W once more per chunk
 * after the first; vocabulary slices (a negative chunk) write grad_W once and
 * accumulate an fp32 [N, D] grad_H in the workspace instead (one rounding to
 * dt at the end), at the cost of grad_W summed in one tensor-core sweep over
 * all N rows. */
FLCE_API int64_t flce_default_chunk(int dt, int64_t N, int64_t D, int64_t V);

/* Forward.  H: [N, D], W: [V, D] (row v is the embedding of token v), bias:
 * [V] or NULL, all of dtype dt (FLCE_BF16: tensor cores in bf16 with fp32
 * accumulation; FLCE_F32: tensor cores in tf32 with fp32 accumulation).
 * H and W must be 16-byte aligned and D * sizeof(dt) a multiple of 16.
 * Outputs as in ce_logits_fwd (loss, n_valid, lse, optional loss_rows and
 * label_logit, the latter the fp32 GEMM value of z_{i,y_i}).
 * Requires 0 <= N, 1 <= V < 2^31, 8 <= D.  N == 0 (an empty batch; H,
 * labels, lse and ws may then be NULL) gives loss 0 and n_valid 0, and the
 * backward calls (flce_bwd, flce_fwd_bwd and the shard steps) then write a
 * zero grad_W (left as it is when accumulating) and a zero grad_bias. */
FLCE_API int flce_fwd(const void* H, const void* W, const void* bias, int dt, int64_t N, int64_t D,
             int64_t V, const int64_t* labels, int64_t ignore_index, int reduction,
             int64_t num_label_tokens, float* loss, int64_t* n_valid, float* lse,
             float* loss_rows, float* label_logit, void* ws, size_t ws_bytes,
             int32_t* status, flce_stream_t stream);

/* Backward (fully recomputed: the logits are formed again chunk by chunk).
 * Reads the forward's inputs plus lse and n_valid from flce_fwd and grad_loss
 * ([1] f32 device).  Writes, each optional (NULL skips it):
 *   grad_H    [N, D] dtype dt      = dZ W
 *   grad_W    [V, D] f32           = dZ^T H, added to the existing contents if
 *                                    accumulate_grad_W != 0 (addmm beta = 1)
 *   grad_bias [V]    f32           = sum over rows of dZ (overwritten)
 * dZ is formed per row chunk (or vocabulary slice) in fp32 and rounded to dt
 * before the two gradient contractions.  chunk as in flce_workspace_bytes
 * (0: flce_default_chunk); the workspace must have been sized with the same
 * chunk.  A negative chunk with fp32 inputs returns FLCE_ENOSUP, one that is
 * not a multiple of 256 FLCE_ESHAPE. */
FLCE_API int flce_bwd(const void* H, const void* W, const void* bias, int dt, int64_t N, int64_t D,
             int64_t V, const int64_t* labels, int64_t ignore_index, int reduction,
             int64_t num_label_tokens, const float* lse, const int64_t* n_valid,
             const float* grad_loss, int64_t chunk, void* grad_H, float* grad_W,
             int accumulate_grad_W, float* grad_bias, void* ws, size_t ws_bytes,
             int32_t* status, flce_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Vocabulary-parallel fused linear cross-entropy                           */
/* ------------------------------------------------------------------------ */
/* "Loss Parallel" of torchtitan PR #996 (review: TP with Loss Parallel): each
 * rank holds rows [vocab_offset, vocab_offset + V_shard) of W (and of the
 * bias) and all of H and the labels (global ids in [0, V_total)).  A forward
 * step is:
 *   1. flce_fwd_shard     per row: m, s = base-2 max and sum of 2^(z*log2e - m)
 *                         over the shard's columns; zy = the label logit if the
 *                         label lies in the shard, else 0
 *   2. all-reduce MAX of m over the ranks                     -> m_global
 *   3. flce_shard_rescale s_scaled = s * 2^(m - m_global)
 *   4. all-reduce SUM of s_scaled and of zy                   -> s_global, zy_global
 *   5. flce_shard_finish  lse = (m_global + log2 s_global) ln 2, loss rows,
 *                         reduction (identical on every rank)
 * and the backward is flce_bwd_shard with the global lse (the shard's columns
 * of dZ), followed by an all-reduce SUM of the fp32 grad_H partials; grad_W and
 * grad_bias stay with their shard.  Workspaces: flce_workspace_bytes(dt, N, D,
 * V_shard, chunk).  The collectives are the caller's (e.g. NCCL). */
FLCE_API int flce_fwd_shard(const void* H, const void* W_shard, const void* bias_shard, int dt,
                            int64_t N, int64_t D, int64_t V_shard, int64_t vocab_offset,
                            int64_t V_total, const int64_t* labels, int64_t ignore_index,
                            float* m_local, float* s_local, float* zy_local, void* ws,
                            size_t ws_bytes, int32_t* status, flce_stream_t stream);

/* s_scaled[i] = s_local[i] * 2^(m_local[i] - m_global[i]) (0 when m_local[i] is -inf). */
FLCE_API int flce_shard_rescale(const float* m_local, const float* s_local,
                                const float* m_global, int64_t N, float* s_scaled,
                                flce_stream_t stream);

/* lse, per-row loss (loss_rows may be NULL: ws then needs 4N bytes rounded up
 * to 256) and the reduced loss and n_valid from the reduced m, s and zy. */
FLCE_API int flce_shard_finish(const float* m_global, const float* s_global,
                               const float* zy_global, const int64_t* labels, int64_t N,
                               int64_t V_total, int64_t ignore_index, int reduction,
                               int64_t num_label_tokens, float* lse, float* loss_rows,
                               float* loss, int64_t* n_valid, void* ws, size_t ws_bytes,
                               int32_t* status, flce_stream_t stream);

/* Backward of one shard: as flce_bwd over the shard's columns, with the
 * global lse and n_valid; grad_H_partial is this shard's term of grad_H,
 * written as fp32 [N, D] whatever dt is, so that the ranks' partials are
 * summed in fp32 and rounded to the input dtype once, after the sum (a sum
 * of partials already rounded to bf16 would add one rounding per rank). */
FLCE_API int flce_bwd_shard(const void* H, const void* W_shard, const void* bias_shard, int dt,
                            int64_t N, int64_t D, int64_t V_shard, int64_t vocab_offset,
                            int64_t V_total, const int64_t* labels, int64_t ignore_index,
                            int reduction, int64_t num_label_tokens, const float* lse,
                            const int64_t* n_valid, const float* grad_loss, int64_t chunk,
                            void* grad_H_partial, float* grad_W_shard, int accumulate_grad_W,
                            float* grad_bias_shard, void* ws, size_t ws_bytes, int32_t* status,
                            flce_stream_t stream);

/* CE on a vocabulary shard of given logits: logits_shard [N, ld] holds the
 * columns [vocab_offset, vocab_offset + V_shard) of the full [N, V_total]
 * logits; labels are global ids.  The forward writes the same per-row m_local,
 * s_local, zy_local as flce_fwd_shard (then steps 2-5 above); the backward
 * writes the shard's columns of dZ (in place or not, as ce_logits_bwd) from
 * the global lse and n_valid. */
FLCE_API int ce_logits_fwd_shard(const void* logits_shard, int dt, int64_t N, int64_t V_shard,
                                 int64_t ld, int64_t vocab_offset, int64_t V_total,
                                 const int64_t* labels, int64_t ignore_index, float* m_local,
                                 float* s_local, float* zy_local, int32_t* status,
                                 flce_stream_t stream);

FLCE_API int ce_logits_bwd_shard(const void* logits_shard, int dt, int64_t N, int64_t V_shard,
                                 int64_t ld, int64_t vocab_offset, int64_t V_total,
                                 const int64_t* labels, int64_t ignore_index, int reduction,
                                 int64_t num_label_tokens, const float* lse,
                                 const int64_t* n_valid, const float* grad_loss,
                                 int inplace_grad, void* grad_logits, int64_t ld_grad,
                                 int32_t* status, flce_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Fused linear cross-entropy, forward and backward in one call             */
/* ------------------------------------------------------------------------ */

/* Workspace bytes for flce_fwd_bwd.  chunk > 0: rows per chunk as for
 * flce_workspace_bytes; chunk <= 0 (a negative value included): the row chunk
 * of the library default.  The one-call path always chunks rows: each chunk's
 * lse must be complete before its gradient is formed. */
FLCE_API size_t flce_fwd_bwd_workspace_bytes(int dt, int64_t N, int64_t D, int64_t V,
                                             int64_t chunk);

/* Loss and gradients in one call, with the gradient formed while the logits of
 * each chunk are at hand: the eager-gradient variant of Liger-Kernel issue
 * #533 "Gradient checkpointing for grad_weight in LFCE" (feature pitch: the
 * gradients are computed in the forward and only scaled in the backward).
 * It costs 6NDV flops instead of the 8NDV of flce_fwd + flce_bwd: per chunk
 * the forward contraction also stores the chunk's logits (as base-2 offsets
 * from each 256-column tile's maximum, in dtype dt) into the workspace, dZ is
 * formed from them in place once the chunk's lse is known, and grad_H, grad_W,
 * grad_bias follow as in flce_bwd.  grad_loss ([1] f32 device) may be NULL,
 * meaning g = 1 (scale later with flce_grad_scale).  Outputs as flce_fwd
 * (loss, n_valid, lse, optional loss_rows) and flce_bwd (grad_H, grad_W,
 * grad_bias, each optional).  ws: flce_fwd_bwd_workspace_bytes bytes. */
FLCE_API int flce_fwd_bwd(const void* H, const void* W, const void* bias, int dt, int64_t N,
                          int64_t D, int64_t V, const int64_t* labels, int64_t ignore_index,
                          int reduction, int64_t num_label_tokens, const float* grad_loss,
                          int64_t chunk, float* loss, int64_t* n_valid, float* lse,
                          float* loss_rows, void* grad_H, float* grad_W, int accumulate_grad_W,
                          float* grad_bias, void* ws, size_t ws_bytes, int32_t* status,
                          flce_stream_t stream);

/* *n_valid = number of labels[0..N) that are not ignore_index and lie in
 * [0, V) (device pointers).  Data-parallel training sums it over ranks and
 * passes the total as num_label_tokens, so that the per-rank losses and
 * gradients add up to those of the global mean. */
FLCE_API int flce_count_valid(const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index,
                              int64_t* n_valid, flce_stream_t stream);

/* x[0..n) *= *g for x of dtype dt (device pointers); when *g == 1 nothing is
 * written.  Applies the incoming gradient to gradients computed with g = 1. */
FLCE_API int flce_grad_scale(void* x, int dt, int64_t n, const float* g, flce_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H */
