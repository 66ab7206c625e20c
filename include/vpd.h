/*
 * vpd.h -- C ABI of the GB300 (sm_103a) per-token vocabulary softmax
 * divergence library (libvpd): generalized Jensen-Shannon divergence JSD_beta,
 * forward/reverse KL, entropy and selected (top-k) log-probabilities between
 * language-model logits, each with its closed-form backward.
 *
 * Sources (web pages), cited below by short name:
 *   [JSD page]  DeepSpeed pull request #8958, "[VocabTP] Add vocabulary-parallel
 *               generalized JSD with Triton kernels".
 *   [ops page]  DeepSpeed pull request #8791, "Add vocabulary-parallel logprobs,
 *               entropy and KL ops".
 *   [OPSD page] DeepSpeedExamples pull request #1019, "Add an opt-in
 *               vocabulary-parallel KL route to OPSD".
 *
 * Notation for one token row r of logits s (student) and t (teacher), or x:
 *   S_x = { j : x_j > -inf },  m_x = max_{S_x} x_j,  Z_x = sum_{S_x} e^{x_j - m_x},
 *   L_x = ln Z_x,  ln p_j = (s_j - m_s) - L_s,  ln q_j = (t_j - m_t) - L_t,
 *   M_j = (1 - beta) p_j + beta q_j.
 * The max and the log-sum-exp are kept separate ([ops page], "How"). Natural
 * logarithms throughout; every output is float32.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Ownership: the caller owns every buffer. The library allocates no device or
 *   host memory for its calls and keeps no state between them besides one
 *   device error word per GPU (see vpd_device_status), a 4 MiB scratch array
 *   per GPU for vpd_jsd_linear_fwd_noalloc, and, per device and calling
 *   thread, a side stream with its events (vpd_jsd_fwd / vpd_jsd_fwdbwd) and
 *   the events of vpd_jsd_fwdbwd_teacher_stream, created on first use.
 *   Pointers documented as "device" must be device-accessible addresses on the
 *   current CUDA device.
 * Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *   default stream) and the call returns without waiting, except where stated.
 * Errors: argument, dtype and shape problems are detected on the host before
 *   anything is launched, and the call returns the matching code with nothing
 *   written. A launch failure returns VPD_ERR_CUDA. vpd_last_error() gives a
 *   one-line description of the last failure on the calling thread.
 * Rows: N = 0 is a no-op. V = 0 gives NaN rows (no distribution).
 * Special rows ([ops page], "How" and the review thread "Prevent NaN gradients
 *   from fully masked padding rows"): a row that is fully -inf in any input of
 *   the op has no distribution; its output is NaN and its gradient exactly 0,
 *   so masking the output afterwards is safe. A row whose KL is +inf (the
 *   target has mass on a token the other side masks, decided by logit
 *   finiteness, [ops page], "Tests") also gets a zero gradient. A row holding
 *   NaN or +inf is outside the contract; it is given a NaN output and a zero
 *   gradient.
 * Temperature, T^2 scaling, masking and reduction over tokens stay with the
 *   caller ([JSD page], "Changes"; [ops page], "Limitations").
 */
#ifndef VPD_H
#define VPD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VPD_ABI_VERSION 1
/* Most vocabulary segments one call accepts. */
#define VPD_MAX_SEGMENTS 256

typedef enum {
    VPD_OK = 0,
    VPD_ERR_ARG = 1,     /* NULL pointer, beta outside [0, 1], k < 1, misaligned pointer ... */
    VPD_ERR_DTYPE = 2,   /* unknown dtype, or student and teacher dtypes differ */
    VPD_ERR_SHAPE = 3,   /* rows/vocab mismatch, stride < vocab, segment widths not summing to vocab */
    VPD_ERR_INDEX = 4,   /* an index outside [0, V) (vpd_logprobs_fwd without err_flag) */
    VPD_ERR_CUDA = 5,    /* a CUDA call or launch failed */
    VPD_ERR_TIMEOUT = 6, /* a bounded device-side wait gave up (see vpd_device_status) */
    VPD_ERR_UNSUPPORTED = 7
} vpd_status;

typedef enum { VPD_F32 = 0, VPD_BF16 = 1, VPD_F16 = 2 } vpd_dtype;

/* A read-only [N, V] logits view. Row r starts at element
 *     (r / rows_per_batch) * batch_stride + (r % rows_per_batch) * row_stride
 * when rows_per_batch > 0, else at r * row_stride (strides in elements).
 * rows_per_batch / batch_stride describe a non-contiguous causal-shift view such
 * as logits[:, :-1, :] of a [B, T, V] tensor ([JSD page], "Changes": non-contiguous
 * causal-shift views). `data` must be aligned to the element size. */
typedef struct {
    const void *data;       /* device pointer to element (0, 0) */
    int32_t dtype;          /* vpd_dtype */
    int64_t rows;           /* N >= 0 */
    int64_t vocab;          /* V >= 0 */
    int64_t row_stride;     /* elements between consecutive rows of a batch, >= V */
    int64_t rows_per_batch; /* 0: plain 2-D view */
    int64_t batch_stride;   /* elements between batches when rows_per_batch > 0 */
} vpd_view;

/* An ordered split of the vocabulary into segments, the single-GPU stand-in for
 * vocabulary shards ([JSD page], "Changes": uneven vocabulary shards and empty
 * local shards). Widths are host memory, each >= 0, summing to V; count <=
 * VPD_MAX_SEGMENTS. Per-segment statistics are merged as the shards' MAX and SUM
 * all-reduces would merge them, an empty or fully -inf segment contributing
 * (-inf, 0) ([ops page], "How" and the review thread "Reject unsupported empty
 * shards consistently across TP ranks"). A NULL pointer or count 0 means one
 * segment spanning the vocabulary. */
typedef struct {
    int32_t count;
    const int64_t *widths;
} vpd_segments;

/* A gradient output: dense [N, V] rows, `row_stride` elements apart, in `dtype`
 * (float32, or bf16/fp16 rounded to nearest even). A NULL vpd_grad pointer or
 * NULL `data` means that gradient is not wanted (e.g. a detached teacher,
 * [JSD page], "Changes"). */
typedef struct {
    void *data;
    int32_t dtype;
    int64_t row_stride;
} vpd_grad;

/* Per-row state saved by a forward for its backward ([ops page], "How": only the
 * inputs and [N] statistics are saved). Float32, row-major, device memory:
 *   JSD and KL:  [N, 6] = (m_s, L_s, m_t, L_t, A, B), A = KL(P_t || M) and
 *                B = KL(P_s || M) with M taken at beta (so at beta = 0, A is the
 *                forward KL and B = 0; at beta = 1, A = 0 and B is the reverse KL).
 *   entropy:     [N, 3] = (m, L, H)
 *   log-probs:   [N, 2] = (m, L)
 * A row with NaN or +inf input stores m = NaN; a fully -inf row stores m = -inf. */
#define VPD_SAVED_PAIR 6
#define VPD_SAVED_ENTROPY 3
#define VPD_SAVED_LOGPROBS 2

/* ---------------------------------------------------------------------------
 * Generalized JSD ([JSD page], "Motivation", "Changes", "Scope and limitations").
 *   JSD_beta = beta * KL(P_t || M) + (1 - beta) * KL(P_s || M),  0 < beta < 1;
 *   beta = 0 is the explicit forward-KL branch KL(P_t || P_s) and beta = 1 the
 *   explicit reverse-KL branch KL(P_s || P_t): branches, not limits.
 * s, t: student and teacher views with the same N, V and dtype; they share the
 *   segment table. beta in [0, 1].
 * ------------------------------------------------------------------------- */

/* Forward. The statistics must be global before the divergence ([JSD page],
 * "Scope and limitations"). At beta = 0 / 1 (the KL branches) the call runs
 * the online single-pass KL kernel of vpd_kl_fwd (same loss and saved
 * layout). Otherwise, under the single-read conditions of vpd_jsd_fwdbwd
 * (aligned rows, V a multiple of 8), a forward-only cluster kernel
 * reads each row pair once and keeps it on chip for both steps, when the row
 * fits in clusters of at most 10 CTAs (V <= 191040 with 227 KB of shared memory
 * per CTA), or of at most 16 when the call has enough rows for the SMs those
 * clusters leave idle to take a share (as in vpd_jsd_fwdbwd); otherwise the
 * pages' design in two input passes: a
 * paired-statistics kernel merges per-segment (max,
 * sum-exp) of both inputs, then a divergence kernel reduces the two
 * KL-to-mixture expectations together ([JSD page], "Changes").
 * On the single-read path a row whose largest finite logit exceeds 2^126 is
 * out of contract and comes back NaN (the streaming path and the oracle give a
 * finite value there); the limit keeps every clamped log-difference finite.
 * Segments: the single-read kernel merges its CTA slices with the same MAX /
 * SUM merge the segments define, so a segmented call takes it too (results
 * equal up to the order of the additions).
 * loss:  device float[N], the per-token divergence.
 * saved: device float[N, 6] (see above), required: it carries the statistics
 *        to the backward (and between the two streaming kernels). */
vpd_status vpd_jsd_fwd(const vpd_view *s, const vpd_view *t, double beta, const vpd_segments *seg,
                       float *loss, float *saved, void *stream);

/* Backward: recomputes P_s, P_t and M from the inputs and the saved statistics,
 * with no saved probability tensors ([JSD page], "Changes"; [ops page], "How").
 *   0 < beta < 1: dS_j = g (1 - beta) p_j (ln p_j - ln M_j - B),
 *                 dT_j = g beta q_j (ln q_j - ln M_j - A);
 *   beta = 0:     dS = g (p - q),  dT_j = g q_j (ln q_j - ln p_j - KL);
 *   beta = 1:     dS_j = g p_j (ln p_j - ln q_j - KL),  dT = g (q - p).
 * Tokens outside the support and rows with a non-finite loss get exactly 0.
 * grad_loss: device float[N], the upstream gradient g (NULL means 1).
 * saved: device float[N, 6] written by vpd_jsd_fwd or vpd_jsd_fwdbwd with the
 *   same inputs and beta.
 * ds, dt: gradient outputs; either may be absent (NULL or NULL data). */
vpd_status vpd_jsd_bwd(const vpd_view *s, const vpd_view *t, double beta, const vpd_segments *seg,
                       const float *grad_loss, const float *saved, const vpd_grad *ds,
                       const vpd_grad *dt, void *stream);

/* Forward and backward in one call, with the upstream gradient given up front.
 * The single-read path runs when V is a multiple of 8, every row of the
 * inputs and gradients starts on a 16-byte boundary, the gradients are
 * float32 or the input dtype, and the row fits on a thread-block cluster
 * (V <= 311296 for bf16 / fp16, V <= 229248 for fp32, whose gradients are
 * stored from registers); any segment table (see vpd_jsd_fwd). There a
 * cluster of up to 16 CTAs holds each row pair on chip and statistics,
 * divergence and gradients come from one HBM read; a row whose finite max
 * exceeds 2^126 is treated as out of contract (NaN, zero gradient). The clusters cannot
 * always cover every SM (at V = 151936, 15 clusters of 9 CTAs use 135 of 152);
 * when the call has many rows per cluster, its last rows (from any row of
 * the view, mid-batch included) go to the streaming kernels on the SMs left
 * idle, on a side stream that
 * forks from `stream` and joins it again before the call's work ends (the
 * share follows the measured per-SM rates of the two paths). Otherwise the
 * call runs the two forward kernels and the backward kernel in turn. With both
 * gradients absent the single-read path is the forward-only kernel. Outputs
 * as vpd_jsd_fwd (loss, and saved, which is required) plus the gradients as
 * vpd_jsd_bwd. */
vpd_status vpd_jsd_fwdbwd(const vpd_view *s, const vpd_view *t, double beta,
                          const vpd_segments *seg, const float *grad_loss, float *loss,
                          float *saved, const vpd_grad *ds, const vpd_grad *dt, void *stream);

/* JSD forward+backward with the teacher logits in a pinned host cache
 * ([OPSD page], "Update: copy teacher-cache chunks from pinned memory"). The
 * teacher rows go to the device in chunks of `chunk_rows` rows, one
 * cudaMemcpy2DAsync each, on `copy_stream` into a ring of up to four staging
 * chunks carved from `staging`, and each chunk's vpd_jsd_fwdbwd runs on
 * `stream` as soon as its rows have arrived, while the next chunks copy.
 * s: device student view, plain 2-D [N, V]. t_host: pinned (page-locked or
 * registered) host memory, [N, V] rows `t_row_stride` elements apart, dtype
 * t_dtype equal to the student's. staging: device memory of at least two
 * chunks (chunk_rows * V elements each), 16-byte aligned, owned by the caller
 * and not touched by other work until `stream` has passed this call. Outputs as
 * vpd_jsd_fwdbwd; dt, when given, is a device [N, V] gradient. Both streams
 * must belong to the current device and be distinct; the copy stream first
 * waits for the work already on `stream`, and `stream` ends after the last
 * chunk. The library keeps nine reusable events per device and calling thread
 * for this ordering (created on the first call). A pageable cache returns
 * VPD_ERR_ARG. */
vpd_status vpd_jsd_fwdbwd_teacher_stream(const vpd_view *s, const void *t_host, int32_t t_dtype,
                                         int64_t t_row_stride, double beta, const float *grad_loss,
                                         float *loss, float *saved, const vpd_grad *ds, const vpd_grad *dt,
                                         void *staging, size_t staging_bytes, int64_t chunk_rows,
                                         void *stream, void *copy_stream);

/* The path a JSD call with these arguments takes, decided on the host with
 * nothing launched: how many rows go to the single-read cluster kernel, how
 * many to the streaming kernels on the SMs its clusters leave idle, and the
 * number of kernel launches. With ds and dt both absent (NULL or NULL data)
 * the answer is for vpd_jsd_fwd with 0 < beta < 1 (the forward-only kernel; at
 * beta = 0 / 1 that call runs the online KL kernel, one launch), otherwise for
 * vpd_jsd_fwdbwd. The data pointers of the views and gradients are not read.
 * fused_rows = 0 means the streaming kernels only. Any output may be NULL. */
vpd_status vpd_jsd_plan(const vpd_view *s, const vpd_view *t, const vpd_segments *seg, const vpd_grad *ds,
                        const vpd_grad *dt, int64_t *fused_rows, int64_t *idle_sm_rows, int32_t *launches);

/* ---------------------------------------------------------------------------
 * Forward / reverse KL ([ops page], "What"): reverse = 0 gives KL(P_t || P_s)
 * (the teacher is the target), reverse = 1 gives KL(P_s || P_t). The forward
 * reads the inputs once in one online pass (running maxima with rescaled
 * sums) on every SM, one CTA per row at a time; as on the single-read kernels
 * a row whose largest finite logit exceeds 2^126 is out of contract and comes
 * back NaN (the rescaling of the running sums would overflow). saved may be
 * NULL.
 * Saved layout and backward are those of the JSD beta = 0 / 1 branches.
 * ------------------------------------------------------------------------- */
vpd_status vpd_kl_fwd(const vpd_view *s, const vpd_view *t, int32_t reverse,
                      const vpd_segments *seg, float *loss, float *saved, void *stream);
vpd_status vpd_kl_bwd(const vpd_view *s, const vpd_view *t, int32_t reverse,
                      const vpd_segments *seg, const float *grad_loss, const float *saved,
                      const vpd_grad *ds, const vpd_grad *dt, void *stream);

/* ---------------------------------------------------------------------------
 * Entropy ([ops page], "What"): H = -sum_{S} p_j ln p_j, one online pass;
 * backward dX_j = -g p_j (ln p_j + H).
 * out: device float[N]; saved: device float[N, 3] or NULL.
 * ------------------------------------------------------------------------- */
vpd_status vpd_entropy_fwd(const vpd_view *x, const vpd_segments *seg, float *out, float *saved,
                           void *stream);
vpd_status vpd_entropy_bwd(const vpd_view *x, const vpd_segments *seg, const float *grad_out,
                           const float *saved, const vpd_grad *dx, void *stream);

/* ---------------------------------------------------------------------------
 * Selected / top-k log-probabilities ([ops page], "What"):
 *   out[r, k] = ln p_{index[r, k]}; a position equal to ignore_index returns 0
 *   and takes no gradient; a selected token with a -inf logit returns -inf and
 *   takes no gradient.
 * index: device int64[N, k] (row-major, k >= 1).
 * out: device float[N, k]; saved: device float[N, 2] or NULL.
 * err_flag: device int32[1] or NULL. Given, the call sets it to 0, and to 1 if
 *   any index outside [0, V) (other than ignore_index) is found; such positions
 *   output NaN, and reading the flag is the caller's synchronisation point.
 *   NULL: the call copies the indices to the host on `stream`, synchronises,
 *   and returns VPD_ERR_INDEX before any launch (nothing written) if one is
 *   out of range. Either way the check is the pages' synchronising index
 *   validation ([ops page], review thread "Provide a path for reusing validated
 *   shard metadata").
 * Backward: dX_j = sum_k g_rk [j == index_rk] - p_j sum_k g_rk over the positions
 *   with a finite output. grad_out: device float[N, k] (NULL means 1).
 * ------------------------------------------------------------------------- */
vpd_status vpd_logprobs_fwd(const vpd_view *x, const vpd_segments *seg, const int64_t *index,
                            int32_t k, int64_t ignore_index, float *out, float *saved,
                            int32_t *err_flag, void *stream);
vpd_status vpd_logprobs_bwd(const vpd_view *x, const vpd_segments *seg, const int64_t *index,
                            int32_t k, int64_t ignore_index, const float *grad_out,
                            const float *saved, const vpd_grad *dx, void *stream);

/* ---------------------------------------------------------------------------
 * Vocabulary-parallel JSD / KL ([ops page], "How"; [JSD page], "Changes"): each
 * process holds one ordered vocabulary shard [N, V_k] of both inputs (V_k may
 * be 0) and the forward exchanges only [N]-sized statistics, through three
 * all-reduces that the caller runs on the [N, 2] float buffer xbuf (NCCL or
 * any collective library; the library itself communicates with nobody):
 *   vpd_jsd_shard_stats       local statistics into saved; xbuf = (m_s, m_t)
 *   -> all-reduce MAX (xbuf)
 *   vpd_jsd_shard_rescale     saved keeps the global maxima; xbuf = the
 *                             shard's sums rescaled to them
 *   -> all-reduce SUM (xbuf)
 *   vpd_jsd_shard_divergence  saved gets the global log-sum-exps; loss and
 *                             xbuf get the shard's partial (A, B)
 *   -> all-reduce SUM (xbuf)
 *   vpd_jsd_shard_finish      loss = the per-token value, saved = [N, 6] as
 *                             vpd_jsd_fwd writes it, identical on every shard
 * The backward needs no exchange: vpd_jsd_bwd on the shard with that saved
 * gives the shard's columns of dS and dT. beta = 0 / 1 are the forward /
 * reverse KL branches (a support violation on any shard makes the row +inf).
 * A row outside the contract on any shard travels as +inf through the MAX and
 * NaN through the SUMs, so every process ends with the same NaN row.
 * saved: device float[N, 6]; xbuf: device float[N, 2]; all on `stream`.
 * ------------------------------------------------------------------------- */
vpd_status vpd_jsd_shard_stats(const vpd_view *s, const vpd_view *t, float *saved, float *xbuf, void *stream);
vpd_status vpd_jsd_shard_rescale(int64_t rows, float *saved, float *xbuf, void *stream);
vpd_status vpd_jsd_shard_divergence(const vpd_view *s, const vpd_view *t, double beta, float *loss,
                                    float *saved, float *xbuf, void *stream);
vpd_status vpd_jsd_shard_finish(int64_t rows, double beta, float *saved, const float *xbuf, float *loss,
                                void *stream);

/* ---------------------------------------------------------------------------
 * Two thin ops on the selected log-probabilities ([ops page], "What": the
 * teacher top-k forward KL written with the log-prob op; "How": the
 * cross-entropy op that validates its shard layout the same way), each with an
 * optional temperature T > 0 that divides the logits before the softmax (T = 1:
 * none; [OPSD page] divides by it in fp32 before the op). The statistics saved
 * for the backward ([N, 2] as for log-probs, or NULL) are those of x / T.
 * Index checking, err_flag and ignore_index behave as in vpd_logprobs_fwd.
 * ------------------------------------------------------------------------- */

/* Cross-entropy per token: loss[r] = -ln softmax(x_r / T)[labels[r]]; a label
 * equal to ignore_index gives 0 and no gradient; a label whose logit is -inf
 * gives +inf and no gradient. labels: device int64[N]; loss: device float[N].
 * Backward: dx_j = (g / T) (p_j - [j == label]); grad_loss device float[N] or
 * NULL (ones). */
vpd_status vpd_cross_entropy_fwd(const vpd_view *x, const vpd_segments *seg, const int64_t *labels,
                                 int64_t ignore_index, double temperature, float *loss, float *saved,
                                 int32_t *err_flag, void *stream);
vpd_status vpd_cross_entropy_bwd(const vpd_view *x, const vpd_segments *seg, const int64_t *labels,
                                 int64_t ignore_index, double temperature, const float *grad_loss,
                                 const float *saved, const vpd_grad *dx, void *stream);

/* Teacher top-k forward KL per token:
 *   kl[r] = sum_k e^{tl[r,k]} (tl[r,k] - ln softmax(s_r / T)[index[r,k]]),
 * with tl the teacher's log-probabilities at its top-k ids (device float[N, k],
 * computed by the caller; the teacher is detached). Positions equal to
 * ignore_index, and teacher log-probs of -inf, contribute nothing; an id the
 * teacher gives mass but the student masks (-inf logit) makes the row +inf.
 * Backward to the student only: ds_j = (g / T) (p_j W - sum_k e^{tl_k}
 * [j == index_k]) with W = sum_k e^{tl_k} over the contributing positions; a
 * +inf or NaN row gets a zero gradient. grad_kl device float[N] or NULL. */
vpd_status vpd_topk_kl_fwd(const vpd_view *s, const vpd_segments *seg, const int64_t *index, int32_t k,
                           int64_t ignore_index, const float *teacher_logp, double temperature, float *kl,
                           float *saved, int32_t *err_flag, void *stream);
vpd_status vpd_topk_kl_bwd(const vpd_view *s, const vpd_segments *seg, const int64_t *index, int32_t k,
                           int64_t ignore_index, const float *teacher_logp, double temperature,
                           const float *grad_kl, const float *saved, const vpd_grad *ds, void *stream);

/* ---------------------------------------------------------------------------
 * Fused-linear generalized JSD ([JSD page], "Scope and limitations" and [ops
 * page], "Limitations": the fused-linear divergence the pages leave for later).
 * The logits of two linear heads, s = h_s w_s^T and t = h_t w_t^T, are formed
 * tile by tile on the tensor cores and consumed on chip: the [N, V] logits are
 * never written to memory. The divergence, its beta = 0 / 1 branches, the
 * saved [N, 6] statistics and the special values are those of vpd_jsd_fwd /
 * vpd_jsd_bwd applied to s and t, where the logits are the fp32 sums of the
 * exact bf16 products.
 * ------------------------------------------------------------------------- */
typedef struct {
    const void *h_s;   /* device bf16 [rows, hidden_s] student hidden states, row stride ld_hs */
    const void *w_s;   /* device bf16 [vocab, hidden_s] student head weight, row stride ld_ws */
    const void *h_t;   /* device bf16 [rows, hidden_t] teacher hidden states, row stride ld_ht */
    const void *w_t;   /* device bf16 [vocab, hidden_t] teacher head weight, row stride ld_wt */
    int64_t rows;      /* N >= 0 */
    int64_t vocab;     /* V >= 1, a multiple of 8 */
    int64_t hidden_s;  /* a positive multiple of 64 */
    int64_t hidden_t;  /* a positive multiple of 64 */
    int64_t ld_hs, ld_ws, ld_ht, ld_wt; /* row strides in elements: >= the hidden size, multiples of 8 */
} vpd_linear_heads;

/* Workspace sizes (bytes) of vpd_jsd_linear_fwd and of vpd_jsd_linear_bwd
 * with the given gradients wanted (nonzero flags). The backward works through
 * the rows in chunks of 8192 and keeps, per head, that chunk's gradient of the
 * logits split in two bf16 parts (row-major; the contractions read them and
 * the head weight in place, transposed where they need) and the chunk's hidden
 * states transposed. Either output pointer
 * may be NULL. */
vpd_status vpd_jsd_linear_workspace(const vpd_linear_heads *heads, int32_t student_grads,
                                    int32_t teacher_grads, size_t *fwd_bytes, size_t *bwd_bytes);

/* Forward: two passes of tensor-core tiles over the vocabulary, the first for
 * the statistics of both heads (per-chunk (max, sum-exp) partials merged in
 * chunk order), the second for the two KL-to-mixture sums ([JSD page],
 * "Scope and limitations": the mixture needs global statistics).
 * loss: device float[N]; saved: device float[N, 6] as vpd_jsd_fwd's.
 * workspace: device memory of at least the forward size above (caller-owned,
 * 16-byte aligned; its contents on entry do not matter). */
vpd_status vpd_jsd_linear_fwd(const vpd_linear_heads *heads, double beta, float *loss, float *saved,
                              void *workspace, size_t workspace_bytes, void *stream);

/* Backward: recomputes the logits tiles, forms dS and dT as vpd_jsd_bwd does
 * and contracts them on the tensor cores: dh = dS w, dw = dS^T h per head. The
 * gradient of the logits enters the contractions as a bf16 high part plus a
 * bf16 low part (16 bits of mantissa together). Outputs are device float32,
 * dense: dh_s [N, hidden_s], dw_s [V, hidden_s], dh_t [N, hidden_t], dw_t [V,
 * hidden_t]; each may be NULL (not wanted; a detached teacher passes NULL for
 * both of its own). They are overwritten (set to zero, then accumulated).
 * grad_loss: device float[N] or NULL (ones); loss and saved: as written by
 * vpd_jsd_linear_fwd with the same heads and beta. workspace: at least the
 * backward size above for the gradients wanted. */
vpd_status vpd_jsd_linear_bwd(const vpd_linear_heads *heads, double beta, const float *grad_loss,
                              const float *loss, const float *saved, float *dh_s, float *dw_s,
                              float *dh_t, float *dw_t, void *workspace, size_t workspace_bytes,
                              void *stream);

/* Largest forward workspace (bytes) vpd_jsd_linear_fwd_noalloc can serve. */
#define VPD_LINEAR_NOALLOC_MAX_BYTES (4u << 20)

/* vpd_jsd_linear_fwd for callers that cannot allocate device memory: for
 * example an engine that owns all device memory and hands each op only its
 * inputs and outputs, or a latency-critical loop where cudaMalloc / cudaFree
 * would stall the device. The pages have no counterpart of this entry point.
 * Same arguments, results and errors as vpd_jsd_linear_fwd, without the
 * workspace: the statistics partials go to one array of
 * VPD_LINEAR_NOALLOC_MAX_BYTES bytes that the library keeps in device memory
 * for the life of the process (each GPU that loads the library holds one).
 * The partials take 16 bytes per row, vocabulary chunk and column half of a
 * tile; where the array is smaller than the forward workspace
 * vpd_jsd_linear_workspace reports (the fastest plan's), the forward splits the
 * vocabulary into fewer, longer chunks so that they fit, down to one chunk (32
 * bytes per row). So every problem of up to 131072 rows runs, at any
 * vocabulary; more rows return VPD_ERR_SHAPE before anything is launched.
 * Nothing is allocated: no cudaMalloc, no cudaFree. The first call on a
 * device looks up the array's device address on that device (make that device
 * current first); make this first call before any stream capture. Every call
 * shares the one array: calls whose work overlaps on the GPU (other streams,
 * other threads, other devices are separate arrays) race and give undefined
 * results, so serialise them. Nothing from an earlier call needs clearing:
 * every entry a call reads, the same call writes first. */
vpd_status vpd_jsd_linear_fwd_noalloc(const vpd_linear_heads *heads, double beta, float *loss,
                                      float *saved, void *stream);

/* ---------------------------------------------------------------------------
 * Utilities.
 * ------------------------------------------------------------------------- */
/* Name of a status code (static string). */
const char *vpd_status_string(vpd_status status);
/* Description of the last failure on the calling thread ("" if none). */
const char *vpd_last_error(void);
/* VPD_ABI_VERSION of the loaded library. */
int32_t vpd_abi_version(void);
/* Number of kernel launches this library has issued since it was loaded
 * (all threads, all devices); lets a caller count the device work of a call. */
uint64_t vpd_launch_count(void);
/* Test hook for the failure path. The next single-read launch of
 * vpd_jsd_fwdbwd made from this thread withholds the shared-memory copy of row
 * `row` in the first CTA of the cluster that owns it, so that CTA's bounded
 * wait expires (after about two seconds). The kernel then records the timeout,
 * every CTA leaves its row loop, the outputs of that call are unspecified, and
 * vpd_device_status reports VPD_ERR_TIMEOUT; the device stays usable. A
 * negative row clears the hook. Returns VPD_OK. */
vpd_status vpd_test_withhold_copy(int64_t row);
/* Synchronises `stream`, then reads and clears the device error word that the
 * library's kernels set when a bounded wait gives up. The read and the clear
 * are one atomic exchange on the device, ordered on `stream`, so a failure that
 * a kernel on another stream records meanwhile is reported by this call or the
 * next, never lost. Returns VPD_OK, or VPD_ERR_TIMEOUT with the failure
 * described in vpd_last_error(). */
vpd_status vpd_device_status(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* VPD_H */
