/*
 * saf.h — C ABI of libsaf: the hot path of Selective Attention Freezing (SAF)
 * on one GB300 (sm_103a).
 *
 * The method is the one described in "When Can Attention Heads Be Statically
 * Defined?" (close-reading notes of Li, Tai, Fonseca and Cohen):
 *
 *   - dynamic head (§1, the attention equation):
 *       A = softmax_causal(Q K^T / sqrt(d_h)),  out = A V;
 *   - static ("frozen") head (§3, Eq. (3)):
 *       P(i,j) = exp(alpha(j) + rho(i-j)) / Z(i) for j <= i, 0 for j > i,
 *       Z(i)   = sum_{k<=i} exp(alpha(k) + rho(i-k)),      out = P V,
 *     stored as the two length-T vectors alpha, rho;
 *   - one launch per layer runs both kinds of head; a frozen head never reads
 *     Q or K, and its attention backward is dV = P^T dZ (§3.3, App. D.2);
 *   - calibration (§3.1): A_hat = mean_n A_n over N sequences, the variance
 *     score of Eq. (1)  s_var = sum_n ||A_n - A_hat||_F^2 / ((N-1) T^2),
 *     and the first k = round(r L H) heads of all layers in ascending s_var.
 *
 * Indices are 0-based: query i, key j, distance i - j in [0, T).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensor arguments are DEVICE pointers owned by the caller, contiguous,
 *    16-byte aligned, on the current CUDA device.  The only host pointers are
 *    `dims`, `head_is_static`, `handle` outputs and `saf_status_string`.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Argument checks run on the host before anything is
 *    launched and return an error status without touching any buffer.
 *  - Attention calls never allocate: scratch comes from the caller's
 *    workspace, sized by saf_hybrid_attn_workspace_size().  The calibration
 *    handle allocates its state once, in saf_calib_create().
 *  - Every device-side wait in the kernels is bounded.  A wait that runs out
 *    records SAF_ERR_TIMEOUT in a status word that saf_get_device_status()
 *    returns; the kernels then finish without touching more memory.
 *  - Not thread-safe per workspace or handle: concurrent calls must use
 *    different workspaces / handles.
 */
#ifndef SAF_H_
#define SAF_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SAF_API __attribute__((visibility("default")))
#else
#define SAF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum saf_status {
  SAF_OK = 0,
  SAF_ERR_INVALID_ARG = 1,  /* null or misaligned pointer, bad size, k out of range   */
  SAF_ERR_UNSUPPORTED = 2,  /* valid but not implemented: d_h, T > 16384, H > 256, ...  */
  SAF_ERR_CUDA = 3,         /* a CUDA runtime/driver call or a launch failed            */
  SAF_ERR_STATE = 4,        /* calibration state misuse (e.g. finalize with N < 2)      */
  SAF_ERR_TIMEOUT = 5       /* a bounded device wait ran out (read with get_device_status) */
} saf_status;

typedef enum saf_dtype {
  SAF_BF16 = 0,  /* bf16 Q/K/V/out/dout/dQ/dK/dV                                     */
  SAF_F32 = 1    /* fp32 I/O: converted to bf16 in the workspace, computed in bf16,  *
                  * results written back as fp32                                      */
} saf_dtype;

/* Shape of one attention layer.  Q, out, dout, dQ are [B, H, T, d_h]
 * row-major; K, V, dK, dV are [B, H_kv, T, d_h]; lse is [B, H, T] fp32;
 * alpha, rho, dalpha, drho are [H, T] fp32 (only the rows of static heads are
 * read or written).
 *
 * Grouped K/V (the GQA path of "When Can Attention Heads Be Statically
 * Defined?", §3.3 / App. D.2): with H_kv < H, query head h reads K/V head
 * h / (H / H_kv).  A frozen query head still mixes its group's V (only its
 * query path is gone); dK and dV of a K/V head sum the gradients of every
 * query head it serves, and dK of a K/V head that serves no dynamic head is
 * zero.  H_kv = 0 means H_kv = H (one K/V head per query head).
 *
 * The kernels work on whole tiles of 128 rows.  A length T that is not a
 * multiple of 128 runs on copies padded to the next multiple, held in the
 * workspace (zero rows of Q, K, V, dout; alpha and rho padded with -inf;
 * lse of the padded rows 0), and the results are cropped back to T: padded
 * keys lie above the causal diagonal of every real row and padded rows carry
 * dout = 0, so the real rows' outputs and gradients are those of length T.
 * The workspace then holds the padded copies too.
 *
 * B, H or T zero is an empty layer: the attention calls return SAF_OK at once
 * without reading any pointer or launching anything, and the workspace query
 * returns 0. */
typedef struct saf_attn_dims {
  int B;        /* batch size, >= 0                                    */
  int H;        /* query heads in the layer, 0..256                    */
  int T;        /* sequence length, 0..16384 (below: T % 128 != 0)     */
  int d_h;      /* head dimension: 32, 64 or 128                       */
  saf_dtype dtype;
  int H_kv;     /* K/V heads: 0 (= H) or a divisor of H                */
} saf_attn_dims;

/* Bytes of device workspace that saf_hybrid_attn_fwd / _bwd need for `dims`
 * (the larger of the two; want_param_grads != 0 adds the dalpha/drho
 * scratch).  Returns 0 when `dims` is invalid or unsupported. */
SAF_API size_t saf_hybrid_attn_workspace_size(const saf_attn_dims* dims,
                                      int want_param_grads);

/* Forward of the hybrid layer: one persistent launch runs the dynamic heads
 * (causal flash-style online softmax, tcgen05 MMAs) and the static heads
 * (P tiles generated from alpha/rho, shared by the whole batch, times V),
 * preceded by a small pre-pass over alpha/rho that forms Z(i).
 *
 *   Q, K, V        [B,H,T,d_h] (bf16 or fp32 per dims->dtype); Q and K rows of
 *                  static heads are never read (they may hold anything).
 *   alpha, rho     [H,T] fp32; rows of dynamic heads are never read.  -inf is
 *                  allowed (a weight of exactly zero); a row whose every
 *                  logit is -inf gives out = 0 and lse = -inf.
 *   head_is_static HOST array [H]; nonzero marks a frozen head.
 *   out            [B,H,T,d_h], same dtype as Q.
 *   lse            [B,H,T] fp32 or NULL.  Dynamic heads: log sum_j exp(S(i,j));
 *                  static heads: log Z(i).  Needed by the backward.
 *   workspace      device scratch of ws_bytes >= the size query; 256-byte
 *                  aligned.  It also holds the device status word.
 * Returns SAF_OK, or INVALID_ARG / UNSUPPORTED / CUDA. */
SAF_API saf_status saf_hybrid_attn_fwd(const saf_attn_dims* dims,
                               const void* Q, const void* K, const void* V,
                               const float* alpha, const float* rho,
                               const uint8_t* head_is_static,
                               void* out, float* lse,
                               void* workspace, size_t ws_bytes,
                               void* stream);

/* Backward of the hybrid layer for the loss gradient `dout` of `out`.
 *
 *   Q, K, V, alpha, rho, head_is_static: as in the forward.
 *   out, lse       the forward's outputs (lse must not be NULL here).
 *   dout           [B,H,T,d_h] upstream gradient.
 *   dQ, dK, dV     [B,H,T,d_h] outputs, overwritten.  Dynamic heads: the full
 *                  softmax-attention gradients.  Static heads: dV = P^T dout;
 *                  their dQ and dK are written as zeros.
 *   dalpha, drho   [H,T] fp32 or NULL (both NULL or both set).  When set, the
 *                  gradients of alpha and rho of the static heads, summed over
 *                  the batch, overwrite those rows; dynamic rows are zeroed.
 *                  These are an extension: the paper keeps alpha/rho frozen.
 *   workspace      as in the forward, sized with want_param_grads = 1 when
 *                  dalpha/drho are requested.
 * Returns SAF_OK, or INVALID_ARG / UNSUPPORTED / CUDA. */
SAF_API saf_status saf_hybrid_attn_bwd(const saf_attn_dims* dims,
                               const void* Q, const void* K, const void* V,
                               const void* out, const float* lse,
                               const void* dout,
                               const float* alpha, const float* rho,
                               const uint8_t* head_is_static,
                               void* dQ, void* dK, void* dV,
                               float* dalpha, float* drho,
                               void* workspace, size_t ws_bytes,
                               void* stream);

/* saf_hybrid_attn_fwd without a workspace: for callers that cannot allocate
 * device memory when they run the layer.  An inference engine's plugin, for
 * example, may only enqueue work on the buffers it is handed: the engine has
 * planned all device memory ahead of time (often inside a captured CUDA
 * graph) and an allocation at that point would break its plan.  Such callers
 * pass only inputs and outputs here.  The paper has no counterpart to this
 * call; it is an interface convenience.
 *
 * Arguments and results are those of saf_hybrid_attn_fwd with dims->dtype ==
 * SAF_BF16 and dims->T a multiple of 128 (fp32 I/O and other lengths would
 * need staging buffers: SAF_ERR_UNSUPPORTED).  The
 * scratch (the frozen heads' tables, log Z and the status word) lives in one
 * file-scope device array of 4 MiB that every GPU which loads the library
 * holds until the process exits; a shape whose tables need more,
 * n_static * (4 T + 130) * 4 bytes plus at most 1.5 KiB of status word and
 * alignment, is rejected with SAF_ERR_UNSUPPORTED before anything is launched
 * (15 frozen heads fit at T = 16384, 16 fit at T = 16256, 16 at T = 16384 do
 * not).  Nothing is allocated: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call on a device shares the one array and it keeps the last
 * call's contents, so calls whose work overlaps on the GPU (different streams,
 * or several host threads) race on it: serialise them.  The status word is
 * cleared at the start of every call but cannot be read back through
 * saf_get_device_status (there is no workspace to name). */
SAF_API saf_status saf_hybrid_attn_fwd_noalloc(const saf_attn_dims* dims,
                                       const void* Q, const void* K, const void* V,
                                       const float* alpha, const float* rho,
                                       const uint8_t* head_is_static,
                                       void* out, float* lse, void* stream);

/* Calibration state for `num_heads` heads (all layers, flat index
 * l * H + h) of sequence length T (a positive multiple of 4, <= 16384).
 * Allocates the per-element running mean and M2 (2 * num_heads * T * T fp32)
 * on the current device.  *handle receives an opaque pointer. */
SAF_API saf_status saf_calib_create(void** handle, int num_heads, int T);

/* saf_calib_create with options.  flags = SAF_CALIB_TRACK_KL also keeps, per
 * element, the sum over samples of x log x (one more num_heads * T * T fp32
 * array), which saf_calib_finalize_kl needs; flags = 0 is saf_calib_create. */
#define SAF_CALIB_TRACK_KL 1u
SAF_API saf_status saf_calib_create_ex(void** handle, int num_heads, int T, unsigned flags);

/* Streams n more calibration samples into the state (§3.1).
 *   A  device fp32 [n, head_count, T, T]: the causal attention probabilities of
 *      heads head_begin .. head_begin+head_count-1 for n sequences.  Only the
 *      lower triangle j <= i is read; entries above the diagonal are treated
 *      as zero.
 * All heads in the range must have seen the same number of samples so far
 * (SAF_ERR_STATE otherwise).  n = 0 or head_count = 0 changes nothing and
 * returns SAF_OK (A is then not read).  Per element the kernel keeps a count, a mean
 * and a sum of squared deviations (Welford's update, merged with Chan et
 * al.'s pairwise formula), so chunked calls match a one-shot call. */
SAF_API saf_status saf_calib_accumulate(void* handle, const float* A, int n,
                                int head_begin, int head_count, void* stream);

/* k = round(r * num_heads) with exact halves rounded to even. */
SAF_API int saf_calib_num_select(double r, int num_heads);

/* Finishes the reduction.  Every head must have the same N >= 2 samples
 * (SAF_ERR_STATE otherwise); 0 <= k <= num_heads (INVALID_ARG otherwise).
 *   A_hat     device fp32 [num_heads, T, T] or NULL: the mean pattern, exact
 *             zeros above the diagonal.
 *   s_var     device fp32 [num_heads]: Eq. (1).
 *   selected  device int32 [k] (may be NULL when k == 0): the k heads with the
 *             smallest s_var in ascending (s_var, flat index) order; ties go to
 *             the lower index.  The order compares the fp32 values written
 *             to s_var. */
SAF_API saf_status saf_calib_finalize(void* handle, int k, float* A_hat, float* s_var,
                              int32_t* selected, void* stream);

/* The row-wise forward-KL selector that the notes compare with s_var (§3.1,
 * App. B.2; its formula is not printed, the reading here is the mean over
 * samples and rows):  s_kl = (1/(N T)) sum_n sum_i KL(A_n(i,:) || A_hat(i,:)),
 * computed from the tracked state as sum_n x log x - N A_hat log A_hat, summed
 * in fp64.  Needs a handle made with SAF_CALIB_TRACK_KL (SAF_ERR_STATE
 * otherwise) and the same N >= 1 samples for every head.
 *   s_kl      device fp32 [num_heads].
 *   selected  device int32 [k]: the k heads with the smallest s_kl in
 *             ascending (s_kl, index) order (NULL when k == 0). */
SAF_API saf_status saf_calib_finalize_kl(void* handle, int k, float* s_kl, int32_t* selected,
                                 void* stream);

/* Sharp-mean pattern ("When Can Attention Heads Be Statically Defined?", one
 * of the candidate fixed patterns of §3, compared in §5.1 / Fig. 3): when the
 * handle has been fed pre-softmax logits instead of probabilities (the same
 * [n, head_count, T, T] layout; the lower triangle j <= i must be finite,
 * the rest is ignored), the pattern is the causal softmax of each row of the
 * logits' mean over the N >= 1 samples.
 *   pattern  device fp32 [num_heads, T, T]: each row a causal distribution,
 *            exact zeros above the diagonal.
 * SAF_ERR_STATE if no samples were accumulated or heads differ in N. */
SAF_API saf_status saf_calib_finalize_sharp(void* handle, float* pattern, void* stream);

/* Compact pattern fit ("When Can Attention Heads Be Statically Defined?",
 * §3 Eq. (3)/(4) and App. A.2).  For each candidate head, alpha and rho are
 * fitted to its mean pattern A_hat by `steps` Adam steps (rate `lr`, beta =
 * (0.9, 0.999), eps = 1e-8) on the row-averaged cross-entropy, starting from
 * the log of A_hat's column and diagonal means; the gradient uses only the
 * column and diagonal sums of A_hat (Eq. (4)).  Then the candidates are
 * walked in the given order and the first k whose fitted pattern has mean row
 * KL(A_hat || P_hat) <= kl_max (0.2 nat in the paper) are selected; a head
 * over the gate is skipped.
 *   A_hat       device fp32 [num_heads, T, T] (e.g. from saf_calib_finalize);
 *               T <= 4096.
 *   candidates  device int32 [n_candidates]: head indices in priority order
 *               (ascending s_var: saf_calib_finalize with k = num_heads).
 *   alpha, rho  device fp32 [n_candidates, T]: the fitted vectors.
 *   kl          device fp32 [n_candidates]: mean row KL of each fit, in nats.
 *   selected    device int32 [k] (NULL when k == 0); n_selected device int32
 *               [1]: how many heads passed (<= k; the rest of `selected` is
 *               left untouched).
 * One CTA per candidate; no workspace is needed. */
SAF_API saf_status saf_fit_compact(const float* A_hat, int num_heads, int T,
                           const int32_t* candidates, int n_candidates, int k,
                           float kl_max, int steps, float lr,
                           float* alpha, float* rho, float* kl,
                           int32_t* selected, int32_t* n_selected, void* stream);

/* Forget all accumulated samples (the allocation is kept). */
SAF_API saf_status saf_calib_reset(void* handle);

/* Free the state (synchronises the device first).  NULL is accepted. */
SAF_API saf_status saf_calib_destroy(void* handle);

/* Reads (and clears) the device status word kept in an attention workspace
 * (`is_calib_handle` = 0) or in a calibration handle (`is_calib_handle` = 1).
 * Every saf_hybrid_attn_fwd / _bwd call clears the word of its workspace when
 * it starts, so the word describes the latest call on that workspace.
 * Synchronises `stream`.  Returns SAF_OK or SAF_ERR_TIMEOUT when a bounded
 * wait ran out in a kernel; *site (if not NULL) receives a code for where it
 * happened (0 when none). */
SAF_API saf_status saf_get_device_status(void* workspace_or_handle, int is_calib_handle,
                                 int* site, void* stream);

/* Static string naming a status code. */
SAF_API const char* saf_status_string(saf_status status);

/* Number of this library's kernel launches made by the most recent
 * saf_hybrid_attn_fwd / _bwd / saf_calib_* call on this host thread. */
SAF_API int saf_last_launch_count(void);

/* Kernel trace (per host thread; for profiling, off by default).
 * saf_trace_enable(1) clears the record and starts recording: every kernel
 * this library launches from the thread is then bracketed by two CUDA events
 * on its launch stream (up to 65536 launches).  saf_trace_enable(0) stops
 * recording and clears the record.  saf_trace_get(i, ...) waits for the i-th
 * recorded launch to finish and returns its kernel name (a static string) and
 * its duration in milliseconds between the two events. */
SAF_API saf_status saf_trace_enable(int enable);
SAF_API int saf_trace_count(void);
SAF_API saf_status saf_trace_get(int index, const char** kernel, float* ms);

/* Failure-path testing (off by default; the paper has no counterpart).  With
 * hold != 0, the forward launches that follow on any host thread withhold the
 * first Q tile of their first CTA, so that the kernel's bounded waits on it
 * run out (after 2 s): that CTA records SAF_ERR_TIMEOUT and a site in the
 * workspace's status word, abandons its remaining waits, lets its copies and
 * tensor-core products finish, frees its tensor memory and returns; its
 * outputs are then undefined and the next call on the context runs normally.
 * hold = 0 restores normal operation.  Nothing faults, traps or hangs: the
 * forward only takes its own abort path. */
SAF_API saf_status saf_debug_forward_hold(int hold);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* SAF_H_ */
