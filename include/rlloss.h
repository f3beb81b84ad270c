/*
 * rlloss — fused LM-head projection + RL policy loss (GMPO, GSPO-token,
 * top-entropy-quantile mask) with its gradients, for one NVIDIA GB300 GPU.
 *
 * C ABI.  Plain pointers and sizes only.  All tensor pointers are DEVICE
 * pointers owned by the caller; the library never allocates or frees device
 * memory and keeps no pointer after a call returns.  Every call is
 * asynchronous on the given CUDA stream (a cudaStream_t passed as void*; NULL
 * = legacy default stream).  Gradients are overwritten, not accumulated.
 *
 * What is computed (sources: the pages' titles and sections):
 *   logits l = X W^T (+ b)  — "Add GMPO to fused linear GRPO loss", Summary
 *       (the fused linear path never materialises [tokens, vocab] logits);
 *   z = l / temperature; per token the target log-prob logp = z_y - lse(z)
 *       and the entropy H = lse - sum p z, streamed over the vocabulary with
 *       running (max, sum e^(z-m), sum e^(z-m) z) — "support
 *       top_entropy_quantile in fused linear GRPO loss", Details;
 *   optional entropy mask: keep active tokens with H >= quantile(active H,
 *       1 - q) over the whole batch — same page, Details;
 *   GMPO: per-token log ratio clipped one-sided in log space to
 *       [-eps_low, +eps_high] by the sign of the advantage, per-sequence
 *       geometric mean r_i = exp(masked_mean(clipped lr)), loss
 *       mean_i(-A_i r_i ebar_i + beta KL_i) with K3 KL — "Add GMPO ...",
 *       Summary and Details;
 *   GSPO-token: s_i = exp(masked_mean(logp - old)), token ratio with s_i's
 *       value and its own log-prob's gradient, loss
 *       -sum_t min(s A_t, clip(s, 1-eps_low, 1+eps_high) A_t) — Tinker
 *       "GSPO", the ratio and objective formulas;
 *   gradients dX, dW, db of the loss through the LM head.
 *
 * Layouts (row-major, contiguous): X [N, H], W [V, H], b [V] with N = B*T
 * (sequence i owns rows i*T .. i*T+T-1); dtype of X, W, b per cfg.dtype
 * (bf16 or fp32).  targets int64 [N] in [0, V).  old_logp, ref_logp fp32 [N].
 * adv fp32 [B] (applied on the sequence's active tokens), or [N] with
 * RLLOSS_FLAG_ADV_PER_TOKEN.  mask uint8 [N],
 * nonzero = completion token (active).  Outputs fp32 unless noted.
 *
 * Errors.  Functions return RLLOSS_OK or a synchronous error code BEFORE any
 * launch (invalid configuration, null or misaligned pointers, too small a
 * workspace), or RLLOSS_ECUDA when a launch failed.  Problems only visible on
 * the device (a bounded wait that ran out, a target id outside [0, V), a GSPO
 * sequence without active tokens, a non-finite loss) are OR-ed into a status
 * word inside the workspace; read it with rlloss_get_device_status after the
 * stream has been synchronised.  No kernel traps.
 */
#ifndef RLLOSS_H
#define RLLOSS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
#define RLLOSS_OK 0
#define RLLOSS_EINVAL 1        /* invalid configuration, size or pointer */
#define RLLOSS_EUNSUPPORTED 2  /* valid request this build does not implement */
#define RLLOSS_EWORKSPACE 3    /* workspace too small or misaligned */
#define RLLOSS_ECUDA 4         /* a CUDA call or kernel launch failed */

/* device status bits (rlloss_get_device_status) */
#define RLLOSS_DEV_ETIMEOUT 0x10    /* a bounded on-device wait ran out; results invalid */
#define RLLOSS_DEV_ENONFINITE 0x20  /* the loss came out NaN or infinite */
#define RLLOSS_DEV_EBADTARGET 0x40  /* a target id outside [0, V); its logp is NaN */
#define RLLOSS_DEV_EEMPTYSEQ 0x80   /* GSPO sequence with no active token; it contributes 0 */
#define RLLOSS_DEV_EBOUNDS 0x100    /* builds with -DRLLOSS_DEBUG only: an index or TMA coordinate
                                       check failed and that access was skipped; results invalid */

/* cfg.dtype */
#define RLLOSS_BF16 0
#define RLLOSS_FP32 1
#define RLLOSS_FP8_E4M3 2   /* forward-only scoring (rlloss_forward_e4m3): X, W as e4m3 bytes with
                               per-row fp32 scales; the pages name no fp8 path, this is ours */
/* cfg.loss_type */
#define RLLOSS_GMPO 0
#define RLLOSS_GSPO_TOKEN 1
/* cfg.is_level: importance-sampling level.  GMPO clips at token level before
 * the sequence aggregation, so GMPO with RLLOSS_IS_SEQUENCE is rejected with
 * RLLOSS_EINVAL ("Add GMPO ...", Details).  GSPO ignores it. */
#define RLLOSS_IS_TOKEN 0
#define RLLOSS_IS_SEQUENCE 1
/* cfg.flags */
#define RLLOSS_FLAG_FORCE_ENTROPY_PATH 0x1u  /* run the quantile/mask path even at q = 1 */
#define RLLOSS_FLAG_ADV_PER_TOKEN 0x4u       /* adv holds N per-token advantages (GSPO only; Tinker
                                                "GSPO", Input tensors: advantages (N,)); each token's
                                                objective uses its own A_n, tokens outside the mask
                                                included */
#define RLLOSS_FLAG_SINGLE_CTA_TILES 0x2u    /* forward / recompute kernels on 128-row single-CTA
                                                tiles instead of 256-row CTA-pair tiles (same
                                                results; for comparison) */
#define RLLOSS_FLAG_ALL_ROWS 0x8u            /* run the forward and the backward over every row.
                                                By default rlloss_fwd_bwd (1) skips the forward of
                                                row tiles in which every row is masked, when no
                                                per-token logp / entropy output is requested and
                                                advantages are per sequence: such rows enter
                                                neither the loss nor the gradients; and (2) drops
                                                before the backward the rows whose coefficient
                                                c_n = dL/dlogp_n is zero (tokens outside the mask,
                                                clipped tokens without KL, clipped GSPO sequences):
                                                they add exactly nothing to dX, dW, db ("Add GMPO
                                                ...", Details: the gradients are sums over tokens
                                                of c_n times per-token terms).  Same results up to
                                                fp32 summation order; for comparison */
#define RLLOSS_FLAG_ACCUMULATE 0x10u         /* rlloss_fwd_bwd adds its gradients to the values
                                                already in dX, dW and db instead of overwriting
                                                them (gradient accumulation over micro-batches).
                                                Each element receives the call's contribution in a
                                                fixed order, so repeated calls from the same
                                                initial values give the same bits.  Ignored by the
                                                forward-only entries */
#define RLLOSS_FLAG_RECOMPUTE 0x20u          /* recompute the logits of every backward row.  By
                                                default, with bf16 operands, no bias and without
                                                ACCUMULATE, rlloss_fwd_bwd has the forward also
                                                write each logit's unnormalised probability 2^t
                                                (bf16) for the row tiles that fit the chunk buffer
                                                (the memory the recompute's dlogits chunk would
                                                use), and forms dX and dW of those rows from them
                                                with no second logits GEMM; rows outside those
                                                tiles, or whose log-sum-exp lies outside about
                                                [-55, 66] nats, are recomputed.  Same results up
                                                to bf16 rounding of the dlogits; for comparison */

#define RLLOSS_NMETRICS 8
/* out_metrics layout:
 *  [0] clip fraction: GMPO clipped active tokens / active tokens;
 *      GSPO sequences whose ratio lies strictly outside the clip range / B
 *      (Tinker "GSPO", Output diagnostics: gspo_clipped_fraction:mean)
 *  [1] clip count (tokens for GMPO, sequences for GSPO)
 *  [2] K3 KL mean over active tokens (0 when beta == 0)
 *  [3] number of active tokens
 *  [4] entropy threshold (NaN when the mask is off or no token is active)
 *  [5] active tokens kept by the entropy mask
 *  [6] mean over sequences of the sequence log ratio (GMPO: mean clipped lr;
 *      GSPO: log s_i — gspo_sequence_log_ratio:mean)
 *  [7] mean over sequences of the sequence ratio (GMPO r_i, GSPO s_i)
 * GMPO means in [6], [7] run over sequences with at least one active token. */

typedef struct {
  int32_t B, T, H, V;       /* sequences, tokens per sequence, hidden size, vocabulary */
  int32_t dtype;            /* RLLOSS_BF16 or RLLOSS_FP32 for X, W, b; RLLOSS_FP8_E4M3 for
                               rlloss_forward_e4m3 only */
  int32_t loss_type;        /* RLLOSS_GMPO or RLLOSS_GSPO_TOKEN */
  int32_t is_level;         /* RLLOSS_IS_TOKEN or RLLOSS_IS_SEQUENCE */
  float eps_low, eps_high;  /* GMPO: log-space bounds [-eps_low, +eps_high] ("Add GMPO ...",
                               Details); GSPO: ratio clip [1-eps_low, 1+eps_high] (Tinker
                               "GSPO", Choosing clipping thresholds: 3e-4, 4e-4) */
  float beta;               /* K3 KL weight; 0 = off (GMPO only) */
  float temperature;        /* > 0; logits are divided by it before softmax and entropy */
  float top_entropy_quantile; /* q in [0, 1]; 1 = mask off ("support top_entropy_quantile",
                                 Details); GMPO only */
  int32_t has_bias;         /* b present */
  uint32_t flags;           /* RLLOSS_FLAG_* */
  int32_t chunk_rows;       /* rows per backward chunk; 0 = library default */
} rlloss_cfg;

/* Bytes of device workspace rlloss_fwd_bwd needs for cfg (0 if cfg is
 * invalid).  Depends on the current device's SM count.  Pure host call. */
size_t rlloss_workspace_bytes(const rlloss_cfg* cfg);

/* Bytes of device workspace rlloss_loss_from_logp needs (0 if invalid). */
size_t rlloss_loss_workspace_bytes(const rlloss_cfg* cfg);

/* The whole fused path: forward (LM head + streamed log-softmax, target
 * log-prob, entropy), entropy mask, loss and metrics, and backward.
 * dX, dW and db are overwritten, or added to with RLLOSS_FLAG_ACCUMULATE.
 *   X, W: [N,H], [V,H] of cfg.dtype; b: [V] or NULL when !has_bias.
 *   targets [N] int64; old_logp [N]; ref_logp [N] (NULL when beta == 0);
 *   adv [B]; mask [N].
 *   out_loss [1]; out_metrics [RLLOSS_NMETRICS]; dX [N,H] fp32;
 *   dW [V,H] fp32; db [V] fp32 (NULL when !has_bias; required otherwise).
 *   out_logp [N], out_entropy [N] fp32 and out_entropy_mask [N] uint8 are
 *   optional (NULL = not written).
 *   workspace: device buffer of at least rlloss_workspace_bytes(cfg) bytes,
 *   256-byte aligned; it also holds the device status word.
 * Pointers must be 16-byte aligned.  Returns RLLOSS_* codes as above.
 * The backward needs G = (c/tau)(onehot(y) - softmax) for every row with
 * c_n != 0 ("Add GMPO ...", Details: the input, weight and bias gradients).
 * With bf16 operands and without ACCUMULATE it takes the softmax from the
 * forward, which stores each logit's unnormalised probability 2^t (bf16) in a
 * buffer of the workspace (cfg.chunk_rows rows, by default one or two waves of
 * row tiles), for the row tiles that fit; other rows have their logits
 * recomputed.  Without an entropy mask, with per-sequence advantages and T a
 * multiple of 256, a batch larger than that buffer runs in groups of whole
 * sequences that fit it (sequences are coupled only through B and sums), so
 * every row's probabilities are stored; the results equal the one-pass call
 * up to fp32 summation order.  The stored-probability dX and dW run over the
 * 128-row blocks of the buffer that hold a row with c_n != 0 (its other rows
 * with zero factors).  RLLOSS_FLAG_RECOMPUTE recomputes every row. */
int rlloss_fwd_bwd(const rlloss_cfg* cfg, const void* X, const void* W, const void* b,
                   const int64_t* targets, const float* old_logp, const float* ref_logp,
                   const float* adv, const uint8_t* mask, float* out_loss, float* out_metrics,
                   float* dX, float* dW, float* db, float* out_logp, float* out_entropy,
                   uint8_t* out_entropy_mask, void* workspace, size_t workspace_bytes,
                   void* stream);

/* Forward only (scoring): per-token target log-prob, entropy and log-sum-exp
 * of the temperature-scaled logits, streamed over the vocabulary without
 * writing logits (Tinker "GSPO", Output tensors: logprobs; "support
 * top_entropy_quantile in fused linear GRPO loss", Details: entropy from the
 * streamed accumulators).  Uses cfg.B, T, H, V, dtype, temperature,
 * has_bias, flags; the loss fields are ignored.  out_logp, out_entropy,
 * out_lse: fp32 [N], each optional.  workspace: at least
 * rlloss_forward_workspace_bytes(cfg) bytes, 256-byte aligned. */
size_t rlloss_forward_workspace_bytes(const rlloss_cfg* cfg);
int rlloss_forward(const rlloss_cfg* cfg, const void* X, const void* W, const void* b,
                   const int64_t* targets, float* out_logp, float* out_entropy, float* out_lse,
                   void* workspace, size_t workspace_bytes, void* stream);

/* rlloss_forward with e4m3 operands (cfg.dtype = RLLOSS_FP8_E4M3): the
 * tensor cores take X and W as 8-bit floats (OCP e4m3, finite-only) and the
 * logit of token n and vocabulary row v is
 *     (sum_h X8[n][h] * W8[v][h]) * x_scale[n] * w_scale[v] (+ b[v]),
 * then scaled by 1/temperature as in rlloss_forward.  X8 [N,H] and W8 [V,H]
 * are row-major bytes (H a multiple of 16); x_scale [N], w_scale [V] and b
 * [V] (NULL when !has_bias) are fp32.  The products and their fp32 sums are
 * exact up to fp32 rounding, so the results equal those of the dequantized
 * inputs X8*x_scale, W8*w_scale to fp32 accuracy; how the caller quantizes
 * is its own choice.  Workspace: rlloss_forward_workspace_bytes(cfg).
 * RLLOSS_FLAG_SINGLE_CTA_TILES is not supported here (RLLOSS_EUNSUPPORTED). */
int rlloss_forward_e4m3(const rlloss_cfg* cfg, const void* X8, const float* x_scale, const void* W8,
                        const float* w_scale, const float* b, const int64_t* targets, float* out_logp,
                        float* out_entropy, float* out_lse, void* workspace, size_t workspace_bytes,
                        void* stream);

/* The loss stage alone, from given per-token log-probs (no LM head): entropy
 * mask (if q < 1), loss, metrics and dL/dlogp.
 *   logp [N] fp32; entropy [N] fp32 (required when q < 1 or the
 *   FORCE_ENTROPY_PATH flag is set, else may be NULL); old_logp, ref_logp,
 *   adv, mask as for rlloss_fwd_bwd.  out_dlogp [N] fp32 = dL/dlogp_n
 *   (optional); out_entropy_mask [N] uint8 (optional).  cfg.H, cfg.V,
 *   cfg.dtype, cfg.has_bias and cfg.temperature are ignored. */
int rlloss_loss_from_logp(const rlloss_cfg* cfg, const float* logp, const float* entropy,
                          const float* old_logp, const float* ref_logp, const float* adv,
                          const uint8_t* mask, float* out_loss, float* out_metrics,
                          float* out_dlogp, uint8_t* out_entropy_mask, void* workspace,
                          size_t workspace_bytes, void* stream);

/* The loss stage of rlloss_loss_from_logp for callers that cannot allocate
 * device memory: code that runs while another component is capturing a CUDA
 * graph, plugins that are handed only the tensors they read and write, and
 * runtimes whose memory pool is reserved in full up front.  It takes no
 * workspace.  The pages have no counterpart of this entry point.
 *   Scratch: a file-scope device array of RLLOSS_NOALLOC_SCRATCH_BYTES
 *   (4 MiB) inside the library, which every GPU that loads the library holds
 *   until the process exits.  A problem fits when
 *   rlloss_loss_workspace_bytes(cfg) <= RLLOSS_NOALLOC_SCRATCH_BYTES; callers
 *   should size problems with that comparison.  The loss workspace is about
 *   N + B*(84 + 40*S) + 9.5 KB bytes, each region rounded up to 256 bytes,
 *   with N = B*T and S = min(ceil(16*SMs/B), ceil(T/256)) slices per sequence
 *   (at least 1; SMs of the current device): on a 152-SM GPU, N up to about
 *   4.08e6 tokens when B is small (at most ~100 KB of per-sequence sums), while
 *   many short sequences fill it sooner (B = 34000 with T = 1 does not fit,
 *   each sequence taking at least 124 + T bytes).  A larger problem is
 *   rejected with RLLOSS_ETOOLARGE before any launch; a configuration the
 *   workspace entry rejects gets the same code here (RLLOSS_EINVAL or
 *   RLLOSS_EUNSUPPORTED).
 *   The first call on a device looks up the array's device address with that
 *   device current and caches it; make that first call before any stream
 *   capture.  A device reset (cudaDeviceReset) invalidates the cached
 *   address: a call that meets a CUDA error drops it, so the call after the
 *   error looks it up again.
 *   All calls share the one array, which keeps the last call's contents; each
 *   call clears what must start at zero.  Calls that overlap on the GPU (for
 *   example on two streams) race on the array and must not be issued.
 *   Arguments as for rlloss_loss_from_logp; out_device_status (optional,
 *   device int32) receives this call's device status word (RLLOSS_DEV_*). */
#define RLLOSS_ETOOLARGE 5     /* problem larger than a fixed-size internal scratch */
#define RLLOSS_NOALLOC_SCRATCH_BYTES (4u << 20)   /* size of that scratch */
int rlloss_loss_from_logp_noalloc(const rlloss_cfg* cfg, const float* logp, const float* entropy,
                                  const float* old_logp, const float* ref_logp, const float* adv,
                                  const uint8_t* mask, float* out_loss, float* out_metrics,
                                  float* out_dlogp, uint8_t* out_entropy_mask,
                                  int32_t* out_device_status, void* stream);

/* ---- Vocabulary-parallel form (W split by vocabulary rows over shards).
 * The streamed softmax accumulators of a row are mergeable ("support
 * top_entropy_quantile in fused linear GRPO loss", Details: log-sum-exp and
 * entropy from two online accumulators), so a shard holding W rows
 * [v_begin, v_begin + cfg.V) needs only X, its W rows and the targets:
 *   1. rlloss_forward_shard on every shard -> one row state per token;
 *   2. the caller gathers the states of all shards (an all-gather of
 *      32 B per token and shard) and calls rlloss_loss_from_shards, which
 *      gives lse, logp, entropy, loss, metrics and dL/dlogp for the whole
 *      vocabulary (every shard may run it; the results are the same bits);
 *   3. rlloss_backward_shard on every shard -> its rows of dW and db and its
 *      part of dX; dX is the sum of the parts (an all-reduce).
 * The library makes no collective call: the exchanges are the caller's. */
#define RLLOSS_MAX_SHARDS 4096
#define RLLOSS_STATE_FLOATS 8   /* floats per token in a shard row state */

/* Step 1.  cfg describes the shard: cfg.V = rows of this W shard; b = its
 * bias rows; targets [N] are ids of the whole vocabulary (v_begin >= 0 is
 * the id of the shard's first row).  out_state: [N][RLLOSS_STATE_FLOATS]
 * fp32, 16-byte aligned; its contents are opaque (a softmax reference,
 * sums against it, and the target's logit if the shard holds the target).
 * bf16 or fp32 operands; workspace as for rlloss_forward
 * (rlloss_forward_workspace_bytes of the shard's cfg). */
int rlloss_forward_shard(const rlloss_cfg* cfg, const void* X, const void* W, const void* b,
                         const int64_t* targets, int64_t v_begin, float* out_state, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Bytes of workspace rlloss_loss_from_shards needs (0 if cfg is invalid). */
size_t rlloss_shard_loss_workspace_bytes(const rlloss_cfg* cfg);

/* Step 2.  cfg describes the whole problem (cfg.V = the whole vocabulary;
 * the loss fields as for rlloss_fwd_bwd; H and dtype are not used).
 * states: [nshards][N][RLLOSS_STATE_FLOATS], the shards' outputs of step 1
 * in any fixed order, 16-byte aligned; 1 <= nshards <= RLLOSS_MAX_SHARDS.
 * Outputs: out_loss [1], out_metrics [RLLOSS_NMETRICS], and, each optional,
 * out_lse [N] (natural log; needed by step 3), out_dlogp [N] = dL/dlogp_n
 * (needed by step 3), out_logp, out_entropy [N] fp32, out_entropy_mask [N].
 * A target that no shard holds sets RLLOSS_DEV_EBADTARGET. */
int rlloss_loss_from_shards(const rlloss_cfg* cfg, int32_t nshards, const float* states,
                            const int64_t* targets, const float* old_logp, const float* ref_logp,
                            const float* adv, const uint8_t* mask, float* out_loss, float* out_metrics,
                            float* out_lse, float* out_dlogp, float* out_logp, float* out_entropy,
                            uint8_t* out_entropy_mask, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Bytes of workspace rlloss_backward_shard needs (0 if cfg is invalid). */
size_t rlloss_backward_shard_workspace_bytes(const rlloss_cfg* cfg);

/* Step 3.  cfg, X, W, b, targets, v_begin as in step 1 (the loss fields of
 * cfg are not used; flags RLLOSS_FLAG_ALL_ROWS and RLLOSS_FLAG_ACCUMULATE
 * apply); lse, dlogp [N] from step 2.  Writes (or adds into) dW [cfg.V, H]
 * and db [cfg.V] of this shard and dX [N, H], this shard's part:
 *   G = (dlogp / temperature)(onehot(target) - softmax) over the shard's
 *   columns, dX_shard = G W_shard, dW_shard = G^T X, db_shard = sum_n G.
 * Rows with dlogp = 0 are skipped as in rlloss_fwd_bwd. */
int rlloss_backward_shard(const rlloss_cfg* cfg, const void* X, const void* W, const void* b,
                          const int64_t* targets, int64_t v_begin, const float* lse, const float* dlogp,
                          float* dX, float* dW, float* db, void* workspace, size_t workspace_bytes,
                          void* stream);

/* ---- Batch split over ranks by whole sequences (data parallel).
 * Each rank holds some whole sequences of one batch of B_global sequences.
 * Every per-sequence quantity is then local; what couples the ranks is the
 * batch-global entropy threshold ("support top_entropy_quantile in fused
 * linear GRPO loss", Details: the quantile is taken over the active tokens
 * of the whole batch, not per chunk), the batch size of GMPO's mean over
 * sequences ("Add GMPO to fused linear GRPO loss", Details: per-sample
 * reduction), and sums (metrics, dW, db).  Per step, on every rank:
 *   1. rlloss_forward (its rows) -> logp, entropy, lse;
 *   2. only when top_entropy_quantile < 1: for pass = 0 .. RLLOSS_SELECT_PASSES-1,
 *      rlloss_entropy_hist (this rank's counts), an all-reduce (sum) of the
 *      RLLOSS_SELECT_COUNTS counts over ranks, rlloss_entropy_select (the
 *      summed counts); every rank's select state then holds the same
 *      threshold, bit for bit the one a single device computes for the
 *      whole batch (exact order statistics by radix selection);
 *   3. rlloss_loss_from_logp_dp -> dL/dlogp of its tokens for the whole
 *      batch's loss, the entropy mask of its tokens, and its 8 batch sums;
 *      an all-reduce (sum) of the sums; rlloss_metrics_from_sums -> loss and
 *      metrics of the whole batch;
 *   4. rlloss_backward_shard with the whole vocabulary (v_begin = 0) ->
 *      dX of its rows, and its dW, db parts; dW and db are sums over ranks.
 * A rank that holds no sequence in a step contributes zero counts
 * (rlloss_entropy_hist with N = 0) and zero sums, and skips steps 1, 3, 4.
 * The library makes no collective call: the exchanges are the caller's. */
#define RLLOSS_SELECT_PASSES 4
#define RLLOSS_SELECT_COUNTS 512   /* uint32 counts per pass */
#define RLLOSS_NSUMS 8             /* doubles of batch sums */

/* Bytes of device memory a select state needs (256).  The state is opaque;
 * one state per rank, 16-byte aligned, kept across the passes of one step. */
size_t rlloss_select_state_bytes(void);

/* Pass `pass` (0 .. RLLOSS_SELECT_PASSES-1) of the distributed entropy
 * quantile: writes into counts (device, RLLOSS_SELECT_COUNTS uint32, zeroed
 * by the call) this rank's histogram of its active tokens (mask != 0) under
 * the selection prefixes in select_state (not read at pass 0).  entropy,
 * mask: [N] device (N may be 0).  RLLOSS_EINVAL for a bad pass or pointer. */
int rlloss_entropy_hist(const float* entropy, const uint8_t* mask, int64_t N, int32_t pass,
                        const void* select_state, uint32_t* counts, void* stream);

/* The select step of pass `pass` from counts summed over every rank (device,
 * RLLOSS_SELECT_COUNTS uint32), q = top_entropy_quantile in [0, 1]: updates
 * select_state.  Pass 0 initialises the state (the active-token count is the
 * sum of the counts).  After the last pass the state holds the threshold:
 * linear interpolation between the order statistics at (1-q)(n_act-1) of
 * the batch's active entropies, NaN if no token is active. */
int rlloss_entropy_select(int32_t pass, const uint32_t* counts, float q, void* select_state, void* stream);

/* Copy the threshold held by select_state into *threshold (host).
 * Synchronous; call after the stream has finished the last select step. */
int rlloss_select_threshold(const void* select_state, double* threshold);

/* The loss stage of one rank.  cfg describes this rank's sequences (cfg.B of
 * them, T tokens each); B_global >= cfg.B is the whole batch's sequence
 * count.  select_state: the finished state of step 2 when the entropy mask
 * is on (top_entropy_quantile < 1 or RLLOSS_FLAG_FORCE_ENTROPY_PATH), else
 * NULL; entropy [N] is then required.  Other inputs as for
 * rlloss_loss_from_logp.  Writes out_sums (device, RLLOSS_NSUMS doubles, this
 * rank's share; each entry adds over ranks):
 *   [0] sum of the sequence terms (GMPO: -A_i r_i ebar_i + beta KL_i, before
 *       the 1/B_global of the mean; GSPO: minus the summed objective),
 *   [1] active tokens, [2] clipped tokens (GSPO: clipped sequences),
 *   [3] sum of K3 KL over active tokens, [4] tokens kept by the entropy mask
 *   (GSPO: active tokens), [5] sum of the sequence log ratios and [6] of the
 *   sequence ratios over sequences with tokens, [7] sequences with tokens;
 * and, each optional, out_dlogp [N] = dL/dlogp_n of the whole batch's loss,
 * out_entropy_mask [N].  Workspace: rlloss_loss_workspace_bytes(cfg). */
int rlloss_loss_from_logp_dp(const rlloss_cfg* cfg, int32_t B_global, const void* select_state,
                             const float* logp, const float* entropy, const float* old_logp,
                             const float* ref_logp, const float* adv, const uint8_t* mask,
                             double* out_sums, float* out_dlogp, uint8_t* out_entropy_mask,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Host only, no device access: the whole batch's loss (*out_loss) and
 * metrics (out_metrics [RLLOSS_NMETRICS], the layout of rlloss_fwd_bwd) from
 * the batch sums added over ranks (sums: host, RLLOSS_NSUMS doubles) and the
 * threshold of step 2 (NaN without the entropy mask). */
int rlloss_metrics_from_sums(const rlloss_cfg* cfg, int32_t B_global, const double* sums, double threshold,
                             float* out_loss, float* out_metrics);

/* Copy the device status word of ``workspace`` (the one a previous call used)
 * into *status.  Synchronous; call after the stream has finished.  Returns
 * RLLOSS_ECUDA if the copy failed. */
int rlloss_get_device_status(const void* workspace, int32_t* status);

/* Copy into *rows the number of rows the last rlloss_fwd_bwd on ``workspace``
 * ran its backward over: the rows with c_n != 0, or every row under
 * RLLOSS_FLAG_ALL_ROWS (see there).  Synchronous; call after the stream
 * has finished.  Returns RLLOSS_ECUDA if the copy failed.  (Our addition, for
 * reporting executed work; the pages have no counterpart.) */
int rlloss_get_backward_rows(const void* workspace, int32_t* rows);

/* Copy into *rows the number of rows the last rlloss_fwd_bwd on ``workspace``
 * formed dX and dW for from the forward's stored probabilities (rows with
 * c_n != 0; 0 under RLLOSS_FLAG_RECOMPUTE, with fp32 operands or
 * ACCUMULATE).  The rows counted by rlloss_get_backward_rows are the others
 * with c_n != 0, recomputed.  Synchronous; call
 * after the stream has finished.  Returns RLLOSS_ECUDA if the copy failed.
 * (Our addition, for reporting executed work; the pages have no
 * counterpart.) */
int rlloss_get_stored_rows(const void* workspace, int32_t* rows);

/* Copy into *rows the number of buffer rows the stored-probability dX and dW
 * of the last rlloss_fwd_bwd on ``workspace`` ran over: whole 128-row blocks
 * of the stored-probability buffer holding a row counted by
 * rlloss_get_stored_rows (so at least that count, and a multiple of 128 per
 * sequence group).  Synchronous; call after the stream has finished.  Returns
 * RLLOSS_ECUDA if the copy failed.  (Our addition, for reporting executed
 * work; the pages have no counterpart.) */
int rlloss_get_stored_positions(const void* workspace, int32_t* rows);

/* Copy into *tiles the number of row tiles (256 rows each, 128 with
 * RLLOSS_FLAG_SINGLE_CTA_TILES) the last forward on ``workspace`` computed:
 * all of them, or under rlloss_fwd_bwd's tile skipping (see
 * RLLOSS_FLAG_ALL_ROWS) those holding a row with mask != 0.  Synchronous;
 * call after the stream has finished.  (Ours, for reporting executed work.) */
int rlloss_get_forward_tiles(const void* workspace, int32_t* tiles);

/* Launch a kernel that waits on a barrier nothing will complete, with a limit
 * of limit_ns nanoseconds, so the bounded-wait path can be exercised: the
 * status word of ``workspace`` (>= 256 bytes) then carries RLLOSS_DEV_ETIMEOUT.
 * The library has no other use for it. */
int rlloss_selftest_bounded_wait(void* workspace, uint64_t limit_ns, void* stream);

/* Phase timing for benchmarks.  While enabled, rlloss_fwd_bwd records CUDA
 * events on the caller's stream around its phases:
 *   0 forward tensor-core kernel, 1 row merge + entropy mask + loss,
 *   2 backward G producer (all chunks), 3 grouped dX + dW kernels,
 *   4 (unused), 5 everything else (operand split, bias scaling, db).
 * rlloss_phase_times synchronises on the recorded events, writes the summed
 * milliseconds and the launch counts per phase (arrays of nphase <= 6), and
 * clears the record.  rlloss_phase_timing(0/1) switches it off/on and clears. */
#define RLLOSS_NPHASES 6
int rlloss_phase_timing(int enable);
int rlloss_phase_times(float* ms, int32_t* launches, int nphase);

/* Number of kernels this library has launched in this process so far. */
uint64_t rlloss_kernel_launches(void);

/* Static description of a code. */
const char* rlloss_status_str(int code);

#ifdef __cplusplus
}
#endif
#endif /* RLLOSS_H */
