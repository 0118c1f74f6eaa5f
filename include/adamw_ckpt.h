/*
 * adamw_ckpt.h -- C ABI of the GB300 (sm_103a) clipped-AdamW optimizer step
 * and of the step_NNNNNN.bin checkpoint.
 *
 * The library updates a flat float32 training state (weights w, gradient g,
 * Adam moments m and v, n parameters, all resident in GPU memory) once per
 * training step, and packs / writes / reads that state as one checkpoint
 * file.  Sources, cited by page title and section:
 *
 *  [T] "Training as a Recoverable State Transition" (aihero.club, Language
 *      Models from Scratch), section "The Exact Targets of Clipping and AdamW"
 *      -- global L2 clip and AdamW with bias correction and decoupled weight
 *      decay; section "The Checkpoint Contract and a Real Recovery Test" --
 *      save after a complete optimizer step, t counts real updates.
 *  [C] "Grow a Language Model: Checkpoints" (unhomeschool.com), sections
 *      "Format", "Region by region", "Total size", "Why save m & v" -- the
 *      file layout [int32 step][int32 n][n f32 w][n f32 m][n f32 v].
 *  [B] "Grow a Language Model: Backprop" (unhomeschool.com), sections
 *      "Optimizer state" and "Signals & checkpoints" -- w, g, m, v are one
 *      buffer each, allocated once at start-up; the clip kernels
 *      k_grad_norm_partial / k_grad_norm_final / k_grad_scale.
 *  [S] "Checkpoint and Sharded Resume" (AI Engineering from Scratch, phase
 *      19 lesson 80), sections "Atomic write" and "Three failure modes".
 *
 * Conventions for every entry point:
 *  - Return value: ADAMW_OK (0) or a negative ADAMW_E* status; a failing
 *    call leaves a one-line explanation in adamw_last_error() (per thread).
 *  - Device pointers (d_*) point into memory of the device that was current
 *    when the context was created; each holds n float32 values laid out in
 *    the flat parameter order of the offset table.  The caller owns them.
 *    16-byte aligned pointers take the vectorised path; other alignments
 *    are accepted and take a scalar path.
 *  - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls are asynchronous on that stream unless stated.
 *  - The context owns all scratch (device, pinned host), allocated by
 *    adamw_create; the only later allocations are made by setup calls
 *    outside the training loop (adamw_set_decay_mask: the flag bits;
 *    adamw_graph_create: the step graph).  No step allocates, except the
 *    first graph step after such a setup change, which rebuilds its graph.
 *  - A context is not thread-safe: one host thread drives it at a time.
 */
#ifndef ADAMW_CKPT_H
#define ADAMW_CKPT_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ADAMW_API __attribute__((visibility("default")))
#else
#define ADAMW_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define ADAMW_OK 0
#define ADAMW_EINVAL (-1)     /* bad argument: null pointer, size, t < 1 ... */
#define ADAMW_ECUDA (-2)      /* a CUDA runtime call or kernel launch failed */
#define ADAMW_EIO (-3)        /* open/read/write/fsync/rename failed         */
#define ADAMW_EFORMAT (-4)    /* checkpoint header impossible (step/n < 0)   */
#define ADAMW_ESIZE (-5)      /* file size is not 8 + 12 n, or truncated     */
#define ADAMW_EMISMATCH (-6)  /* n in the file differs from the context's n  */
#define ADAMW_ENONFINITE (-7) /* gradient norm inf/nan: update was skipped   */
#define ADAMW_ESTATE (-8)     /* call out of order (e.g. write with no pack) */

/* adamw_create flags. */
#define ADAMW_CREATE_NO_CKPT 1 /* do not allocate the checkpoint staging    */

/* Element types of adamw_clip_step_mixed's gradient and weight copy. */
#define ADAMW_DTYPE_F32 0  /* IEEE binary32                               */
#define ADAMW_DTYPE_BF16 1 /* bfloat16: the top 16 bits of a binary32      */
#define ADAMW_DTYPE_F16 2  /* IEEE binary16                                */

/* adamw_set_launch_options flags. */
#define ADAMW_LAUNCH_NO_PDL 1     /* launch the fused kernel after the norm ends */
#define ADAMW_LAUNCH_NO_ONEPASS 2 /* small states: two launches, not one         */
#define ADAMW_LAUNCH_TEST_BARRIER_TIMEOUT 4 /* tests only: see below          */
#define ADAMW_LAUNCH_STATIC_CHUNKS 8 /* fused, pack: chunks fixed per block     */

/* adamw_clip_step_ex flags. */
#define ADAMW_ZERO_GRAD 1    /* write 0 into g after reading it             */
#define ADAMW_TENSOR_NORMS 2 /* also sum g^2 per tensor of the offset table */

/* ckpt_set_options / ckpt_write_image flags. */
#define CKPT_DIRECT 1 /* write with O_DIRECT when the file system allows it */
#define CKPT_COPY_ENGINE 2 /* staging -> host image by the copy engine       */

/* Checkpoint requests recorded by the signal handlers (ckpt_signals_*). */
#define CKPT_REQ_WRITE 1 /* SIGUSR1: write a checkpoint, keep training     */
#define CKPT_REQ_EXIT 2  /* SIGTERM: write a checkpoint, then stop         */

/* ckpt_step_end actions. */
#define CKPT_ACTION_NONE 0    /* no checkpoint at this step                 */
#define CKPT_ACTION_WRITING 1 /* packed; being written in the background    */
#define CKPT_ACTION_EXIT 2    /* written and durable; the caller should exit */

typedef struct adamw_ctx adamw_ctx;

/*
 * Creates a context for a flat state of n_params float32 values split into
 * n_tensors tensors: tensor k occupies [offsets[k], offsets[k] + numels[k]).
 * Flat order per [C] "Region by region": embeddings, then each layer, then
 * the head.  The table must be sorted, contiguous, without gaps or overlap,
 * cover exactly [0, n_params), and every numel must be > 0; n_params must be
 * in [1, 2^31 - 1] (it is stored as an int32 in the checkpoint header).  The
 * table is copied.  n_tensors = 0 with NULL offsets and numels means one flat
 * tensor of n_params values.
 *
 * Allocates, once ([B] "Optimizer state": every buffer at start-up): the
 * norm-reduction scratch, a pinned host mirror of the norm result and,
 * unless ADAMW_CREATE_NO_CKPT is set, a device staging image and a pinned
 * host image of 8 + 12 n bytes each for the checkpoint.  Uses the current
 * CUDA device.  AdamW hyperparameters start at beta1 = 0.9,
 * beta2 = 0.999, eps = 1e-8 ([T]).  On failure *out is set to NULL.
 */
ADAMW_API int adamw_create(int64_t n_params, const int64_t* offsets,
                 const int64_t* numels, int32_t n_tensors, int32_t flags,
                 adamw_ctx** out);

/* Frees everything the context owns; waits for its pending copies first.
 * NULL is accepted. */
ADAMW_API int adamw_destroy(adamw_ctx* ctx);

/* Replaces beta1, beta2 (each in [0, 1)) and eps (finite, >= 0) for the
 * following steps (the step graph's included); ADAMW_EINVAL otherwise, the
 * previous values kept.  The defaults are the pages' 0.9, 0.999, 1e-8. */
ADAMW_API int adamw_set_hparams(adamw_ctx* ctx, double beta1, double beta2, double eps);

/* Number of parameters and tensors of the context; -1 for a NULL ctx. */
ADAMW_API int64_t adamw_num_params(const adamw_ctx* ctx);
ADAMW_API int32_t adamw_num_tensors(const adamw_ctx* ctx);

/*
 * Global L2 norm of the gradient d_g[0..n) ([T]: all gradients joined into
 * one vector g, ||g||_2).  Two-level deterministic reduction: fixed per-block
 * partial sums of squares (float32 squares summed in short runs, flushed
 * into double), then one fixed-order double sum; bit-identical from run to
 * run for a given n.  If h_norm is not NULL the call waits for the stream
 * and stores the norm there (double); otherwise it returns at once and the
 * result stays in the context (adamw_last_norm).  Returns ADAMW_ENONFINITE
 * (with *h_norm = inf or nan) when waited for and the norm is not finite.
 */
ADAMW_API int grad_global_norm(adamw_ctx* ctx, const float* d_g, double* h_norm,
                     void* stream);

/*
 * One optimizer step, in place on d_w, d_m, d_v ([T]):
 *   norm = ||g||_2;  s = (norm > clip) ? clip / norm : 1
 *   g_hat = s g;  m = beta1 m + (1 - beta1) g_hat;
 *   v = beta2 v + (1 - beta2) g_hat^2
 *   w = w (1 - lr wd) - lr m_hat / (sqrt(v_hat) + eps),
 *   m_hat = m / (1 - beta1^t),  v_hat = v / (1 - beta2^t).
 * t >= 1 is the 1-based index of this update (t counts real optimizer
 * updates only).  clip > 0 (INFINITY disables clipping); lr, wd >= 0.
 * d_g is read only.  The bias-correction scalars are computed on the host in
 * double.  Two kernels on `stream`: the norm reduction's fixed per-block
 * partial sums, then the fused clip-scale + AdamW pass, whose blocks each
 * add up those partials in the same fixed order (the same bits in every
 * block; block 0 records the norm) and then read w, g, m, v once and write
 * w, m, v once.  If the norm is not finite the second kernel leaves w, m, v
 * untouched; the call itself does not wait, so that outcome is reported by
 * adamw_last_norm().  Decay applies to every parameter.
 */
ADAMW_API int adamw_clip_step(adamw_ctx* ctx, float* d_w, const float* d_g, float* d_m,
                    float* d_v, int32_t t, double lr, double wd, double clip,
                    void* stream);

/*
 * adamw_clip_step with the two extensions a training loop needs around it.
 *
 * Gradient accumulation ([B] "Accumulation across micro-batches": backward
 * adds into the gradient buffer, then scale_grads(1 / n_micro), the optimizer
 * step, zero_grads): grad_scale > 0 multiplies the gradient before the norm,
 * the clip and the update, folded into the clip factor at no extra traffic;
 * flags ADAMW_ZERO_GRAD makes the fused kernel write 0 into d_g after reading
 * it (+4 bytes per parameter; a skipped non-finite step leaves g as is);
 * ADAMW_TENSOR_NORMS also computes the per-tensor sums of squares of the raw
 * gradient (adamw_last_tensor_sumsq; not with global_sumsq >= 0).
 *
 * Sharded state (ZeRO-1 style: each rank owns one contiguous range of the
 * flat state and holds the gradient of that range): global_sumsq >= 0 is the
 * sum of g^2 of the whole raw gradient -- the ranks' grad_sumsq values,
 * summed in rank order -- and replaces the local reduction: no norm kernel
 * runs, the clip factor is computed on the host in double, and a non-finite
 * global norm returns ADAMW_ENONFINITE at once with nothing launched.
 * global_sumsq < 0 reduces this context's gradient on the GPU, as
 * adamw_clip_step does (which is this call with grad_scale 1,
 * global_sumsq -1, flags 0).
 */
ADAMW_API int adamw_clip_step_ex(adamw_ctx* ctx, float* d_w, float* d_g, float* d_m,
                                 float* d_v, int32_t t, double lr, double wd,
                                 double clip, double grad_scale, double global_sumsq,
                                 int32_t flags, void* stream);

/*
 * The mixed-precision step ([B] "Where the gradients live": FP16 gradient
 * buffers, ~240 MB at FP16 for 120M parameters; "Framework overhead": the
 * FP16 cuBLAS path).  Weights (the float32 master copy), m and v stay
 * float32 -- they are what step_NNNNNN.bin stores; the gradient d_g has
 * g_dtype (ADAMW_DTYPE_F32 / _BF16 / _F16), read and widened exactly; if
 * d_w_lp is not NULL the new weights are also written there rounded to
 * w_lp_dtype (BF16 or F16, nearest even), the copy the next forward pass
 * reads.  Everything else is as adamw_clip_step_ex (grad_scale,
 * global_sumsq, ADAMW_ZERO_GRAD zeroes the 16-bit g, ADAMW_TENSOR_NORMS).
 * Bytes per parameter with a 16-bit g and a copy: 2 (norm) + 2 + 12 read,
 * 12 + 2 written.  16-bit types or a copy need w, m, v on 16-byte
 * boundaries and d_g (16-bit) and d_w_lp on 8-byte boundaries.
 */
ADAMW_API int adamw_clip_step_mixed(adamw_ctx* ctx, float* d_w, void* d_g, int32_t g_dtype,
                                    float* d_m, float* d_v, void* d_w_lp,
                                    int32_t w_lp_dtype, int32_t t, double lr, double wd,
                                    double clip, double grad_scale, double global_sumsq,
                                    int32_t flags, void* stream);

/* grad_sumsq for a gradient of element type g_dtype (16-bit: 8-byte aligned). */
ADAMW_API int grad_sumsq_typed(adamw_ctx* ctx, const void* d_g, int32_t g_dtype,
                               double* h_sumsq, void* stream);

/*
 * Sum of g^2 over this context's n values of d_g (double, the same
 * deterministic two-level reduction as grad_global_norm); waits for the
 * stream.  For a sharded state, each rank's value is exchanged and summed in
 * rank order to give adamw_clip_step_ex's global_sumsq.  Returns
 * ADAMW_ENONFINITE (with the inf/nan sum stored) if the sum is not finite.
 */
ADAMW_API int grad_sumsq(adamw_ctx* ctx, const float* d_g, double* h_sumsq, void* stream);

/*
 * The sharded step with the exchange on the device ("Checkpoint and Sharded
 * Resume", lesson 80: each rank holds one contiguous shard; the clip needs
 * the norm of the whole gradient).  Per step, on each rank, all on `stream`
 * with no host wait:
 *   1. grad_sumsq_to: the shard's sum of g^2 (double, the deterministic
 *      reduction) written to the device address d_out (8-byte aligned) --
 *      this rank's send buffer of an all-gather;
 *   2. the caller all-gathers one double per rank into d_rank_sumsq[world]
 *      in rank order (e.g. an NCCL all-gather on the same stream);
 *   3. adamw_clip_step_gathered: adds d_rank_sumsq[0..world) in rank order
 *      on the device, takes grad_scale sqrt(sum) as the norm and the clip
 *      factor from it -- the same formula and order as adamw_clip_step_ex
 *      with global_sumsq, so the same bits -- and runs the fused update of
 *      this rank's shard.  A non-finite sum skips the update (the state is
 *      left as it was); adamw_last_norm then reports ADAMW_ENONFINITE and
 *      the global norm.  flags: ADAMW_ZERO_GRAD.
 * g_dtype: ADAMW_DTYPE_F32 / BF16 / F16 (16-bit: 8-byte aligned; then the
 * update needs adamw_clip_step_mixed's alignment and takes no weight copy).
 * Errors: ADAMW_EINVAL (NULL pointers, world < 1, bad scalars), ADAMW_ECUDA.
 */
ADAMW_API int grad_sumsq_to(adamw_ctx* ctx, const void* d_g, int32_t g_dtype, double* d_out,
                            void* stream);
ADAMW_API int adamw_clip_step_gathered(adamw_ctx* ctx, float* d_w, void* d_g, int32_t g_dtype,
                                       float* d_m, float* d_v, int32_t t, double lr, double wd,
                                       double clip, double grad_scale,
                                       const double* d_rank_sumsq, int32_t world, int32_t flags,
                                       void* stream);

/*
 * The sharded step with the exchange on the host ("Training as a
 * Recoverable State Transition", section "The Exact Targets of Clipping and
 * AdamW": the clip uses the norm of all gradients joined into one vector;
 * "Checkpoint and Sharded Resume", lesson 80, section "Manifest schema":
 * each rank owns the contiguous range param_shard_offset /
 * param_shard_numel).  Per step, on each rank: grad_sumsq gives the shard's
 * sum of g^2 on the host; the caller gathers one double per rank, in rank
 * order, into a host array (e.g. a gloo all-gather); then:
 *
 * adamw_rank_total (host only, no GPU needed): S = h_rank_sumsq[0] + ... +
 *   h_rank_sumsq[world - 1], added in rank order in double (the order and
 *   formula of the device form, adamw_clip_step_gathered, so the same bits);
 *   norm = grad_scale sqrt(S); the factor applied to the raw gradient,
 *   grad_scale (norm > clip ? clip / norm : 1), rounded to float once.  Each
 *   output pointer may be NULL.  Errors: ADAMW_EINVAL (NULL array, world < 1,
 *   a negative rank value, clip <= 0, grad_scale not finite and > 0);
 *   ADAMW_ENONFINITE when the norm is inf or nan (outputs still stored, the
 *   factor then grad_scale).
 * adamw_clip_step_ranks: adamw_rank_total, then the fused update of this
 *   rank's shard with that factor (adamw_clip_step_mixed with global_sumsq =
 *   S; no norm kernel runs).  h_rank_sumsq is read before the call returns.
 *   A non-finite global norm returns ADAMW_ENONFINITE with nothing
 *   launched.  flags: ADAMW_ZERO_GRAD (ADAMW_TENSOR_NORMS is refused: the
 *   shard's own reduction does not run).  g_dtype and alignment as
 *   adamw_clip_step_gathered.
 */
ADAMW_API int adamw_rank_total(const double* h_rank_sumsq, int32_t world, double clip,
                               double grad_scale, double* sumsq_out, double* norm_out,
                               float* scale_out);
ADAMW_API int adamw_clip_step_ranks(adamw_ctx* ctx, float* d_w, void* d_g, int32_t g_dtype,
                                    float* d_m, float* d_v, int32_t t, double lr, double wd,
                                    double clip, double grad_scale,
                                    const double* h_rank_sumsq, int32_t world, int32_t flags,
                                    void* stream);

/*
 * One step as a CUDA graph, for states small enough that launch latency
 * dominates (e.g. 65,536 parameters: L2-resident, a few microseconds per
 * kernel).  adamw_graph_create builds, for these buffers, a graph of the norm
 * kernel followed by the fused clip+AdamW kernel -- or, up to 65,536
 * parameters, the one-launch step in its cluster form as one kernel node
 * (see adamw_set_launch_options) -- with
 * the same results bit for bit as
 * adamw_clip_step, and instantiates it; the context owns it (replaced by the
 * next adamw_graph_create, freed by adamw_graph_destroy or adamw_destroy).
 * adamw_graph_step writes step t's scalars (t, lr, wd, clip; bias
 * corrections in double on the host) into the graph's kernel nodes and
 * launches it on `stream` -- one launch per step; it first rebuilds the
 * graph if decay flags or the one-launch option changed since it was made.
 * adamw_last_norm reports its norm.  ADAMW_ESTATE if no graph was created.
 */
ADAMW_API int adamw_graph_create(adamw_ctx* ctx, float* d_w, const float* d_g,
                                 float* d_m, float* d_v);
ADAMW_API int adamw_graph_step(adamw_ctx* ctx, int32_t t, double lr, double wd,
                               double clip, void* stream);
ADAMW_API int adamw_graph_destroy(adamw_ctx* ctx);

/*
 * Per-tensor sums of squares ([T] "The Exact Targets of Clipping and AdamW":
 * record the norms of all parameters to detect numerical faults): g^2 summed
 * over each tensor of the offset table, in table order, computed by the same
 * reduction pass as the global norm at no extra memory traffic (its blocks
 * take contiguous tile ranges and flush a tensor's share where the next
 * tensor starts; the host adds the shares in block order, so the values are
 * bit-stable from run to run).
 * grad_tensor_sumsq: reduces d_g, waits, writes n_tensors doubles to h_out;
 * returns ADAMW_ENONFINITE (with the values stored, inf/nan in the affected
 * tensors) if the global sum is not finite.
 * adamw_last_tensor_sumsq: the per-tensor sums of the last step launched
 * with ADAMW_TENSOR_NORMS (waits for it); ADAMW_ESTATE if the last reduction
 * did not compute them.  Read them before the next step reuses the scratch.
 */
ADAMW_API int grad_tensor_sumsq(adamw_ctx* ctx, const float* d_g, double* h_out,
                                void* stream);
ADAMW_API int adamw_last_tensor_sumsq(adamw_ctx* ctx, double* h_out);

/*
 * Per-group weight decay ("Training as a Recoverable State Transition",
 * section "The Exact Targets of Clipping and AdamW": the lesson decays every
 * parameter, normalisation gains and biases included, and does not claim
 * that this is the best grouping).  decay: one byte per tensor of the
 * context's offset table (n_tensors must equal adamw_num_tensors); 0 exempts
 * that tensor: every later step of this context updates its elements with
 * wd = 0, i.e. its old weight is multiplied by exactly 1.  The norm and the
 * clip stay global.  decay == NULL (n_tensors ignored), or all flags set,
 * restores the default: decay on every parameter.
 * Applies to adamw_clip_step, adamw_clip_step_ex, adamw_clip_step_mixed and
 * the step graph (a graph made before the flags were set or cleared is
 * rebuilt by its next adamw_graph_step; adamw_clip_step_noalloc, having no
 * context, always decays everything).  Without flags the fused kernel is
 * compiled without the flag reads.  The flags are configuration, not state: the checkpoint
 * format has no place for them, so a resumed run sets them again.
 * A setup call, not for the training loop: it waits for all work on the
 * device, then copies one bit per parameter to the device (allocated by
 * the first call that exempts a tensor, n / 8 bytes, freed with the
 * context).  Errors: ADAMW_EINVAL (NULL ctx, n_tensors mismatch),
 * ADAMW_ECUDA.
 */
ADAMW_API int adamw_set_decay_mask(adamw_ctx* ctx, const uint8_t* decay, int32_t n_tensors);

/*
 * Waits for the last norm reduction launched on this context (by
 * grad_global_norm or adamw_clip_step) and reports it: *norm_out (may be
 * NULL) receives the norm of the (scaled) gradient in double, *scale_out
 * (may be NULL) the factor that step applied to the raw gradient
 * (grad_scale times the clip factor).  Returns ADAMW_ENONFINITE if the norm was inf/nan (the
 * step, if any, was skipped), ADAMW_ESTATE if no reduction ran yet.
 */
ADAMW_API int adamw_last_norm(adamw_ctx* ctx, double* norm_out, float* scale_out);

/*
 * Launch options.  By default the fused kernel of adamw_clip_step(_ex) is
 * launched as a programmatic dependent of the norm kernel (sm_90+
 * programmatic dependent launch): it may start while the norm's last blocks
 * finish, warms L2 with its first chunk, and waits in hardware for the norm
 * grid to complete before reading its result; results are unchanged.
 * ADAMW_LAUNCH_NO_PDL launches it in plain stream order instead.  (An
 * instrumentation event between the kernels also implies plain order.)
 * States of up to 2^19 parameters (float32 gradient, 16-byte aligned arrays,
 * no weight copy, no per-tensor norms, no global_sumsq) take the whole step
 * as one launch instead: the same partial sums, the same fixed-order total
 * and the same update, so the same bits, at half the launch cost.  When the
 * stream is being captured into a graph (no launch cost to save), only the
 * cluster form below is used as one kernel node; larger captured steps are
 * two kernel nodes, which take less GPU time there.  Up to 65,536
 * parameters (without ADAMW_ZERO_GRAD) the launch is thread-block clusters
 * of 8 CTAs, each cluster computing the norm itself and meeting at its
 * hardware barrier; otherwise a cooperative grid whose blocks meet at a
 * grid barrier with a bounded wait (about one second) -- a wait that runs
 * out skips the update and makes the next adamw_last_norm return
 * ADAMW_ECUDA.
 * ADAMW_LAUNCH_NO_ONEPASS always uses the two launches.
 * From 2^24 parameters up, the fused kernel and the checkpoint pack hand
 * their chunks out by an atomic counter, so a block that starts late (its
 * SM held by other work) takes fewer and no block's share sets the kernel's
 * end; the results are the same bits.  ADAMW_LAUNCH_STATIC_CHUNKS deals
 * chunks out cyclically by block at every size.
 * ADAMW_LAUNCH_TEST_BARRIER_TIMEOUT (for tests of that path): the next
 * one-launch step runs as the cooperative grid at any one-launch size (a
 * captured step too; in a step graph above 65,536 parameters, whose next
 * step rebuilds the graph with that grid as its node) and waits for one
 * block more than it launched, so its barrier runs out after about a
 * second, as above.  Used once, then cleared.
 */
ADAMW_API int adamw_set_launch_options(adamw_ctx* ctx, int32_t flags);

/*
 * Instrumentation: the next adamw_clip_step on this context records the given
 * events (cudaEvent_t passed as void*; NULL entries skipped) on its stream:
 * ev_begin before the norm kernel, ev_mid between the norm and the fused
 * kernel, ev_end after the fused kernel.  They apply to that one call only.
 * Used to time each kernel inside a longer timed region.
 */
ADAMW_API int adamw_record_events(adamw_ctx* ctx, void* ev_begin, void* ev_mid,
                                  void* ev_end);

/*
 * Checkpoint, part 1 ([C] "Format"; [T] "save after a complete optimizer
 * step"): a kernel on main_stream packs [int32 step][int32 n][w][m][v] into
 * the context's device staging (the header and the w, m, v regions, little-
 * endian, each in a 256-byte aligned slot), then side_stream copies them to
 * their file offsets in the context's pinned host image (8 + 12 n bytes):
 * by a kernel on a quarter of the SMs by default (aligned 16-byte stores
 * into host memory), by the copy engine with CKPT_COPY_ENGINE (see
 * ckpt_set_options).  The
 * caller may launch the next step on main_stream right away: the pack reads
 * w, m, v before it, and the copy reads only the staging image.  A later
 * pack waits for the previous copy.  side_stream may equal main_stream.
 * step is the number of completed updates (>= 0); resume continues with
 * t = step + 1.  ADAMW_ESTATE if the context has no staging.
 */
ADAMW_API int ckpt_pack(adamw_ctx* ctx, int32_t step, const float* d_w,
              const float* d_m, const float* d_v, void* main_stream,
              void* side_stream);

/*
 * Checkpoint, part 2 ([S] "Atomic write"): waits for the copy started by the
 * last ckpt_pack, writes the image to <dir>/step_%06d.bin.tmp, fsyncs it,
 * renames it to <dir>/step_%06d.bin and fsyncs dir.  A crash before the
 * rename leaves any previous file of that name intact.  With CKPT_DIRECT
 * (the default; see ckpt_set_options) the pinned image goes to the disk with
 * O_DIRECT where the file system allows it, else through the page cache.
 * After the rename, rotation (if set) deletes all but the newest `keep`
 * step_*.bin files of dir.  The final path is copied to path_out (may be
 * NULL) if it fits in path_cap bytes.  ADAMW_ESTATE if there is no packed
 * image; ADAMW_EIO on any file error (the .tmp file is removed), and also
 * when the fsync of dir after the rename fails (the file is then in place
 * but the rename may not be durable; a file system that does not sync
 * directories is not an error).
 *
 * ckpt_write blocks the calling thread until the file is durable.
 * ckpt_write_async hands the same work to the context's writer thread and
 * returns at once ([S] "Production patterns": asynchronous writes so that
 * training continues); ckpt_wait blocks until that write is done and returns
 * its status and path (ADAMW_OK and "" if none was started).  One write is in
 * flight at most: ckpt_write_async, ckpt_pack, ckpt_read and
 * ckpt_set_options first wait (on the host) for a write in flight.  A failed
 * asynchronous write not yet reported by ckpt_wait is reported by the next
 * ckpt_write_async.
 */
ADAMW_API int ckpt_write(adamw_ctx* ctx, const char* dir, char* path_out,
                         size_t path_cap);
ADAMW_API int ckpt_write_async(adamw_ctx* ctx, const char* dir);
ADAMW_API int ckpt_wait(adamw_ctx* ctx, char* path_out, size_t path_cap);

/*
 * Writer options: keep >= 1 keeps only the newest `keep` step_*.bin files of
 * the target directory after each write ([S] "Production patterns": rotation
 * keeps the last K checkpoints so the disk does not fill); keep = 0 keeps
 * all.  flags: CKPT_DIRECT, CKPT_COPY_ENGINE, both or 0.  Defaults:
 * keep = 0, CKPT_DIRECT.  CKPT_COPY_ENGINE makes ckpt_pack copy the staging
 * to the pinned image with the copy engine instead of a kernel on the side
 * stream: the copy engine leaves the SMs to the steps running meanwhile,
 * but on GB300 its copy into a pinned image that was just written to a file
 * took 80-116 ms for 1.33 GB where the kernel took 7-14 ms (and the steps
 * lost about 4 ms); the write of the next checkpoint waits for that copy.
 */
ADAMW_API int ckpt_set_options(adamw_ctx* ctx, int32_t keep, int32_t flags);

/*
 * Checkpoint policy at a step boundary ([C] "Five decisions": every 100
 * steps; "SIGTERM & SIGUSR1": finish the step, then write; SIGTERM then
 * exits, SIGUSR1 continues).  Call after the optimizer step of `step`
 * (completed updates) has been launched.  Writes when step > 0 and
 * step % every == 0 (every = 0: only on signals) or when a signal recorded
 * by ckpt_signals_install is pending (the request is consumed).  On a
 * SIGTERM request the write completes before the call returns and
 * *action_out = CKPT_ACTION_EXIT: the caller should stop training; otherwise
 * the write runs in the background (CKPT_ACTION_WRITING) or nothing happens
 * (CKPT_ACTION_NONE).  The library never exits the process itself.
 */
ADAMW_API int ckpt_step_end(adamw_ctx* ctx, int32_t step, const float* d_w,
                            const float* d_m, const float* d_v, void* main_stream,
                            void* side_stream, const char* dir, int32_t every,
                            int32_t* action_out);

/*
 * Installs handlers that record SIGUSR1 (mask bit CKPT_REQ_WRITE) and
 * SIGTERM (CKPT_REQ_EXIT) as checkpoint requests instead of their default
 * actions; the handlers only set a lock-free flag.  ckpt_signals_take
 * returns the pending request bits and clears them (async-signal-safe).
 */
ADAMW_API int ckpt_signals_install(int32_t mask);
ADAMW_API int32_t ckpt_signals_take(void);

/*
 * Resume ([C] "Why save m & v"; [S] "Three failure modes"): opens path,
 * checks that the header is readable, step >= 0, n == the context's n and
 * that the file holds exactly 8 + 12 n bytes; only then reads it into the
 * pinned image and copies w, m, v to d_w, d_m, d_v on `stream`, and waits
 * for those copies.  *step_out receives the stored step.  On any failure
 * the device arrays are not modified.  Errors: ADAMW_EIO (cannot open or
 * read), ADAMW_ESIZE, ADAMW_EFORMAT, ADAMW_EMISMATCH.
 */
ADAMW_API int ckpt_read(adamw_ctx* ctx, const char* path, int32_t* step_out,
              float* d_w, float* d_m, float* d_v, void* stream);

/*
 * One clipped-AdamW step with no context and no allocation, for callers that
 * must not allocate GPU memory: code running under a framework or server that
 * owns all device memory through its own pool, plug-ins handed nothing but
 * their input and output buffers, and latency-critical paths where
 * cudaMalloc / cudaFree would synchronise the device.  The pages have no
 * counterpart: this is a packaging of the same two kernels as
 * adamw_clip_step.
 *
 * Same arguments and arithmetic as adamw_clip_step (n parameters, flat
 * layout, 1-based t, beta1/beta2/eps given per call), same results bit for
 * bit.  If d_norm_out is not NULL, the gradient norm (double) is written to
 * that device address on `stream`; a non-finite norm leaves w, m, v
 * untouched and shows there as inf/nan (the call does not wait, so it cannot
 * return ADAMW_ENONFINITE).
 *
 * Scratch: a 5,120-byte array in the library's static device memory, which
 * every GPU that loads the library keeps until the process exits; it serves
 * any n in [1, 2^31 - 1] (the reduction grid is capped); n outside that range
 * is rejected with ADAMW_EINVAL.  The first call on each device resolves
 * that array's address and the kernels' launch limits (no allocation); make
 * that first call before any stream capture.  Those values are kept for the
 * life of the process: after a cudaDeviceReset (which unloads the library's
 * device code and its array) the kept address is stale, so a caller that
 * resets a device must not call this entry point on it again.  All calls share the one array
 * and it keeps the last call's contents (each call clears the part that must
 * start at zero): calls that overlap on the GPU -- on different streams or
 * from different threads without ordering -- race and give wrong results.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
ADAMW_API int adamw_clip_step_noalloc(float* d_w, const float* d_g, float* d_m,
                                      float* d_v, int64_t n, int32_t t,
                                      double lr, double wd, double clip,
                                      double beta1, double beta2, double eps,
                                      double* d_norm_out, void* stream);

/*
 * Host-only helpers (no GPU needed).
 *
 * ckpt_file_size: 8 + 12 n ([C] "Total size"); -1 if n is outside
 * [0, 2^31 - 1].
 *
 * ckpt_write_host: the atomic writer of ckpt_write applied to host arrays
 * h_w, h_m, h_v of n floats (e.g. a state held on the host).
 *
 * ckpt_probe: validates a file the way ckpt_read does (header, sign, size)
 * without reading the arrays; *step_out and *n_out (may be NULL) receive the
 * header fields.  n_expected < 0 skips the n comparison.
 *
 * ckpt_write_image: the atomic writer applied to a complete host image of
 * `bytes` bytes (header included; the header must describe exactly that
 * size).  With CKPT_DIRECT, an image at a 4096-byte aligned address with
 * capacity >= bytes rounded up to 4096 is written with O_DIRECT when the
 * file system allows it (the padding past `bytes` is written, then cut off).
 *
 * ckpt_rotate: deletes all but the newest `keep` files named
 * step_<digits>.bin in dir (keep = 0: none); *removed (may be NULL) receives
 * the count.
 */
ADAMW_API int64_t ckpt_file_size(int64_t n);
ADAMW_API int ckpt_write_host(const char* dir, int32_t step, int32_t n,
                    const float* h_w, const float* h_m, const float* h_v,
                    char* path_out, size_t path_cap);
ADAMW_API int ckpt_probe(const char* path, int32_t n_expected, int32_t* step_out,
               int32_t* n_out);
ADAMW_API int ckpt_write_image(const char* dir, const void* image, int64_t bytes,
                               int64_t capacity, int32_t flags, char* path_out,
                               size_t path_cap);
ADAMW_API int ckpt_rotate(const char* dir, int32_t keep, int32_t* removed);

/*
 * Sharded checkpoint ([S]: each rank writes its own shard file, a manifest
 * records which rank owns which range).  One directory per checkpoint:
 *   <dir>/step_NNNNNN/rank<R>.bin    shard R in the step_NNNNNN.bin format
 *                                    over its range (its own n in the header)
 *   <dir>/step_NNNNNN/manifest.json  {"world_size", "step",
 *       "wall_clock_seconds", "shards": [{"rank", "path", "sha256",
 *       "param_shard_offset", "param_shard_numel"}], "schema_version": 1}
 * ([S] "Manifest schema").  Every rank writes and fsyncs its file under
 * <dir>/step_NNNNNN.tmp/ and reports its sha256; once all have (the caller
 * synchronises the ranks and gathers the digests), rank 0 calls
 * ckpt_manifest_commit, which writes the manifest there (tmp, fsync, rename),
 * fsyncs, and renames the directory to step_NNNNNN: the checkpoint appears
 * complete or not at all ([S] "Atomic write"; one directory rename instead
 * of one rename per file, so the set is atomic).  Loading refuses
 * ([S] "Three failure modes"): a world size other than expected_world
 * (ADAMW_EMISMATCH), a shard count or rank set that does not match
 * world_size (ADAMW_EMISMATCH), a shard whose size, header or sha256
 * disagrees with the manifest (ADAMW_ESIZE / ADAMW_EFORMAT).
 *
 * ckpt_shard_write: writes the image of the last ckpt_pack of this context
 * (its shard, step = the packed step) as rank<rank>.bin; sha256_hex_out
 * receives 64 hex digits + NUL.  Blocks until durable.
 * ckpt_shard_write_host: the same from host arrays of n floats.
 * ckpt_manifest_commit: rank 0, after every shard is written; offsets,
 * numels: per rank, contiguous from 0; sha256_hex: the ranks' digests
 * concatenated (64 x world hex digits).  path_out receives the directory.
 * ckpt_manifest_load: validates a step directory (digests too if
 * verify_sha256) and returns its step, world size and layout (cap entries).
 * ckpt_shard_read: validates the manifest and this rank's shard (size,
 * header, sha256), then copies the shard into d_w, d_m, d_v (n = the
 * context's n must equal the shard's numel) and waits; the device arrays
 * are untouched on failure.
 */
ADAMW_API int ckpt_shard_write(adamw_ctx* ctx, const char* dir, int32_t rank,
                               char* sha256_hex_out);
ADAMW_API int ckpt_shard_write_host(const char* dir, int32_t step, int32_t rank, int32_t n,
                                    const float* h_w, const float* h_m, const float* h_v,
                                    char* sha256_hex_out);
ADAMW_API int ckpt_manifest_commit(const char* dir, int32_t step, int32_t world,
                                   double wall_clock_seconds, const int64_t* offsets,
                                   const int64_t* numels, const char* sha256_hex,
                                   char* path_out, size_t path_cap);
ADAMW_API int ckpt_manifest_load(const char* step_dir, int32_t expected_world,
                                 int32_t verify_sha256, int32_t* step_out,
                                 int32_t* world_out, int64_t* offsets_out,
                                 int64_t* numels_out, int32_t cap);
ADAMW_API int ckpt_shard_read(adamw_ctx* ctx, const char* step_dir, int32_t rank,
                              int32_t expected_world, int32_t* step_out, float* d_w,
                              float* d_m, float* d_v, void* stream);

/*
 * Resume at another world size ([S] "Three failure modes": the manifest's
 * param_shard_offset and param_shard_numel let the loader put every shard's
 * range back at its place in the flat parameter vector).
 *
 * ckpt_consolidate (host only): validates the manifest of step_dir against
 * expected_world (< 0: any) and every shard's size and header, then writes
 * the flat checkpoint of the whole state, <out_dir>/step_NNNNNN.bin in the
 * ckpt_read format (n = the shards' total, which must fit an int32), by one
 * streaming pass: the w regions of all shards in rank order, then m, then v.
 * Each shard's sha256 is checked on the way (its bytes arrive in file
 * order); a mismatch returns ADAMW_EFORMAT and leaves no file.  The file is
 * made durable like ckpt_write (tmp, fsync, rename, directory fsync).
 * path_out receives its path.
 *
 * ckpt_read_range: like ckpt_read, for a range of a flat checkpoint: the
 * file may hold N >= offset + n parameters (n = the context's); copies
 * w[offset, offset + n), m[...], v[...] to d_w, d_m, d_v and waits.  With
 * ranges from a partition of [0, N) (for example 4-aligned equal shards) any
 * number of ranks resumes from one consolidated file.  ADAMW_EMISMATCH if
 * the range does not fit the file; the device arrays are untouched on
 * failure.
 */
ADAMW_API int ckpt_consolidate(const char* step_dir, int32_t expected_world,
                               const char* out_dir, char* path_out, size_t path_cap);
ADAMW_API int ckpt_read_range(adamw_ctx* ctx, const char* path, int64_t offset,
                              int32_t* step_out, float* d_w, float* d_m, float* d_v,
                              void* stream);

/*
 * SHA-256 (FIPS 180-4) of `bytes` bytes as 64 lowercase hex digits + NUL.
 * Every digest of the library (shard files, manifests' checks) is computed
 * by the system's libcrypto (OpenSSL 3, the CPU's SHA instructions) when it
 * can be loaded at run time, else by the library's own implementation of
 * the standard; both give the same digest.  OSR_SHA256=builtin in the
 * environment, read once at the first digest, selects the library's own.
 * ckpt_sha256_backend: 1 if libcrypto computes the digests, 0 if not.
 */
ADAMW_API int ckpt_sha256_hex(const void* data, int64_t bytes, char* hex_out);
ADAMW_API int ckpt_sha256_backend(void);

/* Name of a status code, and the last failure's explanation (this thread). */
ADAMW_API const char* adamw_strerror(int status);
ADAMW_API const char* adamw_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ADAMW_CKPT_H */
