/*
 * fadam.h - C ABI of the multi-tensor fused Adam/AdamW update over one
 * data-parallel rank's optimizer shard, for NVIDIA GB300 (sm_103a).
 *
 * What the library computes (sources are web pages, cited by title and the
 * construct on the page):
 *   - "Enhance Distributed Fused Adam (#1794)" (apex patch),
 *     DistAdamCapturableFunctor::local_step: per element, with sg the
 *     scaled gradient,
 *       L2 mode:    sg = g*grad_scale + wd*p
 *       AdamW mode: sg = g*grad_scale
 *       m' = beta1*m + (1-beta1)*sg          v' = beta2*v + (1-beta2)*sg^2
 *       u  = (m'/bc1) / (sqrt(v'/bc2) + eps)  (+ wd*p in AdamW mode, old p)
 *       p' = p - lr*u,   p_out = p' cast to the param-out dtype
 *     with bc1 = 1-beta1^step, bc2 = 1-beta2^step when bias correction is
 *     on (operator(), bias-correction block) and 1 otherwise; a noop flag
 *     equal to 1 leaves everything untouched (operator(), early return).
 *     lerp() is not defined on the page; it is read as the moving average
 *     above.  Every operation is one IEEE fp32 operation, not contracted.
 *   - "apex/contrib/optimizers/distributed_fused_adam.py":
 *     step() (regular: the step counter advances by one before the update;
 *     capturable: by (noop != 1), on the device), _local_step() (one call per
 *     group over lists p, m, v, g, p_out), _local_step_with_param_remainders()
 *     and _bf16_rem_to_fp32() (the fp32 master held as a bf16 high half plus
 *     an int16 remainder).
 *   - "[PyTorch] Advance FusedAdam step counter for empty param groups"
 *     (TransformerEngine PR), Fix section: every param group's counter
 *     advances, also a group that holds no tensor on this rank.
 *
 * Design: a plan packs the ragged tensor list once into a balanced work list
 * for a persistent grid; each fadam_step() is then ONE kernel launch on the
 * caller's stream, with no host synchronisation, no allocation and no
 * host-to-device copy, so the capturable form can be captured in a CUDA
 * graph.
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev are device pointers (cudaMalloc, torch CUDA
 *     storage); other pointers are host pointers unless stated.
 *   - The caller owns all tensor memory.  A plan owns only its work list,
 *     its copy of the descriptors and a small device status block.
 *   - Argument checks run on the host before anything is launched.  A
 *     failing check returns a non-zero status and launches nothing; the
 *     message for the calling thread is available from fadam_last_error().
 *   - No entry point traps or asserts on the device.  The only device-side
 *     error (a bounded wait that gives up) is recorded in the plan's status
 *     block and reported by fadam_plan_status().
 *   - Calls on one plan must be ordered (one stream, or ordered streams):
 *     the plan's device status block is shared by its launches.
 */
#ifndef FADAM_H_
#define FADAM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t.  NULL means the legacy default stream. */
typedef struct CUstream_st* fadam_stream;

/* Opaque plan (packed work list for one shard). */
typedef struct fadam_plan fadam_plan;

/* Status codes returned by every entry point. */
typedef int32_t fadam_status;
#define FADAM_OK 0
#define FADAM_EINVAL 1   /* an argument failed its check; nothing launched */
#define FADAM_EDTYPE 2   /* unsupported dtype combination; nothing launched */
#define FADAM_EALIGN 3   /* a pointer is not aligned to its element size */
#define FADAM_ECUDA 4    /* a CUDA runtime call failed (see fadam_last_error) */
#define FADAM_ETIMEOUT 5 /* a bounded device-side wait gave up (device status) */
#define FADAM_ELIMIT 6   /* a size is beyond a documented maximum */

/* Update mode ("mode" argument of the page's kernel; adam_w_mode). */
#define FADAM_MODE_L2 0    /* L2: weight decay folded into the gradient */
#define FADAM_MODE_ADAMW 1 /* decoupled weight decay */

/* Element types. */
#define FADAM_DT_NONE 0 /* no param-out copy */
#define FADAM_DT_F32 1
#define FADAM_DT_BF16 2
#define FADAM_DT_F16 3

/* Plan flags. */
#define FADAM_CAPTURABLE 1u  /* lr, grad_scale, step read from device memory */
#define FADAM_REMAINDERS 2u  /* master = bf16 p (high half) + int16 rem */
#define FADAM_CHECK_FINITE 4u /* screen g*grad_scale for inf/nan first; sets noop */
#define FADAM_STEP_PREADVANCED 8u /* capturable: *step_dev already advanced by the
                                     caller; use it as is and do not write it */
#define FADAM_SCALED_STATES 16u /* 16-bit p, m, v stored with one fp32 scale each
                                   per tensor (fadam_plan_set_state_scales) */
/* An fp32 master (p_dtype FADAM_DT_F32) with both moments, m and v, in bf16
 * or in fp16: TransformerEngine's FusedAdam exp_avg_dtype and
 * exp_avg_sq_dtype (constructor arguments in the adam_bench.py script of
 * "[Performance] FusedAdam capturable kernel is ~1.9x slower than regular
 * Adam on GB300"), taken equal.  m and v are widened to float, the update
 * runs in float as for an fp32 state, p keeps the float result and m, v are
 * rounded to nearest-even when stored.  Not with FADAM_REMAINDERS or
 * FADAM_SCALED_STATES. */
#define FADAM_MOMENTS_BF16 32u
#define FADAM_MOMENTS_F16 64u
/* Reciprocal bias corrections, for the 16-bit state forms (FADAM_DT_BF16 or
 * FADAM_DT_F16 state, plain or FADAM_SCALED_STATES), whose update is bound
 * by instruction issue rather than by memory: each CTA computes 1/bc1 and
 * 1/bc2 once per group (IEEE reciprocals) and the update multiplies the
 * moments of every element by them instead of dividing by bc1 and bc2 (the
 * functor's m/bc1 and v/bc2).  Each bias-corrected moment then carries two
 * roundings instead of one, so results are no longer bit-identical to the
 * division: the update u = m_hat / (sqrt(v_hat) + eps) moves by at most a
 * few float ulps; m and v do not move (they precede any division); p' =
 * p - lr*u moves by a few ulps of lr*u <= |p| + |p'|, so a stored p (or
 * param-out) lands within one unit in its last place plus
 * 2e-6 * max(|p|, |p'|) of the divided result per step (more than one ulp
 * only where the step nearly cancels p).  Once a correction rounds to 1 in
 * float the multiply is exact.  Infinite and NaN inputs give the same
 * non-finite results as the division; the bound holds while m/bc1 and
 * v/bc2 stay finite (where m is within a few ulps of FLT_MAX * bc1, m/bc1
 * may be infinite in one form and finite in the other; likewise v).  Other
 * state forms (fp32 master, remainders, 16-bit moments) are bound by memory,
 * keep the division and ignore the flag. */
#define FADAM_RECIP_BC 128u
/* Diagnostic, for testing the failure path: the grid barrier after the
 * inf/nan screen (FADAM_CHECK_FINITE), or else the one between the two
 * passes of a scaled state (FADAM_SCALED_STATES), of the plan's FIRST step
 * launch (fadam_step, fadam_step_reduce or fadam_step_host_grads) waits for
 * one more CTA than the launch has, so every CTA's wait runs out after its
 * limit (about 2 s).  That step then writes no p, m, v or scales (after the
 * scaled state's first pass, param-out is written), advances no counter,
 * and fadam_plan_status() reports FADAM_ETIMEOUT; the plan's later launches
 * run normally, which shows that a plan recovers from a wait that gave up.
 * fadam_step_noalloc applies it to every call that passes it.  Never set in
 * normal use. */
#define FADAM_TEST_BARRIER_TIMEOUT 0x80000000u

/* Maximum number of param groups in one plan. */
#define FADAM_MAX_GROUPS 32

/* Maximum numbers of gradient sources and extra param-out destinations of
 * the data-parallel exchange (fadam_plan_set_exchange). */
/* reduce_flags of fadam_plan_set_exchange. */
#define FADAM_EXCHANGE_AVERAGE 1    /* divide the sum by R (ReduceOp.AVG) */
#define FADAM_EXCHANGE_ACCUMULATE 2 /* add the reduced value to the shard's g */
#define FADAM_MAX_SOURCES 16
#define FADAM_MAX_DESTS 16

/* One tensor (fragment) of the shard.  Every data pointer is a device
 * pointer to numel contiguous elements, aligned at least to its element
 * size.
 *   p      master parameter in the plan's state dtype (fp32, bf16 or fp16),
 *          updated in place; in FADAM_REMAINDERS mode the bf16 high half of
 *          the master (read only, unless p_out aliases it)
 *   m, v   first and second moments (exp_avg, exp_avg_sq) in the state
 *          dtype (fp32 in FADAM_REMAINDERS mode; bf16 or fp16 with
 *          FADAM_MOMENTS_BF16 / _F16), in place
 *   g      gradient in the plan's g dtype, read only
 *   p_out  param-out copy in the plan's out dtype; NULL iff the out dtype
 *          is FADAM_DT_NONE; may alias p; required (bf16) in remainder mode
 *   rem    int16 remainder, in place; non-NULL iff FADAM_REMAINDERS
 *   group  index of the tensor's param group, 0 <= group < n_groups
 * Tensors must not overlap one another, except that p_out may equal p. */
typedef struct {
  void* p;
  void* m;
  void* v;
  const void* g;
  void* p_out;
  int16_t* rem;
  int64_t numel;
  int32_t group;
  int32_t reserved; /* set to 0 */
} fadam_tensor;

/* One param group's hyper-parameters and scalars.
 *   mode             FADAM_MODE_L2 or FADAM_MODE_ADAMW
 *   bias_correction  0 or 1
 *   beta1, beta2     in [0, 1)
 *   eps              >= 0;  weight_decay: finite
 * Regular plans read the host scalars lr, grad_scale and step (the step
 * already advanced for this update, >= 1 when bias correction is on;
 * fadam_step checks it, since a plan is normally made before the first step).
 * Capturable plans read lr_dev, grad_scale_dev (fp32) and step_dev (int32)
 * instead; step_dev is required for every group, empty or not, and groups
 * may share one counter (it then advances once per step).  lr_dev and
 * grad_scale_dev may be NULL only for a group with no tensor. */
typedef struct {
  int32_t mode;
  int32_t bias_correction;
  float beta1;
  float beta2;
  float eps;
  float weight_decay;
  float lr;
  float grad_scale;
  int32_t step;
  int32_t reserved; /* set to 0 */
  const float* lr_dev;
  const float* grad_scale_dev;
  int32_t* step_dev;
} fadam_group;

/* Read-only facts about a plan. */
typedef struct {
  int64_t n_tensors;
  int64_t n_elements;     /* elements updated per step */
  int64_t n_items;        /* work items in the packed list */
  int64_t n_chunks;       /* chunks of bulk-copy tiles the CTAs share out */
  int32_t grid;           /* CTAs of the persistent launch */
  int32_t block;          /* threads per CTA */
  int32_t blocks_per_sm;  /* resident CTAs per SM at this block size */
  int32_t sm_count;
  int32_t n_groups;
  int32_t device;
  double bytes_per_step;  /* algorithmic HBM bytes of one update (each
                             stream read or written once) */
  double check_bytes_per_step; /* extra bytes of the FADAM_CHECK_FINITE screen */
} fadam_plan_info;

/* Build a plan for a shard: validates every descriptor, packs the ragged
 * tensor list into a balanced work list for a persistent grid sized to the
 * current device, uploads it (synchronously) and allocates the plan's
 * device status block and a 2 KB memo through which each launch hands the
 * next step's bias corrections to the next launch (keyed by betas and
 * step; a launch that finds no matching entry computes them, so results do
 * not depend on it).  Call it before any stream capture.
 *   tensors[n_tensors]  descriptors (host array, copied; n_tensors >= 0)
 *   groups[n_groups]    1 <= n_groups <= FADAM_MAX_GROUPS (host array, copied)
 *   p_dtype             state dtype of p, m and v: FADAM_DT_F32, _BF16 or
 *                       _F16 (the optimizer's `dtype`; 16-bit values are
 *                       widened for the update and rounded to nearest-even
 *                       on store); FADAM_DT_BF16 with FADAM_REMAINDERS
 *                       (then m and v are fp32)
 *   g_dtype             FADAM_DT_F32, FADAM_DT_BF16 or FADAM_DT_F16
 *   out_dtype           FADAM_DT_NONE, _F32, _BF16 or _F16 (_BF16 with remainders)
 *   flags               FADAM_CAPTURABLE | FADAM_REMAINDERS |
 *                       FADAM_CHECK_FINITE | FADAM_STEP_PREADVANCED |
 *                       FADAM_SCALED_STATES (bf16 or fp16 state only; set
 *                       the scales with fadam_plan_set_state_scales) |
 *                       FADAM_MOMENTS_BF16 or FADAM_MOMENTS_F16 (fp32 master
 *                       with m and v in that dtype) | FADAM_RECIP_BC
 *   *plan_out           receives the plan (owned by the caller; free with
 *                       fadam_plan_destroy)
 * Errors: FADAM_EINVAL, FADAM_EDTYPE, FADAM_EALIGN, FADAM_ELIMIT, FADAM_ECUDA;
 * on error *plan_out is set to NULL. */
fadam_status fadam_plan_create(const fadam_tensor* tensors, int64_t n_tensors,
                               const fadam_group* groups, int32_t n_groups,
                               int32_t p_dtype, int32_t g_dtype, int32_t out_dtype,
                               uint32_t flags, fadam_plan** plan_out);

/* Replace the plan's param-group table (same n_groups as at creation).  This
 * is how a regular plan receives each step's host lr, grad_scale and step;
 * it copies the values on the host and touches no device memory, so it may
 * be called between captured launches (the captured launch keeps the values
 * it was captured with).  Errors: FADAM_EINVAL. */
fadam_status fadam_plan_set_groups(fadam_plan* plan, const fadam_group* groups,
                                   int32_t n_groups);

/* One optimizer step over the whole shard: one persistent-grid kernel
 * launch on `stream`, or none when there is nothing to do.  With exchange
 * destinations set (fadam_plan_set_exchange), param-out is also written to
 * every destination.
 *   noop_dev  int32 device flag (may be NULL when FADAM_CHECK_FINITE is not
 *             set).  When it equals 1 nothing is written: not p, m, v, rem,
 *             p_out, nor the step counters; any other value counts as clear
 *             (the page's kernel tests for 1).  The library only ever
 *             writes 1 to it (with FADAM_CHECK_FINITE, when some
 *             g*grad_scale is not finite; the screen runs over the whole
 *             shard before any update).
 * Capturable plans advance every group's *step_dev by (noop != 1) within
 * the same launch and use step+1 in the bias correction (unless
 * FADAM_STEP_PREADVANCED).  No host sync, no allocation: safe to capture.
 * Errors: FADAM_EINVAL, FADAM_EALIGN, FADAM_ECUDA (launch failed). */
fadam_status fadam_step(fadam_plan* plan, int32_t* noop_dev, fadam_stream stream);

/* End-to-end step from host gradients g_host[i] (a host buffer of numel
 * elements of the g dtype per tensor).  When every buffer is page-locked and
 * mapped for the device (cudaHostAlloc / cudaHostRegister, or torch's
 * pin_memory), with the same address alignment modulo 16 bytes as the
 * tensor's device g, the step reads the gradients over the host link
 * itself (zero copy: the transfer overlaps the update of p, m and v, and
 * the tensors' device g buffers are not written).  Otherwise each buffer is
 * copied into the tensor's device g first (cudaMemcpyAsync) and fadam_step()
 * runs.  Then each group's step counter is copied into steps_host[n_groups]
 * (may be NULL), and the call waits for the stream.  Errors: as fadam_step. */
fadam_status fadam_step_host_grads(fadam_plan* plan, const void* const* g_host,
                                   int32_t* noop_dev, int32_t* steps_host,
                                   fadam_stream stream);

/* Gradient norm, step one: the squared L2 norm of the shard's scaled
 * gradient, sum over groups of grad_scale^2 * sum of g^2 over the group's
 * tensors ("apex/contrib/optimizers/distributed_fused_adam.py",
 * _local_grad_norm and grad_norm), written as one double to *sumsq_dev by
 * one launch on `stream`.  grad_scale is the host value of regular plans
 * and *grad_scale_dev of capturable ones.  Accumulation: float within a
 * thread's share of a chunk of tiles (Kahan-compensated) and within a warp,
 * exactly in double wherever a float partial would overflow, underflow or is
 * not finite, double across warps, chunks and CTAs (a fixed order: the
 * result is deterministic).  Across data-parallel ranks, all-reduce
 * (sum) *sumsq_dev before step two.  No allocation, no host sync: safe to
 * capture.  Errors: FADAM_EINVAL (NULL or misaligned sumsq_dev),
 * FADAM_ECUDA. */
fadam_status fadam_grad_sumsq(fadam_plan* plan, double* sumsq_dev, fadam_stream stream);

/* Gradient norm, step two (same source, clip_grad_norm and step()): from
 * the squared norm (summed over ranks), one thread on `stream` writes
 * norm = sqrt(*sumsq_dev) rounded to float into *norm_dev (may be NULL),
 * found_inf = (norm is not finite) as 0 or 1 into *noop_dev (may be NULL:
 * the page copies found_inf into its noop buffer), and, when max_norm > 0,
 * multiplies each distinct grad_scale_dev of a capturable plan by
 * min(1, max_norm / (norm + 1e-6)) (float arithmetic; a NaN coefficient is
 * kept).  Regular plans keep grad_scale on the host (the page reads the
 * norm with .item()): when grad_scales_out_dev is not NULL, the same
 * launch writes each group's grad_scale (as last set with
 * fadam_plan_set_groups) times that coefficient into
 * grad_scales_out_dev[n_groups] (unchanged when max_norm <= 0), for the
 * caller to read back and pass to fadam_plan_set_groups; capturable plans
 * ignore it.  Errors: FADAM_EINVAL, FADAM_EALIGN, FADAM_ECUDA. */
fadam_status fadam_clip_apply(fadam_plan* plan, const double* sumsq_dev, float max_norm,
                              float* norm_dev, int32_t* noop_dev, float* grad_scales_out_dev,
                              fadam_stream stream);

/* The data-parallel exchange around the step, on one GPU
 * ("apex/contrib/optimizers/distributed_fused_adam.py":
 * _start_bucket_grad_sync, the reduce-scatter of every rank's gradient
 * bucket into this rank's shard with ReduceOp.AVG or SUM, and
 * _start_bucket_param_sync, the all-gather of every rank's param shard).
 * A data-parallel group of R ranks is stood in for by R device buffers: the
 * plan's gradients are this rank's shard (the tensors' g pointers all lie in
 * one shard buffer starting at g_shard), and sources[r] is where rank r's
 * contribution to that shard starts, laid out like the shard; each tensor's
 * contribution from rank r is read at g + (sources[r] - g_shard).  Likewise
 * the tensors' p_out pointers lie in one buffer starting at out_shard, and
 * dests[d] is another buffer laid out like it (another rank's place for this
 * shard in its param bucket); every p_out value is also written at
 * p_out + (dests[d] - out_shard).
 *   g_shard, sources[n_sources]   0 <= n_sources <= FADAM_MAX_SOURCES
 *                                 (host array of device pointers, copied);
 *                                 every sources[r] - g_shard a multiple of 16
 *                                 bytes.  The sources are only read.
 *   reduce_flags                  FADAM_EXCHANGE_AVERAGE: the sum divided by
 *                                 R (ReduceOp.AVG), else the sum;
 *                                 FADAM_EXCHANGE_ACCUMULATE: gradient
 *                                 accumulation across reduce-scatters
 *                                 (_finish_bucket_grad_sync: the second and
 *                                 later reduce-scatters of a step add their
 *                                 shard to the gradient shard,
 *                                 grads_shard.add_): the shard's g becomes
 *                                 its old value plus the reduced value
 *                                 rounded to the grad dtype, both widened,
 *                                 one IEEE addition, rounded once to the grad
 *                                 dtype; without it g is overwritten.
 *   out_shard, dests[n_dests]     0 <= n_dests <= FADAM_MAX_DESTS, each
 *                                 dests[d] - out_shard a multiple of 16
 *                                 bytes; needs a param-out dtype.
 * The reduction: the R values of an element widened to float and added in
 * rank order one IEEE addition at a time, divided by R (one IEEE division)
 * when averaging, rounded once (nearest-even) to the grad dtype and stored
 * in the shard's g.  Buffers are owned by the caller and must stay valid
 * while the plan is used; the pointers are copied on the host (no device
 * memory is touched, so this may be called between captured launches;
 * captured launches keep the pointers they were captured with).
 * n_sources = 0 and n_dests = 0 remove the exchange.  Set the flags again
 * (with the same buffers) to switch accumulation on after a step's first
 * reduce-scatter and off for the next step's first.  Errors: FADAM_EINVAL
 * (counts out of range, NULL pointers, destinations without a param-out
 * dtype, unknown reduce_flags bits), FADAM_EALIGN (a difference not a
 * multiple of 16 bytes). */
fadam_status fadam_plan_set_exchange(fadam_plan* plan, const void* g_shard,
                                     const void* const* sources, int32_t n_sources,
                                     int32_t reduce_flags, const void* out_shard,
                                     void* const* dests, int32_t n_dests);

/* The reduce-scatter stand-in alone: one launch that writes this rank's
 * gradient shard (every tensor's g) from the plan's sources, as described
 * at fadam_plan_set_exchange.  It touches nothing else (no state, no step
 * counter, no noop flag), so it can feed fadam_grad_sumsq and
 * fadam_clip_apply before fadam_step.  Safe to capture.  Errors:
 * FADAM_EINVAL (no sources set), FADAM_ECUDA. */
fadam_status fadam_grad_reduce(fadam_plan* plan, fadam_stream stream);

/* The reduce-scatter stand-in fused with the step: one cooperative launch
 * that first writes the gradient shard from the sources (as
 * fadam_grad_reduce; with FADAM_CHECK_FINITE the inf/nan screen of the
 * reduced g*grad_scale happens in the same pass), waits at a bounded grid
 * barrier, then runs the step exactly as fadam_step (param-out also to the
 * plan's destinations).  The gradient shard is written even when the step
 * is skipped (a set noop flag).  Errors: as fadam_step, and FADAM_EINVAL
 * when no sources are set. */
fadam_status fadam_step_reduce(fadam_plan* plan, int32_t* noop_dev, fadam_stream stream);

/* Scaled optimizer state ("apex/contrib/optimizers/distributed_fused_adam.py",
 * _local_step_with_scaled_states and _apply_state_scale): with
 * FADAM_SCALED_STATES the plan's p, m and v (state dtype bf16 or fp16, not
 * the remainder form) hold scaled values, and each tensor has three fp32
 * scales.  A step widens each value and multiplies it by its scale, runs
 * the fp32 update (param-out, if any, is the cast of the new fp32 param),
 * then rescales each of the tensor's three buffers: absmax = the largest
 * magnitude of the new values (NaN if any is NaN), scale = absmax /
 * (largest finite value of the state dtype / 2), reciprocal = 1 / scale
 * where scale > 0 else 0, stored value = new value * reciprocal rounded to
 * nearest even; the new scales replace the old.  Tensors with no elements
 * keep their scales.  Each product, quotient and reciprocal is one IEEE
 * float operation.  For bf16 that target is about 1.7e38, so a buffer whose
 * absmax is below about 0.5 gets a subnormal scale whose reciprocal is
 * infinite (the page's operations do the same).
 *   scales_dev   device float array of 3 * n_tensors: tensor i's scales of
 *                p, m, v at [3i], [3i+1], [3i+2] (i in the order given to
 *                fadam_plan_create), 4-byte aligned, read and rewritten by
 *                every applied step (left as is by a skipped one).
 * The pointer is copied on the host; a scaled plan's steps fail with
 * FADAM_EINVAL until it is set.  A scaled step is one cooperative launch
 * with two passes over the shard and a bounded grid barrier between
 * (the new scales depend on every new value of a tensor).  Errors:
 * FADAM_EINVAL (not a scaled plan, NULL), FADAM_EALIGN. */
fadam_status fadam_plan_set_state_scales(fadam_plan* plan, float* scales_dev);

/* Read (synchronously) and clear the plan's device status word:
 * *device_status = FADAM_OK, or FADAM_ETIMEOUT when a bounded device wait
 * (a grid barrier, or a bulk copy's completion) of some launch since the
 * last read gave up; that launch may be partly applied.  The word is sticky
 * until read, but it does not block the plan: each launch's last CTA resets
 * the barrier counters, so the next launch runs normally whether or not
 * the status was read in between (a scaled-state launch replaces the
 * scales unless one of its own waits gave up).  Errors: FADAM_EINVAL,
 * FADAM_ECUDA. */
fadam_status fadam_plan_status(fadam_plan* plan, int32_t* device_status);

/* Facts about a plan.  Errors: FADAM_EINVAL. */
fadam_status fadam_plan_get_info(const fadam_plan* plan, fadam_plan_info* info);

/* Free a plan (waits for the device first).  NULL is accepted. */
fadam_status fadam_plan_destroy(fadam_plan* plan);

/* One-shot step mirroring the page's kernel signature: packs `tensors`
 * (all in one param group), runs one step and frees its work list in
 * stream order (cudaMallocAsync / cudaFreeAsync).  Regular when lr_dev,
 * step_dev and grad_scale_dev are all NULL (host lr, step, grad_scale);
 * capturable when all three are given.  out_dtype as in fadam_plan_create,
 * p and g dtypes fp32 and g_dtype.  It copies pageable host memory, so it
 * is not for stream capture.  Errors: as fadam_plan_create / fadam_step. */
fadam_status fadam_step_once(const fadam_tensor* tensors, int64_t n_tensors, int32_t mode,
                             int32_t bias_correction, float beta1, float beta2, float eps,
                             float weight_decay, float lr, const float* lr_dev,
                             int32_t step, int32_t* step_dev, float grad_scale,
                             const float* grad_scale_dev, int32_t* noop_dev,
                             int32_t g_dtype, int32_t out_dtype, fadam_stream stream);

/* Step without any device allocation (no counterpart on the pages: this
 * entry point exists for callers of this library, not for the method).
 *
 * Some callers cannot call cudaMalloc: code running while a framework's
 * caching allocator has reserved nearly all device memory (a direct
 * cudaMalloc can fail there), code inside another library's hooks that may
 * only use memory handed to it, and latency-critical loops where
 * cudaMalloc/cudaFree could synchronise the device.  This call packs the
 * shard on the host, as fadam_plan_create does, and runs one step as
 * fadam_step does, but keeps the work list, the status block and the
 * bias-correction memo in a static device array instead of allocated
 * memory: about 340 KB that every GPU which loads this library holds until
 * the process exits.  It calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *
 * Not for stream capture: each call copies its work list from host memory
 * that is freed when the call returns, which a captured graph could not
 * replay.  A call on a capturing stream returns FADAM_EINVAL before any
 * device work; graphs use fadam_plan_create / fadam_step.
 *
 * Limits: at most 4096 work items (roughly one per tensor plus one per CTA
 * of the grid) and 2048 CTAs; a larger shard is rejected with FADAM_ELIMIT
 * and a message from fadam_last_error(), before any device work.  Its list
 * of tile chunks is capped at 4096 entries by making chunks larger, which
 * can leave the CTAs a little less evenly loaded than a plan's.
 * Arguments: as fadam_plan_create, plus noop_dev and stream as fadam_step;
 * the step counters behave as in fadam_step.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current) and keeps it for the life of the
 * process; it does not survive a cudaDeviceReset() of that device, so do
 * not call this entry point on a device after resetting it.  Each call
 * copies its work list into the array and clears the status block on
 * `stream` before the launch.  All calls share the one array and it keeps
 * the last call's contents: calls whose work overlaps on the GPU (unordered
 * streams, or concurrent host threads) race on the work list, the status
 * block and the memo, so issue them in order on one stream.  Errors: as
 * fadam_plan_create and fadam_step, FADAM_ELIMIT beyond the limits above,
 * FADAM_EINVAL on a capturing stream. */
fadam_status fadam_step_noalloc(const fadam_tensor* tensors, int64_t n_tensors,
                                const fadam_group* groups, int32_t n_groups, int32_t p_dtype,
                                int32_t g_dtype, int32_t out_dtype, uint32_t flags,
                                int32_t* noop_dev, fadam_stream stream);

/* One work item of a dry-run packing (see fadam_pack_dry). */
typedef struct {
  int64_t tensor; /* index into the tensors array */
  int64_t offset; /* first element of the run within the tensor */
  int32_t n;      /* elements in the run */
  int32_t vec;    /* alignment of every stream at the run start: 0 none
                     (scalar path), 1 one 4-element vector (128-bit loads),
                     2 also 16 bytes (bulk copies through shared memory) */
} fadam_pack_item;

/* Host-only dry run of the packer, for inspection and tests; needs no GPU
 * and dereferences no tensor pointer (their addresses only decide
 * alignment).  Packs `tensors` for a grid of `grid` CTAs exactly as
 * fadam_plan_create would, writes the item count to *n_items_out, the items
 * to items_out[max_items] (may be NULL) and grid+1 CTA start indices to
 * cta_begin_out (may be NULL): CTA b runs items
 * [cta_begin_out[b], cta_begin_out[b+1]).  Errors: as fadam_plan_create's
 * argument checks, FADAM_ELIMIT when the items exceed max_items. */
fadam_status fadam_pack_dry(const fadam_tensor* tensors, int64_t n_tensors, int32_t n_groups,
                            int32_t p_dtype, int32_t g_dtype, int32_t out_dtype, uint32_t flags,
                            int32_t grid, fadam_pack_item* items_out, int64_t max_items,
                            int32_t* cta_begin_out, int64_t* n_items_out);

/* Host-only dry run of the chunk list, for inspection and tests; needs no
 * GPU and dereferences no tensor pointer.  Packs `tensors` for a grid of
 * `grid` CTAs as fadam_pack_dry does, then builds the list of bulk-tile
 * chunks the CTAs of a launch take in order, at most `max_chunks` long (a
 * plan uses 131072, fadam_step_noalloc 4096): 16 tiles a chunk (more when
 * that keeps the list within max_chunks), tapering at the end of the list
 * to about R / (2 grid) tiles, at least 4, for a chunk that starts with R
 * tiles left; the tapered list is used when it fits max_chunks.  A tile
 * here is 1024 vectors of 4 elements (a pass may copy several at once);
 * only items whose streams are all 16-byte aligned have tiles.  Writes the chunk
 * count to *n_chunks_out and, when chunks_out is not NULL, each chunk as
 * three int32 (item index as in fadam_pack_dry, first tile, tiles) to
 * chunks_out[3 * max_out].  Errors: as fadam_pack_dry, FADAM_EINVAL for
 * max_chunks < 1, FADAM_ELIMIT when the chunks exceed max_out. */
fadam_status fadam_chunk_dry(const fadam_tensor* tensors, int64_t n_tensors, int32_t n_groups,
                             int32_t p_dtype, int32_t g_dtype, int32_t out_dtype, uint32_t flags,
                             int32_t grid, int64_t max_chunks, int32_t* chunks_out,
                             int64_t max_out, int64_t* n_chunks_out);

/* Static description of a status code. */
const char* fadam_status_string(fadam_status status);

/* Message of the last failure in the calling thread ("" when none). */
const char* fadam_last_error(void);

/* Library version, as major*10000 + minor*100 + patch. */
int32_t fadam_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FADAM_H_ */
