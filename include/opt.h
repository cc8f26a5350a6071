/*
 * opt.h -- C ABI of the GB300 (sm_103a) fused optimizer-step library.
 *
 * One optimizer step over a list of parameter tensors, in two calls:
 *
 *   opt_grad_norm      deterministic global gradient 2-norm and inf-norm,
 *                      accumulated beyond fp32, NaN/Inf counted, and the clip
 *                      coefficient derived from it -- all on the device.
 *   opt_adamw_step     fused multi-tensor AdamW, decoupled weight decay
 *   opt_ademamix_step  fused multi-tensor AdEMAMix, decoupled weight decay
 *
 * Sources (page title and section):
 *  - "Fix decoupled weight decay ordering in the CUDA Adam/AdEMAMix kernels"
 *    (bitsandbytes PR #2040), body: decay and update both taken from the old
 *    parameter, p <- p (1 - lr wd) + step_size * update.
 *  - "When Small Updates Disappear" (Topollai), sec. 1.1, 2.1, 3, 6.1, 7.3,
 *    8.1: low-precision optimizer states (BF16, FP8, unsigned E2M2 "FP4"),
 *    nearest and stochastic rounding, a counter-based draw tied to the
 *    element, the fused step that reads and writes each tensor once.
 *  - "perf(training): fused multi-tensor gradient-norm reduction" (NeMo
 *    Automodel PR #3685), 'What' and 'Correctness properties': one launch per
 *    dtype bucket, values widened in registers, host-side chunking from sizes
 *    only with no atomics (bit-identical run to run), NaN counted and the
 *    partial poisoned, the caller owning any cross-rank reduction.
 *  - "Investigate SM103 bias-correction broadcast in 32-bit optimizers"
 *    (bitsandbytes fork issue #7), 'Problem': bias-correction scalars are
 *    uniform, so they are computed once per step on the host and passed in.
 *
 * Conventions for every call:
 *  - Pointers named d_* or held in an opt_tensor_list are DEVICE pointers on
 *    the device that was current when the plan was created; everything else
 *    is host memory.  The caller owns every tensor; a plan owns only its
 *    chunk table and a small workspace (about 16 bytes per 2048 elements).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are stream-ordered and never synchronise, except where
 *    a host output (h_*) is requested.
 *  - Arguments are validated on the host before any launch.  Failures return
 *    a negative status and launch nothing.  There is no CPU fallback.
 *  - Not thread-safe per plan: calls on one plan must not overlap in time on
 *    different host threads.  Concurrent device work on one plan (two streams)
 *    races on the plan's workspace: the norm's slots and completion counter,
 *    and the tile counter from which the FP32-state and LAMB steps' warps
 *    take their tiles (two overlapping steps would split one step's tiles
 *    between them).  Order one plan's calls on one stream, or with events.
 */
#ifndef PS_OPT_H
#define PS_OPT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OPT_ABI_VERSION 2

/* ---- status codes --------------------------------------------------- */
#define OPT_OK            0
#define OPT_ENONFINITE    1   /* a status, not a failure: the gradient norm was
                                 NaN or Inf; a step given this norm changes
                                 nothing */
#define OPT_EINVAL       -1   /* NULL pointer, negative size, bad enum, bad step */
#define OPT_EUNSUPPORTED -2   /* dtype combination not built (e.g. FP8 grads) */
#define OPT_EALIGN       -3   /* a device pointer not 16-byte aligned */
#define OPT_ECUDA        -4   /* a CUDA runtime call failed */
#define OPT_ENOMEM       -5   /* workspace allocation failed */
#define OPT_ELIMIT       -6   /* list exceeds a fixed limit of the norm (see OPT_NORM_MAX_PART, opt_grad_norm_noalloc) */

/* ---- storage types ----------------------------------------------------
 * OPT_F32   IEEE binary32.
 * OPT_BF16  top 16 bits of a binary32 word (2 bytes per element).
 * OPT_E4M3  OCP FP8 E4M3FN: bias 7, 3 fraction bits, largest 448, no Inf,
 *           NaN = S.1111.111 (1 byte per element).  Nearest rounding
 *           saturates to +-448.
 * OPT_E2M2  unsigned 4-bit float: 2 exponent bits (bias 1), 2 fraction bits,
 *           values 0, 1/4, 1/2, 3/4, 1, 1.25 ... 7; no sign, NaN or Inf.
 *           Negative inputs store 0, NaN stores 7.  Two codes per byte: the
 *           LOW nibble holds the even element.  A tensor of n elements needs
 *           ceil(n/2) bytes; for odd n the unused high nibble of the last byte
 *           is written as 0.
 * ("When Small Updates Disappear", sec. 2.1.) */
typedef enum { OPT_F32 = 0, OPT_BF16 = 1, OPT_E4M3 = 2, OPT_E2M2 = 3 } opt_dtype;

/* Rounding of low-precision states on write-back ("When Small Updates
 * Disappear", sec. 3 and 6.1).  Stochastic rounding of value x adds a 16-bit
 * draw r to the 16 bits of x that lie just below the target grid's last kept
 * bit and rounds away from zero iff they carry: probability l / 2^16 where l
 * is those 16 bits.  r comes from Philox4x32-10 (Salmon et al., SC'11) with
 * key = (seed low 32, seed high 32) and counter = (q low 32, q high 32,
 * tensor index, step low 32), q = element index / 4; word (index mod 4)
 * gives the draw for m (its low 16 bits) and for v (its high 16 bits).  The
 * draw therefore depends only on (seed, step, tensor, element), never on the
 * launch shape. */
typedef enum { OPT_ROUND_NEAREST = 0, OPT_ROUND_STOCHASTIC = 1 } opt_round;

/* ---- tensor list ------------------------------------------------------
 * All arrays are HOST arrays of length n; their entries are DEVICE pointers.
 * Supported per-plan state combinations (m_dtype, v_dtype):
 *   (F32, F32), (BF16, BF16), (BF16, E4M3), (BF16, E2M2).
 * param_dtype must be F32; grad_dtype[i] is F32 or BF16 per tensor.  m2 is
 * used only by opt_ademamix_step (FP32 states only); pass NULL otherwise.
 * Every non-NULL pointer must be 16-byte aligned; the AdamW step reads FP32
 * p, m and v faster where they are 32-byte aligned.  Tensors with numel 0 may
 * have NULL pointers.  The plan copies what it needs: the arrays may be
 * freed after opt_plan_create returns.
 *
 * v_scale (optional, NULL = all 1): a per-tensor power of two s_i for a
 * low-precision v.  The stored code then holds v / s_i, so a small second
 * moment early in training is not flushed to 0 by a coarse grid ("When Small
 * Updates Disappear", sec. 2.3 and 5: FP8/FP4 states stall and lose small
 * values).  Both scalings are exact, so the rounding is the same rule on the
 * grid scaled by s_i.  Values that are not positive finite powers of two
 * are rejected (OPT_EINVAL). */
typedef struct opt_tensor_list {
  int32_t n;
  const int64_t* numel;
  void* const* param;
  const void* const* grad;
  void* const* m;
  void* const* v;
  void* const* m2;             /* NULL unless AdEMAMix */
  const int32_t* grad_dtype;   /* per tensor: OPT_F32 or OPT_BF16 */
  int32_t param_dtype;
  int32_t m_dtype;             /* also the dtype of m2 */
  int32_t v_dtype;
  const float* v_scale;        /* per tensor, power of two; NULL = 1 */
} opt_tensor_list;

/* ---- hyperparameters ----------------------------------------------------
 * Step t (1-based) computes, per element, with g the gradient (times the
 * clip coefficient when a norm result is given):
 *   m  <- beta1 m  + (1 - beta1) g
 *   m2 <- beta3 m2 + (1 - beta3) g                       (AdEMAMix)
 *   v  <- beta2 v  + (1 - beta2) g^2
 *   u  <- (m / (1 - beta1^t) [+ alpha m2]) / (sqrt(v / (1 - beta2^t)) + eps)
 *   p  <- p (1 - lr weight_decay) - lr u                  (decay-first)
 * in fp32 arithmetic with the (1 - beta) constants and bias corrections
 * formed once on the host in double and rounded to fp32.  m, v are formed in
 * this order with no fused multiply-add, so that their values before
 * rounding to a low-precision state are reproducible bit for bit. */
typedef struct opt_hparams {
  float lr, beta1, beta2, beta3, alpha, eps, weight_decay;
  int32_t rounding;          /* opt_round; ignored for FP32 states */
  uint64_t seed;             /* stochastic-rounding key */
  int32_t count_unchanged;   /* nonzero: also count v codes left unchanged
                                (read with opt_unchanged_count) */
  int32_t flags;             /* OPT_STEP_* bits; others must be 0 */
} opt_hparams;

/* Periodic state reset ("When Small Updates Disappear", sec. 5: resetting
 * the moments to zero restarts the cycle in which small updates get through,
 * every ~1000 / 300 / 200 steps for BF16 / FP8 / FP4 states).  With this flag
 * the step starts from m = v = 0 (and m2 = 0) instead of the stored states,
 * which it does not read.  Pass step = 1 on the reset step and count up from
 * there, as for a fresh optimizer, so that the bias corrections restart too.
 * With count_unchanged, the reset step compares the new v codes with code 0
 * (the state it started from). */
#define OPT_STEP_RESET_STATES 1

/* Step number from the plan's device step counter (FP32 states only,
 * otherwise OPT_EUNSUPPORTED).  Pass step = 0 (anything else is
 * OPT_EINVAL): the call advances the counter on the device and takes the
 * step it reaches, so a CUDA graph captured around opt_grad_norm and the step
 * replays as step t, t + 1, ... with no host work per step.  One extra
 * one-thread launch forms the step's two bias corrections on the device, in
 * double from the FP32 betas, rounded once to FP32: the value the host forms
 * for the same step, give or take the last bit (the device's pow is not
 * the host's).  The counter starts at 0 (the first counted step is 1); set
 * it with opt_plan_set_step, for example to 1 on a reset step.  Counted and
 * host-numbered steps may be mixed; they do not see each other's numbers. */
#define OPT_STEP_DEVICE_COUNTER 2

/* Wait drill: make the staged step kernel's bounded waits run out on purpose,
 * so that a caller can test its handling of OPT_FLAG_WAIT_TIMEOUT without a
 * GPU fault.  The kernel's producer withholds each thread block's first tile
 * (no copy is issued for it, and nothing completes its stage), so every
 * consumer's first wait runs out after the plan's wait limit
 * (opt_plan_set_wait_limit; set it short, say 1 ms, for a drill).  The step
 * then processes no tile: p and every state are left as they were, and
 * opt_plan_status reports OPT_FLAG_WAIT_TIMEOUT.  Only for AdamW steps that
 * run the staged kernel (low-precision states with stochastic rounding, or
 * BF16 v with nearest rounding); others return OPT_EUNSUPPORTED. */
#define OPT_STEP_WAIT_DRILL 4

/* ---- norm result (48 bytes, written by opt_grad_norm) -------------------
 * sumsq    sum of squares of all finite gradient elements (fp64)
 * norm2    sqrt(sumsq); NaN if any NaN, else +Inf if any +-Inf
 * norm_inf max |g|; NaN if any NaN, else +Inf if any +-Inf
 * clip_coef  (float) min(1, max_norm / (norm2 + 1e-6)) computed in double;
 *          1 when max_norm <= 0 or the norm is not finite
 * status   OPT_OK or OPT_ENONFINITE */
typedef struct opt_norm_result {
  double sumsq, norm2, norm_inf;
  uint64_t nan_count, inf_count;
  float clip_coef;
  int32_t status;
} opt_norm_result;

typedef struct opt_plan opt_plan;

/* ---- library ------------------------------------------------------------ */
int opt_version(void);                 /* OPT_ABI_VERSION */
const char* opt_strerror(int status);  /* static string, never NULL */

/* Validate `list`, build the chunk table (host, from sizes only), allocate
 * the workspace on the current device and upload the tables (synchronous).
 * On success *out owns the plan; destroy it with opt_plan_destroy.  Returns
 * OPT_ELIMIT for a gradient-dtype bucket of more than
 * OPT_NORM_SLOTS * OPT_NORM_MAX_PART (622,592) tensors, whose chunks the
 * norm's slots cannot hold (see OPT_NORM_CHUNK_MIN). */
int opt_plan_create(const opt_tensor_list* list, opt_plan** out);
void opt_plan_destroy(opt_plan* plan);   /* NULL is a no-op; synchronises the device */
/* Plan facts: chunks, elements, device workspace bytes (any may be NULL). */
int opt_plan_info(const opt_plan* plan, int64_t* n_chunks, int64_t* total_numel,
                  int64_t* workspace_bytes);

/* Global gradient norm over every tensor of the plan ("perf(training): fused
 * multi-tensor gradient-norm reduction", 'Correctness properties').  One
 * partial-sum launch per gradient dtype into fixed slots; the CTA that
 * completes last reduces the slots in a fixed order.  Bit-identical run to
 * run for the same inputs and plan.  Writes the result to d_out (device, 48
 * bytes, may be NULL to use the plan's own buffer, whose device address
 * opt_plan_norm_buffer returns).  If h_out is non-NULL the result is also
 * copied to it and the stream is synchronised.
 * Returns OPT_OK, OPT_ENONFINITE (only when h_out is given), or an error. */
int opt_grad_norm(opt_plan* plan, double max_norm, opt_norm_result* d_out,
                  opt_norm_result* h_out, void* stream);
const opt_norm_result* opt_plan_norm_buffer(const opt_plan* plan);

/* One fused step over every tensor of the plan, in place.  d_norm: a device
 * opt_norm_result from opt_grad_norm, or NULL for no clipping.  When
 * d_norm->status is OPT_ENONFINITE the kernels leave p and every state
 * untouched (the step is skipped on the device, no host sync).  step >= 1,
 * or 0 with OPT_STEP_DEVICE_COUNTER.  One launch per gradient-dtype bucket
 * (one more with the device counter). */
int opt_adamw_step(opt_plan* plan, const opt_hparams* hp, int64_t step,
                   const opt_norm_result* d_norm, void* stream);
/* Set the plan's device step counter (OPT_STEP_DEVICE_COUNTER) so that the
 * next counted step is next_step (>= 1, else OPT_EINVAL), in stream order;
 * a launch, so it may itself be captured. */
int opt_plan_set_step(opt_plan* plan, int64_t next_step, void* stream);

/* As opt_adamw_step plus m2 and alpha; needs FP32 states and m2 pointers. */
int opt_ademamix_step(opt_plan* plan, const opt_hparams* hp, int64_t step,
                      const opt_norm_result* d_norm, void* stream);

/* Update-norm clipping, the LAMB / max_unorm path ("Investigate SM103
 * bias-correction broadcast in 32-bit optimizers", 'Problem' and 'B300
 * result': the norm of each tensor's whole update is measured before it is
 * applied; there a cross-CTA atomicAdd made it differ run to run).  With the
 * AdamW direction u = m_hat / (sqrt(v_hat) + eps) of every element and |.| the
 * 2-norm over a tensor, ratio = max_unorm |p| / |u| when |u| > max_unorm |p|
 * (p before the step), else 1; then p <- p (1 - lr wd) - lr ratio u.  The norms
 * come from fixed per-tile slots reduced per tensor in a fixed order: the
 * result is bit-identical run to run.  max_unorm = 0 disables the clipping
 * (the AdamW step, in three passes).  FP32 states only; hp->flags must be 0.
 * The first call allocates a workspace of 16 bytes per 2048 elements. */
int opt_lamb_step(opt_plan* plan, const opt_hparams* hp, int64_t step, float max_unorm,
                  const opt_norm_result* d_norm, void* stream);

/* Number of v codes (FP32 words for FP32 v) the last step with
 * count_unchanged set left bitwise unchanged ("stalled", "When Small Updates
 * Disappear" sec. 1.1).  Copies to host and synchronises the stream; resets
 * the counter. */
int opt_unchanged_count(opt_plan* plan, uint64_t* h_count, void* stream);

/* Error flags raised by this plan's kernels since the last call, then
 * cleared.  0 means every kernel ran to completion.  Copies to host and
 * synchronises the stream.  Returns OPT_OK, OPT_EINVAL (NULL argument) or
 * OPT_ECUDA.
 *
 * OPT_FLAG_WAIT_TIMEOUT: the staged step kernel (low-precision states with
 *   stochastic rounding, and BF16 v with nearest rounding, take their tiles
 *   through shared memory) gave up a wait on its own bulk copies -- each wait
 *   is bounded in time (opt_plan_set_wait_limit), so the kernel never hangs
 *   -- and left part of its tiles unprocessed.  That step's outputs (p and
 *   every state) are then partly updated and must be discarded: restore them
 *   from a copy taken before the step.  Before leaving, the kernel let every
 *   copy it had issued land; the plan itself is intact, and once this call
 *   has cleared the flag it may be used again.
 * OPT_FLAG_DRAIN_TIMEOUT: in addition, one of those final waits for issued
 *   copies ran out too (no healthy GPU takes that long: the limit is the
 *   wait limit plus 10 s), so a thread block may have left with copies
 *   still targeting its shared memory.  Treat the whole CUDA context as
 *   unreliable: discard the step's outputs, destroy every plan, and reset
 *   the device before further work. */
#define OPT_FLAG_WAIT_TIMEOUT 1
#define OPT_FLAG_DRAIN_TIMEOUT 2
int opt_plan_status(opt_plan* plan, int32_t* h_flags, void* stream);

/* Limit, in nanoseconds of the GPU's global timer, of each wait of the
 * staged step kernel on this plan (see OPT_FLAG_WAIT_TIMEOUT); 2 s unless
 * set.  0 <= ns <= 10 s, else OPT_EINVAL.  The register-pipelined step
 * kernels, the norm and the codecs do not wait on anything.  A short limit
 * keeps a wait drill (OPT_STEP_WAIT_DRILL) short.  Host only: takes effect
 * from the next step call. */
int opt_plan_set_wait_limit(opt_plan* plan, uint64_t ns);

/* Copy each tensor's gradient from host memory (pinned for asynchrony) into
 * the plan's device gradient buffers: one cudaMemcpyAsync per tensor. */
int opt_grads_upload(opt_plan* plan, const void* const* h_grad, void* stream);

/* Standalone conversion of n fp32 values to a state format (and back), with
 * the same codecs the step uses ("When Small Updates Disappear", sec. 6-8:
 * the stand-alone cast).  Stochastic rounding draws one 16-bit value per
 * element from the step's generator and key (seed; tensor `tensor_index`,
 * step `step` in the counter), eight elements per generator call: element i
 * takes word (i/2) mod 4 of counter i/8, its low half for even i and its
 * high half for odd i.  d_out holds n elements of `dtype` (ceil(n/2) bytes
 * for E2M2, the unused high nibble of an odd tail 0).  Pointers 16-byte
 * aligned; n >= 0, step >= 0.  Returns OPT_OK, OPT_EINVAL, OPT_EUNSUPPORTED
 * (not BF16, E4M3 or E2M2), OPT_EALIGN or OPT_ECUDA. */
int opt_encode(const float* d_in, void* d_out, int64_t n, int32_t dtype,
               int32_t rounding, uint64_t seed, uint32_t tensor_index,
               int64_t step, void* stream);
int opt_decode(const void* d_in, float* d_out, int64_t n, int32_t dtype, void* stream);

/* ---- gradient norm without allocation ------------------------------------
 * The same global norm as opt_grad_norm (same kernels, same chunk order, so
 * the same result bit for bit), for callers that cannot allocate device
 * memory and therefore cannot build a plan: code running under a framework
 * whose caching allocator owns all device memory, in a runtime with a fixed
 * memory budget reserved up front, or at a point where a synchronising
 * cudaMalloc would stall the pipeline.  This call allocates nothing -- no
 * cudaMalloc, cudaFree or allocating library routine, and no host heap.  The
 * pages describe no such variant; it has no counterpart there.
 *
 * Scratch: one fixed device array inside the library (4,466,432 bytes, held
 * by every GPU that loads the library until the process exits), large enough
 * for OPT_NOALLOC_MAX_TENSORS tensors and OPT_NOALLOC_MAX_CHUNKS chunks of
 * the norm's table (about 8.6e9 elements at OPT_CHUNK_ELEMS per chunk).
 * Larger lists are rejected with OPT_ELIMIT before any GPU work.
 *
 * Inputs: n tensors; numel, grad (device pointers, 16-byte aligned) and
 * grad_dtype (OPT_F32 or OPT_BF16) are HOST arrays, copied into the scratch
 * array on `stream` by cudaMemcpyAsync.  Ordinary (pageable) host arrays may
 * be reused as soon as the call returns; page-locked ones must stay
 * unchanged until `stream` has reached this call.
 * d_out: device, 8-byte aligned, 48 bytes.  Returns OPT_OK or an error
 * status; the norm's own status (OPT_ENONFINITE) is in d_out->status.
 *
 * The first call on each device looks up the scratch array's device address
 * (with that device current) and caches it; make that first call before any
 * stream capture.  Every call shares the one array: calls whose device work
 * overlaps (on two streams, or from two host threads) race and must be
 * serialised by the caller.  Each call overwrites every part of the array it
 * reads, except a completion counter that every call returns to 0, so
 * nothing carries over from an earlier call. */
#define OPT_NOALLOC_MAX_TENSORS 8192
#define OPT_NOALLOC_MAX_CHUNKS 262144
int opt_grad_norm_noalloc(int32_t n, const int64_t* numel, const void* const* grad,
                          const int32_t* grad_dtype, double max_norm,
                          opt_norm_result* d_out, void* stream);

/* ---- host-only helpers (no GPU needed) ----------------------------------- */

/* The norm's chunks.  A gradient-dtype bucket of E elements is cut into
 * chunks of OPT_NORM_CHUNK_MIN elements when E < 2^28, 2 OPT_NORM_CHUNK_MIN
 * when E < 2^29, 4 OPT_NORM_CHUNK_MIN when E < 2^31, OPT_CHUNK_ELEMS
 * otherwise -- doubled while any of the
 * bucket's OPT_NORM_SLOTS slots would own more than OPT_NORM_MAX_PART chunks
 * (slot s owns chunks s, s + OPT_NORM_SLOTS, ...).  A small list then gives
 * every slot's warps many chunks to share, a large one fewer per-chunk costs.
 * The size depends on the sizes alone, so the result stays bit-identical run
 * to run; a bucket whose tensors alone exceed the bound (more than
 * OPT_NORM_SLOTS * OPT_NORM_MAX_PART of them) returns OPT_ELIMIT. */
#define OPT_NORM_CHUNK_MIN 4096
#define OPT_CHUNK_ELEMS 32768
/* Fixed partial-sum slots per gradient-dtype bucket: one CTA of 24 warps each
 * (one per SM of a GB300). */
#define OPT_NORM_SLOTS 152
#define OPT_NORM_MAX_PART 4096

typedef struct opt_chunk {
  uint32_t tensor;   /* index into the list */
  uint32_t len;      /* 1..chunk size of its bucket */
  int64_t start;     /* element offset in the tensor, a multiple of that size */
} opt_chunk;

/* Chunk size of gradient-dtype bucket `bucket` (0: FP32 gradients, 1: BF16)
 * of a list, by the rule above; a positive power of two, or a negative
 * status. */
int64_t opt_norm_chunk_elems(int32_t n, const int64_t* numel, const int32_t* grad_dtype, int32_t bucket);

/* The norm's chunk table, from sizes and gradient dtypes only: bucket 0
 * (FP32 grads) first, then bucket 1 (BF16 grads), each in chunks of its
 * opt_norm_chunk_elems; within a bucket, tensors in list order and chunks in
 * element order.  Writes up to `cap` entries to `out` (may be NULL to count)
 * and the bucket boundaries to bucket_begin[0..2] (chunks of bucket b are
 * [bucket_begin[b], bucket_begin[b+1])).  Returns the chunk count, or a
 * negative status. */
int64_t opt_chunk_table(int32_t n, const int64_t* numel, const int32_t* grad_dtype,
                        opt_chunk* out, int64_t cap, int64_t bucket_begin[3]);

/* Per-step scalars, formed in double and rounded once to fp32.  Returns
 * OPT_EINVAL for step < 1 or hyperparameters outside the ranges
 * torch.optim.AdamW accepts (0 <= beta1, beta2 < 1; 0 <= beta3 <= 1;
 * lr, eps, weight_decay >= 0; all finite).  Every step entry point applies
 * the same check before any launch. */
typedef struct opt_step_scalars {
  float lr, decay;            /* decay = 1 - lr wd */
  float beta1, omb1;          /* omb = 1 - beta */
  float beta2, omb2;
  float beta3, omb3;
  float alpha, eps;
  float inv_bc1, inv_bc2;     /* 1 / (1 - beta^t) */
} opt_step_scalars;
int opt_step_scalars_compute(const opt_hparams* hp, int64_t step, opt_step_scalars* out);

/* Combine per-rank norm results (each rank's opt_grad_norm over its own
 * shard) in rank order: fp64 sum of sumsq in index order, max of norm_inf,
 * sum of counts; then norm2, clip_coef and status as opt_grad_norm defines
 * them.  Deterministic for a fixed rank order ("perf(training): fused
 * multi-tensor gradient-norm reduction", 'Correctness properties': the
 * caller owns the cross-rank scalar reduction). */
int opt_norm_combine(const opt_norm_result* parts, int32_t n, double max_norm,
                     opt_norm_result* out);

#ifdef __cplusplus
}
#endif
#endif /* PS_OPT_H */
