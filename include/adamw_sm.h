/*
 * adamw_sm.h -- C ABI of the GB300 (sm_103a) AdamW optimizer-step library.
 *
 * One optimizer step of decoupled-weight-decay Adam with bias correction over
 * a list of parameter tensors, in one of these storage modes:
 *
 *   ADAMW_MODE_BF16_KAHAN  pure-bf16 AnyPrecisionAdamW with Kahan summation:
 *       bf16 param p, grad g, exp_avg m, exp_avg_sq v and compensation c.
 *       ("[pure bf16 training] w/ AnyPrecisionAdamW and Kahan summation",
 *       transformers PR #21312, "Train from scratch" run recipe: optim
 *       adamw_anyprecision, use_kahan_summation=true, bf16 momentum, variance
 *       and compensation buffers; memory breakdown "bf16 pure" = 10 B/param.)
 *
 *   ADAMW_MODE_MIXED_FP32_MASTER  the per-shard update of a distributed
 *       (ZeRO-style) Adam: fp32 master weights, fp32 m and v, bf16 grad in,
 *       bf16 param out.  ("Distributed optimizer support for BERT", NeMo PR
 *       #5305, "Usage": distributed_fused_adam; memory breakdown "bf16 mixed"
 *       of the transformers PR = 16 B/param.)
 *
 *   ADAMW_MODE_MIXED_BF16_REMAINDER  the same update with the fp32 master
 *       stored as the model's bf16 parameter plus a 16-bit remainder, so the
 *       sharded optimizer state is fp32 m, fp32 v and the remainder: 10 B/param
 *       ("2 FP32 optim state + 1 16-bit master param", memory estimate under
 *       the 4xA40 table of the NeMo PR).  bits(master) = (bits(p16) << 16) +
 *       r16 (r16 signed, integer addition): exact, so the trajectory equals
 *       ADAMW_MODE_MIXED_FP32_MASTER's; p16 is the master rounded to nearest,
 *       ties away from zero.
 *
 *   ADAMW_MODE_BF16_PLAIN  AnyPrecisionAdamW with use_kahan_summation=false:
 *       bf16 p, g, m, v, no compensation buffer (aux unused, may be NULL).
 *
 *   ADAMW_MODE_BF16_KAHAN_FP32_VAR  AnyPrecisionAdamW with bf16 momentum and
 *       compensation and variance_dtype=float32: bf16 p, g, m, c, fp32 v.
 *
 *   ADAMW_MODE_ANYPREC | flags  AnyPrecisionAdamW with every buffer type the
 *       recipe's optim_args name: momentum_dtype, variance_dtype and
 *       compensation_buffer_dtype each bfloat16 or float32, and
 *       use_kahan_summation on or off.  bf16 p and g; ADAMW_ANYPREC_M_FP32,
 *       ADAMW_ANYPREC_V_FP32 and ADAMW_ANYPREC_C_FP32 make exp_avg, exp_avg_sq
 *       and the compensation (aux) fp32, ADAMW_ANYPREC_NO_KAHAN drops the
 *       compensation (aux unused; C_FP32 is then invalid).  Twelve modes,
 *       16..27 less 28..31; 16, 18 and 24 are the same steps as
 *       ADAMW_MODE_BF16_KAHAN, ADAMW_MODE_BF16_KAHAN_FP32_VAR and
 *       ADAMW_MODE_BF16_PLAIN and run those modes' kernels.
 *
 * Arithmetic (identical in every mode up to storage; fp32, one IEEE
 * round-to-nearest per operation, no fused multiply-add):
 *   host, fp64 rounded once to fp32:  step_size = lr / (1 - beta1^t),
 *       sbc2 = sqrt(1 - beta2^t), omb1 = 1 - beta1, omb2 = 1 - beta2,
 *       lrwd = lr * weight_decay
 *   per element:  g *= coef (only when clipping)
 *       m' = beta1*m + omb1*g ;  v' = beta2*v + (omb2*g)*g
 *       (bf16 mode: m', v' rounded to bf16 and used as stored)
 *       den = sqrt(v')/sbc2 + eps ;  upd = step_size*(m'/den) + lrwd*p
 *   bf16 mode:  y = c - upd ; p' = bf16(p + y) ; c' = bf16(y - (p' - p))
 *   mixed mode: master' = master - upd ; p_out = bf16(master')
 *   remainder mode: master = join(p16, r16) ; master' = master - upd ;
 *       (p16', r16') = split(master')
 *   bf16 plain: p' = bf16(p - upd)
 *   bf16 Kahan fp32 variance: as bf16 mode with v' kept in fp32
 *   any precision: as bf16 mode (or bf16 plain without Kahan), each of
 *       m', v', c' rounded to its own storage type and used as stored
 *   clipping:   norm = sqrt(sum g^2) over every tensor of the plan;
 *       coef = min(1, max_grad_norm / (norm + 1e-6)); a non-finite gradient
 *       anywhere sets the non-finite flag and the step writes no state.
 * fp32 -> bf16 rounds to nearest even; subnormals are kept.
 *
 * Threading: a plan may be used from one host thread at a time, and steps on
 * one plan must not overlap on the GPU (they share the plan's workspace).
 * All entry points are asynchronous on the given stream unless stated.
 */
#ifndef ADAMW_SM_H
#define ADAMW_SM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* adamw_stream_t;

/* Storage modes. */
#define ADAMW_MODE_BF16_KAHAN 0
#define ADAMW_MODE_MIXED_FP32_MASTER 1
#define ADAMW_MODE_MIXED_BF16_REMAINDER 2
#define ADAMW_MODE_BF16_PLAIN 3
#define ADAMW_MODE_BF16_KAHAN_FP32_VAR 4
#define ADAMW_MODE_ANYPREC 16      /* | the ADAMW_ANYPREC_* flags below */
#define ADAMW_ANYPREC_M_FP32 1     /* exp_avg stored as fp32             */
#define ADAMW_ANYPREC_V_FP32 2     /* exp_avg_sq stored as fp32          */
#define ADAMW_ANYPREC_C_FP32 4     /* compensation (aux) stored as fp32  */
#define ADAMW_ANYPREC_NO_KAHAN 8   /* no compensation; aux unused        */

/* adamw_plan_create flags. */
#define ADAMW_PLAN_NORM 1     /* allocate the global-norm workspace (clipping)  */
#define ADAMW_PLAN_NO_FUSE 2  /* never run a clipped step as one fused launch   */

/* Status codes (0 = success, negative = error). */
#define ADAMW_OK 0
#define ADAMW_ERR_INVALID_ARG (-1) /* NULL or out-of-range argument       */
#define ADAMW_ERR_MISALIGNED (-2)  /* base not aligned to its element size */
#define ADAMW_ERR_CUDA (-3)        /* a CUDA call failed; see status string */
#define ADAMW_ERR_NO_NORM (-4)     /* clipping asked of a plan without norm */
#define ADAMW_ERR_TOO_LARGE (-5)   /* a size exceeds a documented limit     */
#define ADAMW_ERR_NOT_ACCESSIBLE (-6) /* a buffer the device cannot reach   */

/* One tensor of the list.  Every pointer is owned by the caller and must be
 * dereferenceable by the plan's device: device memory of that device, managed
 * memory, pinned host memory mapped at the same address (cudaHostAlloc under
 * unified addressing), or pageable host memory on devices with pageable-memory
 * access (Grace systems).  Host-resident buffers are read and written by the
 * kernels over the CPU-GPU link (NVLink-C2C on GB300): a gradient list kept in
 * pinned host memory needs no separate host-to-device copy.  The five buffers
 * of one tensor hold `numel` elements each and must not overlap one another
 * (different tensors may not overlap either).
 *              bf16 Kahan          | mixed fp32 master  | mixed remainder
 *   param      bf16 p (read/write) | fp32 master (r/w)  | bf16 p (r/w)
 *   grad       bf16 g (read)       | bf16 g (read)      | bf16 g (read)
 *   exp_avg    bf16 m (r/w)        | fp32 m (r/w)       | fp32 m (r/w)
 *   exp_avg_sq bf16 v (r/w)        | fp32 v (r/w)       | fp32 v (r/w)
 *   aux        bf16 Kahan c (r/w)  | bf16 p out (write) | int16 r (r/w)
 *              bf16 plain          | bf16 Kahan fp32 variance
 *   param      bf16 p (r/w)        | bf16 p (r/w)
 *   exp_avg    bf16 m (r/w)        | bf16 m (r/w)
 *   exp_avg_sq bf16 v (r/w)        | fp32 v (r/w)
 *   aux        unused (NULL ok)    | bf16 Kahan c (r/w)
 *              any precision (ADAMW_MODE_ANYPREC | flags)
 *   param      bf16 p (r/w)
 *   exp_avg    bf16 m, fp32 with ADAMW_ANYPREC_M_FP32 (r/w)
 *   exp_avg_sq bf16 v, fp32 with ADAMW_ANYPREC_V_FP32 (r/w)
 *   aux        bf16 Kahan c, fp32 with ADAMW_ANYPREC_C_FP32 (r/w);
 *              unused (NULL ok) with ADAMW_ANYPREC_NO_KAHAN
 * Element alignment is required (2 B for 16-bit, 4 B for fp32 buffers).  Tensors whose
 * five bases are all 16-byte aligned take the vectorised path; others are
 * still updated correctly, more slowly.  numel may be 0. */
typedef struct {
    void* param;
    const void* grad;
    void* exp_avg;
    void* exp_avg_sq;
    void* aux;
    int64_t numel;
} adamw_tensor_t;

/* Hyperparameters of one step.  beta1, beta2 in [0, 1); eps > 0; lr >= 0;
 * weight_decay >= 0; all finite.  max_grad_norm <= 0 disables clipping. */
typedef struct {
    float lr;
    float beta1;
    float beta2;
    float eps;
    float weight_decay;
    float max_grad_norm;
} adamw_hparams_t;

typedef struct adamw_plan* adamw_plan_t;

/* Facts about a plan, for callers that size launches or count bytes. */
typedef struct {
    int32_t mode;
    int32_t n_tensors;
    int64_t total_elems;   /* sum of numel                                  */
    int32_t grid;          /* CTAs of the update kernel                     */
    int32_t block;         /* threads per CTA                               */
    int64_t n_chunks;      /* pieces of tensors handed to CTAs              */
    int64_t scalar_elems;  /* elements on the unvectorised path             */
    int32_t device;        /* CUDA device the plan lives on                 */
    int32_t has_norm;      /* ADAMW_PLAN_NORM was given                     */
    int32_t norm_grid;     /* CTAs of the norm-partial kernel (0: no norm)  */
    int32_t fused;         /* clipped steps run as one fused launch         */
} adamw_plan_info_t;

/* One piece of a tensor assigned to one CTA (host-side view of the plan). */
typedef struct {
    int32_t tensor;  /* index into the tensor list                      */
    int32_t vec;     /* 1: 16-byte vector path, 0: element path          */
    int64_t offset;  /* first element, relative to the tensor's base     */
    int64_t len;     /* elements                                         */
    int32_t cta;     /* CTA that processes the piece; -1: claimed at run
                        time by whichever CTA runs out of its own first  */
    int32_t pad_;
} adamw_chunk_t;

/* Builds a plan on the current CUDA device: validates the list, splits the
 * flattened element space over a persistent grid (grid = SM count x resident
 * CTAs per SM, fewer for small lists), uploads the tensor table and the chunk
 * table, and (with ADAMW_PLAN_NORM) builds the norm kernel's own partition
 * and allocates the norm workspace.  With ADAMW_PLAN_NORM, a list whose
 * gradients take at most 32 MiB (16.7M parameters) runs its clipped steps as
 * one launch whose grid fits on the device at once: norm partials, a bounded
 * grid barrier, and the update reading g again (from L2 where it fits)
 * (unless ADAMW_PLAN_NO_FUSE; adamw_plan_info_t.fused says which).  Either
 * way the norm is the exact sum of squares up to fp64 rounding; the two
 * paths group the sum differently (different grids), so their norms may
 * differ in the last bits.
 * Synchronous (it allocates and copies).  host_table is read during the call
 * only.  On error *out is left NULL and nothing stays allocated.
 * Errors: INVALID_ARG (NULL out or table with n_tensors > 0, n_tensors < 0,
 * bad mode, numel < 0, NULL buffer with numel > 0), MISALIGNED,
 * NOT_ACCESSIBLE (a buffer the current device cannot dereference: another
 * device's memory, unmapped host memory), CUDA. */
int adamw_plan_create(const adamw_tensor_t* host_table, int32_t n_tensors,
                      int32_t mode, int32_t flags, adamw_plan_t* out);

/* One optimizer step over every tensor of the plan, asynchronous on stream.
 * step = t >= 1, the number of applied updates including this one (a step
 * skipped for a non-finite gradient does not count).
 * d_grad_norm (nullable, device fp64): receives the global gradient L2 norm.
 *   Clipping computes it anyway; without clipping a non-NULL d_grad_norm
 *   costs one extra read of every gradient (and needs ADAMW_PLAN_NORM).
 * d_nonfinite (device int32): receives 1 if any gradient element is inf or
 *   NaN, else 0.  Required when clipping (hp->max_grad_norm > 0): a 1 then
 *   means the step wrote nothing, and the caller must pass the same step
 *   next time.  Nullable without clipping; the state is then still updated
 *   (non-finite values propagate) and the flag only reports it.
 * Errors: INVALID_ARG (NULL plan/hp, step < 1, hyperparameter out of range,
 * clipping with d_nonfinite NULL), NO_NORM (clipping on a plan made without
 * ADAMW_PLAN_NORM), CUDA (launch failure).  An error return launches
 * nothing. */
int adamw_step(adamw_plan_t plan, const adamw_hparams_t* hp, int64_t step,
               double* d_grad_norm, int32_t* d_nonfinite,
               adamw_stream_t stream);

/* adamw_step_device flags. */
#define ADAMW_STEP_CLIP 1 /* clip by d_hp->max_grad_norm (needs ADAMW_PLAN_NORM) */
#define ADAMW_STEP_NORM 2 /* compute the norm into d_grad_norm, no clipping      */

/* adamw_step with every per-step input in device memory, so a sequence of
 * calls can be captured in a CUDA graph and replayed:
 * d_hp (device adamw_hparams_t) is read when the step runs (write a new lr
 * there between replays for a schedule); d_step (device int64) holds the
 * number of updates applied so far: the step uses t = *d_step + 1 and stores
 * t back unless it is skipped.  The step is skipped (nothing written, counter
 * unchanged) when ADAMW_STEP_CLIP is set and a gradient is non-finite, or when
 * the hyperparameters in d_hp are out of range (then *d_nonfinite = -1).
 * d_grad_norm, d_nonfinite: as in adamw_step.  The scalars are computed on
 * the device with the same fp64 operations as the host path, so results are
 * bit-identical to adamw_step with the same t.  Launches: one (every CTA
 * computes the scalars, the last one to finish advances the counter) when
 * neither clipping nor the norm is asked; otherwise the norm pass, a one-CTA
 * prologue and the update.
 * No host synchronisation and no allocation; all pointers are device-
 * accessible memory the caller owns (not checked here).
 * Errors: INVALID_ARG (NULL plan, d_hp or d_step, unknown flag), NO_NORM,
 * CUDA. */
int adamw_step_device(adamw_plan_t plan, const adamw_hparams_t* d_hp, int64_t* d_step,
                      int32_t flags, double* d_grad_norm, int32_t* d_nonfinite,
                      adamw_stream_t stream);

/* The run recipe's learning-rate schedule ("--lr_scheduler_type linear
 * --warmup_steps W", transformers PR #21312, "Train from scratch") for the
 * update `step` (>= 1) of a run of `total` updates: with k = step - 1,
 * base_lr * k / max(1, W) while k < W, then base_lr * max(0, (total - k) /
 * max(1, total - W)); fp64, rounded once to fp32.  The first update of a
 * warm-up therefore has lr 0.  Host-only; returns 0 for step < 1 or negative
 * W or total. */
float adamw_lr_linear_warmup(float base_lr, int64_t step, int64_t warmup, int64_t total);

/* The same schedule on the device, for the device-resident step: writes
 * d_hp->lr for the update *d_step + 1 (d_step as in adamw_step_device),
 * bit-identical to adamw_lr_linear_warmup.  One single-thread launch on
 * stream; capturable in a CUDA graph before adamw_step_device.
 * Errors: INVALID_ARG, CUDA. */
int adamw_lr_linear_warmup_device(adamw_hparams_t* d_hp, const int64_t* d_step, float base_lr,
                                  int64_t warmup, int64_t total, adamw_stream_t stream);

/* The global gradient L2 norm and non-finite flag of the plan's gradients,
 * without an update (the two-stage reduction the clipped step runs first).
 * d_grad_norm and d_nonfinite as in adamw_step (either may be NULL).
 * Errors: INVALID_ARG, NO_NORM, CUDA. */
int adamw_grad_norm(adamw_plan_t plan, double* d_grad_norm,
                    int32_t* d_nonfinite, adamw_stream_t stream);

/* Reads and clears the plan's device status word (synchronises the plan's
 * device first): 0, or a combination of
 *   1  a kernel of this plan gave up on a bounded wait (every device-side
 *      wait in this library is bounded, about a second; the launch then left
 *      its CTA's work undone, so the step is partly applied);
 *   2  (bounds-checked builds only, ADAMW_BUILD_CHECK_BOUNDS) a chunk of the
 *      plan fell outside its tensor's buffers and was skipped.
 * Clearing also realigns the fused step's barrier counter, so the plan is
 * usable again.  Errors: INVALID_ARG, CUDA. */
int adamw_plan_device_status(adamw_plan_t plan, int32_t* out);

/* For failure-path tests only: shifts the fused clipped step's grid-barrier
 * counter by `delta` (synchronous), so that in the next fused launch one
 * CTA's bounded barrier wait runs out and sets the device status.  Never
 * needed in normal use.  Errors: INVALID_ARG, CUDA. */
int adamw_plan_test_skew_barrier(adamw_plan_t plan, int64_t delta);

/* How the library was built: ADAMW_BUILD_CHECK_BOUNDS when every kernel
 * checks each chunk against its tensor's buffers before touching it (a
 * debugging build, compiled with -DADAMW_CHECK_BOUNDS=1), and
 * ADAMW_BUILD_BULK_STAGING when the bf16 Kahan update stages its inputs with
 * cp.async.bulk (-DADAMW_BULK=1). */
#define ADAMW_BUILD_CHECK_BOUNDS 1
#define ADAMW_BUILD_BULK_STAGING 2
int32_t adamw_build_flags(void);

/* For tests of the bounds-checked build only: lengthens update chunk `chunk`
 * of the plan by `delta` elements (synchronous), so that the next update
 * finds it outside its tensor, skips it and sets status bit 2.  Other builds
 * refuse (INVALID_ARG), as they do not check.  Errors: INVALID_ARG, CUDA. */
int adamw_plan_test_corrupt_chunk(adamw_plan_t plan, int64_t chunk, int64_t delta);

/* Releases the plan's device memory (synchronises the plan's device first).
 * NULL is accepted. */
int adamw_plan_destroy(adamw_plan_t plan);

/* Fills *out with facts about the plan.  Errors: INVALID_ARG. */
int adamw_plan_get_info(adamw_plan_t plan, adamw_plan_info_t* out);

/* Host-only (needs no GPU): the partition adamw_plan_create would build for
 * the given list on a grid of `grid` CTAs (the update kernel's grid is
 * adamw_plan_info_t.grid, the norm kernel's norm_grid).  Writes up to `cap` chunks to out
 * (out may be NULL when cap is 0) and the full count to *n_out.
 * Errors: INVALID_ARG, MISALIGNED, TOO_LARGE (cap smaller than the count;
 * *n_out still holds the count). */
int adamw_plan_chunks(const adamw_tensor_t* host_table, int32_t n_tensors,
                      int32_t mode, int32_t grid, adamw_chunk_t* out,
                      int64_t cap, int64_t* n_out);

/* Host-only: the five per-step fp32 scalars of step t, in the order
 * step_size, sbc2, omb1, omb2, lrwd.  Errors: INVALID_ARG. */
int adamw_step_scalars(const adamw_hparams_t* hp, int64_t step, float out5[5]);

/* One step over a tensor table the caller already holds in DEVICE memory
 * (d_table: n_tensors adamw_tensor_t entries, read during the call).  The
 * table is copied to the host, so unlike adamw_step this call BLOCKS the
 * host until `stream` has reached that copy (one device-to-host read of the
 * table per call); the step itself is then queued asynchronously.  The plan
 * built for the table is kept in a cache of up to 8 plans keyed by the
 * table's bytes, the mode and the current device, so passing the same table
 * every step builds the plan (and allocates) once.  Other arguments and
 * errors as adamw_plan_create and adamw_step (d_nonfinite is required when
 * clipping; cached plans carry the norm workspace, so clipping is always
 * available).  Thread-safe with respect to the cache; the buffers named by a
 * cached table must outlive its use. */
int adamw_step_table(const adamw_tensor_t* d_table, int32_t n_tensors, int32_t mode,
                     const adamw_hparams_t* hp, int64_t step, double* d_grad_norm,
                     int32_t* d_nonfinite, adamw_stream_t stream);

/* Destroys every plan adamw_step_table cached (synchronising their devices)
 * and returns how many there were. */
int adamw_step_table_cache_clear(void);

/* Measurement aid: copies `bytes` from src to dst (device pointers) with the
 * library's 16-byte-vector streaming copy kernel, asynchronously.  Used to
 * measure the HBM copy ceiling the update kernel is compared with.
 * bytes >= 0; both pointers 16-byte aligned and bytes a multiple of 16.
 * Errors: INVALID_ARG, MISALIGNED, CUDA. */
int adamw_copy_probe(void* dst, const void* src, int64_t bytes,
                     adamw_stream_t stream);

/* Largest tensor list adamw_grad_norm_noalloc accepts. */
#define ADAMW_NOALLOC_MAX_TENSORS 4096

/* The global gradient L2 norm and non-finite flag of a tensor list, like
 * adamw_grad_norm, for callers that cannot allocate device memory: code whose
 * device memory is all handed to a caching allocator (a raw cudaMalloc then
 * fails or fragments that pool), and code that must not synchronise the
 * device (cudaMalloc and cudaFree may).  It needs no plan (plan creation
 * allocates) and allocates nothing: its scratch is a fixed file-scope device
 * array of about 76 KiB in this library, which every GPU that loads the
 * library keeps until the process exits.  The source pages have no
 * counterpart; this is a utility of this library.
 * host_table: host array of n_tensors entries (pageable or pinned), read
 *   during the call only: the entries travel to the device as kernel launch
 *   parameters, which the runtime copies when the launch is made, so the
 *   array may be changed or freed as soon as the call returns.  Only .grad
 *   (device bf16, 2-byte aligned) and .numel are used.
 * d_grad_norm (nullable, device fp64) and d_nonfinite (nullable, device
 *   int32) receive the norm and the flag, as in adamw_grad_norm.
 * The first call on a device sets that device up (looks up the scratch
 * address and the grid size) with it current.  All calls share the one
 * scratch array, which keeps the last call's contents (nothing in it needs
 * to start at zero): calls that overlap on the GPU, on any streams, race.
 * The sum runs in a fixed order for a given device, but not the order of
 * adamw_grad_norm, so the two norms agree to fp64 rounding, not bit for bit.
 * Errors: INVALID_ARG (n_tensors < 0, NULL table or grad with numel > 0,
 * numel < 0), TOO_LARGE (n_tensors > ADAMW_NOALLOC_MAX_TENSORS, or a device
 * index of 64 or more), MISALIGNED (odd grad address), CUDA. */
int adamw_grad_norm_noalloc(const adamw_tensor_t* host_table, int32_t n_tensors,
                            double* d_grad_norm, int32_t* d_nonfinite,
                            adamw_stream_t stream);

/* Text for a status code; for ADAMW_ERR_CUDA it also names the last CUDA
 * error seen by this thread.  Never NULL; valid until the next call from the
 * same thread. */
const char* adamw_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* ADAMW_SM_H */
