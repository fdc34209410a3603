/*
 * lamb.h -- C ABI of the GB300 (sm_103a) LAMB optimizer-step library.
 *
 * One call of lamb_step() performs one LAMB optimizer step on one
 * data-parallel rank's ZeRO-2 shard of optimizer state, on one GPU.
 *
 * The method.  LAMB (You, Li, Reddi et al., "Large Batch Optimization for
 * Deep Learning: Training BERT in 76 minutes", ICLR 2020) is Adam with a
 * per-tensor ("layer-wise") trust ratio.  MegaScale adopts it so the batch can
 * grow 4x without losing accuracy ("MegaScale: Scaling Large Language Model
 * Training to More Than 10,000 GPUs", guided-reading digest, section 2: the
 * step size is scaled tensor by tensor through a trust ratio; the same
 * digest's section 8, Table 3, credits it with +3.0 MFU points).  The state
 * it updates is the rank's ZeRO-2 shard (digest section 3, "Data parallelism
 * (ZeRO-2 style)", and the "Terms" entry for ZeRO-2: optimizer state and
 * gradients sharded over the data-parallel ranks).  For tensor i with n_i
 * elements, at step t:
 *
 *   per element   g' = c * g / S                       (S: loss scale)
 *                 m  = b1 m + (1 - b1) g'
 *                 v  = b2 v + (1 - b2) g'^2
 *                 r  = (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps) + wd_i w
 *   per tensor    trust_i = ||w|| / ||r||, or 1 if either norm is 0
 *                 (||w|| over the weights before the update)
 *                 w  = w - lr * trust_i * r ;   w16 = bf16_round_nearest_even(w)
 *   global        G = ||g / S|| over every tensor of the shard (the reported
 *                 grad norm, before clipping); c = clip / G if clip > 0 and
 *                 G > clip, else 1; any inf/NaN grad skips the whole step.
 *
 * Memory.  Every state and grad buffer lives in device memory, is allocated
 * and owned by the caller (for example as torch tensors) and must stay valid
 * for the life of the handle (state) or until lamb_step returns (grads).  The
 * handle owns only its work table and a small device scratch area (one fp64
 * per work item or per CTA of one kernel's grid, whichever is more, one fp64
 * pair per work item, a few words per tensor, a few scalars) plus
 * a small pinned host area; lamb_destroy frees them.
 *
 * Threads and streams.  A handle is bound to the device that was current at
 * lamb_create and to the stream given there; every call enqueues its work on
 * that stream.  A handle must not be used from two host threads at once.
 *
 * Errors.  Every int-returning call returns LAMB_OK (0) or a negative code;
 * lamb_last_error() then gives a message for the calling thread.
 */
#ifndef LAMB_GB300_H
#define LAMB_GB300_H

#include <stdint.h>

#if defined(__GNUC__)
#define LAMB_API __attribute__((visibility("default")))
#else
#define LAMB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define LAMB_OK 0
#define LAMB_ERR_INVALID (-1) /* bad argument: NULL, negative size, t < 1, ... */
#define LAMB_ERR_ALIGN (-2)   /* a device pointer is not 16-byte aligned */
#define LAMB_ERR_CUDA (-3)    /* a CUDA runtime call or a kernel launch failed */
#define LAMB_ERR_NOMEM (-4)   /* device or pinned host allocation failed */
#define LAMB_NOT_READY 1      /* lamb_step_result without waiting: not finished yet */

/* Grad element types (all grads of one handle have the same type). */
#define LAMB_GRAD_BF16 0
#define LAMB_GRAD_FP16 1

typedef struct lamb_handle lamb_handle;

/* Hyperparameters fixed for the life of a handle.
 *   beta1, beta2  moment decay rates, each in [0, 1)
 *   eps           added to sqrt of the corrected second moment, >= 0
 *   weight_decay  wd applied to tensors whose wd flag is 1, >= 0
 *   grad_dtype    LAMB_GRAD_BF16 or LAMB_GRAD_FP16 */
typedef struct {
  float beta1;
  float beta2;
  float eps;
  float weight_decay;
  int32_t grad_dtype;
} lamb_hparams;

/* Outcome of one step.
 *   skipped          1 if some grad was inf or NaN; the step then wrote
 *                    nothing (w, m, v and w16 are bit-identical to before) and
 *                    the step number did not advance; 0 otherwise
 *   grad_norm        ||g / S|| over the whole shard, before clipping; +inf
 *                    when skipped
 *   loss_scale       the S this step divided the grads by
 *   next_loss_scale  the S the next step will use: with a dynamic loss scaler
 *                    (lamb_set_loss_scaler) the scale the next backward pass
 *                    must multiply the loss by; otherwise equal to loss_scale
 *   t                the step number this step used for its bias corrections */
typedef struct {
  int32_t skipped;
  int32_t reserved;
  double grad_norm;
  float loss_scale;
  float next_loss_scale;
  int64_t t;
} lamb_result;

/* Dynamic loss scaling, kept on the GPU (see lamb_set_loss_scaler).
 *   init_scale       S of the first step after enabling (finite, > 0)
 *   growth_factor    S *= growth_factor after growth_interval clean steps in a
 *                    row (>= 1; a product that is not finite is dropped)
 *   backoff_factor   S *= backoff_factor after a skipped step (in (0, 1])
 *   growth_interval  clean steps in a row before S grows (>= 1)
 *   min_scale, max_scale  S never goes below min_scale after a backoff nor
 *                    above max_scale after a growth (0 <= min <= init <= max;
 *                    max may be +inf) */
typedef struct {
  float init_scale;
  float growth_factor;
  float backoff_factor;
  int32_t growth_interval;
  float min_scale;
  float max_scale;
} lamb_loss_scaler;

/* One entry of the multi-tensor work table (see lamb_plan).
 *   tensor >= 0: elements [begin, begin + count) of that tensor;
 *   tensor == -1: a pack of whole small tensors, whose ids are
 *                 pack_ids[begin .. begin + count). */
typedef struct {
  int64_t begin;
  int32_t count;
  int32_t tensor;
} lamb_work_item;

/*
 * Create a handle over n_tensors tensors (n_tensors >= 0).
 *
 *   sizes[i]     element count of tensor i (>= 0; host array)
 *   wd_flags[i]  1 if tensor i takes weight decay, 0 if not (for example
 *                LayerNorm gains and biases); host array
 *   w[i], m[i], v[i]  device pointers to tensor i's fp32 master weights and
 *                first / second moments (updated in place by lamb_step)
 *   w_bf16[i]    device pointer to tensor i's bf16 weight copy (written by
 *                lamb_step)
 *   hp           hyperparameters (host struct, copied)
 *   stream       the cudaStream_t every call enqueues on (NULL: the legacy
 *                default stream)
 *
 * The four pointer arrays are host arrays of device pointers; each pointer of
 * a non-empty tensor must be non-NULL and 16-byte aligned (LAMB_ERR_ALIGN
 * otherwise).  The work table is built, uploaded and the call returns after
 * the uploads complete.  On success *out receives the handle.
 */
LAMB_API int lamb_create(lamb_handle** out, int32_t n_tensors, const int64_t* sizes,
                         const uint8_t* wd_flags, float* const* w, float* const* m,
                         float* const* v, uint16_t* const* w_bf16, const lamb_hparams* hp,
                         void* stream);

/*
 * Create a handle over one rank's shard of a data-parallel (ZeRO-2) group
 * whose shard boundaries may cut tensors.  ZeRO-2 gives each data-parallel
 * rank a contiguous slice of the flattened optimizer state (MegaScale
 * guided-reading digest, section 3, "Data parallelism (ZeRO-2 style)", and
 * the "Terms" entry for ZeRO-2), so the first and the last tensor of a shard
 * can be pieces of tensors that other ranks also hold.  LAMB's trust ratio
 * needs ||w|| and ||r|| of the whole tensor, and the clip factor and the skip
 * decision need the grad norm of the whole model, so such a group takes the
 * step in three phases with two exchanges between them (the split step,
 * lamb_split_norms / lamb_split_moments / lamb_split_apply below).
 *
 *   n_tensors ... w_bf16, hp, stream   as for lamb_create (the sizes are the
 *                 local pieces' element counts)
 *   exchange_slot  host array of n_tensors ints: -1 for a tensor this rank
 *                 holds whole, or k in [0, n_slots) for a piece of a tensor
 *                 shared with other ranks (each k given to at most one local
 *                 tensor; the ranks sharing a tensor use the same k).  May be
 *                 NULL when n_slots is 0.  Such tensors are never packed.
 *   norm_exchange  device pointer to 2 doubles, caller-owned, 8-byte aligned:
 *                 the grad-norm partials {sum of g^2 of the grads as given
 *                 (before dividing by S), inf/NaN count}, written by
 *                 lamb_split_norms, to be summed over the group in place
 *   tensor_exchange  device pointer to 2 * n_slots doubles, caller-owned,
 *                 8-byte aligned: {sum w^2, sum r^2} of slot k at [2k, 2k+1],
 *                 written by lamb_split_moments (entries of slots this rank
 *                 does not hold are left as they are: the caller zeroes them
 *                 before summing), to be summed over the group in place
 *
 * A handle made by lamb_create has neither buffer and cannot take split
 * steps.  One made here takes ordinary steps (lamb_step, lamb_step_async) only
 * while no tensor has an exchange slot; with one, they return
 * LAMB_ERR_INVALID, since a shared tensor's trust ratio needs the group's sums.
 */
LAMB_API int lamb_create_sharded(lamb_handle** out, int32_t n_tensors, const int64_t* sizes,
                                 const uint8_t* wd_flags, float* const* w, float* const* m,
                                 float* const* v, uint16_t* const* w_bf16,
                                 const int32_t* exchange_slot, int32_t n_slots,
                                 double* norm_exchange, double* tensor_exchange,
                                 const lamb_hparams* hp, void* stream);

/*
 * The split step, for a handle made by lamb_create_sharded.  Every call only
 * enqueues work on the handle's stream; between the calls the caller sums the
 * exchange buffers over the data-parallel group (for example with an
 * all-reduce on the same stream, or through host memory after waiting for
 * the stream), and every rank then continues with the same sums:
 *
 *   lamb_split_norms(h, grads, loss_scale)
 *       reads this shard's grads and writes norm_exchange = {sum g^2, 0 or
 *       1}.  loss_scale as for lamb_step (ignored while a dynamic loss scaler
 *       is on).                              -> sum norm_exchange over the group
 *   lamb_split_moments(h, lr, t, clip)
 *       forms the grad norm ||g / S||, the clip factor and the skip decision
 *       from the summed norm_exchange (a non-zero inf/NaN count skips the
 *       step on every rank), then updates m and v, finishes every whole
 *       tensor (its trust ratio; small whole tensors are also applied here,
 *       and on a shard of at most 8 waves of work items -- lamb_get_info's
 *       fused -- every whole tensor) and writes the {sum w^2, sum r^2} of
 *       each shared piece to its slot of tensor_exchange.  t >= 1 fixes the step number; 0 takes the GPU's
 *       counter (see lamb_step_async).          -> sum tensor_exchange over the group
 *   lamb_split_apply(h, &seq)
 *       forms the trust ratio of each shared tensor from its summed slot and
 *       applies the update and the bf16 copy (to the shared tensors, and to
 *       the whole ones lamb_split_moments has not applied); seq (may be
 *       NULL) receives the step's sequence number for lamb_step_result.
 *
 * The calls must come in this order (LAMB_ERR_INVALID otherwise, with nothing
 * enqueued).  In between, the handle refuses (LAMB_ERR_INVALID) every call
 * that would start another step or change what this one reads or copies:
 * lamb_step, lamb_step_async, lamb_set_step, lamb_set_loss_scaler,
 * lamb_set_speculative and lamb_snapshot_async.  The result of
 * a group of one rank, with no exchange at all, equals lamb_step's.
 */
LAMB_API int lamb_split_norms(lamb_handle* h, const void* const* grads, float loss_scale);
LAMB_API int lamb_split_moments(lamb_handle* h, float lr, int64_t t, float clip);
LAMB_API int lamb_split_apply(lamb_handle* h, int64_t* seq);

/*
 * One LAMB step.
 *
 *   grads       host array of n_tensors device pointers to this step's grads
 *               (grad_dtype elements, 16-byte aligned, read only)
 *   lr          learning rate (finite)
 *   t           step number, >= 1 (bias corrections use b1^t and b2^t)
 *   clip        global grad-norm clip threshold; <= 0 disables clipping
 *   loss_scale  S > 0 (finite); grads are divided by S (ignored while a
 *               dynamic loss scaler is on)
 *   out         receives {skipped, grad_norm, loss_scale, next_loss_scale}
 *
 * Enqueues the step's kernels on the handle's stream -- the grad-norm
 * kernel, then one persistent moments-and-apply kernel when the work table
 * holds at most 8 waves of items (lamb_get_info's fused), else the moments
 * and per-tensor norms kernel and the apply kernel; in speculative mode
 * (lamb_set_speculative) one kernel and the redo kernel -- and waits for the
 * outcome record, which the GPU writes into pinned host memory: the call
 * returns when the step has finished on the GPU.  The skip decision is taken
 * on the GPU; the host never reads it in the middle of a step.  Each step's grad-pointer set is matched against four
 * device slots, so alternating among up to four grad buffers costs no upload;
 * a new set is written by a small kernel, never by a copy (a copy could queue
 * behind unrelated bulk transfers on the copy engine).
 *
 * Errors: LAMB_ERR_INVALID and LAMB_ERR_ALIGN are found before anything is
 * enqueued, and the state is untouched.  LAMB_ERR_CUDA means that a launch, a
 * copy or the wait failed, or that a bounded wait on the GPU gave up (the
 * apply kernel's staged copies from HBM, or a tensor's trust ratio or the
 * step's scalars published by another CTA, never arrived); the state may
 * then be partly updated and should be restored from a snapshot.
 */
LAMB_API int lamb_step(lamb_handle* h, const void* const* grads, float lr, int64_t t, float clip,
                       float loss_scale, lamb_result* out);

/*
 * Asynchronous step: the same step as lamb_step, but the step number lives on
 * the GPU and the call returns as soon as the work is enqueued, so the host
 * never waits for the GPU between steps.
 *
 *   grads, lr, clip, loss_scale   as for lamb_step
 *   seq         receives the step's sequence number (may be NULL), which
 *               lamb_step_result takes
 *
 * The step number t is a counter on the GPU: the grad-norm kernel reads it,
 * forms the bias corrections 1/(1 - beta1^t) and 1/(1 - beta2^t) in fp64, and
 * advances it only if the step is not skipped, so the caller never has to
 * learn the skip decision before enqueueing the next step.  A new handle's
 * counter is 1; lamb_set_step sets it.  lamb_step (with an explicit t) also
 * leaves the counter at t + 1 after a clean step and at t after a skipped
 * one, so the two calls can be mixed.
 *
 * The outcome {skipped, grad_norm, loss_scale, next_loss_scale, t} is
 * written by the GPU into a slot of a pinned, device-mapped ring owned by the
 * handle; the last 64 steps' outcomes stay readable.  Grad buffers must stay
 * valid and unchanged until the step has finished on the GPU (for example
 * until the next work on the handle's stream that writes them).
 *
 * Errors: LAMB_ERR_INVALID and LAMB_ERR_ALIGN before anything is enqueued;
 * LAMB_ERR_CUDA if a launch fails.  A bounded wait on the GPU that gives up
 * (see lamb_step) is reported by lamb_step_result for that step.
 */
LAMB_API int lamb_step_async(lamb_handle* h, const void* const* grads, float lr, float clip,
                             float loss_scale, int64_t* seq);

/*
 * Outcome of a step enqueued by lamb_step_async (or lamb_step).
 *
 *   seq   the step's sequence number; one of the last 64 steps enqueued on
 *         the handle (older ones: LAMB_ERR_INVALID, their slot was reused)
 *   wait  != 0: block until the step has finished; 0: return LAMB_NOT_READY
 *         (a positive value) at once if it has not
 *   out   receives the outcome
 *
 * Returns LAMB_ERR_CUDA, with the state of that step undefined, if a bounded
 * wait on the GPU gave up during it (see lamb_step).
 */
LAMB_API int lamb_step_result(lamb_handle* h, int64_t seq, int32_t wait, lamb_result* out);

/* What a handle was built with (for accounting and tests).
 *   n_params         elements over all tensors
 *   one_pass_params  elements the moments kernel finishes in one pass (packed
 *                    small tensors and tensors of a single work item, unless
 *                    shared with other ranks): their update re-reads the
 *                    moments from cache, so they move 30 bytes per element
 *                    over HBM instead of 42
 *   chunk_elems      the chunk size of the work table
 *   n_items          work items in the table
 *   fused            1: an ordinary step runs the moments and apply passes as
 *                    one persistent kernel (chosen when the work table holds
 *                    at most 8 waves of items per resident CTA; the monitor
 *                    then reports the apply kernel's time as 0); 0: as two
 *                    kernels */
typedef struct {
  int64_t n_params;
  int64_t one_pass_params;
  int64_t chunk_elems;
  int64_t n_items;
  int32_t fused;
  int32_t speculative;  /* 1 while speculative mode is on (lamb_set_speculative) */
} lamb_info;
LAMB_API int lamb_get_info(lamb_handle* h, lamb_info* out);

/*
 * Speculative mode (opt-in): a second, caller-owned set of m and v buffers
 * lets a step read the grads once instead of twice.
 *
 *   m2[i], v2[i]  device pointers, n_i floats each, 16-byte aligned, distinct
 *                 from every m and v; both arrays NULL turns the mode off
 *
 * In this mode one persistent kernel reads g, m, v and w, sums the grad norm
 * on the way and writes the new m and v into the set the step did not start
 * from, computed as if the step were neither skipped nor clipped; once the
 * last moments item is done the grad norm is known, and the same kernel
 * applies the update from the written set: 40 bytes per parameter over HBM
 * instead of 42, and one kernel instead of two.  If the step turns out
 * clipped, a second kernel redoes it from the untouched set (62 bytes per
 * parameter for that step), so the mode pays only when clipping is rare or
 * off.  A skipped step leaves the state where it was.  Results equal an
 * ordinary step's bit for bit except the grad norm, which is summed in
 * another order (within the parity tolerance).
 *
 * After a step that is not skipped the state (the current m and v) lives in
 * the other set: lamb_state_buffers tells which.  lamb_snapshot_async copies
 * the current set (it waits for the handle's stream to learn which).
 * Turning the mode off (or switching to other buffers) first moves the state
 * back into m and v.  Split steps and tensors with exchange slots are not
 * supported in this mode (LAMB_ERR_INVALID).  The caller owns both sets.
 */
LAMB_API int lamb_set_speculative(lamb_handle* h, float* const* m2, float* const* v2);

/* Speculative mode: *which = 0 if the state is in m, v, 1 if it is in m2, v2
 * (waits for the handle's stream).  Always 0 when the mode is off. */
LAMB_API int lamb_state_buffers(lamb_handle* h, int32_t* which);

/* Sets the GPU's step counter (the t of the next lamb_step_async), t >= 1,
 * in stream order on the handle's stream. */
LAMB_API int lamb_set_step(lamb_handle* h, int64_t t);

/* Device address of the dynamic loss scale (one fp32 on the handle's device,
 * valid for the life of the handle): the scale the next step divides by while
 * a dynamic loss scaler is on, updated by each step's grad-norm kernel.  A
 * framework that never waits for lamb_step_result can read it on the GPU, in
 * order on the handle's stream, to scale the next loss. */
LAMB_API int lamb_loss_scale_device(lamb_handle* h, const float** scale);

/*
 * Turn dynamic loss scaling on (cfg non-NULL) or off (NULL).  While it is on,
 * lamb_step ignores its loss_scale argument: the scale lives on the GPU, each
 * step divides its grads by it, and the grad-norm kernel updates it right
 * after deciding whether the step is skipped -- backoff after a skipped step,
 * growth after growth_interval clean steps in a row -- with no host round
 * trip.  lamb_result reports the scale a step used and the next one, which
 * the next backward pass must use.  Enabling resets the scale to init_scale
 * and the clean-step count to 0.  The scale is fp32, as at the interface.
 */
LAMB_API int lamb_set_loss_scaler(lamb_handle* h, const lamb_loss_scaler* cfg);

/*
 * Snapshot of the optimizer state into host memory: the first stage of
 * MegaScale's two-stage checkpoint (guided-reading digest, section 6: a quick
 * device-to-host copy that pauses training only briefly, followed by a
 * background write from host memory to storage).
 *
 *   host_w, host_m, host_v  host arrays of n_tensors host pointers that
 *                receive each tensor's fp32 w, m and v (size n_i floats;
 *                page-locked memory makes the copies asynchronous)
 *   stream       the cudaStream_t the copies are enqueued on, normally one
 *                other than the handle's so that they overlap other work
 *
 * The copies start once everything already enqueued on the handle's stream
 * has finished, so they capture the state between two steps.  The call
 * returns at once.  The next lamb_step makes its state-writing kernels wait
 * for the copies on the GPU (its grad-norm kernel still overlaps them), so a
 * step never changes the state under a running snapshot; no host wait is
 * needed.  Several snapshots may be outstanding at once (on any streams):
 * the next step waits for all of them.  lamb_snapshot_wait blocks until every
 * outstanding copy is in host memory.
 */
LAMB_API int lamb_snapshot_async(lamb_handle* h, float* const* host_w, float* const* host_m,
                                 float* const* host_v, void* stream);
LAMB_API int lamb_snapshot_wait(lamb_handle* h);

/* Free everything the handle owns (after waiting for its stream).  NULL is a
 * no-op.  Caller-owned buffers are untouched. */
LAMB_API int lamb_destroy(lamb_handle* h);

/* Message for the last non-zero return on the calling thread ("" if none).
 * The pointer stays valid until the next call on this thread. */
LAMB_API const char* lamb_last_error(void);

/* Diagnostic: copy the per-tensor trust ratios of the last step that was not
 * skipped into host_out[0 .. n_tensors) (1.0 for empty tensors and before the
 * first step).  Waits for the handle's stream. */
LAMB_API int lamb_get_trust(lamb_handle* h, float* host_out, int32_t n_tensors);

/*
 * CUDA event monitor (after the per-rank CUDA-event timing of MegaScale's
 * guided-reading digest, section 7: critical segments are timed with CUDA
 * events instead of host timers, so timing forces no synchronisation and can
 * stay on).  With timing enabled, every step records four events on the
 * handle's stream, around its three phases; each of the last 64 steps keeps
 * its own events.  Events between kernels keep a kernel from launching while
 * the one before it drains, so a monitored step can be a little slower.
 *
 *   lamb_set_timing    enable != 0 turns the monitor on (creating the events),
 *                      0 turns it off
 *   lamb_step_kernel_times  ms[0..3) receive the device durations, in
 *                      milliseconds, of step seq's phases, waiting for them
 *                      if needed: the grad-norm kernel, the moments kernel
 *                      (or the fused moments-and-apply kernel), the apply
 *                      kernel (0 when fused); in speculative mode 0, the
 *                      one-pass kernel and the redo kernel
 *                      (LAMB_ERR_INVALID if that step was not timed or is
 *                      older than the last 64)
 *   lamb_kernel_times  the same for the last step enqueued
 */
LAMB_API int lamb_set_timing(lamb_handle* h, int32_t enable);
LAMB_API int lamb_step_kernel_times(lamb_handle* h, int64_t seq, float* ms);
LAMB_API int lamb_kernel_times(lamb_handle* h, float* ms);

/*
 * Host-only view of a work table like the one lamb_create builds (no GPU
 * needed).
 *
 * Tensors larger than small_max elements are split into chunks of at most
 * chunk_elems elements whose starts are multiples of 8 elements; tensors of
 * 1 .. small_max elements are packed whole, in order, into packs of at most
 * max(chunk_elems, small_max) elements and pack_max tensors; empty tensors
 * get no work.  Pack items come first, then the tensors of a single chunk,
 * then the chunks of the others, each tensor's chunks contiguous and each
 * group in tensor order.  lamb_create picks chunk_elems itself:
 * the fewest whole waves of one item per resident CTA of the GPU that keep
 * chunks at most 32768 elements, and the chunk size that fills them (never
 * below 2048).
 *
 *   chunk_elems             0 (= 32768) or a multiple of 256 in [2048, 2^30]
 *   items, items_cap        output array for the work items (may be NULL)
 *   pack_ids, pack_cap      output array for packed tensor ids (may be NULL)
 *   n_items, n_pack_ids     receive the full counts
 *
 * Returns LAMB_ERR_INVALID (with the counts still set) when a capacity is too
 * small for a non-NULL output array.
 */
LAMB_API int lamb_plan(int32_t n_tensors, const int64_t* sizes, int64_t chunk_elems,
                       lamb_work_item* items, int64_t items_cap, int32_t* pack_ids,
                       int64_t pack_cap, int64_t* n_items, int64_t* n_pack_ids);

/* The constants lamb_plan uses (any output may be NULL): the largest and the
 * smallest chunk size, the largest packed tensor, and tensors per pack. */
LAMB_API void lamb_plan_limits(int64_t* chunk_elems, int64_t* min_chunk_elems,
                               int64_t* small_max, int64_t* pack_max);

/*
 * Allocation-free grad-norm pass.  The pages have no counterpart of this
 * entry point: it exists for callers that cannot allocate device memory when
 * they need the check -- for example a framework whose caching allocator has
 * already reserved nearly all of HBM, so that a raw cudaMalloc behind its back
 * would fail or fragment its pool, or an out-of-memory recovery path that must
 * look for inf/NaN grads exactly when no memory is left.
 *
 * It computes what lamb_step's first kernel computes, for grads the caller
 * passes, without a handle:
 *   out[0] = ||g / S|| over all tensors (+inf if any grad is inf or NaN)
 *   out[1] = clip factor c = clip / out[0] if clip > 0 and out[0] > clip, else 1
 *            (0 when a grad is not finite)
 *   out[2] = 1.0 if any grad is inf or NaN, else 0.0
 *
 *   n_tensors   0 .. LAMB_NOALLOC_MAX_TENSORS; more is rejected with
 *               LAMB_ERR_INVALID and a message naming the limit
 *   sizes       host array of element counts (>= 0)
 *   grads       host array of device pointers (grad_dtype elements, 16-byte
 *               aligned; may be NULL for empty tensors)
 *   out         device pointer to 3 doubles (8-byte aligned), written by the
 *               kernel when the stream reaches it
 *   stream      cudaStream_t the work is enqueued on (NULL: legacy default)
 *
 * It allocates nothing: no cudaMalloc, no cudaFree, no pinned memory.  Its
 * scratch (tensor table, per-CTA partial sums, completion ticket) is one
 * fixed device array of LAMB_NOALLOC_SCRATCH_BYTES inside this library.  The
 * tensor table is written by small kernels whose launch arguments carry the
 * entries, so nothing is read from host memory after the call returns.
 *
 * First call on each device.  It looks up that array's device address, sizes
 * the grid and loads this entry point's kernels, with the device current.
 * Under CUDA's lazy module loading (the default) that first call is also
 * when the array and the kernels' code are placed in the device's memory, and
 * they stay there until the process exits; it can therefore fail for lack of
 * memory.  A caller that needs this entry point when memory is exhausted
 * (for example an out-of-memory recovery path) should make one call at
 * start-up, while memory is free (n_tensors = 0 is enough), and make that
 * first call before any stream capture.  Later calls take no device memory.
 *
 * Every call reuses the same array and clears its ticket and flag first, so
 * calls whose work overlaps on the GPU (on different streams or host threads
 * without ordering between them) race and give wrong results; calls in one
 * stream are ordered and safe.  The call returns once the work is enqueued.
 */
#define LAMB_NOALLOC_MAX_TENSORS 8192
#define LAMB_NOALLOC_SCRATCH_BYTES (256 + 1024 * 8 + LAMB_NOALLOC_MAX_TENSORS * 16)
LAMB_API int lamb_grad_norm_noalloc(int32_t n_tensors, const int64_t* sizes,
                                    const void* const* grads, int32_t grad_dtype,
                                    float loss_scale, float clip, double* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LAMB_GB300_H */
