/*
 * Reference ("oracle") implementation of one LAMB optimizer step on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library under optimizer_step_gb300/) never calls it and shares no code,
 * header, table or helper with it.
 *
 * What it computes (plain restatement, no blocking or fusion beyond the
 * method's own order):
 *
 *   LAMB -- You, Li, Reddi et al., "Large Batch Optimization for Deep Learning:
 *   Training BERT in 76 minutes" (ICLR 2020), the layer-wise adaptive Adam
 *   update -- as adopted by MegaScale ("MegaScale: Scaling Large Language Model
 *   Training to More Than 10,000 GPUs", guided-reading digest, section 2: the
 *   step size is scaled layer by layer, which is what lets the batch grow 4x).
 *   The step runs on one data-parallel rank's ZeRO-2 shard of optimizer state
 *   (same digest, section 3 "Data parallelism (ZeRO-2 style)" and the "Terms"
 *   entry for ZeRO-2): every tensor the rank owns is updated locally.
 *
 *   Order of operations, tensor by tensor:
 *     unscale      g^ = g / S                       (S = loss scale)
 *     finite check any g not finite -> skip (state untouched, grad_norm = +inf)
 *     global norm  G  = sqrt(sum over all tensors of g^^2)
 *     clip         c  = clip / G if (clip > 0 and G > clip) else 1
 *     moments      g' = c g^;  m = b1 m + (1-b1) g';  v = b2 v + (1-b2) g'^2
 *     bias corr.   m^ = m / (1 - b1^t);  v^ = v / (1 - b2^t)
 *     direction    r  = m^ / (sqrt(v^) + eps) + wd_i w
 *     trust        trust_i = ||w|| / ||r||, or 1 if either norm is 0
 *                  (||w|| of the weights before this step)
 *     update       w = w - lr trust_i r
 *     copy         w16 = bf16 round-to-nearest-even of the updated fp32 w
 *
 * Precision: every elementwise quantity is carried in fp64 from the fp32 /
 * bf16 / fp16 inputs and rounded once to fp32 when m, v and w are stored.
 * Norms accumulate in fp64.  Build without FMA contraction
 * (-ffp-contract=off) so the results do not depend on the host ISA.
 *
 * Parity pins (see tests/test_oracle_pins.py): closed forms at t=1 and at t=2
 * with dyadic betas, pure weight decay, zero-weight and zero-direction
 * tensors, scale invariance of the trust ratio, bit-exact power-of-two loss
 * scaling, clip equivalences, per-tensor independence, inf/NaN skip, and the
 * bf16/fp16 conversions against library routines.  The t=1 closed form, the
 * grad norm under active clipping, the power-of-two loss scale and the
 * inf/NaN skip are pinned again on tensors of more than one 65,536-element
 * block (the block-by-block path), with weight-decay flags mixed.
 */
#ifndef LAMB_ORACLE_H
#define LAMB_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Grad element encodings (bit patterns held in uint16_t). */
#define ORACLE_GRAD_BF16 0
#define ORACLE_GRAD_FP16 1

/*
 * One LAMB step over n_tensors tensors, in place.
 *
 *   sizes[i]        element count of tensor i (>= 0)
 *   wd_flags[i]     1: tensor i takes weight decay, 0: it does not
 *   w, m, v         fp32 state arrays, one per tensor (host memory)
 *   w16             bf16 copy of w written after the update (bit patterns)
 *   g               grads as bf16 or fp16 bit patterns (grad_dtype)
 *   update_mask     NULL = update every tensor; otherwise only tensors with
 *                   update_mask[i] != 0 are updated (the global grad norm is
 *                   still taken over all tensors, and the state pointers of
 *                   unmasked tensors may be NULL)
 *   n_threads       0 = all hardware threads
 *   skipped         out: 1 if any grad was inf/NaN (nothing written), else 0
 *   grad_norm       out: norm of the unscaled, pre-clip grads (+inf on skip)
 *   trust_out       optional out (n_tensors): trust ratio of each updated
 *                   tensor (left untouched for skipped steps / unmasked ones)
 *
 * Returns 0, or -1 on an invalid argument.
 */
int oracle_lamb_step(int32_t n_tensors, const int64_t* sizes, const uint8_t* wd_flags,
                     float* const* w, float* const* m, float* const* v,
                     uint16_t* const* w16, const uint16_t* const* g, int32_t grad_dtype,
                     double beta1, double beta2, double eps, double weight_decay,
                     double lr, int64_t t, double clip, double loss_scale,
                     const uint8_t* update_mask, int32_t n_threads,
                     int32_t* skipped, double* grad_norm, double* trust_out);

/*
 * Dynamic loss scaling between steps (the scale is fp32, as the loss scale
 * crosses the library's interface as fp32).  After a step that saw an inf or
 * NaN grad: scale *= backoff, clamped below at min_scale, and the count of
 * clean steps restarts.  After a clean step: the count grows by one, and when
 * it reaches growth_interval the scale is multiplied by growth (kept only if
 * the product is finite, clamped above at max_scale) and the count restarts.
 * Updates *scale and *good_steps in place.
 */
void oracle_loss_scale_update(float* scale, int32_t* good_steps, int32_t found_inf,
                              float growth, float backoff, int32_t growth_interval,
                              float min_scale, float max_scale);

/* Decode one bf16 / fp16 bit pattern to double (IEEE 754 binary16 and the
 * top half of binary32, written out from their definitions). */
double oracle_decode_grad(uint16_t bits, int32_t grad_dtype);

/* Round an fp32 value to bf16, round-to-nearest-even, NaN stays NaN. */
uint16_t oracle_bf16_rne(float x);

/* Bulk forms of the two conversions above (for tests). */
void oracle_decode_grad_n(const uint16_t* bits, int64_t n, int32_t grad_dtype, double* out);
void oracle_bf16_rne_n(const float* x, int64_t n, uint16_t* out);

#ifdef __cplusplus
}
#endif

#endif /* LAMB_ORACLE_H */
