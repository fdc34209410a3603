// The kernels of one LAMB step on sm_103a.
//
// LAMB (You et al., ICLR 2020) as adopted by MegaScale ("MegaScale: Scaling
// Large Language Model Training to More Than 10,000 GPUs", guided-reading
// digest, section 2: a step size scaled layer by layer through a trust ratio),
// on one rank's ZeRO-2 shard (digest section 3).  The step is purely memory-bound (about 25 flops,
// one sqrt and one divide per element against 42 bytes), so there is no
// tensor-core work here: what matters is coalesced 128-bit traffic, enough
// bytes in flight per SM, and no extra passes over HBM.
//
// The exact method needs three passes, because r needs the global clip factor
// and the update needs the whole tensor's ||r||:
//   A  grad_norm_kernel  reads g (2 B/elem): sum of g^2, inf/NaN flag, one
//      partial per CTA; its last CTA (atomic ticket, no waiting) publishes the
//      step: ||g/S||, the clip factor, the skip flag, t and the bias
//      corrections.
//   B  moments_kernel    reads g, m, v, w and writes m, v (22 B/elem); forms
//      per-tensor sum w^2 and sum r^2; the last CTA of each tensor (ticket)
//      turns them into trust_i.
//   C  apply_tma_kernel  reads m, v, w (staged through shared memory by TMA
//      bulk copies) and writes w and the bf16 copy (18 B/elem); r is
//      recomputed with the same function as in B, so the r applied is
//      bit-identical to the r whose norm was taken.
// On a shard of few waves of work items, B and C run as one persistent
// kernel (moments_kernel<DT, true, false>): apply items follow the moments
// items from the same counter and wait, bounded, for their tensor's trust
// ratio.  In the opt-in speculative mode (a second m/v buffer set) one kernel
// (spec_step_kernel) does A and B in one read of the inputs and then C, and a
// redo kernel repeats B and C for a step that turns out clipped.  In a split
// step (a ZeRO-2 group whose shards cut tensors) A only writes this shard's
// partials for the group to sum, finalize_kernel publishes the step from the
// sums, B writes each shared tensor's sum w^2 and sum r^2 for the group to
// sum, and exchange_trust_kernel turns those into trust ratios before C.
// Small tensors (packs) are finished inside B by the warp that owns them, and
// tensors of a single work item (at most one chunk) by the CTA that owns it,
// so they cost 30 B/elem instead of 42: the second pass over them hits cache.
// Recomputing r costs the same bytes as storing it (B +4 B write, C reads r
// instead of m and v), and avoids a 4 B/param scratch buffer.
//
// Work is split by the host-built table of work items (chunks of large
// tensors; packs of small tensors, a warp per tensor).  Grids are persistent
// (a few CTAs per SM): the grad-norm kernel's CTAs walk sub-items blockIdx.x,
// blockIdx.x + gridDim.x, ...; the other kernels take items greedily from an
// atomic counter, which balanced better on GB300, the moments pass from the
// table's start and the separate apply kernel from its end (so each starts
// where the other left data in L2).  Every reduction has a fixed order, so
// results are deterministic run to run.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lamb_internal.h"

namespace lambgb {
namespace {

// Launch shape.  The unroll factors are the 8-element vectors each thread has
// in flight per loop trip; the min-blocks values cap registers so that many
// CTAs stay resident per SM (bytes in flight, not instruction count, bound a
// streaming kernel).  They can be overridden at build time for tuning sweeps.
#ifndef LAMB_UNROLL_B
#define LAMB_UNROLL_B 1
#endif
#ifndef LAMB_MINBLOCKS_B
#define LAMB_MINBLOCKS_B 3
#endif
#ifndef LAMB_UNROLL_C
#define LAMB_UNROLL_C 1
#endif
#ifndef LAMB_MINBLOCKS_C
#define LAMB_MINBLOCKS_C 3
#endif
#ifndef LAMB_MINBLOCKS_A
#define LAMB_MINBLOCKS_A 4
#endif
// Resident CTAs per SM the persistent grids use (at most what fits): more
// concurrent streams per SM than this measured slower on GB300.
#ifndef LAMB_CTAS_PER_SM_A
#define LAMB_CTAS_PER_SM_A 3
#endif
#ifndef LAMB_CTAS_PER_SM_B
#define LAMB_CTAS_PER_SM_B 3
#endif
#ifndef LAMB_CTAS_PER_SM_C
#define LAMB_CTAS_PER_SM_C 4
#endif
// 1: the moments and apply kernels take work items from an atomic counter
// (greedy balance of ragged items); 0: static round-robin.  Results do not
// depend on it: every partial is stored per item and summed in item order.
#ifndef LAMB_DYNAMIC_BC
#define LAMB_DYNAMIC_BC 1
#endif
// 1: the apply kernel walks the work table from its end.  It then starts on
// the items the moments kernel finished last, whose m, v and w are still in
// L2, and ends on the first items, which the next step's moments kernel
// takes first.  Elements are independent, so results do not depend on it.
#ifndef LAMB_REVERSE_C
#define LAMB_REVERSE_C 1
#endif
// 1: the moments and apply kernels are launched as programmatic dependents
// of the kernel before them (PDL): their CTAs start while that kernel drains,
// take their first work item and prefetch its first bytes into L2, and only
// then wait (griddepcontrol.wait) for it to finish before reading what it
// wrote.  0: ordinary stream order.
#ifndef LAMB_PDL
#define LAMB_PDL 1
#endif
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Lets dependent grids launch (once every CTA of this grid has called it or
// exited); they still wait for this grid to finish before using its results.
__device__ __forceinline__ void pdl_trigger() {
#if LAMB_PDL
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}
// Waits until the grids this one depends on have finished and their memory
// writes are visible (returns at once when launched without a dependency).
__device__ __forceinline__ void pdl_wait() {
#if LAMB_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
// Hint: bring [p, p + bytes) into L2 (p 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  if (bytes) asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------------------ memory access
// Everything is streamed once per kernel and the step's footprint is far
// larger than L2.  LAMB_LD_POLICY / LAMB_ST_POLICY pick the cache policy of
// the 128-bit accesses: loads 0 evict-first (.cs), 1 default, 2 cache-global
// (.cg), 3 last-use (.lu), 4 default with a 256-byte L2 prefetch; stores 0
// evict-first (.cs), 1 default (write-back), 2 .cg.  On GB300 the evict-first
// loads measured about 2% slower than the others over the whole step; the
// 256-byte prefetch with write-back stores was the fastest on ragged shards.
#ifndef LAMB_LD_POLICY
#define LAMB_LD_POLICY 4
#endif
#ifndef LAMB_ST_POLICY
#define LAMB_ST_POLICY 1
#endif
template <class T>
__device__ __forceinline__ T ld_policy(const T* p) {
#if LAMB_LD_POLICY == 0
  return __ldcs(p);
#elif LAMB_LD_POLICY == 1
  return *p;
#elif LAMB_LD_POLICY == 2
  return __ldcg(p);
#elif LAMB_LD_POLICY == 3
  return __ldlu(p);
#else
  T r;
  static_assert(sizeof(T) == 16, "128-bit accesses only");
  uint32_t* q = reinterpret_cast<uint32_t*>(&r);
  asm volatile("ld.global.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3])
               : "l"(p));
  return r;
#endif
}
template <class T>
__device__ __forceinline__ void st_policy(T* p, T x) {
#if LAMB_ST_POLICY == 0
  __stcs(p, x);
#elif LAMB_ST_POLICY == 1
  *p = x;
#else
  __stcg(p, x);
#endif
}
__device__ __forceinline__ uint4 ld_u4(const void* p) {
  return ld_policy(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ float4 ld_f4(const float* p) {
  return ld_policy(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ void st_f4(float* p, float4 x) {
  st_policy(reinterpret_cast<float4*>(p), x);
}
__device__ __forceinline__ void st_u4(void* p, uint4 x) {
  st_policy(reinterpret_cast<uint4*>(p), x);
}

// ----------------------------------------------------------- grad decoding
// Two 16-bit grads packed in one 32-bit word -> two floats (exact).
template <int DT>
__device__ __forceinline__ float2 decode2(uint32_t x);
template <>
__device__ __forceinline__ float2 decode2<LAMB_GRAD_BF16>(uint32_t x) {
  return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
}
template <>
__device__ __forceinline__ float2 decode2<LAMB_GRAD_FP16>(uint32_t x) {
  return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(x & 0xFFFFu))),
                     __half2float(__ushort_as_half(static_cast<unsigned short>(x >> 16))));
}
template <int DT>
__device__ __forceinline__ float decode1(uint16_t x) {
  return decode2<DT>(uint32_t(x) | (uint32_t(x) << 16)).x;
}

// 1 if either 16-bit half of x has an all-ones exponent (inf or NaN).
template <int DT>
__device__ __forceinline__ uint32_t nonfinite2(uint32_t x) {
  constexpr uint32_t kExp = DT == LAMB_GRAD_BF16 ? 0x7F807F80u : 0x7C007C00u;
  const uint32_t u = ~x & kExp;  // a half is 0 here iff its exponent is all ones
  return uint32_t((u & 0xFFFFu) == 0u) | uint32_t((u >> 16) == 0u);
}

// Squares of grads.  A bf16 grad spans fp32's exponent range, so its square
// can underflow (|g| below about 1e-19) or, summed with others, overflow
// (|g| from about 1e18) in fp32.  Grads are squared in fp32 a few vectors at
// a time; a partial that is not in [2^-90, 2^120] (while some grad of it is
// not zero) is recomputed in fp64 on a separate, rare path.  Inside that
// range nothing overflowed, and squares that underflowed weigh at most
// 2^-30 of the partial.  fp16 squares are always normal fp32 numbers, so
// fp16 grads never take the fp64 path.  (Choosing per pair instead, with
// fp64 code inline, let the compiler predicate that code into every pair,
// which made the grad-norm kernel twelve times slower on GB300.)
// The fast path also leaves the inf/NaN test to the rare path: an inf or NaN
// grad makes its fp32 partial inf or NaN, which is never inside the range,
// so the words of such a partial are tested there, exactly.
template <int DT>
__device__ __forceinline__ bool partial_out_of_range(float acc, uint32_t any_bits) {
  if (!(acc <= 0x1p120f)) return true;  // overflow, inf or NaN
  return DT == LAMB_GRAD_BF16 && acc < 0x1p-90f && (any_bits & 0x7FFF7FFFu) != 0u;
}

// The squares of the eight grads in four words, in fp64, and their inf/NaN
// flag (the rare path; not inlined, and given the words by value, so that the
// fast path keeps its words in registers and carries no fp64 code).
struct SquaresFp64 {
  double sq;
  uint32_t bad;
};

template <int DT>
__device__ __noinline__ SquaresFp64 squares8_fp64(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  const uint32_t w[4] = {a, b, c, d};
  SquaresFp64 r{0.0, 0u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = decode2<DT>(w[i]);
    r.sq = fma(double(f.x), double(f.x), r.sq);
    r.sq = fma(double(f.y), double(f.y), r.sq);
    r.bad |= nonfinite2<DT>(w[i]);
  }
  return r;
}

// The same for the 4 * K words of a trip (K vectors); ORs the inf/NaN flag.
template <int DT, int K>
__device__ __forceinline__ double trip_squares_fp64(const uint32_t (&w)[4 * K], uint32_t& bad) {
  double t = 0.0;
#pragma unroll
  for (int u = 0; u < K; ++u) {
    const SquaresFp64 r = squares8_fp64<DT>(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
    t += r.sq;
    bad |= r.bad;
  }
  return t;
}

// -------------------------------------------------------------- reductions
__device__ __forceinline__ double warp_sum(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Fixed-shape block sum; the result is valid in every thread.
__device__ __forceinline__ double block_sum(double x, double* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  x = warp_sum(x);
  if (lane == 0) red[warp] = x;
  __syncthreads();
  double y = lane < kWarps ? red[lane] : 0.0;
  y = warp_sum(y);
  __syncthreads();
  return y;
}

__device__ __forceinline__ double2 block_sum2(double a, double b, double2* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_sum(a);
  b = warp_sum(b);
  if (lane == 0) red[warp] = make_double2(a, b);
  __syncthreads();
  double2 y = lane < kWarps ? red[lane] : make_double2(0.0, 0.0);
  y.x = warp_sum(y.x);
  y.y = warp_sum(y.y);
  __syncthreads();
  return y;
}

__device__ __forceinline__ float trust_of(double sum_w2, double sum_r2) {
  const double wn = sqrt(sum_w2), rn = sqrt(sum_r2);
  return (wn > 0.0 && rn > 0.0) ? float(wn / rn) : 1.0f;
}

// fp32 -> bf16 bit pattern, round to nearest even (CUDA's conversion).
__device__ __forceinline__ uint32_t bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// ------------------------------------------------------ per-element math
// Explicitly rounded operations (never contracted), so kernels B and C get
// bit-identical r from the same stored m, v and w.
struct Elem {
  float b1, b2, omb1, omb2, c1, c2, eps, gs;
  __device__ __forceinline__ void moments(float g, float& m, float& v) const {
    const float gp = __fmul_rn(g, gs);
    m = __fmaf_rn(b1, m, __fmul_rn(omb1, gp));
    v = __fmaf_rn(b2, v, __fmul_rn(omb2, __fmul_rn(gp, gp)));
  }
  __device__ __forceinline__ float direction(float m, float v, float w, float wd) const {
    const float den = __fadd_rn(__fsqrt_rn(__fmul_rn(v, c2)), eps);
    return __fmaf_rn(wd, w, __fdiv_rn(__fmul_rn(m, c1), den));
  }
};

__device__ __forceinline__ float4 get4(const float (&a)[8], int h) {
  return make_float4(a[4 * h], a[4 * h + 1], a[4 * h + 2], a[4 * h + 3]);
}
__device__ __forceinline__ void put4(float (&a)[8], int h, float4 x) {
  a[4 * h] = x.x;
  a[4 * h + 1] = x.y;
  a[4 * h + 2] = x.z;
  a[4 * h + 3] = x.w;
}

// ------------------------------------------------------- item scheduling
// Hands out work items to the CTAs of the moments and apply kernels: either
// greedily from an atomic counter (reset by the grad-norm kernel's last CTA
// before either kernel runs) or round-robin.  All threads of the CTA call
// next() together; it returns the same item to all of them, or a value
// >= n_items when the kernel's work is done.
struct ItemQueue {
  uint32_t* counter;
  int32_t n_items;
  int32_t* slot;  // shared memory
  int32_t rr;
  __device__ __forceinline__ int32_t next() {
#if LAMB_DYNAMIC_BC
    __syncthreads();  // everyone has read the previous item
    if (threadIdx.x == 0) *slot = int32_t(atomicAdd(counter, 1u));
    __syncthreads();
    return *slot;
#else
    const int32_t it = rr;
    rr += gridDim.x;
    return it;
#endif
  }
};

// ===================================================== A: grad norm pass
// Sum of raw g^2 and the inf/NaN flag over elements [0, n) of one grad array,
// thread tid of nthr, added to the thread's fp64 total.  Each thread has up to
// kLoadsA 16-byte loads in flight and sums at most 128 squares in fp32 before
// folding them into fp64 (a chunk gives each thread at most 16 vectors; a
// packed tensor of at most 4096 elements gives each lane at most 16).
#ifndef LAMB_LOADS_A
#define LAMB_LOADS_A 8
#endif
constexpr int kLoadsA = LAMB_LOADS_A;

template <int DT>
__device__ __forceinline__ void sumsq_range(const uint16_t* __restrict__ g, int64_t n, int tid,
                                            int nthr, double& total, uint32_t& bad) {
  const int64_t nv = n >> 3;
  for (int64_t k0 = tid; k0 < nv; k0 += int64_t(kLoadsA) * nthr) {
    uint32_t w[4 * kLoadsA];
#pragma unroll
    for (int u = 0; u < kLoadsA; ++u) {
      const int64_t k = k0 + int64_t(u) * nthr;
      const uint4 q = k < nv ? ld_u4(g + 8 * k) : make_uint4(0u, 0u, 0u, 0u);
      w[4 * u] = q.x;
      w[4 * u + 1] = q.y;
      w[4 * u + 2] = q.z;
      w[4 * u + 3] = q.w;
    }
    float acc = 0.0f;
    uint32_t any = 0;
#pragma unroll
    for (int j = 0; j < 4 * kLoadsA; ++j) {
      const float2 f = decode2<DT>(w[j]);
      acc = __fmaf_rn(f.x, f.x, acc);
      acc = __fmaf_rn(f.y, f.y, acc);
      if (DT == LAMB_GRAD_BF16) any |= w[j];
    }
    total += partial_out_of_range<DT>(acc, any) ? trip_squares_fp64<DT, kLoadsA>(w, bad)
                                                : double(acc);
  }
  for (int64_t j = (nv << 3) + tid; j < n; j += nthr) {  // fewer than 8: fp64 squares
    const uint16_t x = g[j];
    const double f = double(decode1<DT>(x));
    total = fma(f, f, total);
    bad |= nonfinite2<DT>(uint32_t(x) | (uint32_t(x) << 16));
  }
}

// The host's copy of a step's outcome, written by the step's publisher into
// its slot of the pinned, device-mapped result ring (the host cleared the
// slot when it enqueued the step; a bounded wait that gives up sets its
// error field).  Writing it one kernel later instead, off the publishing
// CTA's path, measured the same on GB300.
__device__ __forceinline__ void write_record(const StepScalars* sc, ResultRecord* slot) {
  volatile ResultRecord* r = slot;
  r->grad_norm = sc->grad_norm;
  r->t_used = sc->t_used;
  r->scale_used = sc->scale_used;
  r->scale_next = sc->scale_next;
  r->skipped = sc->skip;
}

// Publishes one step's scalars from the sum of raw g^2 over the shard (or the
// data-parallel group) and the inf/NaN flag: the grad norm ||g/S||, the clip
// factor, the skip flag, the step number t and its bias corrections (from
// beta^t in fp64, rounded once to fp32; t and beta^t advance only on a step
// that is not skipped), the dynamic loss scale, the host's copy of the
// outcome, and the item counters of the next step.
//
// Called by all 32 lanes of one warp with the same arguments; lane 0 writes
// and its return value (clipped) is the one to use.  fp64 is slow on GB300
// (a division takes about half a microsecond on one thread, and this runs on
// the step's critical path), so the five divisions run at once, one per lane,
// and there is no pow: ||g/S|| = sqrt(s)/S; the clipped grad factor
// c/S = (clip/||g/S||)/S, taken as clip/sqrt(s) (equal up to rounding); the
// unclipped one 1/S; and 1/(1-beta1^t), 1/(1-beta2^t).
__device__ bool publish_step(const DevTables& T, const NormArgs& na, const ScaleArgs& sa, double s,
                             bool nf, int lane) {
  StepScalars* sc = T.sc;
  const float S = sa.dynamic ? sc->scale : sa.fixed;
  const double loss_scale = double(S);
  const bool host_t = na.t_host > 0;
  const int64_t t = host_t ? na.t_host : sc->t_next;
  const double p1 = host_t ? na.p1_host : sc->p1_next;  // beta1^t
  const double p2 = host_t ? na.p2_host : sc->p2_next;  // beta2^t
  const double rs = sqrt(s);
  double num = 1.0, den = 1.0;
  if (lane == 0) {
    num = rs;
    den = loss_scale;
  } else if (lane == 1) {
    num = double(na.clip);
    den = rs;
  } else if (lane == 2) {
    den = loss_scale;
  } else if (lane == 3) {
    den = 1.0 - p1;
  } else if (lane == 4) {
    den = 1.0 - p2;
  }
  const double q = num / den;
  const double gn = __shfl_sync(0xffffffffu, q, 0);
  const double clip_gscale = __shfl_sync(0xffffffffu, q, 1);
  const double inv_scale = __shfl_sync(0xffffffffu, q, 2);
  const double c1 = __shfl_sync(0xffffffffu, q, 3);
  const double c2 = __shfl_sync(0xffffffffu, q, 4);
  if (lane != 0) return false;
  bool clipped = false;
  if (nf) {
    sc->skip = 1;
    sc->grad_norm = __longlong_as_double(0x7FF0000000000000ll);  // +inf
    sc->gscale = 0.0f;
  } else {
    clipped = na.clip > 0.0f && gn > double(na.clip);
    sc->skip = 0;
    sc->grad_norm = gn;
    sc->gscale = float(clipped ? clip_gscale : inv_scale);
  }
  sc->scale_used = S;
  sc->t_used = t;
  sc->c1 = float(c1);
  sc->c2 = float(c2);
  sc->t_next = nf ? t : t + 1;
  sc->p1_next = nf ? p1 : p1 * double(na.b1);
  sc->p2_next = nf ? p2 : p2 * double(na.b2);
  if (sa.dynamic) {
    // Loss scale for the next step: back off after an overflow, grow after
    // `interval` clean steps in a row (fp32 products, clamped).
    float next = S;
    if (nf) {
      next = __fmul_rn(S, sa.backoff);
      if (next < sa.min_scale) next = sa.min_scale;
      sc->good_steps = 0;
    } else if (++sc->good_steps == sa.interval) {
      const float grown = __fmul_rn(S, sa.growth);
      if (isfinite(grown)) next = grown > sa.max_scale ? sa.max_scale : grown;
      sc->good_steps = 0;
    }
    sc->scale = next;
  }
  sc->scale_next = sa.dynamic ? sc->scale : S;
  if (na.slot) write_record(sc, na.slot);
  sc->error = 0;  // no wait of this step has given up yet
  // Item counters of the next step's moments and apply kernels (the other
  // parity; this step's were reset one step ago, so this step's kernels can
  // take items before the kernel that publishes the step has finished).
  T.queue[1 - na.parity] = 0u;
  T.queue[3 - na.parity] = 0u;
  return clipped;
}

// Each chunk item is cut into na.split equal sub-items (8-element aligned)
// so that the grid's CTAs get nearly equal shares even when the work table
// holds only a wave or two of items; a pack item is one sub-item.  A CTA owns
// sub-items blockIdx.x, blockIdx.x + gridDim.x, ...; it stages up to kStageA
// of them at a time in shared memory (one thread per sub-item loads its item
// and grad pointer, so there is one dependent-load latency per batch, not per
// sub-item), then streams their whole 8-element vectors as one flat list:
// each thread takes vectors tid, tid + 256, ... with kLoadsA 16-byte loads
// in flight, across sub-item boundaries.  Each thread keeps one fp64 total
// (fp32 partial sums of at most 8 * kLoadsA squares folded in after every
// trip); one block reduction per CTA gives the CTA's partial, and the CTA
// that finishes last (atomic ticket, nobody waits) adds the gridDim.x
// partials in CTA order and publishes the step's scalars: the grad norm, the
// clip factor, the skip flag, the step number t and its bias corrections,
// the dynamic loss scale, and the host's copy of the outcome.
constexpr int kStageA = 32;  // one warp stages the sub-items and scans their lengths
static_assert(kStageA == 32, "the staging scan is one warp's shuffle scan");

template <int DT>
__global__ void __launch_bounds__(kThreads, LAMB_MINBLOCKS_A) grad_norm_kernel(DevTables T, NormArgs na,
                                                                               ScaleArgs sa) {
  __shared__ double red[kWarps];
  __shared__ int is_last;
  __shared__ const uint16_t* s_g[kStageA];  // first element of each staged sub-item
  __shared__ int32_t s_len[kStageA];        // its element count (0: none)
  __shared__ int32_t s_pack[kStageA];       // pack item index, or -1
  __shared__ int64_t s_vend[kStageA];       // inclusive prefix of whole-vector counts
  pdl_trigger();  // the moments kernel may launch and take its first items
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t bad = 0;
  double total = 0.0;
  const int32_t split = na.split;
  const int64_t n_sub = int64_t(T.n_items) * split;
  const int64_t stride = int64_t(kStageA) * gridDim.x;
  for (int64_t first = blockIdx.x; first < n_sub; first += stride) {
    if (threadIdx.x < kStageA) {
      const int64_t vi = first + int64_t(threadIdx.x) * gridDim.x;
      const uint16_t* g = nullptr;
      int32_t len = 0, pack = -1;
      if (vi < n_sub) {
        const int32_t it = int32_t(vi / split);
        const int32_t part = int32_t(vi - int64_t(it) * split);
        const lamb_work_item wi = T.items[it];
        if (wi.tensor >= 0) {
          const int64_t per = ((int64_t(wi.count) + split - 1) / split + 7) & ~int64_t(7);
          const int64_t b = int64_t(part) * per;
          const int64_t e = min(int64_t(wi.count), b + per);
          if (b < e) {
            g = static_cast<const uint16_t*>(T.grads[wi.tensor]) + wi.begin + b;
            len = int32_t(e - b);
          }
        } else if (part == 0) {
          pack = it;
        }
      }
      s_g[threadIdx.x] = g;
      s_len[threadIdx.x] = len;
      s_pack[threadIdx.x] = pack;
      // Inclusive prefix of whole vectors over the staged sub-items (warp 0).
      int64_t nv = len >> 3;
#pragma unroll
      for (int o = 1; o < kStageA; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, nv, o);
        if (lane >= o) nv += y;
      }
      s_vend[threadIdx.x] = nv;
    }
    __syncthreads();
    const int64_t nvec = s_vend[kStageA - 1];
    // The thread's current staged sub-item, kept in registers: its vectors
    // are [jbeg, jend) of the flat list and start at jg (a thread's vectors
    // only increase, so it only moves forward).
    int j = 0;
    int64_t jbeg = 0, jend = s_vend[0];
    const uint4* jg = reinterpret_cast<const uint4*>(s_g[0]);
    for (int64_t v0 = threadIdx.x; v0 < nvec; v0 += int64_t(kLoadsA) * kThreads) {
      uint32_t w[4 * kLoadsA];
#pragma unroll
      for (int u = 0; u < kLoadsA; ++u) {
        const int64_t v = v0 + int64_t(u) * kThreads;
        uint4 q = make_uint4(0u, 0u, 0u, 0u);
        if (v < nvec) {
          while (v >= jend) {
            ++j;
            jbeg = jend;
            jend = s_vend[j];
            jg = reinterpret_cast<const uint4*>(s_g[j]);
          }
          q = ld_policy(jg + (v - jbeg));
        }
        w[4 * u] = q.x;
        w[4 * u + 1] = q.y;
        w[4 * u + 2] = q.z;
        w[4 * u + 3] = q.w;
      }
      float acc = 0.0f;
      uint32_t any = 0;
#pragma unroll
      for (int h = 0; h < 4 * kLoadsA; ++h) {
        const float2 f = decode2<DT>(w[h]);
        acc = __fmaf_rn(f.x, f.x, acc);
        acc = __fmaf_rn(f.y, f.y, acc);
        if (DT == LAMB_GRAD_BF16) any |= w[h];
      }
      total += partial_out_of_range<DT>(acc, any) ? trip_squares_fp64<DT, kLoadsA>(w, bad)
                                                  : double(acc);
    }
    // The last (fewer than 8) elements of each staged sub-item: one thread
    // each, squares in fp64.
    if (threadIdx.x < kStageA) {
      const int32_t len = s_len[threadIdx.x];
      const uint16_t* g = s_g[threadIdx.x];
      for (int32_t e = len & ~7; e < len; ++e) {
        const uint16_t x = g[e];
        const double f = double(decode1<DT>(x));
        total = fma(f, f, total);
        bad |= nonfinite2<DT>(uint32_t(x) | (uint32_t(x) << 16));
      }
    }
    // Staged pack items: a warp per small tensor.
    for (int jj = 0; jj < kStageA; ++jj) {
      const int32_t it = s_pack[jj];
      if (it < 0) continue;
      const lamb_work_item wi = T.items[it];
      for (int k = warp; k < wi.count; k += kWarps) {
        const int32_t ti = T.pack_ids[wi.begin + k];
        sumsq_range<DT>(static_cast<const uint16_t*>(T.grads[ti]), T.td[ti].n, lane, 32, total,
                        bad);
      }
    }
    __syncthreads();  // the staging arrays are refilled next
  }
  const double cta_sum = block_sum(total, red);
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    T.item_g2[blockIdx.x] = cta_sum;
    if (bad) atomicOr(&T.sc->nonfinite, 1u);
    __threadfence();
    const uint32_t prev = atomicAdd(&T.sc->ticket, 1u);
    is_last = prev == gridDim.x - 1;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  double s = 0.0;
  for (int32_t i = threadIdx.x; i < int32_t(gridDim.x); i += kThreads) s += __ldcg(&T.item_g2[i]);
  s = block_sum(s, red);
  if (warp != 0) return;
  uint32_t nf = 0;
  if (lane == 0) {
    nf = atomicExch(&T.sc->nonfinite, 0u);
    T.sc->ticket = 0u;  // ready for the next step
  }
  nf = __shfl_sync(0xffffffffu, nf, 0);
  if (na.partial) {
    // Split step: this shard's partials go out to be summed over the group;
    // the finalize kernel publishes the step once they come back.
    if (lane == 0) {
      T.xn[0] = s;
      T.xn[1] = nf ? 1.0 : 0.0;
    }
  } else {
    publish_step(T, na, sa, s, nf != 0u, lane);
  }
}

// Split step: the group's summed {sum of raw g^2, inf/NaN count} -> the
// step's scalars, exactly as the grad-norm kernel's last CTA forms them.
__global__ void finalize_kernel(DevTables T, NormArgs na, ScaleArgs sa) {
  // A programmatic dependent of the kernel before it (the grad-norm kernel,
  // or the collective that summed the partials): wait for its writes.
  pdl_wait();
  // one warp (publish_step's lanes)
  publish_step(T, na, sa, T.xn[0], !(T.xn[1] == 0.0), int(threadIdx.x & 31));
}

// Split step: trust ratio of each tensor shared with other ranks, from the
// group's summed {sum w^2, sum r^2} of its exchange slot.
__global__ void exchange_trust_kernel(DevTables T) {
  const int32_t i = int32_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= T.n_tensors || T.sc->skip) return;
  const int32_t k = T.td[i].xslot;
  if (k >= 0) T.trust[i] = trust_of(T.xt[2 * k], T.xt[2 * k + 1]);
}

// ================================================ B: moments + norms pass
// Moments, direction and norms for elements [begin, begin + n) of one tensor:
// m and v are read from (mi, vi) and the new ones written to (mo, vo) (the
// same arrays except in speculative mode); thread tid of nthr takes 8-element
// vectors tid, tid + nthr, ...  With G2 it also sums the raw g^2 and the
// inf/NaN flag of the grads it reads (speculative mode's grad norm).
template <int DT, bool G2>
__device__ __forceinline__ void moments_range_io(const float* mi, const float* vi, float* mo,
                                                 float* vo, const float* __restrict__ w, float wd,
                                                 const uint16_t* __restrict__ g, int64_t begin,
                                                 int64_t n, int tid, int nthr, const Elem& e,
                                                 float& sw, float& sr, float& sg, double& sgd,
                                                 uint32_t& bad) {
  mi += begin;
  vi += begin;
  mo += begin;
  vo += begin;
  w += begin;
  g += begin;
  const int64_t nv = n >> 3;
  constexpr int kUnroll = LAMB_UNROLL_B;
  for (int64_t k0 = tid; k0 < nv; k0 += int64_t(kUnroll) * nthr) {
    uint4 gq[kUnroll];
    float mr[kUnroll][8], vr[kUnroll][8], wr[kUnroll][8];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t k = k0 + int64_t(u) * nthr;
      if (k < nv) {
        gq[u] = ld_u4(g + 8 * k);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          put4(mr[u], h, ld_f4(mi + 8 * k + 4 * h));
          put4(vr[u], h, ld_f4(vi + 8 * k + 4 * h));
          put4(wr[u], h, ld_f4(w + 8 * k + 4 * h));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t k = k0 + int64_t(u) * nthr;
      if (k < nv) {
        const uint32_t wv[4] = {gq[u].x, gq[u].y, gq[u].z, gq[u].w};
        float pv = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = decode2<DT>(wv[j]);
          if (G2) {
            pv = __fmaf_rn(f.x, f.x, pv);
            pv = __fmaf_rn(f.y, f.y, pv);
          }
          e.moments(f.x, mr[u][2 * j], vr[u][2 * j]);
          e.moments(f.y, mr[u][2 * j + 1], vr[u][2 * j + 1]);
        }
        if (G2) {  // this vector's squares: fp32, or fp64 when out of range
          if (partial_out_of_range<DT>(pv, wv[0] | wv[1] | wv[2] | wv[3])) {
            const SquaresFp64 r = squares8_fp64<DT>(wv[0], wv[1], wv[2], wv[3]);
            sgd += r.sq;
            bad |= r.bad;
          } else {
            sg = __fadd_rn(sg, pv);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float r = e.direction(mr[u][q], vr[u][q], wr[u][q], wd);
          sw = __fmaf_rn(wr[u][q], wr[u][q], sw);
          sr = __fmaf_rn(r, r, sr);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          st_f4(mo + 8 * k + 4 * h, get4(mr[u], h));
          st_f4(vo + 8 * k + 4 * h, get4(vr[u], h));
        }
      }
    }
  }
  for (int64_t j = (nv << 3) + tid; j < n; j += nthr) {
    float mj = mi[j], vj = vi[j];
    const float wj = w[j];
    const uint16_t x = g[j];
    const float f = decode1<DT>(x);
    if (G2) {  // fewer than 8: fp64 squares
      sgd = fma(double(f), double(f), sgd);
      bad |= nonfinite2<DT>(uint32_t(x) | (uint32_t(x) << 16));
    }
    e.moments(f, mj, vj);
    const float r = e.direction(mj, vj, wj, wd);
    sw = __fmaf_rn(wj, wj, sw);
    sr = __fmaf_rn(r, r, sr);
    mo[j] = mj;
    vo[j] = vj;
  }
}

// The same, in place on the tensor's m and v.
template <int DT>
__device__ __forceinline__ void moments_range(const TensorDesc& d, const uint16_t* __restrict__ g,
                                              int64_t begin, int64_t n, int tid, int nthr,
                                              const Elem& e, float& sw, float& sr) {
  float sg = 0.0f;
  double sgd = 0.0;
  uint32_t bad = 0;
  moments_range_io<DT, false>(d.m, d.v, d.m, d.v, d.w, d.wd, g, begin, n, tid, nthr, e, sw, sr,
                              sg, sgd, bad);
}

// Apply for elements [begin, begin + n) of one tensor (kernel C, and packed
// tensors in kernel B): w <- w - step * r, then the bf16 copy.
__device__ __forceinline__ void apply_range(const TensorDesc& d, int64_t begin, int64_t n, int tid,
                                            int nthr, const Elem& e, float step) {
  const float* __restrict__ m = d.m + begin;
  const float* __restrict__ v = d.v + begin;
  float* __restrict__ w = d.w + begin;
  uint16_t* __restrict__ w16 = d.w16 + begin;
  const float wd = d.wd;
  const int64_t nv = n >> 3;
  constexpr int kUnroll = LAMB_UNROLL_C;
  for (int64_t k0 = tid; k0 < nv; k0 += int64_t(kUnroll) * nthr) {
    float mr[kUnroll][8], vr[kUnroll][8], wr[kUnroll][8];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t k = k0 + int64_t(u) * nthr;
      if (k < nv) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          put4(mr[u], h, ld_f4(m + 8 * k + 4 * h));
          put4(vr[u], h, ld_f4(v + 8 * k + 4 * h));
          put4(wr[u], h, ld_f4(w + 8 * k + 4 * h));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t k = k0 + int64_t(u) * nthr;
      if (k < nv) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float r = e.direction(mr[u][q], vr[u][q], wr[u][q], wd);
          wr[u][q] = __fmaf_rn(-step, r, wr[u][q]);
        }
        uint32_t packed[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)  // element 2j in the low half (lower address)
          packed[j] = bf16_bits(wr[u][2 * j]) | (bf16_bits(wr[u][2 * j + 1]) << 16);
#pragma unroll
        for (int h = 0; h < 2; ++h) st_f4(w + 8 * k + 4 * h, get4(wr[u], h));
        st_u4(w16 + 8 * k, make_uint4(packed[0], packed[1], packed[2], packed[3]));
      }
    }
  }
  for (int64_t j = (nv << 3) + tid; j < n; j += nthr) {
    const float r = e.direction(m[j], v[j], w[j], wd);
    const float wn = __fmaf_rn(-step, r, w[j]);
    w[j] = wn;
    w16[j] = static_cast<uint16_t>(bf16_bits(wn));
  }
}

// The first bytes of a chunk item's g, m, v and w, prefetched into L2 by one
// thread while the kernel waits for the grad-norm kernel to finish.
constexpr int64_t kPrefetchElems = 4096;

template <int DT>
__device__ __forceinline__ void prefetch_item(const DevTables& T, int32_t it) {
  const lamb_work_item wi = T.items[it];
  if (wi.tensor < 0) return;
  const TensorDesc d = T.td[wi.tensor];
  const uint32_t n = uint32_t(min(int64_t(wi.count), kPrefetchElems) & ~int64_t(7));
  prefetch_l2(static_cast<const uint16_t*>(T.grads[wi.tensor]) + wi.begin, n * 2u);
  prefetch_l2(d.m + wi.begin, n * 4u);
  prefetch_l2(d.v + wi.begin, n * 4u);
  prefetch_l2(d.w + wi.begin, n * 4u);
}

// Waits (thread 0, bounded) until tensor i's trust ratio of this step is
// published, then lets the whole CTA go on; false if the wait gave up.
constexpr uint32_t kReadyPolls = 1u << 22;

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ bool wait_ready(const uint32_t* flag, uint32_t tag, int* shared_ok) {
  if (threadIdx.x == 0) {
    uint32_t polls = 0;
    bool ok = true;
    while (ld_acquire(flag) != tag) {
      if (++polls > kReadyPolls) {
        ok = false;
        break;
      }
      __nanosleep(100);
    }
    *shared_ok = ok ? 1 : 0;
  }
  __syncthreads();
  return *shared_ok != 0;
}

// B (and, when FUSED, C too).  Items [0, n_items) of the work table are
// moments items; with FUSED, virtual items [n_items, 2 n_items) are the apply
// items of the same table, taken from the same counter after every moments
// item has been handed out.  An apply item waits (bounded) until its tensor's
// trust ratio is published by the CTA that finished the tensor's last
// moments item; that CTA is running and never waits, so the wait ends.  CTAs
// that run out of moments items so start applying finished tensors while the
// last moments items drain, instead of idling until a second kernel starts.
//
// REDO (speculative mode only; launched after the speculative kernel, with
// FUSED): runs only when that step turned out clipped (not skipped).  It
// then reads m and v from the buffer set the step started from, which the
// speculative pass left untouched, and writes the clipped moments over the
// other set, which then holds the state; it uses the apply counters.
template <int DT, bool FUSED, bool REDO>
__global__ void __launch_bounds__(kThreads, LAMB_MINBLOCKS_B) moments_kernel(DevTables T, Hyper hp) {
  __shared__ double2 red[kWarps];
  __shared__ int is_last;
  __shared__ int32_t slot;
  __shared__ int ready_ok;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t n_virtual = FUSED ? 2 * T.n_items : T.n_items;
  // Before the wait: take the first item (this step's counter was reset one
  // step ago) and prefetch its first bytes; nothing the grad-norm kernel
  // writes is read here.
  ItemQueue q{&T.queue[REDO ? 2 + hp.parity : hp.parity], n_virtual, &slot, int32_t(blockIdx.x)};
  int32_t it = q.next();
  if (!REDO && threadIdx.x == 0 && it < T.n_items) prefetch_item<DT>(T, it);
  pdl_wait();
  pdl_trigger();  // the apply kernel may launch as this grid drains
  const StepScalars* sc = T.sc;
  if (sc->skip) return;
  if (REDO && sc->spec_ok) return;
  const int32_t src = REDO ? sc->src : 0;  // REDO: read set src, write the other
  const Elem e{hp.b1, hp.b2, hp.omb1, hp.omb2, sc->c1, sc->c2, hp.eps, sc->gscale};
  // This tensor's m, v to read and to write, and a descriptor whose m, v are
  // the written ones (for the update).
  auto io = [&](const TensorDesc& d, const float*& mi, const float*& vi, TensorDesc& dout) {
    dout = d;
    mi = d.m;
    vi = d.v;
    if (REDO) {
      mi = src ? d.m2 : d.m;
      vi = src ? d.v2 : d.v;
      dout.m = src ? d.m : d.m2;
      dout.v = src ? d.v : d.v2;
    }
  };
  for (; it < n_virtual; it = q.next()) {
    if (FUSED && it >= T.n_items) {
      // ---- an apply item of a tensor with several items
      const lamb_work_item wi = T.items[it - T.n_items];
      if (wi.tensor < 0) continue;  // packs were finished in their moments item
      const TensorDesc d0 = T.td[wi.tensor];
      if (d0.n_items == 1) continue;  // so were tensors of one item
      if (d0.xslot >= 0) continue;    // shared: applied after the group's exchange
      if (!wait_ready(&T.ready[wi.tensor], hp.tag, &ready_ok)) {
        if (threadIdx.x == 0) {
          atomicOr(reinterpret_cast<unsigned int*>(&T.sc->error), 1u);
          if (hp.slot) static_cast<volatile ResultRecord*>(hp.slot)->error = 1;
        }
        continue;
      }
      const float* mi;
      const float* vi;
      TensorDesc d;
      io(d0, mi, vi, d);
      const float step = __fmul_rn(hp.lr, __ldcg(&T.trust[wi.tensor]));
      apply_range(d, wi.begin, wi.count, threadIdx.x, kThreads, e, step);
      continue;
    }
    const lamb_work_item wi = T.items[it];
    if (wi.tensor >= 0) {
      const float* mi;
      const float* vi;
      TensorDesc d;
      io(T.td[wi.tensor], mi, vi, d);
      float sw = 0.0f, sr = 0.0f, sg = 0.0f;
      double sgd = 0.0;
      uint32_t bad = 0;
      moments_range_io<DT, false>(mi, vi, d.m, d.v, d.w, d.wd,
                                  static_cast<const uint16_t*>(T.grads[wi.tensor]), wi.begin,
                                  wi.count, threadIdx.x, kThreads, e, sw, sr, sg, sgd, bad);
      const double2 s = block_sum2(sw, sr, red);
      if (d.n_items == 1) {
        if (d.xslot >= 0) {  // shared with other ranks: out for summing
          if (threadIdx.x == 0) {
            T.xt[2 * d.xslot] = s.x;
            T.xt[2 * d.xslot + 1] = s.y;
          }
          continue;
        }
        // A tensor of one item is finished here, in one pass: every thread
        // re-reads only the elements it has just written or read itself (the
        // same thread-to-element map in both loops), so the update reads
        // cache, not HBM, and the apply pass skips the item.
        const float tr = trust_of(s.x, s.y);
        if (threadIdx.x == 0) T.trust[wi.tensor] = tr;
        apply_range(d, wi.begin, wi.count, threadIdx.x, kThreads, e, __fmul_rn(hp.lr, tr));
        continue;
      }
      if (threadIdx.x == 0) {
        T.item_wr[it] = s;
        __threadfence();
        const uint32_t prev = atomicAdd(&T.tensor_ticket[wi.tensor], 1u);
        is_last = prev == uint32_t(d.n_items - 1);
      }
      __syncthreads();
      if (is_last) {
        // Last chunk of this tensor: sum its chunks' partials in item order.
        __threadfence();
        double a = 0.0, b = 0.0;
#pragma unroll 8
        for (int32_t k = threadIdx.x; k < d.n_items; k += kThreads) {
          const double2 x = __ldcg(&T.item_wr[d.first_item + k]);
          a += x.x;
          b += x.y;
        }
        const double2 tot = block_sum2(a, b, red);
        if (threadIdx.x == 0) {
          if (d.xslot >= 0) {  // shared with other ranks: out for summing
            T.xt[2 * d.xslot] = tot.x;
            T.xt[2 * d.xslot + 1] = tot.y;
          } else {
            T.trust[wi.tensor] = trust_of(tot.x, tot.y);
            if (FUSED) {  // publish: the tensor's apply items may start
              __threadfence();
              st_release(&T.ready[wi.tensor], hp.tag);
            }
          }
          T.tensor_ticket[wi.tensor] = 0u;
        }
      }
    } else {
      // A packed small tensor belongs to one warp, which finishes it here:
      // moments and norms, trust, then the update.  Each lane re-reads only
      // the elements it has just written or read itself (same lane-to-element
      // map in both passes), so the second pass hits cache, not HBM, and needs
      // no synchronisation; the apply pass skips pack items.
      for (int k = warp; k < wi.count; k += kWarps) {
        const int32_t ti = T.pack_ids[wi.begin + k];
        const float* mi;
        const float* vi;
        TensorDesc d;
        io(T.td[ti], mi, vi, d);
        float sw = 0.0f, sr = 0.0f, sg = 0.0f;
        double sgd = 0.0;
        uint32_t bad = 0;
        moments_range_io<DT, false>(mi, vi, d.m, d.v, d.w, d.wd,
                                    static_cast<const uint16_t*>(T.grads[ti]), 0, d.n, lane, 32,
                                    e, sw, sr, sg, sgd, bad);
        const double a = warp_sum(double(sw)), b = warp_sum(double(sr));
        const float tr = trust_of(a, b);
        if (lane == 0) T.trust[ti] = tr;
        apply_range(d, 0, d.n, lane, 32, e, __fmul_rn(hp.lr, tr));
      }
    }
  }
#ifdef LAMB_TEST_APPLY_REPORTS_WAIT_ERROR
  // Test builds only: CTA 0 reports a given-up wait after finishing its work
  // normally (no wait actually runs out), so that the host's handling of the
  // error can be tested.
  if (FUSED && !REDO) {
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      atomicOr(reinterpret_cast<unsigned int*>(&T.sc->error), 1u);
      if (hp.slot) static_cast<volatile ResultRecord*>(hp.slot)->error = 1;
    }
  }
#endif
}

// ============================ speculative mode: the grad-norm pass folded in
// One persistent grid per step, for a handle with a second set of m and v
// buffers.  Items [0, n_items) are moments items: each reads g, m, v and w
// once, sums the raw g^2 and the inf/NaN flag on the way (what the grad-norm
// kernel reads g for), and writes m' and v' -- computed as if the step were
// neither skipped nor clipped -- to the set the step did not start from, so
// the state stays untouched until the step is known to stand.  The CTA that
// finishes the last moments item adds the per-item g^2 partials in item
// order, publishes the step (publish_step) and releases a flag; the apply
// items [n_items, 2 n_items) wait (bounded) for the flag and, if the step
// stands, apply the update from the written set, which then holds the state.
// A clipped step is redone by the REDO moments kernel launched after this
// one; a skipped step leaves the state where it was.  Apply items are handed
// out only after every moments item, and moments items never wait, so every
// wait ends.  Trust ratios, norms and moments use the same functions and the
// same item-ordered sums as an ordinary step, so a step that stands matches
// it bit for bit (the grad norm is summed in a different order).
template <int DT>
__global__ void __launch_bounds__(kThreads, LAMB_MINBLOCKS_B) spec_step_kernel(DevTables T, Hyper hp,
                                                                               NormArgs na,
                                                                               ScaleArgs sa) {
  __shared__ double2 red[kWarps];
  __shared__ double red1[kWarps];
  __shared__ double warp_g2[kWarps];
  __shared__ int is_last;
  __shared__ int is_final;
  __shared__ int32_t slot;
  __shared__ int ready_ok;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t n = T.n_items;
  StepScalars* sc = T.sc;
  ItemQueue q{&T.queue[hp.parity], 2 * n, &slot, int32_t(blockIdx.x)};
  bool have_state = false, have_apply = false, stands = false;
  Elem e{};
  int32_t src = 0;
  for (int32_t it = q.next(); it < 2 * n; it = q.next()) {
    if (it < n) {
      if (!have_state) {
        // The scalars that do not depend on the grad norm, read only after
        // taking a moments item: the step's publisher (which needs this
        // item finished first) advances them for the next step.
        const bool host_t = na.t_host > 0;
        const double p1 = host_t ? na.p1_host : sc->p1_next;
        const double p2 = host_t ? na.p2_host : sc->p2_next;
        const float S = sa.dynamic ? sc->scale : sa.fixed;
        e = Elem{hp.b1, hp.b2, hp.omb1, hp.omb2, float(1.0 / (1.0 - p1)),
                 float(1.0 / (1.0 - p2)), hp.eps, float(1.0 / double(S))};
        src = sc->cur;
        have_state = true;
      }
      const lamb_work_item wi = T.items[it];
      uint32_t bad = 0;
      double item_g2 = 0.0;
      if (wi.tensor >= 0) {
        const TensorDesc d = T.td[wi.tensor];
        float sw = 0.0f, sr = 0.0f, sg = 0.0f;
        double sgd = 0.0;
        moments_range_io<DT, true>(src ? d.m2 : d.m, src ? d.v2 : d.v, src ? d.m : d.m2,
                                   src ? d.v : d.v2, d.w, d.wd,
                                   static_cast<const uint16_t*>(T.grads[wi.tensor]), wi.begin,
                                   wi.count, threadIdx.x, kThreads, e, sw, sr, sg, sgd, bad);
        const double2 s = block_sum2(sw, sr, red);
        item_g2 = block_sum(double(sg) + sgd, red1);
        if (d.n_items == 1) {
          if (threadIdx.x == 0) T.trust_spec[wi.tensor] = trust_of(s.x, s.y);
        } else {
          if (threadIdx.x == 0) {
            T.item_wr[it] = s;
            __threadfence();
            const uint32_t prev = atomicAdd(&T.tensor_ticket[wi.tensor], 1u);
            is_last = prev == uint32_t(d.n_items - 1);
          }
          __syncthreads();
          if (is_last) {
            __threadfence();
            double a = 0.0, b = 0.0;
            for (int32_t k = threadIdx.x; k < d.n_items; k += kThreads) {
              const double2 x = __ldcg(&T.item_wr[d.first_item + k]);
              a += x.x;
              b += x.y;
            }
            const double2 tot = block_sum2(a, b, red);
            if (threadIdx.x == 0) {
              T.trust_spec[wi.tensor] = trust_of(tot.x, tot.y);
              T.tensor_ticket[wi.tensor] = 0u;
            }
          }
        }
      } else {
        // A pack: a warp per small tensor (moments, norms, trust; the update
        // waits for the apply items).  The pack's g^2 is summed per warp in
        // the warp's tensor order, then over the warps in warp order.
        double wg = 0.0;
        for (int k = warp; k < wi.count; k += kWarps) {
          const int32_t ti = T.pack_ids[wi.begin + k];
          const TensorDesc d = T.td[ti];
          float sw = 0.0f, sr = 0.0f, sg = 0.0f;
          double sgd = 0.0;
          moments_range_io<DT, true>(src ? d.m2 : d.m, src ? d.v2 : d.v, src ? d.m : d.m2,
                                     src ? d.v : d.v2, d.w, d.wd,
                                     static_cast<const uint16_t*>(T.grads[ti]), 0, d.n, lane, 32,
                                     e, sw, sr, sg, sgd, bad);
          const double a = warp_sum(double(sw)), b = warp_sum(double(sr));
          wg += warp_sum(double(sg) + sgd);
          if (lane == 0) T.trust_spec[ti] = trust_of(a, b);
        }
        if (lane == 0) warp_g2[warp] = wg;
        __syncthreads();
        if (threadIdx.x == 0) {
          double t = 0.0;
          for (int k = 0; k < kWarps; ++k) t += warp_g2[k];
          item_g2 = t;
        }
      }
      bad = __syncthreads_or(bad);
      // One more moments item done; the CTA that finishes the last one
      // publishes the step.
      if (threadIdx.x == 0) {
        T.item_g2[it] = item_g2;
        if (bad) atomicOr(&sc->nonfinite, 1u);
        __threadfence();
        const uint32_t prev = atomicAdd(&sc->items_done, 1u);
        is_final = prev == uint32_t(n - 1);
      }
      __syncthreads();
      if (is_final) {
        __threadfence();
        double g2 = 0.0;
        for (int32_t k = threadIdx.x; k < n; k += kThreads) g2 += __ldcg(&T.item_g2[k]);
        g2 = block_sum(g2, red1);
        if (warp == 0) {
          uint32_t nf = 0;
          if (lane == 0) {
            nf = atomicExch(&sc->nonfinite, 0u);
            sc->items_done = 0u;
          }
          nf = __shfl_sync(0xffffffffu, nf, 0);
          const int32_t cur = sc->cur;
          const bool clipped = publish_step(T, na, sa, g2, nf != 0u, lane);
          if (lane == 0) {
            sc->src = cur;
            sc->spec_ok = (!nf && !clipped) ? 1 : 0;
            sc->cur = nf ? cur : 1 - cur;
            __threadfence();
            st_release(&sc->published, hp.tag);
            if (na.slot) static_cast<volatile ResultRecord*>(na.slot)->state_buf = sc->cur;
          }
        }
      }
      continue;
    }
    // ---- an apply item: wait until the step is published
    if (!have_apply) {
      if (!wait_ready(&sc->published, hp.tag, &ready_ok)) {
        if (threadIdx.x == 0) {
          atomicOr(reinterpret_cast<unsigned int*>(&sc->error), 1u);
          if (hp.slot) static_cast<volatile ResultRecord*>(hp.slot)->error = 1;
        }
        break;
      }
      stands = __ldcg(&sc->spec_ok) != 0;
      src = __ldcg(&sc->src);
      e = Elem{hp.b1, hp.b2, hp.omb1, hp.omb2, __ldcg(&sc->c1), __ldcg(&sc->c2), hp.eps, 0.0f};
      have_apply = true;
    }
    if (!stands) continue;  // skipped (nothing to do) or clipped (the redo kernel's job)
    const lamb_work_item wi = T.items[it - n];
    // The step stands: its trust ratios become the last step's (lamb_get_trust).
    if (wi.tensor >= 0) {
      TensorDesc d = T.td[wi.tensor];
      d.m = src ? d.m : d.m2;  // the set this step wrote
      d.v = src ? d.v : d.v2;
      const float tr = __ldcg(&T.trust_spec[wi.tensor]);
      if (threadIdx.x == 0 && wi.begin == 0) T.trust[wi.tensor] = tr;
      apply_range(d, wi.begin, wi.count, threadIdx.x, kThreads, e, __fmul_rn(hp.lr, tr));
    } else {
      for (int k = warp; k < wi.count; k += kWarps) {
        const int32_t ti = T.pack_ids[wi.begin + k];
        TensorDesc d = T.td[ti];
        d.m = src ? d.m : d.m2;
        d.v = src ? d.v : d.v2;
        const float tr = __ldcg(&T.trust_spec[ti]);
        if (lane == 0) T.trust[ti] = tr;
        apply_range(d, 0, d.n, lane, 32, e, __fmul_rn(hp.lr, tr));
      }
    }
  }
}

// ========================================================= C: apply pass
// LAMB_TMA_C=1 (default): the TMA-staged apply kernel below; 0: this one.
#ifndef LAMB_TMA_C
#define LAMB_TMA_C 1
#endif
#if !LAMB_TMA_C
__global__ void __launch_bounds__(kThreads, LAMB_MINBLOCKS_C) apply_kernel(DevTables T, Hyper hp) {
  __shared__ int32_t slot;
  ItemQueue q{&T.queue[2 + hp.parity], T.n_items, &slot, int32_t(blockIdx.x)};
  int32_t it = q.next();  // before the wait: the counter was reset one step ago
  pdl_wait();
  const StepScalars* sc = T.sc;
  if (sc->skip) return;
  const Elem e{hp.b1, hp.b2, hp.omb1, hp.omb2, sc->c1, sc->c2, hp.eps, 0.0f};
  for (; it < T.n_items; it = q.next()) {
    const lamb_work_item wi = T.items[LAMB_REVERSE_C ? T.n_items - 1 - it : it];
    if (wi.tensor < 0) continue;  // packs were finished by the moments kernel
    const TensorDesc d = T.td[wi.tensor];
    if (d.n_items == 1 && d.xslot < 0) continue;  // so were tensors of one item
    if (hp.only_shared && d.xslot < 0) continue;  // the fused kernel applied it
    const float step = __fmul_rn(hp.lr, T.trust[wi.tensor]);
    apply_range(d, wi.begin, wi.count, threadIdx.x, kThreads, e, step);
  }
}
#endif

// ====================== C, TMA-staged: m, v, w through shared memory (default)
// Per item, pieces of kTmaPiece elements of m, v and w are bulk-copied
// (cp.async.bulk, one elected thread) into a ring of kTmaStages stages, each
// with an mbarrier that completes on the bytes arriving; all threads wait on
// it (bounded), apply from shared memory, and release the stage with
// __syncthreads before it is refilled.  Tails of fewer than 8 elements take
// the plain path.  4 stages of 24 KB (2 CTAs per SM) measured 0.7% faster
// than apply_kernel's 128-bit loads on GB300; deeper rings at 1 CTA per SM
// were much slower.  LAMB_TMA_C=0 builds the plain kernel instead.  If a
// wait gives up (only if copies never arrive), the CTA records an error in
// StepScalars, lets its copies in flight land (bounded) and leaves; the host
// reports the step as failed.
#if LAMB_TMA_C
constexpr int kTmaPiece = kThreads * 8;  // 2048 elements: 8 per thread
#ifndef LAMB_TMA_STAGES
#define LAMB_TMA_STAGES 4
#endif
constexpr int kTmaStages = LAMB_TMA_STAGES;
constexpr uint32_t kTmaPolls = 1u << 22;
constexpr size_t kTmaSmem = size_t(kTmaStages) * 3 * kTmaPiece * sizeof(float);

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Waits for the given phase parity; false after kTmaPolls polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kTmaPolls; ++i) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__global__ void __launch_bounds__(kThreads, LAMB_MINBLOCKS_C) apply_tma_kernel(DevTables T,
                                                                               Hyper hp) {
  extern __shared__ __align__(128) unsigned char tma_smem[];
  __shared__ __align__(8) uint64_t full[kTmaStages];
  __shared__ int32_t slot;
  float* stage_buf = reinterpret_cast<float*>(tma_smem);  // [stage][m|v|w][piece]
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTmaStages; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Before the wait: take the first item (the counter was reset one step ago).
  ItemQueue q{&T.queue[2 + hp.parity], T.n_items, &slot, int32_t(blockIdx.x)};
  int32_t it = q.next();  // its __syncthreads also publishes the mbarrier init
  pdl_wait();
  const StepScalars* sc = T.sc;
  if (sc->skip) return;
  const Elem e{hp.b1, hp.b2, hp.omb1, hp.omb2, sc->c1, sc->c2, hp.eps, 0.0f};
  uint32_t parity = 0;  // bit s: the phase to wait for on stage s
  bool ok = true;
  for (; it < T.n_items && ok; it = q.next()) {
    const lamb_work_item wi = T.items[LAMB_REVERSE_C ? T.n_items - 1 - it : it];
    if (wi.tensor < 0) continue;  // packs were finished by the moments kernel
    const TensorDesc d = T.td[wi.tensor];
    if (d.n_items == 1 && d.xslot < 0) continue;  // so were tensors of one item
    if (hp.only_shared && d.xslot < 0) continue;  // the fused kernel applied it
    const float step = __fmul_rn(hp.lr, T.trust[wi.tensor]);
    const int64_t body = (int64_t(wi.count) >> 3) << 3;  // elements in whole vectors
    const int npieces = int((body + kTmaPiece - 1) / kTmaPiece);
    auto issue = [&](int p) {
      const int s = p % kTmaStages;
      const int64_t at = int64_t(p) * kTmaPiece;
      const uint32_t n = uint32_t(min(int64_t(kTmaPiece), body - at));
      const uint32_t bytes = n * uint32_t(sizeof(float));
      float* base = stage_buf + size_t(s) * 3 * kTmaPiece;
      mbar_expect_tx(&full[s], 3u * bytes);
      bulk_g2s(base, d.m + wi.begin + at, bytes, &full[s]);
      bulk_g2s(base + kTmaPiece, d.v + wi.begin + at, bytes, &full[s]);
      bulk_g2s(base + 2 * kTmaPiece, d.w + wi.begin + at, bytes, &full[s]);
    };
    if (threadIdx.x == 0)
      for (int p = 0; p < npieces && p < kTmaStages; ++p) issue(p);
    for (int p = 0; p < npieces; ++p) {
      const int s = p % kTmaStages;
      const bool arrived = mbar_wait(&full[s], (parity >> s) & 1u);
      if (__syncthreads_or(!arrived)) {  // the same decision in every thread
        ok = false;
        if (threadIdx.x == 0) {
          atomicOr(reinterpret_cast<unsigned int*>(&T.sc->error), 1u);
          if (hp.slot) static_cast<volatile ResultRecord*>(hp.slot)->error = 1;
          // Let the copies still in flight (pieces p .. p+stages-1) land,
          // again bounded, before leaving.
          for (int r = p; r < npieces && r < p + kTmaStages; ++r) {
            const int rs = r % kTmaStages;
            mbar_wait(&full[rs], (parity >> rs) & 1u);
          }
        }
        break;
      }
      parity ^= 1u << s;
      const int64_t at = int64_t(p) * kTmaPiece;
      const int64_t n = min(int64_t(kTmaPiece), body - at);
      const int j = threadIdx.x * 8;
      if (j < n) {
        const float* base = stage_buf + size_t(s) * 3 * kTmaPiece;
        float mr[8], vr[8], wr[8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          put4(mr, h, *reinterpret_cast<const float4*>(base + j + 4 * h));
          put4(vr, h, *reinterpret_cast<const float4*>(base + kTmaPiece + j + 4 * h));
          put4(wr, h, *reinterpret_cast<const float4*>(base + 2 * kTmaPiece + j + 4 * h));
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
          wr[k] = __fmaf_rn(-step, e.direction(mr[k], vr[k], wr[k], d.wd), wr[k]);
        uint32_t packed[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          packed[k] = bf16_bits(wr[2 * k]) | (bf16_bits(wr[2 * k + 1]) << 16);
        float* wg = d.w + wi.begin + at + j;
#pragma unroll
        for (int h = 0; h < 2; ++h) st_f4(wg + 4 * h, get4(wr, h));
        st_u4(d.w16 + wi.begin + at + j, make_uint4(packed[0], packed[1], packed[2], packed[3]));
      }
      __syncthreads();  // stage s is free again
      if (threadIdx.x == 0 && p + kTmaStages < npieces) issue(p + kTmaStages);
    }
    if (ok) apply_range(d, wi.begin + body, wi.count - body, threadIdx.x, kThreads, e, step);
  }
#ifdef LAMB_TEST_APPLY_REPORTS_WAIT_ERROR
  // Test builds only: CTA 0 reports a given-up wait after finishing its work
  // normally (no copy is in flight), so that the host's handling of the
  // error can be tested without any wait actually running out.
  __syncthreads();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    atomicOr(reinterpret_cast<unsigned int*>(&T.sc->error), 1u);
    if (hp.slot) static_cast<volatile ResultRecord*>(hp.slot)->error = 1;
  }
#endif
}
#endif

}  // namespace

// ---------------------------------------------------------------- launchers
int max_blocks_per_sm(int kernel, int grad_dtype) {
  int nb = 0;
  cudaError_t err = cudaSuccess;
  const bool fp16 = grad_dtype == LAMB_GRAD_FP16;
  if (kernel == 0) {
    err = fp16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                     &nb, grad_norm_kernel<LAMB_GRAD_FP16>, kThreads, 0)
               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                     &nb, grad_norm_kernel<LAMB_GRAD_BF16>, kThreads, 0);
  } else if (kernel == 1) {
    // The fused and the plain moments kernel share one launch shape: take
    // the smaller of the two.
    int nf = 0;
    err = fp16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                     &nb, moments_kernel<LAMB_GRAD_FP16, false, false>, kThreads, 0)
               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                     &nb, moments_kernel<LAMB_GRAD_BF16, false, false>, kThreads, 0);
    if (err == cudaSuccess)
      err = fp16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                       &nf, moments_kernel<LAMB_GRAD_FP16, true, false>, kThreads, 0)
                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                       &nf, moments_kernel<LAMB_GRAD_BF16, true, false>, kThreads, 0);
    if (nf < nb) nb = nf;
    if (err == cudaSuccess)
      err = fp16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                       &nf, spec_step_kernel<LAMB_GRAD_FP16>, kThreads, 0)
                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                       &nf, spec_step_kernel<LAMB_GRAD_BF16>, kThreads, 0);
    if (nf < nb) nb = nf;
  } else {
#if LAMB_TMA_C
    err = cudaFuncSetAttribute(apply_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               int(kTmaSmem));
    if (err == cudaSuccess)
      err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, apply_tma_kernel, kThreads,
                                                          kTmaSmem);
#else
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, apply_kernel, kThreads, 0);
#endif
  }
  if (err != cudaSuccess) return -int(err);
  const int cap = kernel == 0 ? LAMB_CTAS_PER_SM_A : kernel == 1 ? LAMB_CTAS_PER_SM_B
                                                                 : LAMB_CTAS_PER_SM_C;
  return nb < cap ? nb : cap;
}

int launch_grad_norm(const DevTables& T, int grid, int grad_dtype, const NormArgs& na,
                     const ScaleArgs& sa, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (grad_dtype == LAMB_GRAD_FP16)
    grad_norm_kernel<LAMB_GRAD_FP16><<<grid, kThreads, 0, s>>>(T, na, sa);
  else
    grad_norm_kernel<LAMB_GRAD_BF16><<<grid, kThreads, 0, s>>>(T, na, sa);
  return int(cudaGetLastError());
}

int launch_spec_step(const DevTables& T, int grid, int grad_dtype, const Hyper& hp,
                     const NormArgs& na, const ScaleArgs& sa, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (grad_dtype == LAMB_GRAD_FP16)
    spec_step_kernel<LAMB_GRAD_FP16><<<grid, kThreads, 0, s>>>(T, hp, na, sa);
  else
    spec_step_kernel<LAMB_GRAD_BF16><<<grid, kThreads, 0, s>>>(T, hp, na, sa);
  return int(cudaGetLastError());
}

__global__ void set_cur_kernel(StepScalars* sc, int32_t cur) { sc->cur = cur; }

int launch_set_cur(StepScalars* sc, int32_t cur, void* stream) {
  set_cur_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(sc, cur);
  return int(cudaGetLastError());
}

__global__ void set_step_kernel(StepScalars* sc, int64_t t, double p1, double p2) {
  sc->t_next = t;
  sc->p1_next = p1;
  sc->p2_next = p2;
}

int launch_exchange_trust(const DevTables& T, void* stream) {
  const int blocks = T.n_tensors > 0 ? (T.n_tensors + kThreads - 1) / kThreads : 1;
  exchange_trust_kernel<<<blocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(T);
  return int(cudaGetLastError());
}

int launch_set_step(StepScalars* sc, int64_t t, double p1, double p2, void* stream) {
  set_step_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(sc, t, p1, p2);
  return int(cudaGetLastError());
}

namespace {
// Launch configuration of a kernel that depends programmatically (PDL) on
// the kernel before it in the stream.
struct DependentLaunch {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  DependentLaunch(int grid, size_t smem, void* stream, int block = kThreads) {
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(unsigned(block));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = LAMB_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
};
}  // namespace

int launch_finalize(const DevTables& T, const NormArgs& na, const ScaleArgs& sa, void* stream) {
  DependentLaunch L(1, 0, stream, 32);  // one warp
  const cudaError_t e = cudaLaunchKernelEx(&L.cfg, finalize_kernel, T, na, sa);
  return e != cudaSuccess ? int(e) : int(cudaGetLastError());
}

int launch_moments(const DevTables& T, int grid, int grad_dtype, const Hyper& hp, bool fused,
                   void* stream) {
  DependentLaunch L(grid, 0, stream);
  cudaError_t e;
  if (grad_dtype == LAMB_GRAD_FP16)
    e = fused ? cudaLaunchKernelEx(&L.cfg, moments_kernel<LAMB_GRAD_FP16, true, false>, T, hp)
              : cudaLaunchKernelEx(&L.cfg, moments_kernel<LAMB_GRAD_FP16, false, false>, T, hp);
  else
    e = fused ? cudaLaunchKernelEx(&L.cfg, moments_kernel<LAMB_GRAD_BF16, true, false>, T, hp)
              : cudaLaunchKernelEx(&L.cfg, moments_kernel<LAMB_GRAD_BF16, false, false>, T, hp);
  return e != cudaSuccess ? int(e) : int(cudaGetLastError());
}

int launch_apply(const DevTables& T, int grid, const Hyper& hp, void* stream) {
#if LAMB_TMA_C
  DependentLaunch L(grid, kTmaSmem, stream);
  const cudaError_t e = cudaLaunchKernelEx(&L.cfg, apply_tma_kernel, T, hp);
#else
  DependentLaunch L(grid, 0, stream);
  const cudaError_t e = cudaLaunchKernelEx(&L.cfg, apply_kernel, T, hp);
#endif
  return e != cudaSuccess ? int(e) : int(cudaGetLastError());
}

int launch_spec_redo(const DevTables& T, int grid, int grad_dtype, const Hyper& hp, void* stream) {
  DependentLaunch L(grid, 0, stream);
  const cudaError_t e =
      grad_dtype == LAMB_GRAD_FP16
          ? cudaLaunchKernelEx(&L.cfg, moments_kernel<LAMB_GRAD_FP16, true, true>, T, hp)
          : cudaLaunchKernelEx(&L.cfg, moments_kernel<LAMB_GRAD_BF16, true, true>, T, hp);
  return e != cudaSuccess ? int(e) : int(cudaGetLastError());
}

}  // namespace lambgb
