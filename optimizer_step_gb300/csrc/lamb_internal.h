// Internal declarations shared by the host side (plan builder, C ABI) and the
// kernels of the LAMB step library.  Not part of the public interface.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include <vector_types.h>

#include "lamb.h"

namespace lambgb {

// Work-table shape.  Large tensors are cut into chunks of at most
// chunk_elems elements (a multiple of 256, so every chunk start keeps 16-byte
// alignment of the fp32 and 16-bit arrays); tensors up to kSmallMax elements
// are packed whole, one warp per tensor, at most max(chunk_elems, kSmallMax)
// elements and kPackMax tensors a pack.  lamb_create picks chunk_elems from
// the shard size and the GPU (choose_chunk): whole waves of one item per
// resident CTA; kChunkElems is the largest value.
constexpr int64_t kChunkElems = 32768;
constexpr int64_t kMinChunkElems = 2048;
constexpr int64_t kSmallMax = 4096;
constexpr int64_t kPackMax = 64;
// The grad-norm kernel cuts each chunk item into sub-items: about
// kSplitTarget per CTA of its grid, at most kMaxSplit per item, each at least
// kMinSubItem elements.
#ifndef LAMB_SPLIT_TARGET
#define LAMB_SPLIT_TARGET 6
#endif
constexpr int64_t kSplitTarget = LAMB_SPLIT_TARGET;
constexpr int64_t kMaxSplit = 16;
constexpr int64_t kMinSubItem = 1024;

// Chunk size for n_params elements on a GPU with cta_slots resident CTAs.
int64_t choose_chunk(int64_t n_params, int64_t cta_slots);

struct Plan {
  std::vector<lamb_work_item> items;
  std::vector<int32_t> pack_ids;
  std::vector<int32_t> first_item;  // per tensor: index of its first chunk item (-1: packed/empty)
  std::vector<int32_t> n_items;     // per tensor: number of chunk items (0: packed/empty)
};

// Builds the work table; returns false (with a message) on invalid sizes or
// a table too large for 32-bit item indices.  Tensors with no_pack[i] != 0
// (no_pack may be NULL) get chunk items even when small.  tail_shift > 0
// cuts the last tensor of several chunks into chunks 2^tail_shift smaller.
bool build_plan(int32_t n_tensors, const int64_t* sizes, int64_t chunk_elems,
                const uint8_t* no_pack, int tail_shift, Plan* plan, std::string* err);

// Per-tensor record the kernels read (device copy built at create time).
struct TensorDesc {
  float* w;
  float* m;
  float* v;
  uint16_t* w16;
  float* m2;           // speculative mode: the second m and v buffers (else NULL)
  float* v2;
  int64_t n;
  float wd;            // weight_decay if the tensor's flag is set, else 0
  int32_t first_item;  // first chunk item of a chunked tensor
  int32_t n_items;     // number of chunk items (0 for packed tensors)
  int32_t xslot;       // -1, or the exchange slot of a tensor shared with other ranks
};

// Device-resident values of one step, written by the grad-norm kernel's last
// CTA and read by the two later kernels.
struct StepScalars {
  double grad_norm;    // ||g / S|| (+inf if skipped)
  float gscale;        // c / S, the factor turning a raw grad into g'
  int32_t skip;        // 1: a grad was inf/NaN, nothing is written
  uint32_t ticket;     // CTAs of the grad-norm kernel that have finished
  uint32_t nonfinite;  // OR of every CTA's inf/NaN flag
  float scale_used;    // S of this step
  float scale;         // dynamic loss scale for the next step
  int32_t good_steps;  // clean steps in a row since the last growth/backoff
  int32_t error;       // set on the GPU if a bounded wait gave up this step
  float scale_next;    // S the next step uses (scale, or scale_used when it is fixed)
  int32_t pad0;
  float c1, c2;        // 1/(1-beta1^t), 1/(1-beta2^t) of this step
  int64_t t_used;      // the step number t of this step
  int64_t t_next;      // the step number of the next step (advances on clean steps)
  double p1_next;      // beta1^t_next and beta2^t_next (fp64; the host's pow when t
  double p2_next;      //   is set, then one multiplication per step that is not skipped)
  // Speculative mode (second m and v buffers):
  int32_t cur;         // which buffer set holds the state between steps (0: m, v; 1: m2, v2)
  int32_t src;         // the set this step read (the update went to the other one)
  int32_t spec_ok;     // 1: the step was neither skipped nor clipped: the speculative
                       //    moments stand and the apply items of the same kernel run
  uint32_t items_done; // moments items of the speculative kernel finished this step
  uint32_t published;  // tag of the last step whose scalars are published
  uint32_t pad;
};

// The outcome of one step as the host reads it: written by the GPU straight
// into a slot of the handle's pinned, device-mapped result ring (the grad-norm
// kernel's last CTA writes all of it; a CTA of the apply kernel whose bounded
// wait gives up sets error).
struct ResultRecord {
  double grad_norm;
  int64_t t_used;
  float scale_used;
  float scale_next;
  int32_t state_buf;    // speculative mode: the buffer set holding the state after the step
  int32_t pad;
  int32_t skipped;
  int32_t error;
};

// Step-level arguments of the grad-norm kernel.
struct NormArgs {
  float clip;           // <= 0: no clipping
  float b1, b2;         // beta1, beta2 (the bias corrections are formed on the GPU)
  int64_t t_host;       // >= 1: this step's t; 0: take it from StepScalars::t_next
  double p1_host, p2_host;  // beta1^t_host and beta2^t_host (host pow) when t_host >= 1
  ResultRecord* slot;   // device view of this step's result slot
  int32_t split;        // sub-items per chunk item (balances the CTAs)
  int32_t parity;       // this step's sequence number & 1
  int32_t partial;      // 1: only write this shard's {sum g^2, inf/NaN} to DevTables::xn
};

// How the grad-norm kernel finds this step's loss scale.
struct ScaleArgs {
  float fixed;          // S when dynamic == 0
  int32_t dynamic;      // 1: S is StepScalars::scale, updated after the step
  float growth, backoff, min_scale, max_scale;
  int32_t interval;
};

// Device pointers of one handle, passed by value to every kernel.
struct DevTables {
  const lamb_work_item* items;
  const int32_t* pack_ids;
  const TensorDesc* td;
  const void* const* grads;  // per-step grad pointers (device array)
  double* item_g2;           // per CTA of the grad-norm kernel (max(items, its full grid)
                             // entries): sum of raw g^2; per item in speculative mode
  double2* item_wr;          // per chunk item: (sum w^2, sum r^2)
  uint32_t* tensor_ticket;   // per tensor: chunk items finished this step
  float* trust;              // per tensor: trust ratio of the last step that was not skipped
  float* trust_spec;         // speculative mode: per tensor, this step's trust ratio before the
                             //   step is known to stand (copied into trust if it does)
  StepScalars* sc;
  uint32_t* queue;           // [4] item counters: moments [parity], apply [2 + parity]
  double* xn;                // split step: {sum of raw g^2, inf/NaN flag} (caller-owned)
  double* xt;                // split step: {sum w^2, sum r^2} per exchange slot (caller-owned)
  uint32_t* ready;           // per tensor: tag of the step whose trust ratio is published
  int32_t n_items;
  int32_t n_tensors;
};

struct Hyper {
  float b1, b2, omb1, omb2;  // beta1, beta2, 1-beta1, 1-beta2
  float eps, lr;
  ResultRecord* slot;        // device view of this step's result slot
  int32_t parity;            // this step's sequence number & 1: which item counters it uses
  uint32_t tag;              // non-zero, different for consecutive steps: trust-ready flags
  int32_t only_shared;       // apply pass of a split step after the fused kernel: only the
                             // tensors shared with other ranks are left to apply
  int32_t pad;
};

// Sets the calling thread's message returned by lamb_last_error().
void set_last_error(const std::string& msg);

// Kernel launchers (lamb_kernels.cu).  Each returns the launch's error code.
// max_blocks_per_sm: CTAs per SM a kernel's persistent grid uses (what fits,
// capped per kernel); kernel 0 norm, 1 moments, 2 apply; negative: CUDA error.
int max_blocks_per_sm(int kernel, int grad_dtype);
int launch_grad_norm(const DevTables& T, int grid, int grad_dtype, const NormArgs& na,
                     const ScaleArgs& sa, void* stream);
// Sets StepScalars::t_next (the step number of the next step) and its
// powers beta1^t, beta2^t on the stream.
int launch_set_step(StepScalars* sc, int64_t t, double p1, double p2, void* stream);
// Split step: forms the step's scalars from the group's summed DevTables::xn
// (what the grad-norm kernel's last CTA does in an ordinary step).
int launch_finalize(const DevTables& T, const NormArgs& na, const ScaleArgs& sa, void* stream);
// Split step: trust ratios of exchanged tensors from the group's summed xt.
int launch_exchange_trust(const DevTables& T, void* stream);
// fused: one persistent kernel takes the apply items too (ordinary steps).
int launch_moments(const DevTables& T, int grid, int grad_dtype, const Hyper& hp, bool fused,
                   void* stream);
// Speculative mode: the step's one pass (moments into the other buffer set
// with the grad norm summed on the way, then the update if the step is
// neither skipped nor clipped), and the redo of a clipped step (moments from
// the untouched set with the clip factor, then the update; returns at once
// otherwise).  Both launch with the grid of the moments kernel.
int launch_spec_step(const DevTables& T, int grid, int grad_dtype, const Hyper& hp,
                     const NormArgs& na, const ScaleArgs& sa, void* stream);
int launch_spec_redo(const DevTables& T, int grid, int grad_dtype, const Hyper& hp, void* stream);
// Sets StepScalars::cur on the stream (speculative mode on or off).
int launch_set_cur(StepScalars* sc, int32_t cur, void* stream);
int launch_apply(const DevTables& T, int grid, const Hyper& hp, void* stream);

// Writes n grad pointers into the device array dst on the stream, by kernel
// launches rather than a copy (lamb_ptrs.cu).  Returns the CUDA error code.
int write_grad_ptrs(const void** dst, const void* const* src, int32_t n, void* stream);

// Device grad-pointer arrays a handle keeps, so that alternating between a
// few grad buffers (double buffering) needs no upload after the first use.
constexpr int kGradSlots = 4;

}  // namespace lambgb
