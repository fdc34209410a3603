// C ABI of the LAMB step library: argument checks, the handle's device and
// pinned memory, and the per-step launch sequence.  The interface contract is
// documented in include/lamb.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <new>
#include <string>
#include <vector>

#include "lamb_internal.h"

using namespace lambgb;

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(e == cudaErrorMemoryAllocation ? LAMB_ERR_NOMEM : LAMB_ERR_CUDA,
              std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) +
                  ")");
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Makes the handle's device current for the duration of a call and restores
// the caller's device afterwards.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

}  // namespace

void lambgb::set_last_error(const std::string& msg) { g_last_error = msg; }

// Steps whose outcome stays readable after they are enqueued (lamb_step_result).
static constexpr int kResultRing = 64;

// Ordinary steps run the moments and apply passes as one persistent kernel
// when the work table holds at most this many waves of items (one item per
// resident CTA), and as two kernels above that; 0 never fuses.  On GB300 the
// fused kernel took 10% off a 16.8 M-param step and 3% off a 67 M-param one
// (2 and 4.5 waves), tied on the 1.8 B-param shard and was 0.9% slower on the
// 4,000-tensor ragged shard (73 waves), where the separate apply kernel's
// staged copies and its walk from the table's end pay more.  Split steps
// always use two kernels, with the exchange between them.
#ifndef LAMB_FUSED_MAX_WAVES
#define LAMB_FUSED_MAX_WAVES 8
#endif
// A fused shard's last tensor of several chunks gets chunks 2^LAMB_TAIL_SHIFT
// times smaller, so that the kernel's last items end closer together.
#ifndef LAMB_TAIL_SHIFT
#define LAMB_TAIL_SHIFT 1
#endif

struct lamb_handle {
  int device = 0;
  cudaStream_t stream = nullptr;
  lamb_hparams hp{};
  int32_t n_tensors = 0;
  Plan plan;
  std::vector<int64_t> sizes;
  void* dev_block = nullptr;       // every device table and scratch array
  ResultRecord* ring = nullptr;    // pinned, device-mapped: one outcome per step
  ResultRecord* ring_dev = nullptr;  // the device's view of ring
  cudaEvent_t ring_ev[kResultRing] = {};  // recorded after each step's last kernel
  int64_t next_seq = 0;            // sequence number of the next step
  int32_t split_a = 1;             // grad-norm sub-items per chunk item
  bool has_shared = false;         // some tensor has an exchange slot (split steps only)
  int64_t chunk = 0;               // chunk size of the work table
  bool fused = false;              // ordinary steps: moments and apply in one kernel
  bool spec = false;               // speculative mode: second m, v buffers given
  int split_phase = 0;             // split step: 0 none, 1 norms enqueued, 2 moments enqueued
  float split_scale = 1.0f;        // split step: the fixed loss scale of phase 1
  float split_lr = 0.0f;           // split step: the learning rate of phase 2
  const void** grad_slot[kGradSlots] = {};        // device pointer arrays
  std::vector<const void*> slot_ptrs[kGradSlots];  // what each slot holds (empty: unused)
  int next_slot = 0;
  DevTables T{};
  int grid[3] = {0, 0, 0};
  ScaleArgs scaler{};         // dynamic == 1 while a dynamic loss scaler is on
  std::vector<TensorDesc> td_host;       // the tensors' device pointers
  cudaEvent_t snap_start = nullptr;      // handle stream: state is between steps
  cudaEvent_t snap_done = nullptr;       // snapshot stream: copies finished
  bool snap_pending = false;             // the next step must wait for snap_done
  bool timing = false;        // CUDA event monitor on
  int64_t timed_from = -1;    // first step timed since the monitor was turned on
  cudaEvent_t ev[kResultRing][4] = {};  // per result slot: before / after each kernel
};

namespace {

void destroy_events(lamb_handle* h) {
  for (auto& slot : h->ev)
    for (auto& e : slot) {
      if (e) cudaEventDestroy(e);
      e = nullptr;
    }
  h->timing = false;
  h->timed_from = -1;
}

// Records monitor event k of result slot r on the handle's stream (no-op when
// timing is off).
cudaError_t mark(lamb_handle* h, int r, int k) {
  return h->timing ? cudaEventRecord(h->ev[r][k], h->stream) : cudaSuccess;
}

// Frees what lamb_create allocated (everything may be NULL).
void release(lamb_handle* h) {
  for (auto& e : h->ring_ev) {
    if (e) cudaEventDestroy(e);
    e = nullptr;
  }
  if (h->ring) cudaFreeHost(h->ring);
  if (h->dev_block) cudaFree(h->dev_block);
  h->ring = nullptr;
  h->dev_block = nullptr;
}

// Calls that change what a step reads, or copy the state, must not fall
// between the phases of a split step.
bool check_no_split(lamb_handle* h, int* rc) {
  if (h->split_phase == 0) return true;
  *rc = fail(LAMB_ERR_INVALID, "a split step is in progress");
  return false;
}

// Ordinary steps need every trust ratio from this shard alone: none may be
// shared with other ranks.
bool check_unshared(lamb_handle* h, int* rc) {
  if (!h->has_shared) return true;
  *rc = fail(LAMB_ERR_INVALID, "the shard has tensors shared with other ranks: step it with "
                               "the split step");
  return false;
}

bool check_step_args(lamb_handle* h, const void* const* grads, float lr, float clip,
                     float loss_scale, int* rc) {
  if (!(loss_scale > 0.0f) || !std::isfinite(loss_scale)) {
    *rc = fail(LAMB_ERR_INVALID, "loss_scale must be finite and > 0");
    return false;
  }
  if (!std::isfinite(lr)) {
    *rc = fail(LAMB_ERR_INVALID, "lr must be finite");
    return false;
  }
  if (std::isnan(clip)) {
    *rc = fail(LAMB_ERR_INVALID, "clip is NaN");
    return false;
  }
  if (h->n_tensors > 0 && !grads) {
    *rc = fail(LAMB_ERR_INVALID, "grads is NULL");
    return false;
  }
  for (int32_t i = 0; i < h->n_tensors; ++i) {
    if (h->sizes[size_t(i)] == 0) continue;
    if (!grads[i]) {
      *rc = fail(LAMB_ERR_INVALID, "grads[" + std::to_string(i) + "] is NULL");
      return false;
    }
    if (!aligned16(grads[i])) {
      *rc = fail(LAMB_ERR_ALIGN, "grads[" + std::to_string(i) + "] is not 16-byte aligned");
      return false;
    }
  }
  return true;
}

// Clears the result-ring slot of step seq before the step is enqueued.  If
// the step that used the slot last (seq - 64) has not finished on the GPU,
// waits for it first.
int claim_slot(lamb_handle* h, int64_t seq) {
  const int r = int(seq % kResultRing);
  if (seq >= kResultRing) {
    const cudaError_t ce = cudaEventSynchronize(h->ring_ev[r]);
    if (ce != cudaSuccess) return cuda_fail(ce, "waiting for a result slot");
  }
  std::memset(h->ring + r, 0, sizeof(ResultRecord));
  std::atomic_thread_fence(std::memory_order_release);
  return LAMB_OK;
}

int select_grads(lamb_handle* h, const void* const* grads) {
  // Find this step's grad pointers among the device slots, or write them
  // into the next slot.  The write is a kernel on the handle's stream, so it
  // runs after every earlier step has finished reading that slot.
  const size_t nt = size_t(h->n_tensors);
  int slot = -1;
  for (int k = 0; k < kGradSlots && slot < 0; ++k) {
    if (h->slot_ptrs[k].size() == nt &&
        std::memcmp(h->slot_ptrs[k].data(), grads, nt * sizeof(void*)) == 0)
      slot = k;
  }
  if (slot < 0) {
    slot = h->next_slot;
    h->next_slot = (h->next_slot + 1) % kGradSlots;
    h->slot_ptrs[slot].clear();
    const int rc = write_grad_ptrs(h->grad_slot[slot], grads, h->n_tensors, h->stream);
    if (rc) return cuda_fail(cudaError_t(rc), "writing grad pointers");
    h->slot_ptrs[slot].assign(grads, grads + nt);
  }
  h->T.grads = h->grad_slot[slot];
  return LAMB_OK;
}

Hyper make_hyper(const lamb_handle* h, float lr, int64_t seq) {
  Hyper hy;
  hy.b1 = h->hp.beta1;
  hy.b2 = h->hp.beta2;
  hy.omb1 = float(1.0 - double(h->hp.beta1));
  hy.omb2 = float(1.0 - double(h->hp.beta2));
  hy.eps = h->hp.eps;
  hy.lr = lr;
  hy.slot = h->ring_dev + seq % kResultRing;
  hy.parity = int32_t(seq & 1);
  hy.tag = uint32_t(seq % 0xFFFFFFFEll) + 1u;
  hy.only_shared = 0;
  hy.pad = 0;
  return hy;
}

NormArgs make_norm_args(const lamb_handle* h, float clip, int64_t t_host, int64_t seq,
                        int32_t partial) {
  NormArgs na;
  na.clip = clip;
  na.b1 = h->hp.beta1;
  na.b2 = h->hp.beta2;
  na.t_host = t_host;
  na.p1_host = t_host > 0 ? std::pow(double(h->hp.beta1), double(t_host)) : 0.0;
  na.p2_host = t_host > 0 ? std::pow(double(h->hp.beta2), double(t_host)) : 0.0;
  na.slot = partial ? nullptr : h->ring_dev + seq % kResultRing;
  na.split = h->split_a;
  na.parity = int32_t(seq & 1);
  na.partial = partial;
  return na;
}

int wait_for_snapshot(lamb_handle* h) {
  if (h->snap_pending) {
    // A snapshot of the state taken before this step may still be copying:
    // the kernels that write the state wait for it (on the GPU only).
    const cudaError_t ce = cudaStreamWaitEvent(h->stream, h->snap_done, 0);
    if (ce != cudaSuccess) return cuda_fail(ce, "waiting for the snapshot copies");
    h->snap_pending = false;
  }
  return LAMB_OK;
}

// Enqueues one step (arguments already checked) on the handle's stream: the
// grad pointers if new, the step's kernels (grad norm, then the fused
// moments-and-apply kernel or the moments and apply kernels; in speculative
// mode the one-pass kernel and the redo kernel), and the event of its result
// slot.  t_host >= 1 fixes the step number; 0 takes it from the device
// counter.
int enqueue_step(lamb_handle* h, const void* const* grads, float lr, int64_t t_host, float clip,
                 float loss_scale, int64_t* seq_out) {
  cudaError_t ce;
  int rc = select_grads(h, grads);
  if (rc) return rc;
  const int64_t seq = h->next_seq;
  const int r = int(seq % kResultRing);
  if ((rc = claim_slot(h, seq)) != LAMB_OK) return rc;
  const Hyper hy = make_hyper(h, lr, seq);
  const NormArgs na = make_norm_args(h, clip, t_host, seq, 0);
  if ((ce = mark(h, r, 0)) != cudaSuccess) return cuda_fail(ce, "event record");
  ScaleArgs sa = h->scaler;
  sa.fixed = loss_scale;
  if (h->spec) {
    // One pass that also sums the grad norm, then the redo of a clipped step
    // (which returns at once otherwise).
    if ((rc = wait_for_snapshot(h)) != LAMB_OK) return rc;
    if ((ce = mark(h, r, 1)) != cudaSuccess) return cuda_fail(ce, "event record");
    rc = launch_spec_step(h->T, h->grid[1], h->hp.grad_dtype, hy, na, sa, h->stream);
    if (rc) return cuda_fail(cudaError_t(rc), "speculative step kernel launch");
    if ((ce = mark(h, r, 2)) != cudaSuccess) return cuda_fail(ce, "event record");
    rc = launch_spec_redo(h->T, h->grid[1], h->hp.grad_dtype, hy, h->stream);
    if (rc) return cuda_fail(cudaError_t(rc), "redo kernel launch");
  } else {
    rc = launch_grad_norm(h->T, h->grid[0], h->hp.grad_dtype, na, sa, h->stream);
    if (rc) return cuda_fail(cudaError_t(rc), "grad-norm kernel launch");
    if ((rc = wait_for_snapshot(h)) != LAMB_OK) return rc;
    if ((ce = mark(h, r, 1)) != cudaSuccess) return cuda_fail(ce, "event record");
    rc = launch_moments(h->T, h->grid[1], h->hp.grad_dtype, hy, h->fused, h->stream);
    if (rc) return cuda_fail(cudaError_t(rc), "moments kernel launch");
    if ((ce = mark(h, r, 2)) != cudaSuccess) return cuda_fail(ce, "event record");
    if (!h->fused) {
      rc = launch_apply(h->T, h->grid[2], hy, h->stream);
      if (rc) return cuda_fail(cudaError_t(rc), "apply kernel launch");
    }
  }
  if ((ce = mark(h, r, 3)) != cudaSuccess) return cuda_fail(ce, "event record");
  if ((ce = cudaEventRecord(h->ring_ev[r], h->stream)) != cudaSuccess)
    return cuda_fail(ce, "event record");
  h->next_seq = seq + 1;
  if (h->timing && h->timed_from < 0) h->timed_from = seq;
  *seq_out = seq;
  return LAMB_OK;
}

// Speculative mode: waits for the handle's stream and reads which buffer set
// (0: m, v; 1: the second set) holds the state.
int current_set(lamb_handle* h, int32_t* cur) {
  cudaError_t ce = cudaStreamSynchronize(h->stream);
  if (ce == cudaSuccess)
    ce = cudaMemcpy(cur, reinterpret_cast<char*>(h->T.sc) + offsetof(StepScalars, cur),
                    sizeof(int32_t), cudaMemcpyDeviceToHost);
  return ce == cudaSuccess ? LAMB_OK : cuda_fail(ce, "reading which buffer set holds the state");
}

// Uploads the per-tensor records (after a change of the second buffer set).
int upload_tensor_descs(lamb_handle* h) {
  if (h->td_host.empty()) return LAMB_OK;
  cudaError_t ce = cudaMemcpyAsync(const_cast<TensorDesc*>(h->T.td), h->td_host.data(),
                                   h->td_host.size() * sizeof(TensorDesc),
                                   cudaMemcpyHostToDevice, h->stream);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(h->stream);
  return ce == cudaSuccess ? LAMB_OK : cuda_fail(ce, "uploading the tensor records");
}

// Copies a finished step's outcome out of its ring slot.
int read_result(lamb_handle* h, int64_t seq, lamb_result* out) {
  const ResultRecord* rec = h->ring + seq % kResultRing;
  std::atomic_thread_fence(std::memory_order_acquire);
  const volatile ResultRecord* v = rec;
  out->skipped = v->skipped;
  out->reserved = 0;
  out->grad_norm = v->grad_norm;
  out->loss_scale = v->scale_used;
  out->next_loss_scale = v->scale_next;
  out->t = v->t_used;
  if (v->error)
    return fail(LAMB_ERR_CUDA, "a bounded wait on the GPU gave up (staged copies or a "
                               "published result did not arrive); the state of this step "
                               "is undefined");
  return LAMB_OK;
}

}  // namespace

extern "C" {

LAMB_API const char* lamb_last_error(void) { return g_last_error.c_str(); }

LAMB_API int lamb_create_sharded(lamb_handle** out, int32_t n_tensors, const int64_t* sizes,
                                 const uint8_t* wd_flags, float* const* w, float* const* m,
                                 float* const* v, uint16_t* const* w_bf16,
                                 const int32_t* exchange_slot, int32_t n_slots,
                                 double* norm_exchange, double* tensor_exchange,
                                 const lamb_hparams* hp, void* stream) {
  g_last_error.clear();
  if (!out) return fail(LAMB_ERR_INVALID, "out is NULL");
  *out = nullptr;
  if (!hp) return fail(LAMB_ERR_INVALID, "hparams is NULL");
  if (n_tensors < 0) return fail(LAMB_ERR_INVALID, "n_tensors must be >= 0");
  if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
    return fail(LAMB_ERR_INVALID, "beta1 and beta2 must lie in [0, 1)");
  if (!(hp->eps >= 0.0f) || !std::isfinite(hp->eps))
    return fail(LAMB_ERR_INVALID, "eps must be finite and >= 0");
  if (!(hp->weight_decay >= 0.0f) || !std::isfinite(hp->weight_decay))
    return fail(LAMB_ERR_INVALID, "weight_decay must be finite and >= 0");
  if (hp->grad_dtype != LAMB_GRAD_BF16 && hp->grad_dtype != LAMB_GRAD_FP16)
    return fail(LAMB_ERR_INVALID, "grad_dtype must be LAMB_GRAD_BF16 or LAMB_GRAD_FP16");
  if (n_tensors > 0 && (!sizes || !wd_flags || !w || !m || !v || !w_bf16))
    return fail(LAMB_ERR_INVALID, "sizes, wd_flags and the pointer arrays must be non-NULL");
  if (n_slots < 0) return fail(LAMB_ERR_INVALID, "n_slots must be >= 0");
  if (n_slots > 0 && !exchange_slot)
    return fail(LAMB_ERR_INVALID, "exchange_slot is NULL but n_slots > 0");
  if (n_slots > 0 && !tensor_exchange)
    return fail(LAMB_ERR_INVALID, "tensor_exchange is NULL but n_slots > 0");
  if ((reinterpret_cast<uintptr_t>(norm_exchange) & 7u) ||
      (reinterpret_cast<uintptr_t>(tensor_exchange) & 7u))
    return fail(LAMB_ERR_ALIGN, "the exchange buffers must be 8-byte aligned");
  std::vector<uint8_t> no_pack(size_t(std::max(n_tensors, 0)), 0);
  if (exchange_slot) {
    std::vector<uint8_t> used(size_t(n_slots), 0);
    for (int32_t i = 0; i < n_tensors; ++i) {
      const int32_t k = exchange_slot[i];
      if (k < -1 || k >= n_slots)
        return fail(LAMB_ERR_INVALID, "exchange_slot[" + std::to_string(i) + "] must be -1 or in [0, n_slots)");
      if (k < 0) continue;
      if (used[size_t(k)])
        return fail(LAMB_ERR_INVALID, "exchange slot " + std::to_string(k) + " is given to two tensors");
      used[size_t(k)] = 1;
      no_pack[size_t(i)] = 1;
    }
  }
  for (int32_t i = 0; i < n_tensors; ++i) {
    if (sizes[i] < 0) return fail(LAMB_ERR_INVALID, "sizes[" + std::to_string(i) + "] < 0");
    if (sizes[i] == 0) continue;
    if (!w[i] || !m[i] || !v[i] || !w_bf16[i])
      return fail(LAMB_ERR_INVALID, "tensor " + std::to_string(i) + " has a NULL pointer");
    if (!aligned16(w[i]) || !aligned16(m[i]) || !aligned16(v[i]) || !aligned16(w_bf16[i]))
      return fail(LAMB_ERR_ALIGN,
                  "tensor " + std::to_string(i) + " has a pointer not 16-byte aligned");
  }

  // Resident CTAs of the widest kernel, which set the work-table granularity.
  int dev = 0, sms = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (ce != cudaSuccess) return cuda_fail(ce, "querying the device");
  int per_sm[3];
  for (int k = 0; k < 3; ++k) {
    per_sm[k] = max_blocks_per_sm(k, hp->grad_dtype);
    if (per_sm[k] <= 0)
      return cuda_fail(per_sm[k] < 0 ? cudaError_t(-per_sm[k]) : cudaErrorInvalidConfiguration,
                       "occupancy query");
  }
  int64_t n_params = 0;
  for (int32_t i = 0; i < n_tensors; ++i) n_params += sizes[i];

  lamb_handle* h = new (std::nothrow) lamb_handle();
  if (!h) return fail(LAMB_ERR_NOMEM, "host allocation failed");
  std::string err;
  const int64_t chunk = choose_chunk(n_params, int64_t(sms) * per_sm[1]);
  if (!build_plan(n_tensors, sizes, chunk, no_pack.data(), 0, &h->plan, &err)) {
    delete h;
    return fail(LAMB_ERR_INVALID, err);
  }
  // A shard of few waves runs the fused kernel; its last tensor then gets
  // half-size chunks (measured on GB300: 132.3 -> 130.5 us at 16.8 M params,
  // a tie at 4.2 M and 67 M; on a 1.8 B-param shard, which runs three
  // kernels, the same split cost 0.85%).
  const bool fused = !h->plan.items.empty() &&
                     int64_t(h->plan.items.size()) <=
                         int64_t(LAMB_FUSED_MAX_WAVES) * int64_t(per_sm[1]) * sms;
  if (fused && !build_plan(n_tensors, sizes, chunk, no_pack.data(), LAMB_TAIL_SHIFT, &h->plan,
                           &err)) {
    delete h;
    return fail(LAMB_ERR_INVALID, err);
  }
  h->n_tensors = n_tensors;
  h->chunk = chunk;
  h->hp = *hp;
  h->stream = static_cast<cudaStream_t>(stream);
  h->sizes.assign(sizes, sizes + n_tensors);
  h->device = dev;

  // Host copies of the per-tensor records.
  const size_t nt = size_t(n_tensors), ni = h->plan.items.size(), np = h->plan.pack_ids.size();
  std::vector<TensorDesc> td(nt);
  for (size_t i = 0; i < nt; ++i) {
    td[i].w = w[i];
    td[i].m = m[i];
    td[i].v = v[i];
    td[i].w16 = w_bf16[i];
    td[i].n = sizes[i];
    td[i].wd = wd_flags[i] ? hp->weight_decay : 0.0f;
    td[i].first_item = h->plan.first_item[i];
    td[i].n_items = h->plan.n_items[i];
    td[i].xslot = exchange_slot ? exchange_slot[i] : -1;
    if (td[i].xslot >= 0) h->has_shared = true;
    td[i].m2 = nullptr;
    td[i].v2 = nullptr;
  }
  std::vector<float> ones(nt, 1.0f);
  h->td_host = td;

  // One device allocation, carved into 256-byte aligned regions.
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + std::max<size_t>(bytes, 1), 256);
    return at;
  };
  const size_t o_td = carve(nt * sizeof(TensorDesc));
  const size_t o_items = carve(ni * sizeof(lamb_work_item));
  const size_t o_pack = carve(np * sizeof(int32_t));
  size_t o_slot[kGradSlots];
  for (auto& o : o_slot) o = carve(nt * sizeof(void*));
  // item_g2 holds one partial per CTA of the grad-norm kernel (whose grid can
  // exceed the item count: it cuts items into sub-items) and one per item in
  // speculative mode.
  const int64_t g2_entries = std::max<int64_t>(ni, int64_t(per_sm[0]) * sms);
  const size_t o_g2 = carve(size_t(g2_entries) * sizeof(double));
  const size_t o_wr = carve(ni * sizeof(double2));
  const size_t o_ticket = carve(nt * sizeof(uint32_t));
  const size_t o_trust = carve(nt * sizeof(float));
  const size_t o_trust_spec = carve(nt * sizeof(float));
  const size_t o_sc = carve(sizeof(StepScalars));
  const size_t o_queue = carve(4 * sizeof(uint32_t));
  const size_t o_ready = carve(nt * sizeof(uint32_t));
  ce = cudaMalloc(&h->dev_block, off);
  if (ce != cudaSuccess) {
    delete h;
    return cuda_fail(ce, "cudaMalloc of the work table");
  }
  void* ring = nullptr;
  ce = cudaHostAlloc(&ring, kResultRing * sizeof(ResultRecord), cudaHostAllocMapped);
  if (ce == cudaSuccess) {
    h->ring = static_cast<ResultRecord*>(ring);
    std::memset(ring, 0, kResultRing * sizeof(ResultRecord));
    void* dv = nullptr;
    ce = cudaHostGetDevicePointer(&dv, ring, 0);
    h->ring_dev = static_cast<ResultRecord*>(dv);
  }
  for (int k = 0; k < kResultRing && ce == cudaSuccess; ++k)
    ce = cudaEventCreateWithFlags(&h->ring_ev[k], cudaEventDisableTiming);
  if (ce != cudaSuccess) {
    release(h);
    delete h;
    return cuda_fail(ce, "allocating the result ring");
  }
  char* base = static_cast<char*>(h->dev_block);
  for (int k = 0; k < kGradSlots; ++k)
    h->grad_slot[k] = reinterpret_cast<const void**>(base + o_slot[k]);
  DevTables& T = h->T;
  T.td = reinterpret_cast<const TensorDesc*>(base + o_td);
  T.items = reinterpret_cast<const lamb_work_item*>(base + o_items);
  T.pack_ids = reinterpret_cast<const int32_t*>(base + o_pack);
  T.grads = h->grad_slot[0];
  T.item_g2 = reinterpret_cast<double*>(base + o_g2);
  T.item_wr = reinterpret_cast<double2*>(base + o_wr);
  T.tensor_ticket = reinterpret_cast<uint32_t*>(base + o_ticket);
  T.trust = reinterpret_cast<float*>(base + o_trust);
  T.trust_spec = reinterpret_cast<float*>(base + o_trust_spec);
  T.sc = reinterpret_cast<StepScalars*>(base + o_sc);
  T.queue = reinterpret_cast<uint32_t*>(base + o_queue);
  T.ready = reinterpret_cast<uint32_t*>(base + o_ready);
  T.xn = norm_exchange;
  T.xt = tensor_exchange;
  T.n_items = int32_t(ni);
  T.n_tensors = n_tensors;

  auto up = [&](size_t o, const void* src, size_t bytes) {
    return bytes ? cudaMemcpyAsync(base + o, src, bytes, cudaMemcpyHostToDevice, h->stream)
                 : cudaSuccess;
  };
  int krc = 0;
  if ((ce = cudaMemsetAsync(h->dev_block, 0, off, h->stream)) != cudaSuccess ||
      (ce = up(o_td, td.data(), nt * sizeof(TensorDesc))) != cudaSuccess ||
      (ce = up(o_items, h->plan.items.data(), ni * sizeof(lamb_work_item))) != cudaSuccess ||
      (ce = up(o_pack, h->plan.pack_ids.data(), np * sizeof(int32_t))) != cudaSuccess ||
      (ce = up(o_trust, ones.data(), nt * sizeof(float))) != cudaSuccess ||
      (krc = launch_set_step(T.sc, 1, double(hp->beta1), double(hp->beta2), h->stream)) != 0 ||
      (ce = cudaStreamSynchronize(h->stream)) != cudaSuccess) {
    if (krc) ce = cudaError_t(krc);
    release(h);
    delete h;
    return cuda_fail(ce, "uploading the work table");
  }

  // Persistent grids: as many CTAs as fit at once, never more than the items
  // (the grad-norm kernel: never more than its sub-items).
  int64_t n_chunk_items = 0;
  for (const auto& it : h->plan.items) n_chunk_items += it.tensor >= 0;
  for (int k = 0; k < 3; ++k) {
    const int64_t full = int64_t(per_sm[k]) * sms;
    h->grid[k] = int(std::max<int64_t>(1, std::min<int64_t>(full, int64_t(ni))));
  }
  h->fused = fused;
  // Sub-items per chunk item for the grad-norm kernel: about kSplitTarget per
  // CTA of its full grid, sub-items of at least kMinSubItem elements.
  {
    const int64_t full = int64_t(per_sm[0]) * sms;
    int64_t split = n_chunk_items > 0 ? (kSplitTarget * full + n_chunk_items - 1) / n_chunk_items
                                      : 1;
    const int64_t chunk_cap = std::max<int64_t>(1, chunk / kMinSubItem);
    split = std::max<int64_t>(1, std::min<int64_t>(split, std::min<int64_t>(kMaxSplit, chunk_cap)));
    h->split_a = int32_t(split);
    h->grid[0] = int(std::max<int64_t>(
        1, std::min<int64_t>(full, int64_t(ni - n_chunk_items) + n_chunk_items * split)));
  }
  if (int64_t(h->grid[0]) > g2_entries || int64_t(h->grid[1]) > g2_entries) {
    release(h);
    delete h;
    return fail(LAMB_ERR_INVALID, "internal: a grid exceeds its partial-sum array");
  }
  *out = h;
  return LAMB_OK;
}

LAMB_API int lamb_create(lamb_handle** out, int32_t n_tensors, const int64_t* sizes,
                         const uint8_t* wd_flags, float* const* w, float* const* m,
                         float* const* v, uint16_t* const* w_bf16, const lamb_hparams* hp,
                         void* stream) {
  return lamb_create_sharded(out, n_tensors, sizes, wd_flags, w, m, v, w_bf16, nullptr, 0,
                             nullptr, nullptr, hp, stream);
}

LAMB_API int lamb_step(lamb_handle* h, const void* const* grads, float lr, int64_t t, float clip,
                       float loss_scale, lamb_result* out) {
  g_last_error.clear();
  if (!h) return fail(LAMB_ERR_INVALID, "handle is NULL");
  if (h->split_phase != 0) return fail(LAMB_ERR_INVALID, "a split step is in progress");
  if (!out) return fail(LAMB_ERR_INVALID, "out is NULL");
  if (t < 1) return fail(LAMB_ERR_INVALID, "t must be >= 1");
  int rc = LAMB_OK;
  if (!check_unshared(h, &rc) || !check_step_args(h, grads, lr, clip, loss_scale, &rc)) return rc;
  std::memset(out, 0, sizeof *out);
  out->loss_scale = loss_scale;
  out->next_loss_scale = loss_scale;
  // An empty shard still runs the (empty) kernels: the grad norm is 0 and a
  // dynamic loss scale still advances.
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  int64_t seq = 0;
  if ((rc = enqueue_step(h, grads, lr, t, clip, loss_scale, &seq)) != LAMB_OK) return rc;
  const cudaError_t ce = cudaEventSynchronize(h->ring_ev[seq % kResultRing]);
  if (ce != cudaSuccess) return cuda_fail(ce, "waiting for the step");
  return read_result(h, seq, out);
}

LAMB_API int lamb_step_async(lamb_handle* h, const void* const* grads, float lr, float clip,
                             float loss_scale, int64_t* seq) {
  g_last_error.clear();
  if (!h) return fail(LAMB_ERR_INVALID, "handle is NULL");
  if (h->split_phase != 0) return fail(LAMB_ERR_INVALID, "a split step is in progress");
  int rc = LAMB_OK;
  if (!check_unshared(h, &rc) || !check_step_args(h, grads, lr, clip, loss_scale, &rc)) return rc;
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  int64_t s = 0;
  if ((rc = enqueue_step(h, grads, lr, 0, clip, loss_scale, &s)) != LAMB_OK) return rc;
  if (seq) *seq = s;
  return LAMB_OK;
}

LAMB_API int lamb_step_result(lamb_handle* h, int64_t seq, int32_t wait, lamb_result* out) {
  g_last_error.clear();
  if (!h || !out) return fail(LAMB_ERR_INVALID, "NULL argument");
  if (seq < 0 || seq >= h->next_seq)
    return fail(LAMB_ERR_INVALID, "no step with sequence number " + std::to_string(seq));
  if (seq < h->next_seq - kResultRing)
    return fail(LAMB_ERR_INVALID, "the outcome of step " + std::to_string(seq) +
                                      " was overwritten: only the last " +
                                      std::to_string(kResultRing) + " steps are kept");
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  cudaEvent_t ev = h->ring_ev[seq % kResultRing];
  const cudaError_t ce = wait ? cudaEventSynchronize(ev) : cudaEventQuery(ev);
  if (ce == cudaErrorNotReady) return LAMB_NOT_READY;
  if (ce != cudaSuccess) return cuda_fail(ce, "waiting for the step");
  return read_result(h, seq, out);
}

LAMB_API int lamb_split_norms(lamb_handle* h, const void* const* grads, float loss_scale) {
  g_last_error.clear();
  if (!h) return fail(LAMB_ERR_INVALID, "handle is NULL");
  if (!h->T.xn)
    return fail(LAMB_ERR_INVALID, "no norm exchange buffer: create the handle with "
                                  "lamb_create_sharded");
  if (h->split_phase != 0) return fail(LAMB_ERR_INVALID, "a split step is already in progress");
  if (h->spec) return fail(LAMB_ERR_INVALID, "split steps do not run in speculative mode");
  int rc = LAMB_OK;
  if (!check_step_args(h, grads, 0.0f, 0.0f, loss_scale, &rc)) return rc;
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  if ((rc = select_grads(h, grads)) != LAMB_OK) return rc;
  const int64_t seq = h->next_seq;
  const int r = int(seq % kResultRing);
  cudaError_t ce = mark(h, r, 0);
  if (ce != cudaSuccess) return cuda_fail(ce, "event record");
  ScaleArgs sa = h->scaler;
  sa.fixed = loss_scale;
  rc = launch_grad_norm(h->T, h->grid[0], h->hp.grad_dtype, make_norm_args(h, 0.0f, 0, seq, 1),
                        sa, h->stream);
  if (rc) return cuda_fail(cudaError_t(rc), "grad-norm kernel launch");
  h->split_scale = loss_scale;
  h->split_phase = 1;
  return LAMB_OK;
}

LAMB_API int lamb_split_moments(lamb_handle* h, float lr, int64_t t, float clip) {
  g_last_error.clear();
  if (!h) return fail(LAMB_ERR_INVALID, "handle is NULL");
  if (h->split_phase != 1) return fail(LAMB_ERR_INVALID, "call lamb_split_norms first");
  if (t < 0) return fail(LAMB_ERR_INVALID, "t must be >= 1, or 0 for the GPU's step counter");
  if (!std::isfinite(lr)) return fail(LAMB_ERR_INVALID, "lr must be finite");
  if (std::isnan(clip)) return fail(LAMB_ERR_INVALID, "clip is NaN");
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  const int64_t seq = h->next_seq;
  const int r = int(seq % kResultRing);
  int rc = claim_slot(h, seq);
  if (rc != LAMB_OK) return rc;
  ScaleArgs sa = h->scaler;
  sa.fixed = h->split_scale;
  rc = launch_finalize(h->T, make_norm_args(h, clip, t, seq, 0), sa, h->stream);
  if (rc) return cuda_fail(cudaError_t(rc), "finalize kernel launch");
  if ((rc = wait_for_snapshot(h)) != LAMB_OK) return rc;
  cudaError_t ce = mark(h, r, 1);
  if (ce != cudaSuccess) return cuda_fail(ce, "event record");
  // A shard of few waves runs the fused kernel here too: it applies every
  // tensor this rank holds whole, and lamb_split_apply only the shared ones.
  rc = launch_moments(h->T, h->grid[1], h->hp.grad_dtype, make_hyper(h, lr, seq), h->fused,
                      h->stream);
  if (rc) return cuda_fail(cudaError_t(rc), "moments kernel launch");
  h->split_lr = lr;
  h->split_phase = 2;
  return LAMB_OK;
}

LAMB_API int lamb_split_apply(lamb_handle* h, int64_t* seq_out) {
  g_last_error.clear();
  if (!h) return fail(LAMB_ERR_INVALID, "handle is NULL");
  if (h->split_phase != 2) return fail(LAMB_ERR_INVALID, "call lamb_split_moments first");
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  const int64_t seq = h->next_seq;
  const int r = int(seq % kResultRing);
  cudaError_t ce = mark(h, r, 2);
  if (ce != cudaSuccess) return cuda_fail(ce, "event record");
  // After the fused kernel only shared tensors are left to apply; with none,
  // there is nothing to launch.
  if (!(h->fused && !h->has_shared)) {
    int rc = launch_exchange_trust(h->T, h->stream);
    if (rc) return cuda_fail(cudaError_t(rc), "trust kernel launch");
    Hyper hy = make_hyper(h, h->split_lr, seq);
    hy.only_shared = h->fused ? 1 : 0;
    rc = launch_apply(h->T, h->grid[2], hy, h->stream);
    if (rc) return cuda_fail(cudaError_t(rc), "apply kernel launch");
  }
  if ((ce = mark(h, r, 3)) != cudaSuccess) return cuda_fail(ce, "event record");
  if ((ce = cudaEventRecord(h->ring_ev[r], h->stream)) != cudaSuccess)
    return cuda_fail(ce, "event record");
  h->next_seq = seq + 1;
  if (h->timing && h->timed_from < 0) h->timed_from = seq;
  h->split_phase = 0;
  if (seq_out) *seq_out = seq;
  return LAMB_OK;
}

LAMB_API int lamb_get_info(lamb_handle* h, lamb_info* out) {
  g_last_error.clear();
  if (!h || !out) return fail(LAMB_ERR_INVALID, "NULL argument");
  std::memset(out, 0, sizeof *out);
  for (const TensorDesc& d : h->td_host) {
    out->n_params += d.n;
    if (d.n > 0 && d.xslot < 0 && (d.n_items == 0 || d.n_items == 1)) out->one_pass_params += d.n;
  }
  out->chunk_elems = h->chunk;
  out->n_items = int64_t(h->plan.items.size());
  out->fused = h->fused ? 1 : 0;
  out->speculative = h->spec ? 1 : 0;
  return LAMB_OK;
}

LAMB_API int lamb_set_speculative(lamb_handle* h, float* const* m2, float* const* v2) {
  g_last_error.clear();
  if (!h) return fail(LAMB_ERR_INVALID, "handle is NULL");
  if (h->split_phase != 0) return fail(LAMB_ERR_INVALID, "a split step is in progress");
  const bool on = m2 || v2;
  if (on && h->n_tensors > 0 && (!m2 || !v2))
    return fail(LAMB_ERR_INVALID, "give both m2 and v2, or neither");
  if (on) {
    for (int32_t i = 0; i < h->n_tensors; ++i) {
      const TensorDesc& d = h->td_host[size_t(i)];
      if (d.xslot >= 0)
        return fail(LAMB_ERR_INVALID, "speculative mode does not take tensors shared with other "
                                      "ranks (split steps)");
      if (d.n == 0) continue;
      if (!m2[i] || !v2[i])
        return fail(LAMB_ERR_INVALID, "tensor " + std::to_string(i) + " has a NULL m2 or v2");
      if (!aligned16(m2[i]) || !aligned16(v2[i]))
        return fail(LAMB_ERR_ALIGN,
                    "tensor " + std::to_string(i) + " has an m2 or v2 not 16-byte aligned");
      if (m2[i] == d.m || m2[i] == d.v || v2[i] == d.m || v2[i] == d.v || m2[i] == v2[i])
        return fail(LAMB_ERR_INVALID,
                    "tensor " + std::to_string(i) + ": m2 and v2 must be buffers of their own");
    }
  }
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  if (h->spec) {
    // Bring the state back into m and v if it lives in the second set.
    int32_t cur = 0;
    int rc = current_set(h, &cur);
    if (rc != LAMB_OK) return rc;
    if (cur) {
      cudaError_t ce = cudaSuccess;
      for (const TensorDesc& d : h->td_host) {
        if (d.n == 0) continue;
        const size_t bytes = size_t(d.n) * sizeof(float);
        if ((ce = cudaMemcpyAsync(d.m, d.m2, bytes, cudaMemcpyDeviceToDevice, h->stream)) !=
                cudaSuccess ||
            (ce = cudaMemcpyAsync(d.v, d.v2, bytes, cudaMemcpyDeviceToDevice, h->stream)) !=
                cudaSuccess)
          return cuda_fail(ce, "moving the state back into m and v");
      }
    }
    for (TensorDesc& d : h->td_host) d.m2 = d.v2 = nullptr;
    h->spec = false;
  }
  if (on) {
    for (int32_t i = 0; i < h->n_tensors; ++i) {
      h->td_host[size_t(i)].m2 = m2[i];
      h->td_host[size_t(i)].v2 = v2[i];
    }
  }
  const int krc = launch_set_cur(h->T.sc, 0, h->stream);
  if (krc) return cuda_fail(cudaError_t(krc), "resetting the buffer set");
  int rc = upload_tensor_descs(h);
  if (rc != LAMB_OK) return rc;
  h->spec = on && !h->plan.items.empty();
  if (on && !h->spec) {  // an empty shard has nothing to speculate on
    for (TensorDesc& d : h->td_host) d.m2 = d.v2 = nullptr;
    return upload_tensor_descs(h);
  }
  return LAMB_OK;
}

LAMB_API int lamb_state_buffers(lamb_handle* h, int32_t* which) {
  g_last_error.clear();
  if (!h || !which) return fail(LAMB_ERR_INVALID, "NULL argument");
  *which = 0;
  if (!h->spec) return LAMB_OK;
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  return current_set(h, which);
}

LAMB_API int lamb_set_step(lamb_handle* h, int64_t t) {
  g_last_error.clear();
  if (!h) return fail(LAMB_ERR_INVALID, "handle is NULL");
  if (t < 1) return fail(LAMB_ERR_INVALID, "t must be >= 1");
  int rc = LAMB_OK;
  if (!check_no_split(h, &rc)) return rc;
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  rc = launch_set_step(h->T.sc, t, std::pow(double(h->hp.beta1), double(t)),
                       std::pow(double(h->hp.beta2), double(t)), h->stream);
  return rc ? cuda_fail(cudaError_t(rc), "setting the step number") : LAMB_OK;
}

LAMB_API int lamb_loss_scale_device(lamb_handle* h, const float** scale) {
  g_last_error.clear();
  if (!h || !scale) return fail(LAMB_ERR_INVALID, "NULL argument");
  *scale = &h->T.sc->scale;
  return LAMB_OK;
}

LAMB_API int lamb_set_loss_scaler(lamb_handle* h, const lamb_loss_scaler* cfg) {
  g_last_error.clear();
  if (!h) return fail(LAMB_ERR_INVALID, "handle is NULL");
  int rc = LAMB_OK;
  if (!check_no_split(h, &rc)) return rc;
  if (!cfg) {
    h->scaler = ScaleArgs{};
    return LAMB_OK;
  }
  if (!(cfg->init_scale > 0.0f) || !std::isfinite(cfg->init_scale) ||
      !(cfg->growth_factor >= 1.0f) || !std::isfinite(cfg->growth_factor) ||
      !(cfg->backoff_factor > 0.0f && cfg->backoff_factor <= 1.0f) ||
      cfg->growth_interval < 1 || !(cfg->min_scale >= 0.0f) ||
      !(cfg->min_scale <= cfg->init_scale) || !(cfg->init_scale <= cfg->max_scale))
    return fail(LAMB_ERR_INVALID,
                "loss scaler: need init > 0 finite, growth >= 1, backoff in (0, 1], "
                "interval >= 1, 0 <= min <= init <= max");
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  // The scale and the clean-step count sit next to each other in StepScalars.
  struct {
    float scale;
    int32_t good_steps;
  } init{cfg->init_scale, 0};
  static_assert(offsetof(StepScalars, good_steps) == offsetof(StepScalars, scale) + 4,
                "scale and good_steps must be adjacent");
  cudaError_t ce = cudaMemcpyAsync(reinterpret_cast<char*>(h->T.sc) + offsetof(StepScalars, scale),
                                   &init, sizeof init, cudaMemcpyHostToDevice, h->stream);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(h->stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "initialising the loss scale");
  h->scaler.dynamic = 1;
  h->scaler.growth = cfg->growth_factor;
  h->scaler.backoff = cfg->backoff_factor;
  h->scaler.min_scale = cfg->min_scale;
  h->scaler.max_scale = cfg->max_scale;
  h->scaler.interval = cfg->growth_interval;
  return LAMB_OK;
}

LAMB_API int lamb_set_timing(lamb_handle* h, int32_t enable) {
  g_last_error.clear();
  if (!h) return fail(LAMB_ERR_INVALID, "handle is NULL");
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  if (!enable) {
    cudaError_t ce = cudaStreamSynchronize(h->stream);
    destroy_events(h);
    return ce == cudaSuccess ? LAMB_OK : cuda_fail(ce, "waiting for the stream");
  }
  if (h->timing) return LAMB_OK;
  for (auto& slot : h->ev)
    for (auto& e : slot) {
      cudaError_t ce = cudaEventCreate(&e);
      if (ce != cudaSuccess) {
        destroy_events(h);
        return cuda_fail(ce, "cudaEventCreate");
      }
    }
  h->timing = true;
  h->timed_from = -1;
  return LAMB_OK;
}

LAMB_API int lamb_step_kernel_times(lamb_handle* h, int64_t seq, float* ms) {
  g_last_error.clear();
  if (!h || !ms) return fail(LAMB_ERR_INVALID, "NULL argument");
  if (!h->timing || h->timed_from < 0 || seq < h->timed_from || seq >= h->next_seq ||
      seq < h->next_seq - kResultRing)
    return fail(LAMB_ERR_INVALID, "step " + std::to_string(seq) +
                                      " was not timed: enable the monitor first; only the "
                                      "last 64 steps are kept");
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  cudaEvent_t* ev = h->ev[seq % kResultRing];
  for (int k = 0; k < 3; ++k) {
    cudaError_t ce = cudaEventSynchronize(ev[k + 1]);
    if (ce == cudaSuccess) ce = cudaEventElapsedTime(&ms[k], ev[k], ev[k + 1]);
    if (ce != cudaSuccess) return cuda_fail(ce, "reading monitor events");
  }
  return LAMB_OK;
}

LAMB_API int lamb_kernel_times(lamb_handle* h, float* ms) {
  g_last_error.clear();
  if (!h || !ms) return fail(LAMB_ERR_INVALID, "NULL argument");
  if (!h->timing || h->timed_from < 0)
    return fail(LAMB_ERR_INVALID, "no timed step: enable the monitor and run a step first");
  return lamb_step_kernel_times(h, h->next_seq - 1, ms);
}

LAMB_API int lamb_snapshot_async(lamb_handle* h, float* const* host_w, float* const* host_m,
                                 float* const* host_v, void* stream) {
  g_last_error.clear();
  if (!h) return fail(LAMB_ERR_INVALID, "handle is NULL");
  int rc = LAMB_OK;
  if (!check_no_split(h, &rc)) return rc;  // the state is half-updated until split_apply
  if (h->n_tensors > 0 && (!host_w || !host_m || !host_v))
    return fail(LAMB_ERR_INVALID, "host pointer arrays must be non-NULL");
  for (int32_t i = 0; i < h->n_tensors; ++i) {
    if (h->td_host[size_t(i)].n > 0 && (!host_w[i] || !host_m[i] || !host_v[i]))
      return fail(LAMB_ERR_INVALID, "tensor " + std::to_string(i) + " has a NULL host pointer");
  }
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  cudaError_t ce = cudaSuccess;
  if (!h->snap_start) ce = cudaEventCreateWithFlags(&h->snap_start, cudaEventDisableTiming);
  if (ce == cudaSuccess && !h->snap_done)
    ce = cudaEventCreateWithFlags(&h->snap_done, cudaEventDisableTiming);
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaEventCreate");
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // Copies start once everything enqueued on the handle's stream is done.
  if ((ce = cudaEventRecord(h->snap_start, h->stream)) != cudaSuccess ||
      (ce = cudaStreamWaitEvent(cs, h->snap_start, 0)) != cudaSuccess)
    return cuda_fail(ce, "ordering the snapshot after the last step");
  // A snapshot still pending (perhaps on another stream) is chained in, so
  // that snap_done below covers every outstanding copy.
  if (h->snap_pending && (ce = cudaStreamWaitEvent(cs, h->snap_done, 0)) != cudaSuccess)
    return cuda_fail(ce, "ordering after the previous snapshot");
  int32_t cur = 0;  // speculative mode: the set holding the state (the host waits to learn it)
  if (h->spec) {
    rc = current_set(h, &cur);
    if (rc != LAMB_OK) return rc;
  }
  for (int32_t i = 0; i < h->n_tensors; ++i) {
    const TensorDesc& d = h->td_host[size_t(i)];
    if (d.n == 0) continue;
    const size_t bytes = size_t(d.n) * sizeof(float);
    const float* m = cur ? d.m2 : d.m;
    const float* v = cur ? d.v2 : d.v;
    if ((ce = cudaMemcpyAsync(host_w[i], d.w, bytes, cudaMemcpyDeviceToHost, cs)) != cudaSuccess ||
        (ce = cudaMemcpyAsync(host_m[i], m, bytes, cudaMemcpyDeviceToHost, cs)) != cudaSuccess ||
        (ce = cudaMemcpyAsync(host_v[i], v, bytes, cudaMemcpyDeviceToHost, cs)) != cudaSuccess)
      return cuda_fail(ce, "enqueueing snapshot copies");
  }
  if ((ce = cudaEventRecord(h->snap_done, cs)) != cudaSuccess)
    return cuda_fail(ce, "event record");
  h->snap_pending = true;
  return LAMB_OK;
}

LAMB_API int lamb_snapshot_wait(lamb_handle* h) {
  g_last_error.clear();
  if (!h) return fail(LAMB_ERR_INVALID, "handle is NULL");
  if (!h->snap_done) return LAMB_OK;
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  const cudaError_t ce = cudaEventSynchronize(h->snap_done);
  return ce == cudaSuccess ? LAMB_OK : cuda_fail(ce, "waiting for the snapshot");
}

LAMB_API int lamb_get_trust(lamb_handle* h, float* host_out, int32_t n_tensors) {
  g_last_error.clear();
  if (!h || !host_out) return fail(LAMB_ERR_INVALID, "NULL argument");
  if (n_tensors != h->n_tensors) return fail(LAMB_ERR_INVALID, "n_tensors does not match");
  if (n_tensors == 0) return LAMB_OK;
  DeviceGuard dg(h->device);
  if (!dg.ok) return fail(LAMB_ERR_CUDA, "cannot make the handle's device current");
  cudaError_t ce = cudaStreamSynchronize(h->stream);
  if (ce == cudaSuccess)
    ce = cudaMemcpy(host_out, h->T.trust, size_t(n_tensors) * sizeof(float),
                    cudaMemcpyDeviceToHost);
  return ce == cudaSuccess ? LAMB_OK : cuda_fail(ce, "reading trust ratios");
}

LAMB_API int lamb_destroy(lamb_handle* h) {
  g_last_error.clear();
  if (!h) return LAMB_OK;
  int rc = LAMB_OK;
  {
    DeviceGuard dg(h->device);
    cudaError_t ce = cudaStreamSynchronize(h->stream);
    if (ce != cudaSuccess) rc = cuda_fail(ce, "waiting for the stream");
    destroy_events(h);
    if (h->snap_done) {
      cudaEventSynchronize(h->snap_done);
      cudaEventDestroy(h->snap_done);
    }
    if (h->snap_start) cudaEventDestroy(h->snap_start);
    release(h);
  }
  delete h;
  return rc;
}

}  // extern "C"
