// Multi-tensor work table: lets thousands of ragged tensors go through one
// launch per kernel.  Built once per handle on the host.
//
// Large tensors (more than kSmallMax elements) become chunk items of at most
// chunk_elems elements, split evenly so the last chunk is not a sliver; chunk
// starts are multiples of 8 elements so 128-bit loads stay aligned.  Small
// tensors are packed whole, in tensor order, into pack items that one CTA
// handles a warp per tensor, so a 1-element tensor does not cost a CTA.  Pack
// items come first in the table: their latency-bound work then overlaps the
// first wave of chunk work instead of trailing at the end of a kernel.
#include <algorithm>
#include <cstring>
#include <limits>

#include "lamb_internal.h"

namespace lambgb {

// Whole waves of work: the fewest rounds of one item per resident CTA that
// keep chunks at most kChunkElems, and the chunk size that fills them.  Small
// shards then give each CTA one or two large items instead of several small
// ones, which matters because each item costs a chain of dependent latencies
// (table, data, block reduction, ticket); large shards get full-size chunks.
int64_t choose_chunk(int64_t n_params, int64_t cta_slots) {
  const int64_t slots = std::max<int64_t>(1, cta_slots);
  const int64_t waves = std::max<int64_t>(1, (n_params + slots * kChunkElems - 1) /
                                                 (slots * kChunkElems));
  int64_t c = (n_params + waves * slots - 1) / (waves * slots);
  c = (c + 255) / 256 * 256;
  return std::min(kChunkElems, std::max(kMinChunkElems, c));
}

bool build_plan(int32_t n_tensors, const int64_t* sizes, int64_t chunk_elems,
                const uint8_t* no_pack, int tail_shift, Plan* plan, std::string* err) {
  plan->items.clear();
  plan->pack_ids.clear();
  plan->first_item.assign(size_t(std::max(n_tensors, 0)), -1);
  plan->n_items.assign(size_t(std::max(n_tensors, 0)), 0);
  if (n_tensors < 0) {
    *err = "n_tensors must be >= 0";
    return false;
  }
  if (n_tensors > 0 && !sizes) {
    *err = "sizes is NULL";
    return false;
  }
  if (chunk_elems < kMinChunkElems || chunk_elems > (int64_t(1) << 30) || chunk_elems % 256) {
    *err = "chunk_elems must be a multiple of 256 in [2048, 2^30]";
    return false;
  }
  const int64_t pack_budget = std::max(chunk_elems, kSmallMax);
  const int64_t kMaxItems = std::numeric_limits<int32_t>::max();

  // Packs of small tensors first, in tensor order.
  int64_t pack_begin = 0, pack_elems = 0;
  auto close_pack = [&]() {
    const int64_t count = int64_t(plan->pack_ids.size()) - pack_begin;
    if (count > 0) plan->items.push_back({pack_begin, int32_t(count), -1});
    pack_begin = int64_t(plan->pack_ids.size());
    pack_elems = 0;
  };
  for (int32_t i = 0; i < n_tensors; ++i) {
    const int64_t n = sizes[i];
    if (n < 0) {
      *err = "sizes[" + std::to_string(i) + "] is negative";
      return false;
    }
    if (n == 0 || n > kSmallMax || (no_pack && no_pack[i])) continue;
    if (pack_elems + n > pack_budget || int64_t(plan->pack_ids.size()) - pack_begin >= kPackMax)
      close_pack();
    plan->pack_ids.push_back(i);
    pack_elems += n;
  }
  close_pack();

  // Then the chunks of every large tensor (and of every small one that must
  // not be packed), each tensor's chunks contiguous: first the tensors of a
  // single chunk (the moments kernel finishes them in one pass, a chain of
  // latencies that should not trail at the end of the kernel), then the rest.
  // The last tensor of several chunks ends the table; with tail_shift its
  // chunks are 2^tail_shift times smaller, so that the last items of a
  // kernel that has only a few waves of them finish closer together.
  int32_t last_multi = -1;
  for (int32_t i = 0; i < n_tensors; ++i)
    if (sizes[i] > chunk_elems) last_multi = i;
  for (int pass = 0; pass < 2; ++pass)
  for (int32_t i = 0; i < n_tensors; ++i) {
    const int64_t n = sizes[i];
    if (n == 0 || (n <= kSmallMax && !(no_pack && no_pack[i]))) continue;
    if ((n <= chunk_elems) != (pass == 0)) continue;
    const int64_t c = i == last_multi ? std::max<int64_t>(kMinChunkElems, chunk_elems >> tail_shift)
                                      : chunk_elems;
    const int64_t nchunks = (n + c - 1) / c;
    int64_t per = (n + nchunks - 1) / nchunks;
    per = (per + 7) / 8 * 8;
    if (int64_t(plan->items.size()) + nchunks > kMaxItems) {
      *err = "work table exceeds 2^31-1 items";
      return false;
    }
    plan->first_item[size_t(i)] = int32_t(plan->items.size());
    int32_t made = 0;
    for (int64_t b = 0; b < n; b += per) {
      plan->items.push_back({b, int32_t(std::min(per, n - b)), i});
      ++made;
    }
    plan->n_items[size_t(i)] = made;
  }
  if (int64_t(plan->items.size()) > kMaxItems) {
    *err = "work table exceeds 2^31-1 items";
    return false;
  }
  return true;
}

}  // namespace lambgb

extern "C" {

LAMB_API int lamb_plan(int32_t n_tensors, const int64_t* sizes, int64_t chunk_elems,
                       lamb_work_item* items, int64_t items_cap, int32_t* pack_ids,
                       int64_t pack_cap, int64_t* n_items, int64_t* n_pack_ids) {
  lambgb::Plan plan;
  std::string err;
  if (chunk_elems == 0) chunk_elems = lambgb::kChunkElems;
  if (!lambgb::build_plan(n_tensors, sizes, chunk_elems, nullptr, 0, &plan, &err)) {
    lambgb::set_last_error(err);
    return LAMB_ERR_INVALID;
  }
  const int64_t ni = int64_t(plan.items.size()), np = int64_t(plan.pack_ids.size());
  if (n_items) *n_items = ni;
  if (n_pack_ids) *n_pack_ids = np;
  if ((items && items_cap < ni) || (pack_ids && pack_cap < np)) {
    lambgb::set_last_error("output capacity too small");
    return LAMB_ERR_INVALID;
  }
  if (items && ni) std::memcpy(items, plan.items.data(), size_t(ni) * sizeof(lamb_work_item));
  if (pack_ids && np) std::memcpy(pack_ids, plan.pack_ids.data(), size_t(np) * sizeof(int32_t));
  return LAMB_OK;
}

LAMB_API void lamb_plan_limits(int64_t* chunk_elems, int64_t* min_chunk_elems,
                               int64_t* small_max, int64_t* pack_max) {
  if (chunk_elems) *chunk_elems = lambgb::kChunkElems;
  if (min_chunk_elems) *min_chunk_elems = lambgb::kMinChunkElems;
  if (small_max) *small_max = lambgb::kSmallMax;
  if (pack_max) *pack_max = lambgb::kPackMax;
}

}  // extern "C"
