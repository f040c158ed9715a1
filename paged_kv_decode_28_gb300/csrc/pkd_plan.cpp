// pkd_plan.cpp -- the host split-KV scheduler ("plan" of the plan/run split).
//
// The pages ask for a load-balanced, tile-based split of requests of very
// different lengths over a launch whose shape never changes, computed on the
// host before CUDA-graph capture (2026 guide, "What FlashInfer is", idea 3;
// deep dive, "The Architecture, Unpacked" and "It In Action", step 1).  The
// rule implemented here:
//   * a chunk is up to 64 keys of one (request b, kv head h) row: 64 / P whole
//     pages for page size P <= 64, or 64 keys inside one page for P > 64;
//   * rows r = b * Hk + h, in order, contribute their chunks to one list of W
//     chunks; CTA c of G takes list positions [c q, (c + 1) q), q = ceil(W / G);
//   * an item is a maximal run of one row's chunks that fall to one CTA.  Its
//     index is its partial-state slot.  Rows with one item write the final
//     output; rows with several, or none (empty request), are merged.
// Every CTA streams at most q chunks, so the longest CTA is within one chunk of
// the mean whatever the length mix.
#include <stdint.h>

#include <string>

#include "pkd_plan.h"

namespace pkd {

int chunk_keys_for(int page_size) {
  if (page_size <= 0) return -1;
  if (page_size <= kChunkKeysHost) return (kChunkKeysHost / page_size) * page_size;
  if (page_size % kChunkKeysHost != 0) return -1;
  return kChunkKeysHost;
}

int compute_plan(const int32_t* indptr, const int32_t* last, int batch, int num_kv_heads,
                 int page_size, int num_ctas, int32_t* items4, int max_items, int32_t* cta_begin,
                 int32_t* row_begin, int32_t* row_count, int32_t* merge_rows, int32_t* kv_len,
                 PlanCounts* counts, std::string* err) {
  if (batch < 0 || num_kv_heads <= 0 || num_ctas <= 0 || !indptr || (batch > 0 && !last)) {
    *err = "plan: invalid batch, num_kv_heads, num_ctas or NULL table";
    return kPlanInvalid;
  }
  const int ck = chunk_keys_for(page_size);
  if (ck < 0) {
    *err = "plan: page_size must be 1..64 or a multiple of 64 (got " + std::to_string(page_size) + ")";
    return kPlanUnsupported;
  }
  if (indptr[0] != 0) {
    *err = "plan: kv_indptr[0] must be 0";
    return kPlanInvalid;
  }
  int64_t total_chunks = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t n = static_cast<int64_t>(indptr[b + 1]) - indptr[b];
    if (n < 0) {
      *err = "plan: kv_indptr must be non-decreasing (request " + std::to_string(b) + ")";
      return kPlanInvalid;
    }
    int64_t L = 0;
    if (n > 0) {
      if (last[b] < 1 || last[b] > page_size) {
        *err = "plan: kv_last_page_len[" + std::to_string(b) + "] = " + std::to_string(last[b]) +
               " outside 1..page_size";
        return kPlanInvalid;
      }
      L = (n - 1) * page_size + last[b];
    }
    if (L > INT32_MAX) {
      *err = "plan: a request is longer than 2^31 - 1 keys";
      return kPlanInvalid;
    }
    kv_len[b] = static_cast<int32_t>(L);
    total_chunks += (L + ck - 1) / ck;
  }
  const int64_t W = total_chunks * num_kv_heads;
  const int64_t quota = W > 0 ? (W + num_ctas - 1) / num_ctas : 0;
  int n_items = 0;
  int64_t x = 0;
  const int rows = batch * num_kv_heads;
  for (int r = 0; r < rows; ++r) {
    row_begin[r] = n_items;
    row_count[r] = 0;
    const int b = r / num_kv_heads;
    const int64_t c_b = (static_cast<int64_t>(kv_len[b]) + ck - 1) / ck;
    int64_t k = 0;
    while (k < c_b) {
      const int64_t cta = x / quota;
      const int64_t room = (cta + 1) * quota - x;
      const int64_t take = (c_b - k) < room ? (c_b - k) : room;
      if (n_items >= max_items) {
        *err = "plan: more work items than the plan's capacity";
        return kPlanCapacity;
      }
      int32_t* it = items4 + 4 * static_cast<int64_t>(n_items);
      it[0] = r;
      it[1] = static_cast<int32_t>(k);
      it[2] = static_cast<int32_t>(k + take);
      it[3] = static_cast<int32_t>(cta);
      ++n_items;
      ++row_count[r];
      k += take;
      x += take;
    }
  }
  // CTA ranges
  int i = 0;
  for (int c = 0; c <= num_ctas; ++c) {
    while (i < n_items && items4[4 * i + 3] < c) ++i;
    cta_begin[c] = i;
  }
  int n_merge = 0;
  for (int r = 0; r < rows; ++r)
    if (row_count[r] != 1) merge_rows[n_merge++] = r;
  counts->n_items = n_items;
  counts->n_merge_rows = n_merge;
  counts->chunk_keys = ck;
  counts->quota = static_cast<int>(quota);
  return kPlanOk;
}

}  // namespace pkd
