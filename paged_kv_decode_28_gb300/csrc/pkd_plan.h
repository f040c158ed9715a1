// pkd_plan.h -- host split-KV scheduler interface (no CUDA dependency).
#pragma once

#include <stdint.h>

#include <string>

namespace pkd {

constexpr int kChunkKeysHost = 64;

enum PlanResult { kPlanOk = 0, kPlanInvalid = 1, kPlanUnsupported = 2, kPlanCapacity = 4 };

struct PlanCounts {
  int n_items;
  int n_merge_rows;
  int chunk_keys;
  int quota;
};

// Keys per chunk for a page size, or -1 if the page size is not supported.
int chunk_keys_for(int page_size);

// The split-KV rule.  items4: [max_items][4] (row, chunk_begin, chunk_end, cta);
// cta_begin: [num_ctas + 1]; row_begin, row_count, merge_rows: [batch * num_kv_heads];
// kv_len: [batch].  Returns a PlanResult; *err describes a failure.
int compute_plan(const int32_t* indptr, const int32_t* last, int batch, int num_kv_heads,
                 int page_size, int num_ctas, int32_t* items4, int max_items, int32_t* cta_begin,
                 int32_t* row_begin, int32_t* row_count, int32_t* merge_rows, int32_t* kv_len,
                 PlanCounts* counts, std::string* err);

}  // namespace pkd
