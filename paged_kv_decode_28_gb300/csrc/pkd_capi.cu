// pkd_capi.cu -- the C ABI of libpkd.so (declared in include/pkd.h): argument
// checking, workspace layout, TMA tensor-map encoding and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <string>
#include <vector>

#include "pkd.h"
#include "pkd_host.h"
#include "pkd_internal.h"
#include "pkd_upload.h"
#include "pkd_plan.h"

namespace {
thread_local std::string g_err;
}  // namespace

namespace pkd {
namespace host {

pkd_status fail(pkd_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace host
}  // namespace pkd

namespace {

using pkd::host::aligned16;
using pkd::host::align256;
using pkd::host::cuda_fail;
using pkd::host::elem_bytes;
using pkd::host::fail;
using pkd::host::get_encode;

struct Layout {
  int group = 0, max_rows = 0, max_items = 0, max_work = 0;
  size_t cta_begin = 0, items = 0, merge_rows = 0, row_begin = 0, row_count = 0, kv_len = 0,
         page_begin = 0, empty_rows = 0, row_done = 0, meta_end = 0, part_o = 0, part_lse = 0, pre_o = 0,
         pre_lse = 0, work = 0, total = 0;
};

bool make_layout(int max_batch, int hq, int hk, int d, int G, int max_splits, Layout* L) {
  if (max_batch <= 0 || hq <= 0 || hk <= 0 || d <= 0 || G <= 0 || max_splits < 0) return false;
  if (hq % hk != 0) return false;
  L->group = hq / hk;
  L->max_rows = max_batch * hk;
  L->max_items = L->max_rows + G;
  size_t off = sizeof(pkd::WsHeader);
  L->cta_begin = off;
  off += align256(4ull * (G + 1));
  L->items = off;
  off += align256(16ull * L->max_items);
  L->merge_rows = off;
  off += align256(4ull * L->max_rows);
  L->row_begin = off;
  off += align256(4ull * L->max_rows);
  L->row_count = off;
  off += align256(4ull * L->max_rows);
  L->kv_len = off;
  off += align256(4ull * max_batch);
  L->page_begin = off;
  off += align256(4ull * max_batch);
  L->empty_rows = off;
  off += align256(4ull * L->max_rows);
  L->row_done = off;  // never written by the host: every upload resets the counters to zero
  off += align256(4ull * L->max_rows);
  L->meta_end = off;
  L->part_o = off;
  off += align256(4ull * L->max_items * L->group * d);
  L->part_lse = off;
  off += align256(4ull * L->max_items * L->group);
  L->pre_o = off;
  off += align256(4ull * max_splits * max_batch * hq * d);
  L->pre_lse = off;
  off += align256(4ull * max_splits * max_batch * hq);
  // units of the tile-attention kernel's work-list mode (prefix-tree levels,
  // prefill), uploaded by pkd_plan_tree / pkd_plan_prefill
  L->max_work = 8 * (max_batch + G) > 4096 ? 8 * (max_batch + G) : 4096;
  L->work = off;
  off += align256(sizeof(pkd::TileWork) * static_cast<size_t>(L->max_work));
  L->total = off;
  return true;
}


// Tensor map over a pool of NHD pages [num_pages, tok_extent, Hk, 128] (dims
// dim, head, key, page) or HND pages [num_pages, Hk, tok_extent, 128] (dims
// dim, key, head, page), with a page stride in elements; boxes of 64 (16-bit)
// or 128 (fp8) head-dim elements x box_tok keys of one head of one page,
// 128-byte swizzled.  Either way a box lands in shared memory as box_tok rows.
pkd_status encode_kv_map(CUtensorMap* m, const void* base, int kv_dtype, int hk, int64_t tok_extent,
                         int64_t num_pages, int64_t page_stride_elems, int box_tok, bool hnd) {
  auto enc = get_encode();
  if (!enc) return fail(PKD_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const int e = elem_bytes(kv_dtype);
  const cuuint64_t row = static_cast<cuuint64_t>(pkd::kHeadDim) * e;
  const cuuint64_t n1 = hnd ? static_cast<cuuint64_t>(tok_extent) : static_cast<cuuint64_t>(hk);
  const cuuint64_t n2 = hnd ? static_cast<cuuint64_t>(hk) : static_cast<cuuint64_t>(tok_extent);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(pkd::kHeadDim), n1, n2, static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[3] = {row, n1 * row, static_cast<cuuint64_t>(page_stride_elems) * e};
  const cuuint32_t bx = static_cast<cuuint32_t>(e == 1 ? 128 : 64), bt = static_cast<cuuint32_t>(box_tok);
  cuuint32_t box[4] = {bx, hnd ? bt : 1u, hnd ? 1u : bt, 1u};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUtensorMapDataType dt = kv_dtype == PKD_E4M3   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                           : kv_dtype == PKD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  // a key row of one head is 256 B (16-bit) or 128 B (fp8): promote L2 fills to
  // one row, so no neighbouring head's row is fetched with it
  CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   e == 1 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKD_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return PKD_OK;
}


// CTA pairs of the shared-prefix kernel that fit on the current device at
// once (queried once per device and kernel variant; 0 when unknown).
int resident_prefix_clusters(int q_dtype, int kv_dtype) {
  static std::mutex mu;
  static int cache[64][2][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int qi = q_dtype == PKD_BF16 ? 1 : 0, ki = kv_dtype == PKD_E4M3 ? 1 : 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev][qi][ki] == 0) {
    const int n = pkd::prefix_max_active_clusters(q_dtype, kv_dtype);
    cache[dev][qi][ki] = n > 0 ? n : -1;
  }
  return cache[dev][qi][ki] > 0 ? cache[dev][qi][ki] : 0;
}

// Tensor map over an e4m3 pool whose boxes are `box_cols` codes (128 for K,
// 64 for one CTA's V columns) x box_tok keys of one head of one page, not
// swizzled: a box lands as box_tok rows of box_cols bytes.
pkd_status encode_code_map(CUtensorMap* m, const void* base, int hk, int64_t tok_extent, int64_t num_pages,
                           int64_t page_stride_elems, int box_tok, int box_cols, bool hnd) {
  auto enc = get_encode();
  if (!enc) return fail(PKD_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t row = static_cast<cuuint64_t>(pkd::kHeadDim);
  const cuuint64_t n1 = hnd ? static_cast<cuuint64_t>(tok_extent) : static_cast<cuuint64_t>(hk);
  const cuuint64_t n2 = hnd ? static_cast<cuuint64_t>(hk) : static_cast<cuuint64_t>(tok_extent);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(pkd::kHeadDim), n1, n2, static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[3] = {row, n1 * row, static_cast<cuuint64_t>(page_stride_elems)};
  const cuuint32_t bt = static_cast<cuuint32_t>(box_tok);
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_cols), hnd ? bt : 1u, hnd ? 1u : bt, 1u};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKD_ERR_CUDA, "cuTensorMapEncodeTiled(codes) failed (CUresult %d)", (int)r);
  return PKD_OK;
}

int gcd_int(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

}  // namespace

namespace pkd {
// Lets other translation units of the library report through pkd_last_error().
void set_last_error(const char* msg) { g_err = msg; }
}  // namespace pkd

struct pkd_plan_s {
  int max_batch, hq, hk, d, G, max_splits;
  uint8_t* ws;
  size_t ws_bytes;
  Layout lay;
  std::vector<uint8_t> host;  // mirror of workspace bytes [0, meta_end)
  // last plan
  bool planned = false;
  bool err_word_zeroed = false;  // the first plan clears the device error word
  // pinned staging buffer of the schedule: plan writes it, every run copies it
  // into the workspace with a kernel (so a graph captured around run uploads
  // the latest plan on each replay); stage_done fires after each such copy and
  // plan waits for it before overwriting the buffer
  bool use_pinned = true;
  // one-shot plans (single-request decode): the schedule travels in the
  // upload kernel's parameters instead (no copy engine: capturable)
  bool upload_by_blob = false;
  uint8_t* staging = nullptr;
  uint8_t* staging_dev = nullptr;  // device mapping of the staging buffer
  cudaEvent_t stage_done = nullptr;
  // optional caller events recorded around the decode kernel (timing hook);
  // the stop record goes on a side stream forked after the decode launch
  cudaEvent_t ev_start = nullptr, ev_stop = nullptr;
  cudaStream_t side = nullptr;
  cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
  int debug_flags = 0;  // PKD_DEBUG_* test hooks
  int kv_layout = PKD_LAYOUT_NHD;  // page layout of the pools given to run / cascade_decode
  int plan_gen = 0;                // successful pkd_plan calls
  // work-list units of the last pkd_plan_tree (kind 1) or pkd_plan_prefill
  // (kind 2), uploaded into the workspace's work region from a pinned buffer;
  // work_done fires after each upload and the next one waits for it
  int work_kind = 0, n_work = 0, work_gen = 0;
  pkd::TileWork* work_staging = nullptr;
  cudaEvent_t work_done = nullptr;
  const int32_t* level_pages[pkd::kMaxTreeLevels] = {};
  int tree_pieces = 0;
  int pf_tokens = 0, pf_page_size = 0, pf_dtype = 0;
  ~pkd_plan_s() {
    if (work_done) {
      cudaEventSynchronize(work_done);
      cudaEventDestroy(work_done);
    }
    if (work_staging) cudaFreeHost(work_staging);
    if (side) {
      cudaStreamSynchronize(side);
      cudaStreamDestroy(side);
    }
    if (fork_ev) cudaEventDestroy(fork_ev);
    if (join_ev) cudaEventDestroy(join_ev);
    if (stage_done) {
      cudaEventSynchronize(stage_done);
      cudaEventDestroy(stage_done);
    }
    if (staging) cudaFreeHost(staging);
  }
  int batch = 0, page_size = 0, q_dtype = 0, kv_dtype = 0;
  const int32_t* d_page_indices = nullptr;
  pkd::PlanCounts counts{};
};

extern "C" {

const char* pkd_version(void) { return "pkd 0.1.0 sm_103a"; }

const char* pkd_status_string(int s) {
  switch (s) {
    case PKD_OK: return "ok";
    case PKD_ERR_INVALID_ARG: return "invalid argument";
    case PKD_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKD_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PKD_ERR_CAPACITY_EXCEEDED: return "capacity exceeded";
    case PKD_ERR_CUDA: return "CUDA error";
    case PKD_ERR_DEVICE_CHECK: return "device-side check failed";
    case PKD_ERR_NO_PLAN: return "no plan";
    default: return "unknown status";
  }
}

const char* pkd_last_error(void) { return g_err.c_str(); }

pkd_status pkd_num_ctas(int device, int* num_ctas_out) {
  if (!num_ctas_out) return fail(PKD_ERR_INVALID_ARG, "num_ctas_out is NULL");
  int sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(MultiProcessorCount)");
  *num_ctas_out = sms * pkd::kCtasPerSm;
  return PKD_OK;
}

size_t pkd_workspace_bytes(int max_batch, int num_qo_heads, int num_kv_heads, int head_dim,
                           int num_ctas, int max_prefix_splits) {
  Layout L;
  if (head_dim != pkd::kHeadDim) return 0;
  if (max_prefix_splits > pkd::kMaxPrefixSplits) return 0;
  if (!make_layout(max_batch, num_qo_heads, num_kv_heads, head_dim, num_ctas, max_prefix_splits, &L))
    return 0;
  return L.total;
}

pkd_status pkd_plan_create(pkd_plan_t* plan_out, int max_batch, int num_qo_heads, int num_kv_heads,
                           int head_dim, int num_ctas, int max_prefix_splits, void* d_workspace,
                           size_t workspace_bytes) {
  if (!plan_out) return fail(PKD_ERR_INVALID_ARG, "plan_out is NULL");
  *plan_out = nullptr;
  if (head_dim != pkd::kHeadDim) return fail(PKD_ERR_UNSUPPORTED, "head_dim must be 128 (got %d)", head_dim);
  if (num_kv_heads <= 0 || num_qo_heads <= 0 || num_qo_heads % num_kv_heads != 0)
    return fail(PKD_ERR_INVALID_ARG, "num_qo_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                num_qo_heads, num_kv_heads);
  if (num_qo_heads / num_kv_heads > pkd::kMaxGroup)
    return fail(PKD_ERR_UNSUPPORTED, "group size %d above %d", num_qo_heads / num_kv_heads, pkd::kMaxGroup);
  if (max_prefix_splits < 0 || max_prefix_splits > pkd::kMaxPrefixSplits)
    return fail(PKD_ERR_INVALID_ARG, "max_prefix_splits must be 0..%d", pkd::kMaxPrefixSplits);
  Layout L;
  if (!make_layout(max_batch, num_qo_heads, num_kv_heads, head_dim, num_ctas, max_prefix_splits, &L))
    return fail(PKD_ERR_INVALID_ARG, "invalid limits (max_batch %d, num_ctas %d)", max_batch, num_ctas);
  if (!d_workspace) return fail(PKD_ERR_INVALID_ARG, "d_workspace is NULL");
  if (reinterpret_cast<uintptr_t>(d_workspace) & 255u)
    return fail(PKD_ERR_INVALID_ARG, "d_workspace must be 256-byte aligned");
  if (workspace_bytes < L.total)
    return fail(PKD_ERR_WORKSPACE_TOO_SMALL, "workspace has %zu bytes, needs %zu", workspace_bytes, L.total);
  pkd_plan_s* p = new (std::nothrow) pkd_plan_s();
  if (!p) return fail(PKD_ERR_INVALID_ARG, "out of host memory");
  p->max_batch = max_batch;
  p->hq = num_qo_heads;
  p->hk = num_kv_heads;
  p->d = head_dim;
  p->G = num_ctas;
  p->max_splits = max_prefix_splits;
  p->ws = static_cast<uint8_t*>(d_workspace);
  p->ws_bytes = workspace_bytes;
  p->lay = L;
  p->host.assign(L.meta_end, 0);
  *plan_out = p;
  return PKD_OK;
}

pkd_status pkd_plan_destroy(pkd_plan_t plan) {
  delete plan;
  return PKD_OK;
}

pkd_status pkd_plan_host(const int32_t* h_kv_indptr, const int32_t* h_kv_last_page_len, int batch,
                         int num_kv_heads, int page_size, int num_ctas, int32_t* items, int max_items,
                         int32_t* cta_item_begin, int32_t* row_item_begin, int32_t* row_item_count,
                         int32_t* merge_rows, int32_t* counts) {
  if (!items || !cta_item_begin || !row_item_begin || !row_item_count || !merge_rows || !counts)
    return fail(PKD_ERR_INVALID_ARG, "NULL output array");
  std::vector<int32_t> kv_len(batch > 0 ? batch : 1);
  std::string err;
  pkd::PlanCounts c{};
  int r = pkd::compute_plan(h_kv_indptr, h_kv_last_page_len, batch, num_kv_heads, page_size, num_ctas,
                            items, max_items, cta_item_begin, row_item_begin, row_item_count,
                            merge_rows, kv_len.data(), &c, &err);
  if (r != pkd::kPlanOk) return fail(static_cast<pkd_status>(r), "%s", err.c_str());
  counts[0] = c.n_items;
  counts[1] = c.n_merge_rows;
  counts[2] = c.chunk_keys;
  counts[3] = c.quota;
  return PKD_OK;
}

pkd_status pkd_plan(pkd_plan_t plan, const int32_t* h_kv_indptr, const int32_t* d_kv_page_indices,
                    const int32_t* h_kv_last_page_len, int batch, int num_qo_heads, int num_kv_heads,
                    int head_dim, int page_size, int q_dtype, int kv_dtype, void* stream) {
  if (!plan) return fail(PKD_ERR_INVALID_ARG, "plan is NULL");
  plan->planned = false;
  if (num_qo_heads != plan->hq || num_kv_heads != plan->hk || head_dim != plan->d)
    return fail(PKD_ERR_INVALID_ARG, "heads/head_dim (%d, %d, %d) differ from the plan's (%d, %d, %d)",
                num_qo_heads, num_kv_heads, head_dim, plan->hq, plan->hk, plan->d);
  if (batch < 0) return fail(PKD_ERR_INVALID_ARG, "batch must be >= 0");
  if (batch > plan->max_batch)
    return fail(PKD_ERR_CAPACITY_EXCEEDED, "batch %d above max_batch %d", batch, plan->max_batch);
  const bool ok_pair = (q_dtype == PKD_F16 && kv_dtype == PKD_F16) ||
                       (q_dtype == PKD_BF16 && kv_dtype == PKD_BF16) ||
                       (q_dtype == PKD_BF16 && kv_dtype == PKD_E4M3) ||
                       (q_dtype == PKD_F16 && kv_dtype == PKD_E4M3);
  if (!ok_pair) return fail(PKD_ERR_UNSUPPORTED, "dtype pair (q %d, kv %d) not supported", q_dtype, kv_dtype);
  if (!h_kv_indptr) return fail(PKD_ERR_INVALID_ARG, "h_kv_indptr is NULL");
  if (batch > 0 && h_kv_indptr[batch] > 0 && !d_kv_page_indices)
    return fail(PKD_ERR_INVALID_ARG, "d_kv_page_indices is NULL");
  const Layout& L = plan->lay;
  uint8_t* h = plan->host.data();
  auto* hdr = reinterpret_cast<pkd::WsHeader*>(h);
  auto* cta_begin = reinterpret_cast<int32_t*>(h + L.cta_begin);
  auto* items = reinterpret_cast<int32_t*>(h + L.items);
  auto* merge_rows = reinterpret_cast<int32_t*>(h + L.merge_rows);
  auto* row_begin = reinterpret_cast<int32_t*>(h + L.row_begin);
  auto* row_count = reinterpret_cast<int32_t*>(h + L.row_count);
  auto* kv_len = reinterpret_cast<int32_t*>(h + L.kv_len);
  auto* page_begin = reinterpret_cast<int32_t*>(h + L.page_begin);
  std::string err;
  pkd::PlanCounts c{};
  int r = pkd::compute_plan(h_kv_indptr, h_kv_last_page_len, batch, num_kv_heads, page_size, plan->G,
                            items, L.max_items, cta_begin, row_begin, row_count, merge_rows, kv_len,
                            &c, &err);
  if (r != pkd::kPlanOk) return fail(static_cast<pkd_status>(r), "%s", err.c_str());
  // item flags: bit 0 = row split across several items
  for (int i = 0; i < c.n_items; ++i) {
    const int row = items[4 * i + 0];
    items[4 * i + 3] = row_count[row] > 1 ? pkd::kItemSplit : 0;
  }
  for (int b = 0; b < batch; ++b) page_begin[b] = h_kv_indptr[b];
  auto* empty_rows = reinterpret_cast<int32_t*>(h + L.empty_rows);
  int n_empty = 0;
  for (int r = 0; r < batch * num_kv_heads; ++r)
    if (row_count[r] == 0) empty_rows[n_empty++] = r;
  hdr->n_empty_rows = n_empty;
  hdr->n_items = c.n_items;
  hdr->n_merge_rows = c.n_merge_rows;
  hdr->batch = batch;
  hdr->zero_page = 0;
  if (!plan->err_word_zeroed) {
    cudaError_t ez = cudaMemsetAsync(plan->ws, 0, 4, static_cast<cudaStream_t>(stream));
    if (ez != cudaSuccess) return cuda_fail(ez, "cudaMemsetAsync(error word)");
    plan->err_word_zeroed = true;
  }
  // stage everything after the error word (the error word stays the kernels')
  if (plan->use_pinned) {
    if (!plan->staging) {
      cudaError_t ea = cudaHostAlloc(reinterpret_cast<void**>(&plan->staging), L.meta_end, cudaHostAllocMapped);
      if (ea == cudaSuccess)
        ea = cudaHostGetDevicePointer(reinterpret_cast<void**>(&plan->staging_dev), plan->staging, 0);
      if (ea == cudaSuccess) ea = cudaEventCreateWithFlags(&plan->stage_done, cudaEventDisableTiming);
      if (ea != cudaSuccess) return cuda_fail(ea, "plan staging buffer");
    } else {
      // the copy that read the previous schedule (issued by the last run, or by
      // the last replay of a graph captured around run) is done with the buffer
      cudaError_t ea = cudaEventSynchronize(plan->stage_done);
      if (ea != cudaSuccess) return cuda_fail(ea, "cudaEventSynchronize(plan staging)");
    }
    memcpy(plan->staging + 16, h + 16, L.meta_end - 16);
  } else if (plan->upload_by_blob) {
    // run_common launches the upload with the host copy as its parameter
  } else {
    cudaError_t e = cudaMemcpyAsync(plan->ws + 4, h + 4, L.meta_end - 4, cudaMemcpyHostToDevice,
                                    static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "plan upload");
  }
  plan->planned = true;
  ++plan->plan_gen;
  plan->batch = batch;
  plan->page_size = page_size;
  plan->q_dtype = q_dtype;
  plan->kv_dtype = kv_dtype;
  plan->d_page_indices = d_kv_page_indices;
  plan->counts = c;
  return PKD_OK;
}

}  // extern "C"

namespace {

// The plan's side stream and its fork/join events (created on first use).
pkd_status ensure_side(pkd_plan_t plan) {
  if (plan->side) return PKD_OK;
  cudaError_t e = cudaStreamCreateWithFlags(&plan->side, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&plan->fork_ev, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&plan->join_ev, cudaEventDisableTiming);
  if (e != cudaSuccess) return cuda_fail(e, "side stream/events");
  return PKD_OK;
}

// Cascade settings for run_common: every item writes a partial state and the
// merge pass folds n_pre_splits prefix partials into every row.
struct CascadeMerge {
  int n_pre_splits;
  // the prefix kernel, launched between the decode and merge launches (when
  // n_pre_splits > 0): its CTAs take the SMs the decode grid frees as it drains
  CUtensorMap tmq, tmk, tmv;
  pkd::PrefixParams pp;
};

pkd_status run_common(pkd_plan_t plan, const void* d_q, const void* d_k_cache, const void* d_v_cache,
                      int64_t num_pages, int64_t page_stride_elems, int64_t tok_extent,
                      const float* d_k_scale, const float* d_v_scale, float sm_scale, void* d_out,
                      float* d_lse, void* stream, const int32_t* page_indices_override,
                      const CascadeMerge* cascade = nullptr) {
  if (!plan) return fail(PKD_ERR_INVALID_ARG, "plan is NULL");
  if (!plan->planned) return fail(PKD_ERR_NO_PLAN, "run before a successful plan");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Layout& L = plan->lay;
  if (!d_q || !d_out) return fail(PKD_ERR_INVALID_ARG, "q/out is NULL");
  if (!aligned16(d_q) || !aligned16(d_out)) return fail(PKD_ERR_INVALID_ARG, "q/out must be 16-byte aligned");
  const bool fp8 = plan->kv_dtype == PKD_E4M3;
  if (fp8 && (!d_k_scale || !d_v_scale))
    return fail(PKD_ERR_INVALID_ARG, "an E4M3 cache needs k_scale and v_scale");
  if (!fp8 && (d_k_scale || d_v_scale))
    return fail(PKD_ERR_INVALID_ARG, "k_scale/v_scale apply to an E4M3 cache only");
  const int P = plan->page_size;
  const int box_tok = P <= pkd::kChunkKeys ? P : pkd::kChunkKeys;
  const float scale = (sm_scale > 0.f) ? sm_scale : 1.0f / std::sqrt(static_cast<float>(plan->d));
  uint8_t* ws = plan->ws;
  pkd::DecodeParams p{};
  p.items = reinterpret_cast<const int4*>(ws + L.items);
  p.cta_begin = reinterpret_cast<const int*>(ws + L.cta_begin);
  p.kv_len = reinterpret_cast<const int*>(ws + L.kv_len);
  p.page_begin = reinterpret_cast<const int*>(ws + L.page_begin);
  p.page_indices = page_indices_override ? page_indices_override : plan->d_page_indices;
  p.q = d_q;
  p.out = d_out;
  p.lse = d_lse;
  p.part_o = reinterpret_cast<float*>(ws + L.part_o);
  p.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  p.k_scale = d_k_scale;
  p.v_scale = d_v_scale;
  p.err = reinterpret_cast<unsigned*>(ws);
  p.num_kv_heads = plan->hk;
  p.group = plan->hq / plan->hk;
  p.page_size = P;
  p.pages_per_chunk = P <= pkd::kChunkKeys ? pkd::kChunkKeys / P : 0;
  p.chunk_keys = plan->counts.chunk_keys;
  p.box_tok = box_tok;
  p.num_pages = static_cast<int>(num_pages);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.force_partial = cascade ? 1 : 0;
  p.fused_merge = cascade ? 0 : 1;
  p.row_done = reinterpret_cast<int*>(ws + L.row_done);
  p.row_item_begin = reinterpret_cast<const int*>(ws + L.row_begin);
  p.row_item_count = reinterpret_cast<const int*>(ws + L.row_count);
  p.empty_rows = reinterpret_cast<const int*>(ws + L.empty_rows);
  p.header = reinterpret_cast<const pkd::WsHeader*>(ws);
  p.debug_stall = (plan->debug_flags & PKD_DEBUG_STALL_PIPELINE) ? 1 : 0;
  p.kv_hnd = plan->kv_layout == PKD_LAYOUT_HND ? 1 : 0;
  // under stream capture the records become event-record nodes that fire on every replay
  unsigned rec_flags = cudaEventRecordDefault;
  {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
      rec_flags = cudaEventRecordExternal;
  }
  // Upload the staged schedule with a copy kernel; the decode kernel is
  // launched programmatically after it and waits for it in griddepcontrol.wait.
  // The records that follow the copy (stage_done, the timing start) go on the
  // side stream, forked here, so no node separates the two launches.
  bool joined = true;
  if (plan->use_pinned) {
    pkd_status ss = ensure_side(plan);
    if (ss != PKD_OK) return ss;
    cudaError_t e = pkd::launch_copy16(ws + 16, plan->staging_dev + 16, L.meta_end - 16, st);
    if (e != cudaSuccess) return cuda_fail(e, "plan upload");
    e = cudaEventRecord(plan->fork_ev, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->side, plan->fork_ev, 0);
    if (e == cudaSuccess) e = cudaEventRecordWithFlags(plan->stage_done, plan->side, rec_flags);
    if (e == cudaSuccess && plan->ev_start) e = cudaEventRecordWithFlags(plan->ev_start, plan->side, rec_flags);
    if (e != cudaSuccess) return cuda_fail(e, "upload fork");
    joined = false;
  } else if (plan->upload_by_blob) {
    cudaError_t e = pkd::launch_copy_blob(ws + 16, plan->host.data() + 16, L.meta_end - 16, st);
    if (e != cudaSuccess) return cuda_fail(e, "plan upload");
  }
  // A single shared prefix (the pair kernel, one CTA per SM on most of the
  // GPU, bound by its MMA chain) goes ahead of the suffix decode, whose CTAs
  // start on the SMs it leaves free and read HBM meanwhile.
  const bool prefix_first = cascade && cascade->n_pre_splits > 0 && !cascade->pp.work && plan->counts.n_items > 0;
  if (plan->counts.n_items > 0) {
    if (!d_k_cache || !d_v_cache) return fail(PKD_ERR_INVALID_ARG, "k/v cache is NULL");
    if (!aligned16(d_k_cache) || !aligned16(d_v_cache))
      return fail(PKD_ERR_INVALID_ARG, "k/v cache must be 16-byte aligned");
    if (num_pages <= 0 || num_pages > INT32_MAX) return fail(PKD_ERR_INVALID_ARG, "num_pages out of range");
    if ((page_stride_elems * elem_bytes(plan->kv_dtype)) % 16 != 0 ||
        page_stride_elems < static_cast<int64_t>(P) * plan->hk * plan->d)
      return fail(PKD_ERR_INVALID_ARG, "page_stride_elems must cover a page and be a 16-byte multiple");
    CUtensorMap tmk, tmv;
    pkd_status s = encode_kv_map(&tmk, d_k_cache, plan->kv_dtype, plan->hk, tok_extent, num_pages,
                                 page_stride_elems, box_tok, p.kv_hnd != 0);
    if (s != PKD_OK) return s;
    s = encode_kv_map(&tmv, d_v_cache, plan->kv_dtype, plan->hk, tok_extent, num_pages, page_stride_elems,
                      box_tok, p.kv_hnd != 0);
    if (s != PKD_OK) return s;
    if (plan->ev_start && !plan->use_pinned) {
      cudaError_t er = cudaEventRecordWithFlags(plan->ev_start, st, rec_flags);
      if (er != cudaSuccess) return cuda_fail(er, "cudaEventRecord(timing start)");
    }
    if (prefix_first) {
      cudaError_t e = pkd::launch_prefix(cascade->tmq, cascade->tmk, cascade->tmv, cascade->pp, plan->q_dtype,
                                         plan->kv_dtype, st, true);
      if (e != cudaSuccess) return cuda_fail(e, "prefix kernel launch");
      p.behind_prefix = 1;
    }
    cudaError_t e = pkd::launch_decode(tmk, tmv, p, plan->q_dtype, plan->kv_dtype, plan->G, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    if (plan->ev_stop) {
      // the stop record waits for the decode kernel on the side branch, so
      // that no node sits between the decode and merge launches: a record on
      // the call's stream would cancel the merge's programmatic early launch
      pkd_status ss = ensure_side(plan);
      if (ss != PKD_OK) return ss;
      cudaError_t er = cudaEventRecord(plan->fork_ev, st);
      if (er == cudaSuccess) er = cudaStreamWaitEvent(plan->side, plan->fork_ev, 0);
      if (er == cudaSuccess) er = cudaEventRecordWithFlags(plan->ev_stop, plan->side, rec_flags);
      if (er != cudaSuccess) return cuda_fail(er, "cudaEventRecord(timing stop)");
      joined = false;
    }
  }
  if (cascade && cascade->n_pre_splits > 0 && !prefix_first) {
    // a prefix tree's levels are work-list pairs (after the decode grid); a
    // single shared prefix runs here only when there is no decode grid
    cudaError_t e = cascade->pp.work
                        ? pkd::launch_tile2(cascade->tmq, cascade->tmk, cascade->tmv, cascade->pp, plan->kv_dtype, st,
                                            true)
                        : pkd::launch_prefix(cascade->tmq, cascade->tmk, cascade->tmv, cascade->pp, plan->q_dtype,
                                             plan->kv_dtype, st, true);
    if (e != cudaSuccess) return cuda_fail(e, "prefix kernel launch");
  }
  // plain decode merges its split rows and writes its empty rows in the decode
  // kernel; the merge kernel runs for the cascade and for a plan without items
  if (!cascade && plan->counts.n_items > 0) {
    if (!joined) {  // the side branch rejoins the call's stream
      cudaError_t e = cudaEventRecord(plan->join_ev, plan->side);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(st, plan->join_ev, 0);
      if (e != cudaSuccess) return cuda_fail(e, "side branch join");
    }
    return PKD_OK;
  }
  pkd::MergeParams m{};
  m.merge_rows = reinterpret_cast<const int*>(ws + L.merge_rows);
  m.header = reinterpret_cast<const pkd::WsHeader*>(ws);
  m.row_item_begin = reinterpret_cast<const int*>(ws + L.row_begin);
  m.row_item_count = reinterpret_cast<const int*>(ws + L.row_count);
  m.part_o = p.part_o;
  m.part_lse = p.part_lse;
  m.pre_o = reinterpret_cast<const float*>(ws + L.pre_o);
  m.pre_lse = reinterpret_cast<const float*>(ws + L.pre_lse);
  m.n_pre_splits = cascade ? cascade->n_pre_splits : 0;
  m.out = d_out;
  m.lse = d_lse;
  m.out_dtype = plan->q_dtype;
  m.num_kv_heads = plan->hk;
  m.group = p.group;
  m.all_rows = cascade ? 1 : 0;
  // a fixed grid (graph-static): one CTA per decode CTA for the split rows,
  // two for the cascade, which merges every row.  The grid becomes resident as
  // the decode grid drains; a larger one took longer to launch than its warps
  // saved (batch-64 GQA: merge tail 8.6 us with 4x, 4.2 us with 1x; cascade
  // step 128.3 us with 4x, 124.6 us with 2x, 129 us with 1x)
  cudaError_t e = pkd::launch_merge_rows(m, cascade ? 2 * plan->G : plan->G, st);
  if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
  if (!joined) {  // the side branch rejoins the call's stream
    e = cudaEventRecord(plan->join_ev, plan->side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, plan->join_ev, 0);
    if (e != cudaSuccess) return cuda_fail(e, "side branch join");
  }
  return PKD_OK;
}

// Two work-list units with the same keys: one CTA of the paired-tile kernel.
struct UnitPair {
  pkd::TileWork a, b;
};

// The pairs as the kernel's list, longest key range first: the grid takes
// them in list order, so the long ones do not start last.
std::vector<pkd::TileWork> longest_first(std::vector<UnitPair>& pairs) {
  std::stable_sort(pairs.begin(), pairs.end(),
                   [](const UnitPair& x, const UnitPair& y) { return x.a.t1 - x.a.t0 > y.a.t1 - y.a.t0; });
  std::vector<pkd::TileWork> w;
  w.reserve(2 * pairs.size());
  for (const UnitPair& q : pairs) {
    w.push_back(q.a);
    w.push_back(q.b);
  }
  return w;
}

// Paged prefill: the pairs of one request together (its K/V then stays in L2
// while its query tiles run; spread over the launch, a request's pages were
// read from DRAM 1.29 times on the append-prefill workload), requests in
// order of their longest pair and each request's pairs longest first, so the
// long ones still do not start last.  A request's pairs are contiguous in
// `pairs` (built request by request).
std::vector<pkd::TileWork> by_request_longest_first(std::vector<UnitPair>& pairs) {
  auto len = [](const UnitPair& x) { return x.a.t1 - x.a.t0; };
  auto same_request = [](const UnitPair& x, const UnitPair& y) { return x.a.page_begin == y.a.page_begin && x.a.q_end == y.a.q_end; };
  std::vector<std::vector<UnitPair>> groups;
  for (const UnitPair& q : pairs) {
    if (groups.empty() || !same_request(groups.back().front(), q)) groups.emplace_back();
    groups.back().push_back(q);
  }
  for (auto& g : groups) std::stable_sort(g.begin(), g.end(), [&](const UnitPair& x, const UnitPair& y) { return len(x) > len(y); });
  std::stable_sort(groups.begin(), groups.end(),
                   [&](const std::vector<UnitPair>& x, const std::vector<UnitPair>& y) { return len(x.front()) > len(y.front()); });
  std::vector<pkd::TileWork> w;
  w.reserve(2 * pairs.size());
  for (const auto& g : groups)
    for (const UnitPair& q : g) {
      w.push_back(q.a);
      w.push_back(q.b);
    }
  return w;
}

// Prefix-tree work units (host): validates the levels, cuts each level into
// key-range pieces and pairs each node's 128-row query tiles.  Shared by
// pkd_plan_tree and the host-only pkd_tree_units_host.
pkd_status tree_units(int num_levels, const int32_t* const* h_req_indptr, const int32_t* const* h_kv_indptr,
                      const int32_t* const* h_kv_last_page_len, const int32_t* h_num_nodes, int B, int g,
                      int num_kv_heads, int P, int sms, int max_splits, std::vector<pkd::TileWork>* w,
                      int* pieces_out) {
  if (num_levels < 1 || num_levels > pkd::kMaxTreeLevels)
    return fail(PKD_ERR_UNSUPPORTED, "num_levels %d outside 1..%d", num_levels, pkd::kMaxTreeLevels);
  if (!h_req_indptr || !h_kv_indptr || !h_kv_last_page_len || !h_num_nodes)
    return fail(PKD_ERR_INVALID_ARG, "NULL level array");
  if (max_splits < num_levels)
    return fail(PKD_ERR_CAPACITY_EXCEEDED, "the plan was created with max_prefix_splits %d < %d levels",
                max_splits, num_levels);
  if (g < 1 || pkd::kHeadDim % g != 0) return fail(PKD_ERR_UNSUPPORTED, "group size %d does not divide 128", g);
  if (P < 1) return fail(PKD_ERR_INVALID_ARG, "page_size must be >= 1");
  if (sms < 1) return fail(PKD_ERR_INVALID_ARG, "num_ctas must be >= %d", pkd::kCtasPerSm);
  const int per_tile = 128 / g;  // requests per 128-row query tile
  // validate the levels and find each level's longest node (in key tiles)
  std::vector<int> level_max_tiles(num_levels, 0);
  for (int l = 0; l < num_levels; ++l) {
    const int nn = h_num_nodes[l];
    const int32_t* ri = h_req_indptr[l];
    const int32_t* ki = h_kv_indptr[l];
    const int32_t* lp = h_kv_last_page_len[l];
    if (nn < 1 || !ri || !ki || (!lp && nn > 0)) return fail(PKD_ERR_INVALID_ARG, "level %d: bad node arrays", l);
    if (ri[0] != 0 || ri[nn] != B) return fail(PKD_ERR_INVALID_ARG, "level %d: nodes must cover requests 0..%d", l, B);
    if (ki[0] != 0) return fail(PKD_ERR_INVALID_ARG, "level %d: kv_indptr[0] must be 0", l);
    for (int n = 0; n < nn; ++n) {
      if (ri[n + 1] < ri[n] || ki[n + 1] < ki[n])
        return fail(PKD_ERR_INVALID_ARG, "level %d node %d: decreasing indptr", l, n);
      const int pages = ki[n + 1] - ki[n];
      if (pages > 0 && (lp[n] < 1 || lp[n] > P))
        return fail(PKD_ERR_INVALID_ARG, "level %d node %d: last_page_len %d outside 1..%d", l, n, lp[n], P);
      const int64_t len = pages > 0 ? static_cast<int64_t>(pages - 1) * P + lp[n] : 0;
      if (len > INT32_MAX - 128) return fail(PKD_ERR_INVALID_ARG, "level %d node %d: too many keys", l, n);
      const int tiles = static_cast<int>((len + 127) / 128);
      level_max_tiles[l] = tiles > level_max_tiles[l] ? tiles : level_max_tiles[l];
    }
  }
  // key-range pieces per level.  A CTA's cost per 128-key tile: its pair of
  // query tiles takes ~1.43 times as long as a lone tile (the last, odd tile
  // of a node; ~3.9 against ~2.75 us on GB300).  The launch's cost over the
  // SMs is the average load; each level is cut so that its longest unit's
  // pieces cost at most 3/4 of it (pieces as long as the average next to
  // short ones leave SMs idle at the end), within the plan's piece budget
  // (each level keeps one).
  constexpr int64_t kCostPair = 143, kCostLone = 100;  // per key tile
  int64_t cost = 0;                                    // the launch, with one piece per level
  std::vector<int64_t> level_max_cost(num_levels, 0);  // the costliest unit of each level
  for (int l = 0; l < num_levels; ++l) {
    const int32_t* ri = h_req_indptr[l];
    const int32_t* ki = h_kv_indptr[l];
    const int32_t* lp = h_kv_last_page_len[l];
    for (int n = 0; n < h_num_nodes[l]; ++n) {
      const int pages = ki[n + 1] - ki[n];
      const int64_t len = pages > 0 ? static_cast<int64_t>(pages - 1) * P + lp[n] : 0;
      const int64_t tiles = (len + 127) / 128;
      const int64_t qt = (ri[n + 1] - ri[n] + per_tile - 1) / per_tile;  // query tiles of the node
      cost += ((qt / 2) * kCostPair + (qt % 2) * kCostLone) * tiles;
      const int64_t unit = (qt >= 2 ? kCostPair : kCostLone) * tiles;
      level_max_cost[l] = unit > level_max_cost[l] ? unit : level_max_cost[l];
    }
  }
  cost *= num_kv_heads;
  int64_t target = (3 * cost) / (4 * static_cast<int64_t>(sms));
  target = target > 2 * kCostLone ? target : 2 * kCostLone;
  std::vector<int> S(num_levels, 1);
  int budget = max_splits;
  for (int l = 0; l < num_levels; ++l) {
    int64_t want = (level_max_cost[l] + target - 1) / target;
    want = want < 1 ? 1 : (want > level_max_tiles[l] && level_max_tiles[l] > 0 ? level_max_tiles[l] : want);
    const int cap = budget - (num_levels - 1 - l);
    S[l] = want > cap ? cap : static_cast<int>(want);
    budget -= S[l];
  }
  // units in pairs (two query tiles of one node with the same keys: one CTA
  // per pair and kv head); a node's lone last tile is paired with a tile
  // without rows, which the kernel skips
  std::vector<UnitPair> pairs;
  int piece = 0;
  for (int l = 0; l < num_levels; ++l) {
    const int32_t* ri = h_req_indptr[l];
    const int32_t* ki = h_kv_indptr[l];
    const int32_t* lp = h_kv_last_page_len[l];
    for (int n = 0; n < h_num_nodes[l]; ++n) {
      const int pages = ki[n + 1] - ki[n];
      const int len = pages > 0 ? (pages - 1) * P + lp[n] : 0;
      const int tiles = (len + 127) / 128;
      const int tps = tiles > 0 ? (tiles + S[l] - 1) / S[l] : 0;
      for (int r0 = ri[n]; r0 < ri[n + 1]; r0 += 2 * per_tile) {
        for (int sp = 0; sp < S[l]; ++sp) {
          pkd::TileWork t{};
          t.q0 = r0;
          t.q_end = ri[n + 1];
          t.page_begin = ki[n];
          t.kv_len = len;
          t.t0 = sp * tps < tiles ? sp * tps : tiles;
          t.t1 = (sp + 1) * tps < tiles ? (sp + 1) * tps : tiles;
          t.piece = piece + sp;  // every piece of every request is written (empty ranges as empty states)
          t.level = l;
          t.diag = pkd::kNoCausal;
          pkd::TileWork u = t;
          u.q0 = r0 + per_tile < ri[n + 1] ? r0 + per_tile : ri[n + 1];
          pairs.push_back({t, u});
        }
      }
    }
    piece += S[l];
  }
  *w = longest_first(pairs);
  *pieces_out = piece;
  return PKD_OK;
}

// Paged-prefill work units (host): validates the requests and pairs each
// request's 128-row query tiles.  Shared by pkd_plan_prefill and the
// host-only pkd_prefill_units_host.
pkd_status prefill_units(const int32_t* h_qo_indptr, const int32_t* h_kv_indptr, const int32_t* h_kv_last_page_len,
                         int batch, int g, int page_size, bool causal, std::vector<pkd::TileWork>* w) {
  if (batch < 0) return fail(PKD_ERR_INVALID_ARG, "batch must be >= 0");
  if (page_size < 1) return fail(PKD_ERR_INVALID_ARG, "page_size must be >= 1");
  if (g < 1 || pkd::kHeadDim % g != 0) return fail(PKD_ERR_UNSUPPORTED, "group size %d does not divide 128", g);
  if (!h_qo_indptr || !h_kv_indptr || (batch > 0 && !h_kv_last_page_len))
    return fail(PKD_ERR_INVALID_ARG, "NULL host array");
  if (h_qo_indptr[0] != 0 || h_kv_indptr[0] != 0) return fail(PKD_ERR_INVALID_ARG, "indptr[0] must be 0");
  const int per_tile = 128 / g;  // query tokens per 128-row tile
  std::vector<UnitPair> pairs;
  for (int r = 0; r < batch; ++r) {
    const int q_len = h_qo_indptr[r + 1] - h_qo_indptr[r];
    const int pages = h_kv_indptr[r + 1] - h_kv_indptr[r];
    if (q_len < 0 || pages < 0) return fail(PKD_ERR_INVALID_ARG, "request %d: decreasing indptr", r);
    if (pages > 0 && (h_kv_last_page_len[r] < 1 || h_kv_last_page_len[r] > page_size))
      return fail(PKD_ERR_INVALID_ARG, "request %d: last_page_len %d outside 1..%d", r, h_kv_last_page_len[r],
                  page_size);
    const int64_t len64 = pages > 0 ? static_cast<int64_t>(pages - 1) * page_size + h_kv_last_page_len[r] : 0;
    if (len64 > INT32_MAX - 128) return fail(PKD_ERR_INVALID_ARG, "request %d: too many keys", r);
    const int kv_len = static_cast<int>(len64);
    if (q_len > kv_len)
      return fail(PKD_ERR_INVALID_ARG, "request %d: %d query tokens but %d keys (the new tokens' keys are in "
                  "the cache)", r, q_len, kv_len);
    const int q0 = h_qo_indptr[r], q_end = h_qo_indptr[r + 1];
    const int diag = kv_len - q_len - q0;  // token q sits at position q + diag
    // query tiles in pairs (one CTA for both, every key tile read once for
    // 256 rows): both take the key tiles the later tile's last row sees; a
    // lone last tile is paired with a tile without rows, which the kernel skips
    for (int a = q0; a < q_end; a += 2 * per_tile) {
      const int last_tok = (a + 2 * per_tile < q_end ? a + 2 * per_tile : q_end) - 1;
      const int keys = causal ? last_tok + diag + 1 : kv_len;  // keys the pair's last row sees
      pkd::TileWork t{};
      t.q0 = a;
      t.q_end = q_end;
      t.page_begin = h_kv_indptr[r];
      t.kv_len = kv_len;
      t.t0 = 0;
      t.t1 = (keys + 127) / 128;
      t.piece = -1;
      t.level = 0;
      t.diag = causal ? diag : pkd::kNoCausal;
      pkd::TileWork u = t;
      u.q0 = a + per_tile < q_end ? a + per_tile : q_end;
      pairs.push_back({t, u});
    }
  }
  *w = by_request_longest_first(pairs);
  return PKD_OK;
}

// Copy a unit list out as int32 [n][12] (TileWork's field order).
pkd_status export_units(const std::vector<pkd::TileWork>& w, int32_t* units_out, int max_units,
                               int* n_units_out) {
  static_assert(sizeof(pkd::TileWork) == 12 * sizeof(int32_t), "a unit is 12 int32");
  if (!n_units_out) return fail(PKD_ERR_INVALID_ARG, "n_units_out is NULL");
  *n_units_out = static_cast<int>(w.size());
  if (static_cast<int64_t>(w.size()) > max_units)
    return fail(PKD_ERR_CAPACITY_EXCEEDED, "%zu units above max_units %d", w.size(), max_units);
  if (!w.empty() && !units_out) return fail(PKD_ERR_INVALID_ARG, "units_out is NULL");
  if (!w.empty()) memcpy(units_out, w.data(), sizeof(pkd::TileWork) * w.size());
  return PKD_OK;
}

// Upload work-list units into the workspace's work region: copied into the
// plan's pinned buffer (after the previous upload from it has finished), then
// one cudaMemcpyAsync on `st`.
pkd_status upload_work(pkd_plan_t plan, const std::vector<pkd::TileWork>& w, cudaStream_t st) {
  if (static_cast<int64_t>(w.size()) > plan->lay.max_work)
    return fail(PKD_ERR_CAPACITY_EXCEEDED, "%zu work units above the workspace's %d", w.size(), plan->lay.max_work);
  cudaError_t e = cudaSuccess;
  if (!plan->work_staging) {
    e = cudaHostAlloc(reinterpret_cast<void**>(&plan->work_staging),
                      sizeof(pkd::TileWork) * static_cast<size_t>(plan->lay.max_work), cudaHostAllocDefault);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&plan->work_done, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "work staging buffer");
  } else {
    e = cudaEventSynchronize(plan->work_done);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize(work staging)");
  }
  if (!w.empty()) {
    memcpy(plan->work_staging, w.data(), sizeof(pkd::TileWork) * w.size());
    e = cudaMemcpyAsync(plan->ws + plan->lay.work, plan->work_staging, sizeof(pkd::TileWork) * w.size(),
                        cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "work upload");
  }
  e = cudaEventRecord(plan->work_done, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(work upload)");
  plan->n_work = static_cast<int>(w.size());
  return PKD_OK;
}

// Tensor map over query rows viewed as [rows][Hk][g][128] (rows = requests or
// tokens): a box of 128 / g rows x g heads of one kv head is one 128-row tile.
pkd_status encode_q_tile_map(CUtensorMap* m, const void* q, int q_dtype, int g, int hk, int64_t rows) {
  auto enc = get_encode();
  if (!enc) return fail(PKD_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t qdims[4] = {static_cast<cuuint64_t>(pkd::kHeadDim), static_cast<cuuint64_t>(g),
                         static_cast<cuuint64_t>(hk), static_cast<cuuint64_t>(rows)};
  cuuint64_t qstr[3] = {static_cast<cuuint64_t>(pkd::kHeadDim) * 2, static_cast<cuuint64_t>(g) * pkd::kHeadDim * 2,
                        static_cast<cuuint64_t>(hk) * g * pkd::kHeadDim * 2};
  cuuint32_t qbox[4] = {64u, static_cast<cuuint32_t>(g), 1u, static_cast<cuuint32_t>(128 / g)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, q_dtype == PKD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                   const_cast<void*>(q), qdims, qstr, qbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKD_ERR_CUDA, "cuTensorMapEncodeTiled(q) failed (CUresult %d)", (int)r);
  return PKD_OK;
}

// Checks shared by the tile-attention entry points: 16-bit K/V of q's type, a
// group size dividing 128, a page size the kernel's boxes cover.
pkd_status check_tile_geometry(int q_dtype, int kv_dtype, int g, int P, const char* what) {
  if (kv_dtype == PKD_E4M3 || !(kv_dtype == PKD_F16 || kv_dtype == PKD_BF16) || q_dtype != kv_dtype)
    return fail(PKD_ERR_UNSUPPORTED, "%s is built for f16/bf16 q and K/V of one type", what);
  if (pkd::kHeadDim % g != 0) return fail(PKD_ERR_UNSUPPORTED, "%s needs a group size dividing 128", what);
  if (P <= pkd::kChunkKeys ? (128 % P != 0) : (P % pkd::kChunkKeys != 0))
    return fail(PKD_ERR_UNSUPPORTED, "%s needs a page size dividing 128 or a multiple of 64", what);
  return PKD_OK;
}

// Validate a pool and encode its K/V maps for the tile-attention kernel.
pkd_status tile_kv_maps(pkd_plan_t plan, int kv_dtype, int P, const void* d_k, const void* d_v, int64_t num_pages,
                        int64_t page_stride_elems, CUtensorMap* tmk, CUtensorMap* tmv) {
  if (!d_k || !d_v || !aligned16(d_k) || !aligned16(d_v))
    return fail(PKD_ERR_INVALID_ARG, "k/v cache must be non-NULL and 16-byte aligned");
  if (num_pages <= 0 || num_pages > INT32_MAX) return fail(PKD_ERR_INVALID_ARG, "num_pages out of range");
  if ((page_stride_elems * elem_bytes(kv_dtype)) % 16 != 0 ||
      page_stride_elems < static_cast<int64_t>(P) * plan->hk * plan->d)
    return fail(PKD_ERR_INVALID_ARG, "page_stride_elems must cover a page and be a 16-byte multiple");
  const int box_tok = P <= pkd::kChunkKeys ? P : pkd::kChunkKeys;
  const bool hnd = plan->kv_layout == PKD_LAYOUT_HND;
  pkd_status s = encode_kv_map(tmk, d_k, kv_dtype, plan->hk, P, num_pages, page_stride_elems, box_tok, hnd);
  if (s != PKD_OK) return s;
  return encode_kv_map(tmv, d_v, kv_dtype, plan->hk, P, num_pages, page_stride_elems, box_tok, hnd);
}

// Parameters common to the work-list launches.
pkd::PrefixParams tile_params(pkd_plan_t plan, int P, int64_t num_pages, float sm_scale) {
  pkd::PrefixParams pp{};
  const float scale = (sm_scale > 0.f) ? sm_scale : 1.0f / std::sqrt(static_cast<float>(plan->d));
  pp.num_kv_heads = plan->hk;
  pp.group = plan->hq / plan->hk;
  pp.num_pages = static_cast<int>(num_pages);
  pp.page_size = P;
  pp.box_tok = P <= pkd::kChunkKeys ? P : pkd::kChunkKeys;
  pp.cluster = 1;
  pp.n_splits = 1;
  pp.m_groups = 1;
  pp.scale_log2 = scale * 1.4426950408889634f;
  pp.err = reinterpret_cast<unsigned*>(plan->ws);
  pp.kv_hnd = plan->kv_layout == PKD_LAYOUT_HND ? 1 : 0;
  pp.work = reinterpret_cast<const pkd::TileWork*>(plan->ws + plan->lay.work);
  pp.n_work = plan->n_work;
  for (int l = 0; l < pkd::kMaxTreeLevels; ++l) pp.level_pages[l] = plan->level_pages[l];
  return pp;
}

}  // namespace

extern "C" {

pkd_status pkd_run(pkd_plan_t plan, const void* d_q, const void* d_k_cache, const void* d_v_cache,
                   int64_t num_pages, int64_t page_stride_elems, const float* d_k_scale,
                   const float* d_v_scale, float sm_scale, void* d_out, float* d_lse, void* stream) {
  if (!plan) return fail(PKD_ERR_INVALID_ARG, "plan is NULL");
  return run_common(plan, d_q, d_k_cache, d_v_cache, num_pages, page_stride_elems, plan->page_size,
                    d_k_scale, d_v_scale, sm_scale, d_out, d_lse, stream, nullptr);
}

pkd_status pkd_cascade_decode(pkd_plan_t plan, const int32_t* d_prefix_page_indices,
                              int prefix_num_pages, int prefix_last_page_len, const void* d_q,
                              const void* d_k_cache, const void* d_v_cache, int64_t num_pages,
                              int64_t page_stride_elems, const float* d_k_scale,
                              const float* d_v_scale, float sm_scale, void* d_out, float* d_lse,
                              void* stream) {
  if (!plan) return fail(PKD_ERR_INVALID_ARG, "plan is NULL");
  if (!plan->planned) return fail(PKD_ERR_NO_PLAN, "cascade_decode before a successful plan");
  if (plan->max_splits < 1)
    return fail(PKD_ERR_CAPACITY_EXCEEDED, "the plan was created with max_prefix_splits = 0");
  const int g = plan->hq / plan->hk;
  const int P = plan->page_size;
  const bool fp8 = plan->kv_dtype == PKD_E4M3;
  if (prefix_num_pages < 0) return fail(PKD_ERR_INVALID_ARG, "prefix_num_pages must be >= 0");
  if (prefix_num_pages > 0 && (prefix_last_page_len < 1 || prefix_last_page_len > P))
    return fail(PKD_ERR_INVALID_ARG, "prefix_last_page_len %d outside 1..page_size", prefix_last_page_len);
  if (prefix_num_pages > 0 && !d_prefix_page_indices)
    return fail(PKD_ERR_INVALID_ARG, "d_prefix_page_indices is NULL");
  if (fp8 && (!d_k_scale || !d_v_scale)) return fail(PKD_ERR_INVALID_ARG, "an E4M3 cache needs k_scale and v_scale");
  const int64_t prefix_len64 = prefix_num_pages > 0 ? static_cast<int64_t>(prefix_num_pages - 1) * P + prefix_last_page_len : 0;
  if (prefix_len64 > INT32_MAX) return fail(PKD_ERR_INVALID_ARG, "prefix longer than 2^31 - 1 keys");
  const int prefix_len = static_cast<int>(prefix_len64);
  const int B = plan->batch;
  int n_pre = 0;
  CascadeMerge cm{};
  if (prefix_len > 0 && B > 0) {
    if (!d_q || !aligned16(d_q)) return fail(PKD_ERR_INVALID_ARG, "q must be non-NULL and 16-byte aligned");
    if (!d_k_cache || !d_v_cache || !aligned16(d_k_cache) || !aligned16(d_v_cache))
      return fail(PKD_ERR_INVALID_ARG, "k/v cache must be non-NULL and 16-byte aligned");
    if (num_pages <= 0 || num_pages > INT32_MAX) return fail(PKD_ERR_INVALID_ARG, "num_pages out of range");
    if ((page_stride_elems * elem_bytes(plan->kv_dtype)) % 16 != 0 ||
        page_stride_elems < static_cast<int64_t>(P) * plan->hk * plan->d)
      return fail(PKD_ERR_INVALID_ARG, "page_stride_elems must cover a page and be a 16-byte multiple");
    // Each CTA of the prefix kernel holds R = floor(128 / g) requests (R * g
    // query rows) of one kv head; two CTAs form a pair.  Key-range splits fill
    // the pairs that fit on the GPU at once.
    const int R = pkd::kHeadDim / g;
    const int n_tiles = (prefix_len + 127) / 128;
    const int m_tiles = (B + R - 1) / R;
    const int m_pairs = (m_tiles + 1) / 2;
    int resident = resident_prefix_clusters(plan->q_dtype, plan->kv_dtype);
    if (resident <= 0) resident = plan->G / (2 * pkd::kCtasPerSm);
    int splits = resident / (plan->hk * m_pairs);
    splits = splits < 1 ? 1 : splits;
    splits = splits > plan->max_splits ? plan->max_splits : splits;
    splits = splits > n_tiles ? n_tiles : splits;
    const int tps = (n_tiles + splits - 1) / splits;
    splits = (n_tiles + tps - 1) / tps;
    // boxes of gcd(P, 64) keys never cross a page, whatever the page size
    const int box_tok = gcd_int(P, 64);
    auto enc = get_encode();
    if (!enc) return fail(PKD_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    CUtensorMap tmq, tmk, tmv;
    // q viewed as [B][Hk][g][128]: a box of R requests x g heads of one kv head
    cuuint64_t qdims[4] = {static_cast<cuuint64_t>(pkd::kHeadDim), static_cast<cuuint64_t>(g),
                           static_cast<cuuint64_t>(plan->hk), static_cast<cuuint64_t>(B)};
    cuuint64_t qstr[3] = {static_cast<cuuint64_t>(pkd::kHeadDim) * 2, static_cast<cuuint64_t>(g) * pkd::kHeadDim * 2,
                          static_cast<cuuint64_t>(plan->hq) * pkd::kHeadDim * 2};
    cuuint32_t qbox[4] = {64u, static_cast<cuuint32_t>(g), 1u, static_cast<cuuint32_t>(R)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(&tmq, plan->q_dtype == PKD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     4, const_cast<void*>(d_q), qdims, qstr, qbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKD_ERR_CUDA, "cuTensorMapEncodeTiled(q) failed (CUresult %d)", (int)r);
    const bool hnd = plan->kv_layout == PKD_LAYOUT_HND;
    pkd_status s;
    if (fp8) {
      s = encode_code_map(&tmk, d_k_cache, plan->hk, P, num_pages, page_stride_elems, box_tok, 128, hnd);
      if (s != PKD_OK) return s;
      s = encode_code_map(&tmv, d_v_cache, plan->hk, P, num_pages, page_stride_elems, box_tok, 64, hnd);
    } else {
      s = encode_kv_map(&tmk, d_k_cache, plan->kv_dtype, plan->hk, P, num_pages, page_stride_elems, box_tok, hnd);
      if (s != PKD_OK) return s;
      s = encode_kv_map(&tmv, d_v_cache, plan->kv_dtype, plan->hk, P, num_pages, page_stride_elems, box_tok, hnd);
    }
    if (s != PKD_OK) return s;
    const float scale = (sm_scale > 0.f) ? sm_scale : 1.0f / std::sqrt(static_cast<float>(plan->d));
    pkd::PrefixParams pp{};
    pp.prefix_pages = d_prefix_page_indices;
    pp.n_prefix_pages = prefix_num_pages;
    pp.prefix_len = prefix_len;
    pp.batch = B;
    pp.num_kv_heads = plan->hk;
    pp.group = g;
    pp.num_pages = static_cast<int>(num_pages);
    pp.page_size = P;
    pp.box_tok = box_tok;
    pp.n_splits = splits;
    pp.tiles_per_split = tps;
    pp.m_tiles = m_tiles;
    pp.cluster = 2;
    pp.m_groups = m_pairs;
    pp.req_per_tile = R;
    pp.scale_log2 = scale * 1.4426950408889634f;
    pp.pre_o = reinterpret_cast<float*>(plan->ws + plan->lay.pre_o);
    pp.pre_lse = reinterpret_cast<float*>(plan->ws + plan->lay.pre_lse);
    pp.k_scale = d_k_scale;
    pp.v_scale = d_v_scale;
    pp.err = reinterpret_cast<unsigned*>(plan->ws);
    pp.kv_hnd = hnd ? 1 : 0;
    pp.rows_per_piece = B * plan->hq;
    cm.tmq = tmq;
    cm.tmk = tmk;
    cm.tmv = tmv;
    cm.pp = pp;
    n_pre = splits;
  }
  cm.n_pre_splits = n_pre;
  return run_common(plan, d_q, d_k_cache, d_v_cache, num_pages, page_stride_elems, P, d_k_scale, d_v_scale,
                    sm_scale, d_out, d_lse, stream, nullptr, &cm);
}

pkd_status pkd_prefill_units_host(const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                                  const int32_t* h_kv_last_page_len, int batch, int num_qo_heads,
                                  int num_kv_heads, int page_size, int causal, int32_t* units_out, int max_units,
                                  int* n_units_out) {
  if (num_kv_heads <= 0 || num_qo_heads <= 0 || num_qo_heads % num_kv_heads != 0)
    return fail(PKD_ERR_INVALID_ARG, "num_qo_heads must be a positive multiple of num_kv_heads");
  std::vector<pkd::TileWork> w;
  pkd_status s = prefill_units(h_qo_indptr, h_kv_indptr, h_kv_last_page_len, batch, num_qo_heads / num_kv_heads,
                               page_size, causal != 0, &w);
  if (s != PKD_OK) return s;
  return export_units(w, units_out, max_units, n_units_out);
}

pkd_status pkd_tree_units_host(int num_levels, const int32_t* const* h_req_indptr,
                               const int32_t* const* h_kv_indptr, const int32_t* const* h_kv_last_page_len,
                               const int32_t* h_num_nodes, int batch, int num_qo_heads, int num_kv_heads,
                               int page_size, int num_ctas, int max_prefix_splits, int32_t* units_out,
                               int max_units, int* n_units_out, int* n_pieces_out) {
  if (num_kv_heads <= 0 || num_qo_heads <= 0 || num_qo_heads % num_kv_heads != 0)
    return fail(PKD_ERR_INVALID_ARG, "num_qo_heads must be a positive multiple of num_kv_heads");
  if (batch < 0) return fail(PKD_ERR_INVALID_ARG, "batch must be >= 0");
  if (!n_pieces_out) return fail(PKD_ERR_INVALID_ARG, "n_pieces_out is NULL");
  std::vector<pkd::TileWork> w;
  int pieces = 0;
  pkd_status s = tree_units(num_levels, h_req_indptr, h_kv_indptr, h_kv_last_page_len, h_num_nodes, batch,
                            num_qo_heads / num_kv_heads, num_kv_heads, page_size, num_ctas / pkd::kCtasPerSm,
                            max_prefix_splits, &w, &pieces);
  if (s != PKD_OK) return s;
  *n_pieces_out = pieces;
  return export_units(w, units_out, max_units, n_units_out);
}

pkd_status pkd_plan_tree(pkd_plan_t plan, int num_levels, const int32_t* const* h_req_indptr,
                         const int32_t* const* h_kv_indptr, const int32_t* const* d_kv_page_indices,
                         const int32_t* const* h_kv_last_page_len, const int32_t* h_num_nodes, void* stream) {
  if (!plan) return fail(PKD_ERR_INVALID_ARG, "plan is NULL");
  if (!plan->planned) return fail(PKD_ERR_NO_PLAN, "pkd_plan_tree needs the requests' own pages planned first");
  const int g = plan->hq / plan->hk;
  const int P = plan->page_size;
  pkd_status s = check_tile_geometry(plan->q_dtype, plan->kv_dtype, g, P, "prefix-tree decode");
  if (s != PKD_OK) return s;
  std::vector<pkd::TileWork> w;
  int piece = 0;
  s = tree_units(num_levels, h_req_indptr, h_kv_indptr, h_kv_last_page_len, h_num_nodes, plan->batch, g, plan->hk,
                 P, plan->G / pkd::kCtasPerSm, plan->max_splits, &w, &piece);
  if (s != PKD_OK) return s;
  if (!d_kv_page_indices) return fail(PKD_ERR_INVALID_ARG, "NULL level array");
  for (int l = 0; l < num_levels; ++l)
    if (h_kv_indptr[l][h_num_nodes[l]] > 0 && !d_kv_page_indices[l])
      return fail(PKD_ERR_INVALID_ARG, "level %d: page indices NULL", l);
  s = upload_work(plan, w, static_cast<cudaStream_t>(stream));
  if (s != PKD_OK) return s;
  for (int l = 0; l < pkd::kMaxTreeLevels; ++l) plan->level_pages[l] = l < num_levels ? d_kv_page_indices[l] : nullptr;
  plan->tree_pieces = piece;
  plan->work_kind = 1;
  plan->work_gen = plan->plan_gen;
  return PKD_OK;
}

pkd_status pkd_tree_decode(pkd_plan_t plan, const void* d_q, const void* d_k_cache, const void* d_v_cache,
                           int64_t num_pages, int64_t page_stride_elems, float sm_scale, void* d_out,
                           float* d_lse, void* stream) {
  if (!plan) return fail(PKD_ERR_INVALID_ARG, "plan is NULL");
  if (!plan->planned || plan->work_kind != 1 || plan->work_gen != plan->plan_gen)
    return fail(PKD_ERR_NO_PLAN, "tree_decode needs pkd_plan_tree after the last pkd_plan");
  const int B = plan->batch;
  const int P = plan->page_size;
  const int g = plan->hq / plan->hk;
  CascadeMerge cm{};
  if (B > 0 && plan->n_work > 0) {
    if (!d_q || !aligned16(d_q)) return fail(PKD_ERR_INVALID_ARG, "q must be non-NULL and 16-byte aligned");
    pkd_status s = encode_q_tile_map(&cm.tmq, d_q, plan->q_dtype, g, plan->hk, B);
    if (s != PKD_OK) return s;
    s = tile_kv_maps(plan, plan->kv_dtype, P, d_k_cache, d_v_cache, num_pages, page_stride_elems, &cm.tmk, &cm.tmv);
    if (s != PKD_OK) return s;
    cm.pp = tile_params(plan, P, num_pages, sm_scale);
    cm.pp.batch = B;
    cm.pp.rows_per_piece = B * plan->hq;
    cm.pp.pre_o = reinterpret_cast<float*>(plan->ws + plan->lay.pre_o);
    cm.pp.pre_lse = reinterpret_cast<float*>(plan->ws + plan->lay.pre_lse);
    cm.n_pre_splits = plan->tree_pieces;
  }
  return run_common(plan, d_q, d_k_cache, d_v_cache, num_pages, page_stride_elems, P, nullptr, nullptr, sm_scale,
                    d_out, d_lse, stream, nullptr, &cm);
}

pkd_status pkd_plan_prefill(pkd_plan_t plan, const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                            const int32_t* d_kv_page_indices, const int32_t* h_kv_last_page_len, int batch,
                            int num_qo_heads, int num_kv_heads, int head_dim, int page_size, int q_dtype,
                            int kv_dtype, int causal, void* stream) {
  if (!plan) return fail(PKD_ERR_INVALID_ARG, "plan is NULL");
  if (num_qo_heads != plan->hq || num_kv_heads != plan->hk || head_dim != plan->d)
    return fail(PKD_ERR_INVALID_ARG, "head counts / head_dim differ from the plan's");
  if (batch < 0) return fail(PKD_ERR_INVALID_ARG, "batch must be >= 0");
  if (page_size < 1) return fail(PKD_ERR_INVALID_ARG, "page_size must be >= 1");
  const int g = plan->hq / plan->hk;
  pkd_status s = check_tile_geometry(q_dtype, kv_dtype, g, page_size, "prefill");
  if (s != PKD_OK) return s;
  std::vector<pkd::TileWork> w;
  s = prefill_units(h_qo_indptr, h_kv_indptr, h_kv_last_page_len, batch, g, page_size, causal != 0, &w);
  if (s != PKD_OK) return s;
  if (h_kv_indptr[batch] > 0 && !d_kv_page_indices) return fail(PKD_ERR_INVALID_ARG, "d_kv_page_indices is NULL");
  if (!plan->err_word_zeroed) {  // a plan used for prefill only: the first plan clears the error word
    cudaError_t ez = cudaMemsetAsync(plan->ws, 0, 4, static_cast<cudaStream_t>(stream));
    if (ez != cudaSuccess) return cuda_fail(ez, "cudaMemsetAsync(error word)");
    plan->err_word_zeroed = true;
  }
  s = upload_work(plan, w, static_cast<cudaStream_t>(stream));
  if (s != PKD_OK) return s;
  plan->level_pages[0] = d_kv_page_indices;
  for (int l = 1; l < pkd::kMaxTreeLevels; ++l) plan->level_pages[l] = nullptr;
  plan->pf_tokens = h_qo_indptr[batch];
  plan->pf_page_size = page_size;
  plan->pf_dtype = kv_dtype;
  plan->work_kind = 2;
  return PKD_OK;
}

pkd_status pkd_prefill_run(pkd_plan_t plan, const void* d_q, const void* d_k_cache, const void* d_v_cache,
                           int64_t num_pages, int64_t page_stride_elems, float sm_scale, void* d_out,
                           float* d_lse, void* stream) {
  if (!plan) return fail(PKD_ERR_INVALID_ARG, "plan is NULL");
  if (plan->work_kind != 2) return fail(PKD_ERR_NO_PLAN, "prefill_run before a successful pkd_plan_prefill");
  if (plan->n_work == 0) return PKD_OK;
  if (!d_q || !d_out || !aligned16(d_q) || !aligned16(d_out))
    return fail(PKD_ERR_INVALID_ARG, "q/out must be non-NULL and 16-byte aligned");
  const int P = plan->pf_page_size;
  const int g = plan->hq / plan->hk;
  CUtensorMap tmq, tmk, tmv;
  pkd_status s = encode_q_tile_map(&tmq, d_q, plan->pf_dtype, g, plan->hk, plan->pf_tokens);
  if (s != PKD_OK) return s;
  s = tile_kv_maps(plan, plan->pf_dtype, P, d_k_cache, d_v_cache, num_pages, page_stride_elems, &tmk, &tmv);
  if (s != PKD_OK) return s;
  pkd::PrefixParams pp = tile_params(plan, P, num_pages, sm_scale);
  pp.batch = plan->pf_tokens;
  pp.out = d_out;
  pp.lse = d_lse;
  pp.out_dtype = plan->pf_dtype;
  // not programmatic: the kernel reads K/V that the previous launch on the
  // stream (an append) may have written
  cudaError_t e = pkd::launch_tile2(tmq, tmk, tmv, pp, plan->pf_dtype, static_cast<cudaStream_t>(stream), false);
  if (e != cudaSuccess) return cuda_fail(e, "prefill kernel launch");
  return PKD_OK;
}

pkd_status pkd_append_kv(const void* d_k_new, const void* d_v_new, int new_dtype,
                         const int32_t* d_batch_indices, const int32_t* d_positions, int n_tokens,
                         const int32_t* d_kv_indptr, const int32_t* d_kv_page_indices, int batch,
                         int num_kv_heads, int head_dim, int page_size, void* d_k_cache,
                         void* d_v_cache, int kv_dtype, int kv_layout, int64_t num_pages,
                         int64_t page_stride_elems, const float* d_k_scale,
                         const float* d_v_scale, uint32_t* d_err_word, void* stream) {
  if (n_tokens < 0 || batch < 0 || num_kv_heads <= 0) return fail(PKD_ERR_INVALID_ARG, "bad n_tokens/batch/heads");
  if (kv_layout != PKD_LAYOUT_NHD && kv_layout != PKD_LAYOUT_HND)
    return fail(PKD_ERR_INVALID_ARG, "kv_layout %d (PKD_LAYOUT_NHD or PKD_LAYOUT_HND)", kv_layout);
  if (head_dim != pkd::kHeadDim) return fail(PKD_ERR_UNSUPPORTED, "head_dim %d (128 only)", head_dim);
  if (page_size < 1) return fail(PKD_ERR_INVALID_ARG, "page_size must be >= 1");
  const bool fp8 = kv_dtype == PKD_E4M3;
  if (!fp8 && !(kv_dtype == PKD_F16 || kv_dtype == PKD_BF16))
    return fail(PKD_ERR_UNSUPPORTED, "kv dtype %d", kv_dtype);
  if (!(new_dtype == PKD_F16 || new_dtype == PKD_BF16)) return fail(PKD_ERR_UNSUPPORTED, "new dtype %d", new_dtype);
  if (!fp8 && new_dtype != kv_dtype) return fail(PKD_ERR_UNSUPPORTED, "a 16-bit pool takes values of its own dtype");
  if (fp8 && (!d_k_scale || !d_v_scale)) return fail(PKD_ERR_INVALID_ARG, "an E4M3 pool needs k_scale and v_scale");
  if (n_tokens == 0) return PKD_OK;
  if (!d_k_new || !d_v_new || !d_batch_indices || !d_positions || !d_kv_indptr || !d_kv_page_indices ||
      !d_k_cache || !d_v_cache)
    return fail(PKD_ERR_INVALID_ARG, "NULL buffer");
  if (!aligned16(d_k_new) || !aligned16(d_v_new) || !aligned16(d_k_cache) || !aligned16(d_v_cache))
    return fail(PKD_ERR_INVALID_ARG, "new rows and pools must be 16-byte aligned");
  if (num_pages <= 0 || num_pages > INT32_MAX) return fail(PKD_ERR_INVALID_ARG, "num_pages out of range");
  if ((page_stride_elems * elem_bytes(kv_dtype)) % 16 != 0 ||
      page_stride_elems < static_cast<int64_t>(page_size) * num_kv_heads * head_dim)
    return fail(PKD_ERR_INVALID_ARG, "page_stride_elems must cover a page and be a 16-byte multiple");
  pkd::AppendParams p{};
  p.k_new = d_k_new;
  p.v_new = d_v_new;
  p.batch_indices = d_batch_indices;
  p.positions = d_positions;
  p.kv_indptr = d_kv_indptr;
  p.page_indices = d_kv_page_indices;
  p.k_cache = d_k_cache;
  p.v_cache = d_v_cache;
  p.k_scale = d_k_scale;
  p.v_scale = d_v_scale;
  p.err = d_err_word;
  p.page_stride = page_stride_elems;
  p.n_tokens = n_tokens;
  p.batch = batch;
  p.num_kv_heads = num_kv_heads;
  p.page_size = page_size;
  p.num_pages = static_cast<int>(num_pages);
  p.kv_hnd = kv_layout == PKD_LAYOUT_HND ? 1 : 0;
  cudaError_t e = pkd::launch_append_kv(p, new_dtype, kv_dtype, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append kernel launch");
  return PKD_OK;
}

pkd_status pkd_single_decode(const void* d_q, const void* d_k, const void* d_v, int kv_len,
                             int num_qo_heads, int num_kv_heads, int head_dim, int q_dtype,
                             int kv_dtype, const float* d_k_scale, const float* d_v_scale,
                             float sm_scale, void* d_out, float* d_lse, void* d_workspace,
                             size_t workspace_bytes, void* stream) {
  if (kv_len < 0) return fail(PKD_ERR_INVALID_ARG, "kv_len must be >= 0");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int G = 0;
  pkd_status s = pkd_num_ctas(dev, &G);
  if (s != PKD_OK) return s;
  pkd_plan_t plan = nullptr;
  s = pkd_plan_create(&plan, 1, num_qo_heads, num_kv_heads, head_dim, G, 0, d_workspace, workspace_bytes);
  if (s != PKD_OK) return s;
  // the contiguous [kv_len, Hk, D] tensor is one page; its page size is kv_len
  // rounded up to the 64-key chunk (the TMA map's key extent stays kv_len, so
  // keys past the end read as zeros and are masked)
  const int P = kv_len <= pkd::kChunkKeys ? (kv_len > 0 ? kv_len : 1)
                                          : ((kv_len + pkd::kChunkKeys - 1) / pkd::kChunkKeys) * pkd::kChunkKeys;
  const int32_t indptr[2] = {0, kv_len > 0 ? 1 : 0};
  const int32_t last[1] = {kv_len > 0 ? kv_len : 0};
  const int32_t* zero_page = reinterpret_cast<const int32_t*>(
      static_cast<uint8_t*>(d_workspace) + offsetof(pkd::WsHeader, zero_page));
  // a one-shot plan: the schedule goes in the upload kernel's parameters when
  // it fits (capturable), else by a pageable copy staged before return
  plan->use_pinned = false;
  plan->upload_by_blob = plan->lay.meta_end - 16 <= static_cast<size_t>(pkd::kBlobBytes);
  s = pkd_plan(plan, indptr, zero_page, last, 1, num_qo_heads, num_kv_heads, head_dim, P, q_dtype,
               kv_dtype, stream);
  if (s == PKD_OK) {
    // one page: its stride is never stepped, it only has to cover the page
    const int64_t stride = static_cast<int64_t>(P) * num_kv_heads * head_dim;
    s = run_common(plan, d_q, d_k, d_v, 1, stride, kv_len > 0 ? kv_len : 1, d_k_scale, d_v_scale, sm_scale,
                   d_out, d_lse, stream, zero_page);
  }
  pkd_plan_destroy(plan);
  return s;
}

pkd_status pkd_merge_state(const void* d_v_a, const float* d_s_a, const void* d_v_b, const float* d_s_b,
                           void* d_v_out, float* d_s_out, int64_t n, int num_heads, int head_dim,
                           int v_dtype, void* stream) {
  if (n < 0 || num_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0 || head_dim > 1024)
    return fail(PKD_ERR_INVALID_ARG, "n >= 0, num_heads > 0 and head_dim in 8..1024 (multiple of 8) required");
  if (v_dtype != PKD_F32 && v_dtype != PKD_F16 && v_dtype != PKD_BF16)
    return fail(PKD_ERR_UNSUPPORTED, "merge_state values must be F32, F16 or BF16");
  if (n > 0 && (!d_v_a || !d_s_a || !d_v_b || !d_s_b || !d_v_out || !d_s_out))
    return fail(PKD_ERR_INVALID_ARG, "NULL pointer");
  cudaError_t e = pkd::launch_merge_state(d_v_a, d_s_a, d_v_b, d_s_b, d_v_out, d_s_out, n, num_heads, head_dim,
                                          v_dtype, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge_state kernel launch");
  return PKD_OK;
}

pkd_status pkd_merge_states(const void* d_v, const float* d_s, int64_t n, int k, int num_heads,
                            int head_dim, int v_dtype, void* d_v_out, float* d_s_out, void* stream) {
  if (n < 0 || k < 0 || num_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0 || head_dim > 1024)
    return fail(PKD_ERR_INVALID_ARG, "n, k >= 0, num_heads > 0 and head_dim in 8..1024 (multiple of 8) required");
  if (v_dtype != PKD_F32 && v_dtype != PKD_F16 && v_dtype != PKD_BF16)
    return fail(PKD_ERR_UNSUPPORTED, "merge_states values must be F32, F16 or BF16");
  if (n > 0 && (!d_v_out || !d_s_out || (k > 0 && (!d_v || !d_s))))
    return fail(PKD_ERR_INVALID_ARG, "NULL pointer");
  cudaError_t e = pkd::launch_merge_states(d_v, d_s, n, k, num_heads, head_dim, v_dtype, d_v_out, d_s_out,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge_states kernel launch");
  return PKD_OK;
}

pkd_status pkd_plan_set_timing_events(pkd_plan_t plan, void* start_event, void* stop_event) {
  if (!plan) return fail(PKD_ERR_INVALID_ARG, "plan is NULL");
  if ((start_event == nullptr) != (stop_event == nullptr))
    return fail(PKD_ERR_INVALID_ARG, "give both timing events or neither");
  if (stop_event) {
    pkd_status ss = ensure_side(plan);
    if (ss != PKD_OK) return ss;
  }
  plan->ev_start = static_cast<cudaEvent_t>(start_event);
  plan->ev_stop = static_cast<cudaEvent_t>(stop_event);
  return PKD_OK;
}

pkd_status pkd_plan_set_kv_layout(pkd_plan_t plan, int kv_layout) {
  if (!plan) return fail(PKD_ERR_INVALID_ARG, "plan is NULL");
  if (kv_layout != PKD_LAYOUT_NHD && kv_layout != PKD_LAYOUT_HND)
    return fail(PKD_ERR_INVALID_ARG, "kv_layout %d (PKD_LAYOUT_NHD or PKD_LAYOUT_HND)", kv_layout);
  plan->kv_layout = kv_layout;
  return PKD_OK;
}

pkd_status pkd_plan_set_debug(pkd_plan_t plan, int flags) {
  if (!plan) return fail(PKD_ERR_INVALID_ARG, "plan is NULL");
  if (flags & ~PKD_DEBUG_STALL_PIPELINE) return fail(PKD_ERR_INVALID_ARG, "unknown debug flags 0x%x", flags);
  plan->debug_flags = flags;
  return PKD_OK;
}

pkd_status pkd_check_device_errors(pkd_plan_t plan, uint32_t* flags_out, void* stream) {
  if (!plan || !flags_out) return fail(PKD_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t flags = 0;
  cudaError_t e = cudaMemcpyAsync(&flags, plan->ws, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(plan->ws, 0, 4, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  *flags_out = flags;
  if (flags) return fail(PKD_ERR_DEVICE_CHECK, "device error bits 0x%x", flags);
  return PKD_OK;
}

}  // extern "C"
