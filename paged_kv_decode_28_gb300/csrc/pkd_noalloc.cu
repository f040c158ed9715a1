// pkd_noalloc.cu -- batched paged decode that allocates nothing.
//
// Who needs this: callers that are not allowed to allocate device memory at
// the point where they run decode attention -- for example a serving loop
// whose memory is carved out up front by its own pool allocator (cudaMalloc
// may synchronise the device and fragment the pool), a plugin hosted inside a
// runtime that owns every allocation, or code that must keep a fixed memory
// footprint for predictable latency.  The regular path asks the caller for a
// workspace buffer; this one uses a fixed scratch area compiled into the
// library instead, so the caller only passes inputs and outputs.
//
// The scratch area is a file-scope device array of kNoAllocScratchBytes.  It
// exists once per GPU that loads this library and stays allocated until the
// process exits.  Host code cannot use the array's name as a device address,
// so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it.
//
// The schedule is built on the host into a file-scope host buffer (guarded by
// a mutex) and uploaded with one cudaMemcpyAsync from that pageable buffer.
// For a pageable source the runtime copies the bytes into its own staging
// memory before cudaMemcpyAsync returns, so the host buffer may be reused once
// the call is back.  A copy captured into a CUDA graph would instead read the
// host buffer when the graph replays, so the call refuses to run while its
// stream is capturing.  The kernels are the same decode and merge kernels the
// plan/run path launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <cmath>
#include <mutex>
#include <string>

#include "pkd.h"
#include "pkd_host.h"
#include "pkd_internal.h"
#include "pkd_plan.h"

namespace {

constexpr size_t kNoAllocScratchBytes = PKD_NOALLOC_SCRATCH_BYTES;
constexpr size_t kHostMetaBytes = 256u << 10;  // host staging for the schedule
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_scratch[kNoAllocScratchBytes];

uint8_t g_host_meta[kHostMetaBytes] __attribute__((aligned(256)));
std::mutex g_host_mutex;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

using pkd::host::aligned16;
using pkd::host::align256;
using pkd::host::cuda_fail;
using pkd::host::fail;
using pkd::host::get_encode;

// Scratch layout for one call: the same regions as a plan workspace, sized
// exactly for this batch.
struct NaLayout {
  size_t cta_begin, items, merge_rows, row_begin, row_count, kv_len, page_begin, meta_end, part_o,
      part_lse, total;
  int max_items;
};

NaLayout na_layout(int batch, int hk, int group, int G) {
  NaLayout L{};
  const int rows = batch * hk;
  L.max_items = rows + G;
  size_t off = sizeof(pkd::WsHeader);
  L.cta_begin = off;
  off += align256(4ull * (G + 1));
  L.items = off;
  off += align256(16ull * L.max_items);
  L.merge_rows = off;
  off += align256(4ull * (rows > 0 ? rows : 1));
  L.row_begin = off;
  off += align256(4ull * (rows > 0 ? rows : 1));
  L.row_count = off;
  off += align256(4ull * (rows > 0 ? rows : 1));
  L.kv_len = off;
  off += align256(4ull * (batch > 0 ? batch : 1));
  L.page_begin = off;
  off += align256(4ull * (batch > 0 ? batch : 1));
  L.meta_end = off;
  L.part_o = off;
  off += align256(4ull * L.max_items * group * pkd::kHeadDim);
  L.part_lse = off;
  off += align256(4ull * L.max_items * group);
  L.total = off;
  return L;
}

// Device address of this device's scratch array (looked up once per device).
pkd_status scratch_for_current_device(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PKD_ERR_UNSUPPORTED, "device id %d above %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_scratch_addr[dev]);
  return PKD_OK;
}

// dims (dim, head, key, page) for NHD pages, (dim, key, head, page) for HND;
// a box is box_tok rows of one head of one page either way
pkd_status kv_map(CUtensorMap* m, const void* base, int kv_dtype, int hk, int64_t tok_extent,
                  int64_t num_pages, int64_t page_stride_elems, int box_tok, bool hnd) {
  auto enc = get_encode();
  if (!enc) return fail(PKD_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const int e = kv_dtype == PKD_E4M3 ? 1 : 2;
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
  CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B,
                   e == 1 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKD_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return PKD_OK;
}

}  // namespace

extern "C" pkd_status pkd_decode_noalloc(const int32_t* h_kv_indptr, const int32_t* d_kv_page_indices,
                                         const int32_t* h_kv_last_page_len, int batch, int num_qo_heads,
                                         int num_kv_heads, int head_dim, int page_size, int q_dtype,
                                         int kv_dtype, int kv_layout, const void* d_q, const void* d_k_cache,
                                         const void* d_v_cache, int64_t num_pages, int64_t page_stride_elems,
                                         const float* d_k_scale, const float* d_v_scale, float sm_scale,
                                         void* d_out, float* d_lse, void* stream) {
  // ---- arguments
  if (head_dim != pkd::kHeadDim) return fail(PKD_ERR_UNSUPPORTED, "head_dim must be 128 (got %d)", head_dim);
  if (num_kv_heads <= 0 || num_qo_heads <= 0 || num_qo_heads % num_kv_heads != 0)
    return fail(PKD_ERR_INVALID_ARG, "num_qo_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                num_qo_heads, num_kv_heads);
  const int group = num_qo_heads / num_kv_heads;
  if (group > pkd::kMaxGroup) return fail(PKD_ERR_UNSUPPORTED, "group size %d above %d", group, pkd::kMaxGroup);
  if (batch < 0) return fail(PKD_ERR_INVALID_ARG, "batch must be >= 0");
  const bool ok_pair = (q_dtype == PKD_F16 && kv_dtype == PKD_F16) || (q_dtype == PKD_BF16 && kv_dtype == PKD_BF16) ||
                       (q_dtype == PKD_BF16 && kv_dtype == PKD_E4M3) || (q_dtype == PKD_F16 && kv_dtype == PKD_E4M3);
  if (!ok_pair) return fail(PKD_ERR_UNSUPPORTED, "dtype pair (q %d, kv %d) not supported", q_dtype, kv_dtype);
  if (!h_kv_indptr || (batch > 0 && !h_kv_last_page_len))
    return fail(PKD_ERR_INVALID_ARG, "h_kv_indptr / h_kv_last_page_len is NULL");
  if (batch > 0 && (!d_q || !d_out)) return fail(PKD_ERR_INVALID_ARG, "q/out is NULL");
  if ((d_q && !aligned16(d_q)) || (d_out && !aligned16(d_out)))
    return fail(PKD_ERR_INVALID_ARG, "q/out must be 16-byte aligned");
  const bool fp8 = kv_dtype == PKD_E4M3;
  if (fp8 && (!d_k_scale || !d_v_scale)) return fail(PKD_ERR_INVALID_ARG, "an E4M3 cache needs k_scale and v_scale");
  if (!fp8 && (d_k_scale || d_v_scale))
    return fail(PKD_ERR_INVALID_ARG, "k_scale/v_scale apply to an E4M3 cache only");
  if (pkd::chunk_keys_for(page_size) < 0)
    return fail(PKD_ERR_UNSUPPORTED, "page_size must be 1..64 or a multiple of 64 (got %d)", page_size);
  if (kv_layout != PKD_LAYOUT_NHD && kv_layout != PKD_LAYOUT_HND)
    return fail(PKD_ERR_INVALID_ARG, "kv_layout %d (PKD_LAYOUT_NHD or PKD_LAYOUT_HND)", kv_layout);

  // ---- sizes against the fixed scratch
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(MultiProcessorCount)");
  const int G = sms * pkd::kCtasPerSm;
  const NaLayout L = na_layout(batch, num_kv_heads, group, G);
  if (L.total > kNoAllocScratchBytes)
    return fail(PKD_ERR_CAPACITY_EXCEEDED,
                "no-alloc decode: batch %d x %d kv heads needs %zu bytes of device scratch, the fixed scratch "
                "holds %zu",
                batch, num_kv_heads, L.total, kNoAllocScratchBytes);
  if (L.meta_end > kHostMetaBytes)
    return fail(PKD_ERR_CAPACITY_EXCEEDED,
                "no-alloc decode: batch %d x %d kv heads needs a %zu-byte schedule, the fixed host staging "
                "buffer holds %zu",
                batch, num_kv_heads, L.meta_end, kHostMetaBytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  {
    // the schedule upload reads a host buffer that the next call rewrites: a
    // graph node made of it would replay some later call's schedule
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone)
      return fail(PKD_ERR_UNSUPPORTED, "no-alloc decode cannot run while its stream is being captured");
  }
  uint8_t* ws = nullptr;
  pkd_status s = scratch_for_current_device(&ws);
  if (s != PKD_OK) return s;

  // ---- schedule (host, static buffer) and its upload
  pkd::PlanCounts counts{};
  {
    std::lock_guard<std::mutex> lock(g_host_mutex);
    uint8_t* h = g_host_meta;
    memset(h, 0, sizeof(pkd::WsHeader));
    auto* hdr = reinterpret_cast<pkd::WsHeader*>(h);
    auto* cta_begin = reinterpret_cast<int32_t*>(h + L.cta_begin);
    auto* items = reinterpret_cast<int32_t*>(h + L.items);
    auto* merge_rows = reinterpret_cast<int32_t*>(h + L.merge_rows);
    auto* row_begin = reinterpret_cast<int32_t*>(h + L.row_begin);
    auto* row_count = reinterpret_cast<int32_t*>(h + L.row_count);
    auto* kv_len = reinterpret_cast<int32_t*>(h + L.kv_len);
    auto* page_begin = reinterpret_cast<int32_t*>(h + L.page_begin);
    // the rule's own checks, done here first so that the shared planner's
    // message path is never taken
    if (h_kv_indptr[0] != 0) return fail(PKD_ERR_INVALID_ARG, "kv_indptr[0] must be 0");
    for (int b = 0; b < batch; ++b) {
      const int64_t n = static_cast<int64_t>(h_kv_indptr[b + 1]) - h_kv_indptr[b];
      if (n < 0) return fail(PKD_ERR_INVALID_ARG, "kv_indptr must be non-decreasing (request %d)", b);
      if (n > 0 && (h_kv_last_page_len[b] < 1 || h_kv_last_page_len[b] > page_size))
        return fail(PKD_ERR_INVALID_ARG, "kv_last_page_len[%d] = %d outside 1..page_size", b, h_kv_last_page_len[b]);
      if (n > 0 && (n - 1) * page_size + h_kv_last_page_len[b] > INT32_MAX)
        return fail(PKD_ERR_INVALID_ARG, "request %d is longer than 2^31 - 1 keys", b);
    }
    if (batch > 0 && h_kv_indptr[batch] > 0 && !d_kv_page_indices)
      return fail(PKD_ERR_INVALID_ARG, "d_kv_page_indices is NULL");
    std::string why;
    int r = pkd::compute_plan(h_kv_indptr, h_kv_last_page_len, batch, num_kv_heads, page_size, G, items,
                              L.max_items, cta_begin, row_begin, row_count, merge_rows, kv_len, &counts, &why);
    if (r != pkd::kPlanOk) return fail(static_cast<pkd_status>(r), "no-alloc decode: %s", why.c_str());
    for (int i = 0; i < counts.n_items; ++i) items[4 * i + 3] = row_count[items[4 * i]] > 1 ? pkd::kItemSplit : 0;
    for (int b = 0; b < batch; ++b) page_begin[b] = h_kv_indptr[b];
    hdr->err = 0;  // the shared scratch keeps the previous call's bytes: the error word restarts at 0
    hdr->n_items = counts.n_items;
    hdr->n_merge_rows = counts.n_merge_rows;
    hdr->batch = batch;
    hdr->zero_page = 0;
    // pageable source: the runtime has staged the bytes when cudaMemcpyAsync
    // returns, so the static host buffer may be reused once the lock is released
    e = cudaMemcpyAsync(ws, h, L.meta_end, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(no-alloc schedule)");
  }

  // ---- kernels
  const int box_tok = page_size <= pkd::kChunkKeys ? page_size : pkd::kChunkKeys;
  const float scale = (sm_scale > 0.f) ? sm_scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
  pkd::DecodeParams p{};
  p.items = reinterpret_cast<const int4*>(ws + L.items);
  p.cta_begin = reinterpret_cast<const int*>(ws + L.cta_begin);
  p.kv_len = reinterpret_cast<const int*>(ws + L.kv_len);
  p.page_begin = reinterpret_cast<const int*>(ws + L.page_begin);
  p.page_indices = d_kv_page_indices;
  p.kv_hnd = kv_layout == PKD_LAYOUT_HND ? 1 : 0;
  p.q = d_q;
  p.out = d_out;
  p.lse = d_lse;
  p.part_o = reinterpret_cast<float*>(ws + L.part_o);
  p.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  p.k_scale = d_k_scale;
  p.v_scale = d_v_scale;
  p.err = reinterpret_cast<unsigned*>(ws);
  p.num_kv_heads = num_kv_heads;
  p.group = group;
  p.page_size = page_size;
  p.pages_per_chunk = page_size <= pkd::kChunkKeys ? pkd::kChunkKeys / page_size : 0;
  p.chunk_keys = counts.chunk_keys;
  p.box_tok = box_tok;
  p.num_pages = static_cast<int>(num_pages);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.force_partial = 0;
  if (counts.n_items > 0) {
    if (!d_k_cache || !d_v_cache || !aligned16(d_k_cache) || !aligned16(d_v_cache))
      return fail(PKD_ERR_INVALID_ARG, "k/v cache must be non-NULL and 16-byte aligned");
    if (num_pages <= 0 || num_pages > INT32_MAX) return fail(PKD_ERR_INVALID_ARG, "num_pages out of range");
    if ((page_stride_elems * (fp8 ? 1 : 2)) % 16 != 0 ||
        page_stride_elems < static_cast<int64_t>(page_size) * num_kv_heads * head_dim)
      return fail(PKD_ERR_INVALID_ARG, "page_stride_elems must cover a page and be a 16-byte multiple");
    CUtensorMap tmk, tmv;
    s = kv_map(&tmk, d_k_cache, kv_dtype, num_kv_heads, page_size, num_pages, page_stride_elems, box_tok,
               kv_layout == PKD_LAYOUT_HND);
    if (s != PKD_OK) return s;
    s = kv_map(&tmv, d_v_cache, kv_dtype, num_kv_heads, page_size, num_pages, page_stride_elems, box_tok,
               kv_layout == PKD_LAYOUT_HND);
    if (s != PKD_OK) return s;
    e = pkd::launch_decode(tmk, tmv, p, q_dtype, kv_dtype, G, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
  }
  pkd::MergeParams m{};
  m.merge_rows = reinterpret_cast<const int*>(ws + L.merge_rows);
  m.header = reinterpret_cast<const pkd::WsHeader*>(ws);
  m.row_item_begin = reinterpret_cast<const int*>(ws + L.row_begin);
  m.row_item_count = reinterpret_cast<const int*>(ws + L.row_count);
  m.part_o = p.part_o;
  m.part_lse = p.part_lse;
  m.out = d_out;
  m.lse = d_lse;
  m.out_dtype = q_dtype;
  m.num_kv_heads = num_kv_heads;
  m.group = group;
  m.all_rows = 0;
  e = pkd::launch_merge_rows(m, G, st);
  if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
  return PKD_OK;
}

extern "C" pkd_status pkd_noalloc_device_errors(uint32_t* flags_out, void* stream) {
  if (!flags_out) return fail(PKD_ERR_INVALID_ARG, "flags_out is NULL");
  *flags_out = 0;
  uint8_t* ws = nullptr;
  pkd_status s = scratch_for_current_device(&ws);
  if (s != PKD_OK) return s;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned word = 0;
  e = cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(no-alloc error word)");
  *flags_out = word;
  return word ? fail(PKD_ERR_DEVICE_CHECK, "no-alloc decode: device error bits 0x%x", word) : PKD_OK;
}
