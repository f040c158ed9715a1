// pkd_mla_capi.cu -- the C entry points of multi-latent attention decode
// (declared in include/pkd.h): argument checks, the key-range split, the unit
// upload, tensor maps and the launch of the kernels in pkd_mla.cu.
#include <string.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "pkd.h"
#include "pkd_host.h"
#include "pkd_internal.h"

using pkd::host::aligned16;
using pkd::host::align256;
using pkd::host::cuda_fail;
using pkd::host::fail;
using pkd::host::get_encode;

namespace {

// MLA work units (host): validates the page table, cuts the requests into
// key ranges and lists two units per range (one per half of the 512 output
// dims, adjacent), longest first; rpb[b] .. rpb[b+1]-1 are the partial-state
// pieces of a request that was cut (none for one written directly).  Shared by
// pkd_mla_decode and the host-only pkd_mla_units_host.
pkd_status mla_units(const int32_t* h_kv_indptr, const int32_t* h_kv_last_page_len, int batch, int page_size,
                     int num_sms, std::vector<pkd::TileWork>* w_out, std::vector<int32_t>* rpb_out,
                     bool* any_split_out) {
  if (batch < 0) return fail(PKD_ERR_INVALID_ARG, "batch must be >= 0");
  if (page_size < 1) return fail(PKD_ERR_INVALID_ARG, "page_size must be >= 1");
  if (num_sms <= 0) return fail(PKD_ERR_INVALID_ARG, "num_sms must be > 0");
  if (!h_kv_indptr || (batch > 0 && !h_kv_last_page_len)) return fail(PKD_ERR_INVALID_ARG, "NULL argument");
  if (h_kv_indptr[0] != 0) return fail(PKD_ERR_INVALID_ARG, "kv_indptr[0] must be 0");
  const int P = page_size;
  std::vector<int> lens(batch);
  for (int b = 0; b < batch; ++b) {
    const int pages = h_kv_indptr[b + 1] - h_kv_indptr[b];
    if (pages < 0) return fail(PKD_ERR_INVALID_ARG, "decreasing kv_indptr at %d", b);
    if (pages > 0 && (h_kv_last_page_len[b] < 1 || h_kv_last_page_len[b] > P))
      return fail(PKD_ERR_INVALID_ARG, "request %d: last_page_len %d outside 1..%d", b, h_kv_last_page_len[b], P);
    const int64_t L = pages > 0 ? static_cast<int64_t>(pages - 1) * P + h_kv_last_page_len[b] : 0;
    if (L > INT32_MAX - 64) return fail(PKD_ERR_INVALID_ARG, "request %d: too many keys", b);
    lens[b] = static_cast<int>(L);
  }
  // key ranges: the smallest piece size C (in 32-key tiles, at least 16 =
  // 512 keys) for which cutting every request into pieces of at most C tiles
  // gives at most num_sms pieces, so the units (two output halves per piece)
  // make at most two full waves and the longest unit is as short as possible;
  // a request with one piece is written directly, the others merged
  constexpr int kTileKeys = 32;
  std::vector<int> tiles_of(batch);
  int max_tiles = 1;
  for (int b = 0; b < batch; ++b) {
    tiles_of[b] = (lens[b] + kTileKeys - 1) / kTileKeys;
    max_tiles = tiles_of[b] > max_tiles ? tiles_of[b] : max_tiles;
  }
  auto pieces_for = [&](int C) {
    int64_t cnt = 0;
    for (int b = 0; b < batch; ++b) cnt += tiles_of[b] > C ? (tiles_of[b] + C - 1) / C : 1;
    return cnt;
  };
  int lo = 1, hi = max_tiles;
  while (lo < hi) {
    const int mid = lo + (hi - lo) / 2;
    if (pieces_for(mid) <= num_sms) hi = mid; else lo = mid + 1;
  }
  const int C = lo < 16 ? 16 : lo;
  std::vector<pkd::TileWork>& w = *w_out;
  w.clear();
  std::vector<int32_t>& rpb = *rpb_out;
  rpb.assign(batch + 1, 0);
  int piece = 0;
  bool any_split = false;
  for (int b = 0; b < batch; ++b) {
    const int L = lens[b];
    const int tiles = tiles_of[b];
    const int np = tiles > C ? (tiles + C - 1) / C : 1;
    if (np > 1) any_split = true;
    const int tpp = (tiles + np - 1) / np;
    for (int s = 0; s < np; ++s) {
      for (int hv = 0; hv < 2; ++hv) {
        pkd::TileWork t{};
        t.q0 = b;
        t.q_end = b + 1;
        t.page_begin = h_kv_indptr[b];
        t.kv_len = L;
        t.t0 = s * tpp < tiles ? s * tpp : tiles;
        t.t1 = (s + 1) * tpp < tiles ? (s + 1) * tpp : tiles;
        t.piece = np > 1 ? piece + s : -1;
        t.level = hv;
        w.push_back(t);
      }
    }
    if (np > 1) piece += np;
    rpb[b + 1] = np > 1 ? piece : rpb[b];
  }
  if (piece > batch + num_sms) return fail(PKD_ERR_CAPACITY_EXCEEDED, "%d pieces above capacity", piece);
  // longest units first: CTAs are dispatched in grid order, so the short
  // units fill in behind the long ones
  std::stable_sort(w.begin(), w.end(), [](const pkd::TileWork& x, const pkd::TileWork& y) {
    return (x.t1 - x.t0) > (y.t1 - y.t0);
  });
  *any_split_out = any_split;
  return PKD_OK;
}

}  // namespace

extern "C" {

size_t pkd_mla_workspace_bytes(int max_batch, int num_heads, int num_sms) {
  if (max_batch <= 0 || num_heads <= 0 || num_heads > 128 || num_sms <= 0) return 0;
  const size_t pieces = static_cast<size_t>(max_batch) + num_sms;
  const size_t units = 2 * pieces;
  size_t off = 256;  // error word
  off += align256(sizeof(pkd::TileWork) * units);
  off += align256(4ull * (max_batch + 1));
  off += align256(4ull * pieces * num_heads * 512);
  off += align256(4ull * pieces * num_heads);
  return off;
}

pkd_status pkd_mla_units_host(const int32_t* h_kv_indptr, const int32_t* h_kv_last_page_len, int batch,
                              int page_size, int num_sms, int32_t* units_out, int max_units, int* n_units_out,
                              int32_t* req_piece_begin_out) {
  static_assert(sizeof(pkd::TileWork) == 12 * sizeof(int32_t), "a unit is 12 int32");
  if (!n_units_out || !req_piece_begin_out) return fail(PKD_ERR_INVALID_ARG, "NULL output");
  std::vector<pkd::TileWork> w;
  std::vector<int32_t> rpb;
  bool any_split = false;
  pkd_status s = mla_units(h_kv_indptr, h_kv_last_page_len, batch, page_size, num_sms, &w, &rpb, &any_split);
  if (s != PKD_OK) return s;
  *n_units_out = static_cast<int>(w.size());
  if (static_cast<int64_t>(w.size()) > max_units)
    return fail(PKD_ERR_CAPACITY_EXCEEDED, "%zu units above max_units %d", w.size(), max_units);
  if (!w.empty() && !units_out) return fail(PKD_ERR_INVALID_ARG, "units_out is NULL");
  if (!w.empty()) memcpy(units_out, w.data(), sizeof(pkd::TileWork) * w.size());
  memcpy(req_piece_begin_out, rpb.data(), sizeof(int32_t) * rpb.size());
  return PKD_OK;
}

pkd_status pkd_mla_decode(const void* d_q_nope, const void* d_q_pe, const void* d_ckv_cache,
                          const void* d_kpe_cache, const int32_t* h_kv_indptr, const int32_t* d_kv_page_indices,
                          const int32_t* h_kv_last_page_len, int batch, int num_heads, int page_size,
                          int64_t num_pages, int64_t ckv_page_stride_elems, int64_t kpe_page_stride_elems,
                          float sm_scale, void* d_out, float* d_lse, void* d_workspace, size_t workspace_bytes,
                          int num_sms, void* stream) {
  if (batch < 0 || num_heads <= 0 || num_heads > 128)
    return fail(PKD_ERR_UNSUPPORTED, "num_heads %d outside 1..128 (batch %d)", num_heads, batch);
  if (!(page_size >= 1 && ((page_size <= 32 && 32 % page_size == 0) || page_size % 32 == 0)))
    return fail(PKD_ERR_UNSUPPORTED, "page_size %d: a divisor of 32 or a multiple of 32", page_size);
  if (num_sms <= 0) return fail(PKD_ERR_INVALID_ARG, "num_sms must be > 0");
  const size_t need = pkd_mla_workspace_bytes(batch > 0 ? batch : 1, num_heads, num_sms);
  if (!d_workspace || workspace_bytes < need || !aligned16(d_workspace))
    return fail(PKD_ERR_WORKSPACE_TOO_SMALL, "workspace of %zu bytes, need %zu (16-byte aligned)", workspace_bytes,
                need);
  if (batch == 0) return PKD_OK;
  if (!h_kv_indptr || !h_kv_last_page_len || !d_q_nope || !d_q_pe || !d_out)
    return fail(PKD_ERR_INVALID_ARG, "NULL argument");
  if (!aligned16(d_q_nope) || !aligned16(d_q_pe) || !aligned16(d_out))
    return fail(PKD_ERR_INVALID_ARG, "q / out must be 16-byte aligned");
  std::vector<pkd::TileWork> w;
  std::vector<int32_t> rpb;
  bool any_split = false;
  pkd_status su = mla_units(h_kv_indptr, h_kv_last_page_len, batch, page_size, num_sms, &w, &rpb, &any_split);
  if (su != PKD_OK) return su;
  const int P = page_size;
  if (h_kv_indptr[batch] > 0) {
    if (!d_kv_page_indices || !d_ckv_cache || !d_kpe_cache) return fail(PKD_ERR_INVALID_ARG, "NULL cache");
    if (!aligned16(d_ckv_cache) || !aligned16(d_kpe_cache))
      return fail(PKD_ERR_INVALID_ARG, "caches must be 16-byte aligned");
    if (num_pages <= 0 || num_pages > INT32_MAX) return fail(PKD_ERR_INVALID_ARG, "num_pages out of range");
    if ((ckv_page_stride_elems * 2) % 16 || ckv_page_stride_elems < static_cast<int64_t>(P) * 512 ||
        (kpe_page_stride_elems * 2) % 16 || kpe_page_stride_elems < static_cast<int64_t>(P) * 64)
      return fail(PKD_ERR_INVALID_ARG, "page strides must cover a page and be 16-byte multiples");
  }
  // workspace: error word | units | request piece ranges | partial o | partial lse
  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  const size_t pieces_cap = static_cast<size_t>(batch) + num_sms;
  size_t off = 256;
  const size_t off_work = off;
  off += align256(sizeof(pkd::TileWork) * 2 * pieces_cap);
  const size_t off_rpb = off;
  off += align256(4ull * (batch + 1));
  const size_t off_po = off;
  off += align256(4ull * pieces_cap * num_heads * 512);
  const size_t off_pl = off;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, 4, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ws + off_work, w.data(), sizeof(pkd::TileWork) * w.size(), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ws + off_rpb, rpb.data(), 4ull * (batch + 1), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "MLA schedule upload");
  // tensor maps: q_nope as (64 dims, 8 chunks, H heads, B), q_pe as (64, H, B, 1),
  // ckv as (64 dims, 8 chunks, P tokens, pages), kpe as (64, P, pages, 1)
  auto enc = get_encode();
  if (!enc) return fail(PKD_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const int box = P < 32 ? P : 32;
  const int64_t np = h_kv_indptr[batch] > 0 ? num_pages : 1;
  CUtensorMap tqn, tqp, tckv, tkpe;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  auto encode = [&](CUtensorMap* m, const void* ptr, cuuint64_t d0, cuuint64_t d1, cuuint64_t d2, cuuint64_t d3,
                    cuuint64_t s1, cuuint64_t s2, cuuint64_t s3, cuuint32_t b1, cuuint32_t b2) -> pkd_status {
    cuuint64_t dims[4] = {d0, d1, d2, d3};
    cuuint64_t strides[3] = {s1, s2, s3};
    cuuint32_t boxd[4] = {64u, b1, b2, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, boxd, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKD_ERR_CUDA, "cuTensorMapEncodeTiled (MLA) failed (CUresult %d)", (int)r);
    return PKD_OK;
  };
  const cuuint64_t H = static_cast<cuuint64_t>(num_heads);
  pkd_status s = encode(&tqn, d_q_nope, 64, 8, H, batch, 128, 1024, H * 1024, 1, static_cast<cuuint32_t>(num_heads));
  if (s == PKD_OK) s = encode(&tqp, d_q_pe, 64, H, batch, 1, 128, H * 128, H * 128 * batch,
                              static_cast<cuuint32_t>(num_heads), 1);
  const void* ckv = d_ckv_cache ? d_ckv_cache : d_q_nope;  // no page: the maps are never used
  const void* kpe = d_kpe_cache ? d_kpe_cache : d_q_pe;
  if (s == PKD_OK)
    s = encode(&tckv, ckv, 64, 8, P, np, 128, 1024, static_cast<cuuint64_t>(ckv_page_stride_elems) * 2, 1,
               static_cast<cuuint32_t>(box));
  if (s == PKD_OK)
    s = encode(&tkpe, kpe, 64, P, np, 1, 128, static_cast<cuuint64_t>(kpe_page_stride_elems) * 2,
               static_cast<cuuint64_t>(kpe_page_stride_elems) * 2 * np, static_cast<cuuint32_t>(box), 1);
  if (s != PKD_OK) return s;
  pkd::MlaParams p{};
  p.work = reinterpret_cast<const pkd::TileWork*>(ws + off_work);
  p.n_work = static_cast<int>(w.size());
  p.page_indices = d_kv_page_indices;
  p.num_pages = static_cast<int>(np);
  p.page_size = P;
  p.box_tok = box;
  p.num_heads = num_heads;
  p.batch = batch;
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(192.0f);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.part_o = reinterpret_cast<float*>(ws + off_po);
  p.part_lse = reinterpret_cast<float*>(ws + off_pl);
  p.req_piece_begin = reinterpret_cast<const int*>(ws + off_rpb);
  p.any_split = any_split ? 1 : 0;
  p.out = d_out;
  p.lse = d_lse;
  p.err = reinterpret_cast<unsigned*>(ws);
  p.q_nope = d_q_nope;
  p.q_pe = d_q_pe;
  e = pkd::launch_mla(tqn, tqp, tckv, tkpe, p, st);
  if (e != cudaSuccess) return cuda_fail(e, "MLA kernel launch");
  return PKD_OK;
}

}  // extern "C"
