// pkd_internal.h -- structures shared by the host launchers and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkd {

constexpr int kHeadDim = 128;
constexpr int kChunkKeys = 64;        // keys per split-KV chunk (one pipeline stage)
constexpr int kMaxGroup = 8;          // qo heads per kv head served by one MMA row tile
constexpr int kMaxPrefixSplits = 16;  // cascade: pieces the shared prefix may be cut into
constexpr int kCtasPerSm = 2;         // decode CTAs resident per SM
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // bounded pipeline waits

constexpr unsigned kDevErrPageIndex = 1u;
constexpr unsigned kDevErrWaitTimeout = 2u;

enum DType : int { kF16 = 0, kBF16 = 1, kE4M3 = 2, kF32 = 3 };

// Device header at the start of the workspace (int32 words).
struct WsHeader {
  unsigned err;       // PKD_DEVERR_* bits (written by kernels, never by a plan upload)
  int pad0[3];
  int n_items;        // from byte 16 on, everything is the plan's upload
  int n_merge_rows;
  int batch;
  int zero_page;      // a page index of 0 for single-request decode
  int n_empty_rows;   // rows (request, kv head) without items
  int pad[55];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// One split-KV work item: (row = b * Hk + h, first chunk, end chunk, flags).
// flags bit 0: the row is split across items (write a partial state).
constexpr int kItemSplit = 1;

struct DecodeParams {
  const int4* items;
  const int* cta_begin;   // [G + 1]
  const int* kv_len;      // [B]
  const int* page_begin;  // [B]  (= kv_indptr[b])
  const int* page_indices;
  const void* q;          // [B, Hq, D]
  void* out;              // [B, Hq, D]  (q dtype)
  float* lse;             // [B, Hq] natural log, or nullptr
  float* part_o;          // [slot, g, D] fp32
  float* part_lse;        // [slot, g] base-2 log-sum-exp of the scaled scores
  const float* k_scale;   // [Hk] or nullptr
  const float* v_scale;
  unsigned* err;
  int num_kv_heads;
  int group;
  int page_size;          // plan page size
  int pages_per_chunk;    // page_size <= 64: pages per chunk; else 0
  int chunk_keys;         // keys per chunk
  int box_tok;            // tokens per TMA box
  int num_pages;          // pool pages (index validation)
  float scale_log2;       // sm_scale * log2(e)
  int force_partial;      // cascade: every item writes a partial state
  // fused merge (plain decode): the item that completes a split row merges the
  // row's partial states, and rows without items are written at grid start
  int fused_merge;
  int* row_done;              // [B * Hk] items of the row finished (zero at the start of a run)
  const int* row_item_begin;  // [B * Hk]
  const int* row_item_count;  // [B * Hk]
  const int* empty_rows;      // [header->n_empty_rows]
  const WsHeader* header;
  int debug_stall;            // test hook: the producer issues nothing (waits run out)
  int kv_hnd;                 // pages are [Hk, P, D] (HND) instead of [P, Hk, D] (NHD)
  // launched behind the cascade's prefix kernel, once that kernel has waited
  // for the upload: everything this grid reads was complete before it was
  // launched, so it skips griddepcontrol.wait at the start (which would wait
  // for the prefix kernel) and waits at its end instead
  int behind_prefix;
};

struct MergeParams {
  const int* merge_rows;      // rows to merge (normal mode)
  const WsHeader* header;     // n_merge_rows, batch
  const int* row_item_begin;  // [B * Hk]
  const int* row_item_count;  // [B * Hk]
  const float* part_o;        // [slot, g, D]
  const float* part_lse;      // [slot, g] base 2
  const float* pre_o;         // cascade: [split, B * Hq, D] or nullptr
  const float* pre_lse;       // cascade: [split, B * Hq] base 2
  int n_pre_splits;
  void* out;
  float* lse;
  int out_dtype;
  int num_kv_heads;
  int group;
  int all_rows;               // cascade: every row of the batch
};

constexpr int kMaxTreeLevels = 4;  // shared levels of a prefix tree
constexpr int kNoCausal = 0x7fffffff;

// One unit of the tile-attention kernel's work-list mode (prefix-tree levels,
// prefill): the 128-row query tile of one kv head whose first row-token is q0
// (rows r = (q - q0) * g + j for query token / request q and group head j),
// against 128-key tiles [t0, t1) of one page list.
struct TileWork {
  int q0;          // first query token (prefill) or request (tree) of the tile
  int q_end;       // tokens / requests at or past q_end are not this unit's
  int page_begin;  // the list is pages[level][page_begin ..]
  int kv_len;      // keys in the list
  int t0, t1;      // key tiles of this unit
  int piece;       // output piece (fp32 partial state), or -1: final out / lse
  int level;       // page array
  int diag;        // causal: token q sees keys 0 .. q + diag; kNoCausal: all keys
  int pad[3];
};
static_assert(sizeof(TileWork) == 48, "three 16-byte loads");

// Shared-prefix (cascade level 0) attention on the tensor cores.
struct PrefixParams {
  const int* prefix_pages;  // [n_prefix_pages]
  int n_prefix_pages;
  int prefix_len;           // keys in the prefix
  int batch;
  int num_kv_heads;
  int group;
  int num_pages;
  int page_size;
  int box_tok;              // keys per TMA box (min(page_size, 64))
  int n_splits;             // key-range pieces
  int tiles_per_split;      // 128-key tiles per piece
  int m_tiles;              // query tiles per kv head (one per CTA)
  int cluster;              // CTAs per cluster (2: a pair of the shared-prefix kernel)
  int m_groups;             // shared-prefix kernel: CTA pairs per kv head, ceil(m_tiles / 2)
  int req_per_tile;         // shared-prefix kernel: requests per CTA, floor(128 / group)
  float scale_log2;
  float* pre_o;             // [split, B * Hq, D]
  float* pre_lse;           // [split, B * Hq] base 2
  const float* k_scale;
  const float* v_scale;
  unsigned* err;
  int kv_hnd;               // pages are [Hk, P, D] (HND) instead of [P, Hk, D] (NHD)
  // work-list mode (pkd_tile2.cu): the units come in pairs with the same keys;
  // CTA x takes kv head x % Hk of units work[2 (x / Hk)] and work[2 (x / Hk) + 1];
  // pieces are pre_o[piece][row][D] with rows_per_piece rows
  const TileWork* work;
  int n_work;
  int rows_per_piece;       // query rows (tokens or requests times Hq) per piece
  const int* level_pages[kMaxTreeLevels];
  void* out;                // final-output units: [rows, Hq, D] in out_dtype
  float* lse;               //   and lse [rows, Hq] (natural log) or nullptr
  int out_dtype;
};

// Writing new tokens' K/V rows into the paged cache (pkd_append.cu).
struct AppendParams {
  const void* k_new;          // [n_tokens, Hk, D] in the new dtype (f16 / bf16)
  const void* v_new;
  const int* batch_indices;   // [n_tokens]
  const int* positions;       // [n_tokens]
  const int* kv_indptr;       // [batch + 1] (device)
  const int* page_indices;    // [kv_indptr[batch]]
  void* k_cache;              // pool [num_pages, P, Hk, D] (NHD) or [num_pages, Hk, P, D] (HND), page stride
  void* v_cache;
  const float* k_scale;       // e4m3 pools: [Hk]
  const float* v_scale;
  unsigned* err;              // optional device error word
  int64_t page_stride;        // elements
  int n_tokens;
  int batch;
  int num_kv_heads;
  int page_size;
  int num_pages;
  int kv_hnd;                 // HND pages
};

// Multi-latent attention decode (pkd_mla.cu): one CTA per unit (request,
// output half, key range) given as TileWork {q0 = request, -, page_begin,
// kv_len, t0, t1 (32-key tiles), piece (-1: final output), level = half}.
struct MlaParams {
  const TileWork* work;
  int n_work;
  const int* page_indices;      // CSR page ids (device)
  int num_pages;
  int page_size;
  int box_tok;                  // keys per TMA box: min(page_size, 32)
  int num_heads;                // <= 128
  int batch;
  float scale_log2;             // sm_scale * log2(e)
  float* part_o;                // [piece][H][512] fp32
  float* part_lse;              // [piece][H] base-2
  const int* req_piece_begin;   // [batch + 1]
  int any_split;                // some request has more than one piece
  void* out;                    // [batch][H][512] bf16
  float* lse;                   // [batch][H] natural log, or nullptr
  unsigned* err;
  const void* q_nope;           // [batch][H][512] bf16 (chunks 4..7 are read directly)
  const void* q_pe;             // [batch][H][64] bf16
};

// Launchers (defined in the .cu files; return a cudaError_t).
cudaError_t launch_decode(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p,
                          int q_dtype, int kv_dtype, int grid, cudaStream_t stream);
cudaError_t launch_merge_rows(const MergeParams& p, int grid, cudaStream_t stream);
cudaError_t launch_mla(const CUtensorMap& tq_nope, const CUtensorMap& tq_pe, const CUtensorMap& tckv,
                       const CUtensorMap& tkpe, const MlaParams& p, cudaStream_t stream);
int mla_smem_bytes();
cudaError_t launch_append_kv(const AppendParams& p, int new_dtype, int kv_dtype, cudaStream_t stream);
// dst, src and bytes multiples of 16; src may be mapped pinned host memory
cudaError_t launch_copy16(void* dst, const void* src, int64_t bytes, cudaStream_t stream);
cudaError_t launch_merge_state(const void* va, const float* sa, const void* vb, const float* sb,
                               void* vo, float* so, int64_t n, int heads, int dim, int dtype,
                               cudaStream_t stream);
cudaError_t launch_merge_states(const void* v, const float* s, int64_t n, int k, int heads, int dim,
                                int dtype, void* vo, float* so, cudaStream_t stream);
// shared-prefix attention on CTA pairs (pkd_prefix.cu); e4m3 pools take maps
// of unswizzled code boxes (128 codes of K, 64 of V per row)
cudaError_t launch_prefix(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                          const PrefixParams& p, int q_dtype, int kv_dtype, cudaStream_t stream, bool pdl);
// work-list units in pairs (p.work, p.n_work even): one CTA per pair and kv head
cudaError_t launch_tile2(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                         const PrefixParams& p, int kv_dtype, cudaStream_t stream, bool pdl);
int decode_smem_bytes(int kv_dtype);
int prefix_smem_bytes(int kv_dtype);
int tile2_smem_bytes();
int prefix_max_active_clusters(int q_dtype, int kv_dtype);  // resident CTA pairs (clusters of 2), 0 if unknown

}  // namespace pkd
