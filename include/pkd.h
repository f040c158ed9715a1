/*
 * pkd.h -- batched paged-KV decode attention for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libpkd.so.  Every argument is a plain host value or pointer; device
 * buffers are raw device addresses; a stream is a cudaStream_t passed as
 * `void*` (NULL = the legacy default stream).  No call throws or aborts: each
 * returns a pkd_status, and pkd_last_error() gives the calling thread's last
 * message.
 *
 * Problem statement (FlashInfer pages):
 *   - plan/run split of the batched decode wrapper: plan takes the page table
 *     and the static geometry and runs on the host before CUDA-graph capture;
 *     run takes q and the paged K/V (aquanode.io 2026 guide, "Quickstart",
 *     paragraph on BatchDecodeWithPagedKVCacheWrapper; snackonai.com deep dive,
 *     "The Code, Annotated", snippet one, and "It In Action", step 1);
 *   - the KV pool: fixed-size pages in the NHD layout
 *     [num_pages, page_size, num_kv_heads, head_dim], a request's pages named by
 *     a CSR table (kv_indptr, kv_page_indices, kv_last_page_len) (deep dive,
 *     snippet one; 2026 guide, "What FlashInfer is", idea 1 "block-sparse KV
 *     cache format");
 *   - merge_state / merge_states and cascade (shared-prefix) decode
 *     (2026 guide, "Cascade attention for shared prefixes");
 *   - single-request decode with contiguous K/V (ai-tldr.dev tool card,
 *     "Getting started", step 4).
 *
 * Conventions shared by all calls:
 *   - head_dim must be 128.  num_qo_heads must be a multiple of num_kv_heads,
 *     with a group size g = num_qo_heads / num_kv_heads of at most 8; qo head h
 *     reads kv head h / g.
 *   - q is [batch, num_qo_heads, head_dim], contiguous.  out has q's shape and
 *     dtype; lse is fp32 [batch, num_qo_heads], the natural-log log-sum-exp of
 *     the scaled scores sm_scale * <q, k>.  An empty request gives out = 0 and
 *     lse = -inf.
 *   - sm_scale <= 0 selects 1/sqrt(head_dim).
 *   - Supported (q, kv) dtypes: (F16, F16), (BF16, BF16), (BF16, E4M3),
 *     (F16, E4M3).  An E4M3 cache takes one fp32 scale per kv head for K and for
 *     V (k_scale, v_scale: device arrays [num_kv_heads]); the attended values are
 *     code * scale.
 *   - Device pointers handed to run / cascade_decode must stay valid until the
 *     work on the stream has finished.  Base addresses of q, the caches, out,
 *     and page_stride_elems * element size must be 16-byte multiples.
 */
#ifndef PKD_H
#define PKD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkd_status {
  PKD_OK = 0,
  PKD_ERR_INVALID_ARG = 1,         /* a NULL, negative or inconsistent argument */
  PKD_ERR_UNSUPPORTED = 2,         /* head_dim, group size, dtype pair or page size not built */
  PKD_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes below pkd_workspace_bytes(...) */
  PKD_ERR_CAPACITY_EXCEEDED = 4,   /* batch above the plan's max_batch, or prefix splits above max */
  PKD_ERR_CUDA = 5,                /* a CUDA runtime or driver call failed (message has the name) */
  PKD_ERR_DEVICE_CHECK = 6,        /* a kernel recorded an error (see pkd_check_device_errors) */
  PKD_ERR_NO_PLAN = 7              /* run / cascade_decode before a successful pkd_plan */
} pkd_status;

typedef enum pkd_dtype {
  PKD_F16 = 0,
  PKD_BF16 = 1,
  PKD_E4M3 = 2, /* OCP FP8 E4M3 ("fn"), KV cache only */
  PKD_F32 = 3   /* merge_state / merge_states values only */
} pkd_dtype;

/*
 * Page layout of a K or V pool (the batch-decode wrapper of the 2026 Guide,
 * "When to use it", defaults to NHD; the deep dive, "The Code, Annotated",
 * passes kv_layout="NHD").  Element (page p, slot t, kv head h, dim d) is at
 *   NHD: p * page_stride_elems + (t * num_kv_heads + h) * 128 + d
 *   HND: p * page_stride_elems + (h * page_size + t) * 128 + d
 * HND keeps one head's keys of a page contiguous (page_size * 256 bytes for
 * 16-bit values).
 */
typedef enum pkd_kv_layout {
  PKD_LAYOUT_NHD = 0,
  PKD_LAYOUT_HND = 1
} pkd_kv_layout;

/* Device error bits recorded by the kernels (pkd_check_device_errors). */
#define PKD_DEVERR_PAGE_INDEX 1u    /* a page index outside [0, num_pages): page 0 was read instead */
#define PKD_DEVERR_WAIT_TIMEOUT 2u  /* a pipeline wait gave up after ~2 s; outputs are invalid */

/* Opaque plan: host-side state plus views into the caller's device workspace. */
typedef struct pkd_plan_s* pkd_plan_t;

/* Library version string, e.g. "pkd 0.1.0 sm_103a". */
const char* pkd_version(void);

/* Static text for a status code. */
const char* pkd_status_string(int status);

/* The calling thread's last error message ("" if none).  Valid until the next
 * failing call on this thread. */
const char* pkd_last_error(void);

/*
 * Number of CTAs of the decode launch on `device` (a fixed multiple of its SM
 * count).  The plan partitions work over exactly this many CTAs.  Needs a GPU.
 */
pkd_status pkd_num_ctas(int device, int* num_ctas_out);

/*
 * Bytes of device workspace a plan with these limits needs.  Pure host
 * arithmetic (no GPU needed).  num_ctas: the value pkd_num_ctas returns for
 * the device the plan will run on.  max_prefix_splits: how many pieces
 * pkd_cascade_decode may split the shared prefix into (0 = no cascade; the
 * library uses at most 16).  Returns 0 for invalid arguments.
 */
size_t pkd_workspace_bytes(int max_batch, int num_qo_heads, int num_kv_heads, int head_dim,
                           int num_ctas, int max_prefix_splits);

/*
 * Create a plan object.  d_workspace (device, caller-owned, >= the size above,
 * 256-byte aligned) holds the schedule, split-KV partial results and cascade
 * prefix partials; it must outlive the plan and must not be shared by two
 * plans whose work can overlap on the GPU.  Host-only: no device call is made.
 */
pkd_status pkd_plan_create(pkd_plan_t* plan_out, int max_batch, int num_qo_heads,
                           int num_kv_heads, int head_dim, int num_ctas, int max_prefix_splits,
                           void* d_workspace, size_t workspace_bytes);

/* Free the host-side plan object (the workspace stays the caller's). */
pkd_status pkd_plan_destroy(pkd_plan_t plan);

/*
 * Plan one decode step (the host "plan" of the pages' plan/run split).
 *   h_kv_indptr        host int32 [batch + 1]: kv_indptr[0] = 0, non-decreasing;
 *                      request b owns kv_page_indices[kv_indptr[b] .. kv_indptr[b+1]).
 *   d_kv_page_indices  device int32 [kv_indptr[batch]]: physical page ids.
 *                      Borrowed: it must hold the same contents at every
 *                      pkd_run / pkd_cascade_decode until the next pkd_plan.
 *                      Launches read it through this pointer, and a captured
 *                      graph keeps the pointer of the plan it was captured
 *                      with: re-plans for such a graph pass the same buffer.
 *   h_kv_last_page_len host int32 [batch]: valid tokens in each request's last
 *                      page, 1..page_size (ignored for a request with no page).
 *   page_size          tokens per page: 1..64, or a multiple of 64.
 * The split-KV rule: each (request, kv head) row is cut into chunks of up to 64
 * keys (whole pages for page_size <= 64); the list of all chunks, rows in
 * order r = b * num_kv_heads + h, is divided into num_ctas equal contiguous
 * runs of ceil(total / num_ctas) chunks, one per CTA.  A row that falls to one
 * CTA is written directly; rows split across CTAs are merged by a second pass.
 * plan writes the schedule into a pinned staging buffer owned by the plan;
 * the next pkd_run / pkd_cascade_decode copies it into the workspace with a
 * kernel.  Before overwriting the buffer, plan waits (host-side) for the copy
 * that read the previous schedule, so it blocks only until the GPU has begun
 * the previous step.  The first plan also clears the device error word with
 * one cudaMemsetAsync on `stream`.  plan must not be called during stream
 * capture; the launch shape of run never changes and its copy reads the
 * staging buffer, so a graph captured around run uploads the latest plan on
 * every replay and stays valid across re-plans of the same plan object.
 */
pkd_status pkd_plan(pkd_plan_t plan, const int32_t* h_kv_indptr, const int32_t* d_kv_page_indices,
                    const int32_t* h_kv_last_page_len, int batch, int num_qo_heads,
                    int num_kv_heads, int head_dim, int page_size, int q_dtype, int kv_dtype,
                    void* stream);

/*
 * Run batched paged decode with the last plan: (out, lse) for every request
 * and qo head.
 *   d_q        [batch, num_qo_heads, 128] in the planned q dtype.
 *   d_k_cache, d_v_cache  the K and V pools: page p, slot t, kv head h, dim d at
 *              element p * page_stride_elems + (t * num_kv_heads + h) * 128 + d
 *              (NHD, the default), or + (h * page_size + t) * 128 + d when the
 *              plan's layout is PKD_LAYOUT_HND (pkd_plan_set_kv_layout).
 *              page_stride_elems = page_size * num_kv_heads * 128 for separate
 *              pools, 2 * that for one interleaved [pages, 2, page] pool
 *              (then d_v_cache = d_k_cache + page_size * num_kv_heads * 128).
 *   num_pages  pages in each pool; page ids must lie in [0, num_pages).
 *   d_k_scale, d_v_scale  fp32 [num_kv_heads] for an E4M3 cache, else NULL.
 *   d_out      [batch, num_qo_heads, 128] q dtype;  d_lse fp32 [batch, num_qo_heads] or NULL.
 * Enqueues two kernels on `stream`: the schedule upload, then decode
 * (launched programmatically, so it may be scheduled before the upload ends,
 * and waits for it in-kernel).  The decode kernel also merges the split rows
 * (the CTA that finishes a row's last item folds its partial states) and
 * writes the rows of empty requests; a plan without any work item enqueues
 * the merge kernel instead of decode.  Grids depend only on the plan object;
 * event records go on a side stream of the plan that rejoins `stream`
 * (created on the first call).  No allocation, no host sync: capturable in a
 * CUDA graph.
 */
pkd_status pkd_run(pkd_plan_t plan, const void* d_q, const void* d_k_cache, const void* d_v_cache,
                   int64_t num_pages, int64_t page_stride_elems, const float* d_k_scale,
                   const float* d_v_scale, float sm_scale, void* d_out, float* d_lse, void* stream);

/*
 * Cascade (shared-prefix) decode: every request attends one shared prefix page
 * list and its own pages (the last plan's table, which holds only the private
 * suffixes); the two attention states are merged per (request, qo head).
 *   d_prefix_page_indices  device int32 [prefix_num_pages] (prefix_num_pages >= 0).
 *   prefix_last_page_len   valid tokens in the prefix's last page (1..page_size).
 * The prefix is attended once per kv head for all requests (a dense
 * [batch * g, 128] x [128, prefix_len] product on the tensor cores, 256 query
 * rows per pair of SMs), not once per request.  Every dtype pair, group size
 * and page size pkd_plan accepts is supported; E4M3 pools take k_scale /
 * v_scale as in pkd_run (their codes are widened exactly to q's type for the
 * products).  Other arguments as pkd_run.  The plan must have been created
 * with max_prefix_splits >= 1.  Enqueues the schedule upload, the prefix
 * kernel (it waits for the upload, then lets the next grid launch), the
 * suffix decode (launched programmatically behind it: its first CTAs start on
 * the SMs the prefix kernel leaves free, every item writes a partial state,
 * and the grid finishes only after the prefix kernel has) and the merge of the
 * prefix and suffix states.  With no suffix keys the decode grid is left out.
 * Capturable like pkd_run.
 */
pkd_status pkd_cascade_decode(pkd_plan_t suffix_plan, const int32_t* d_prefix_page_indices,
                              int prefix_num_pages, int prefix_last_page_len, const void* d_q,
                              const void* d_k_cache, const void* d_v_cache, int64_t num_pages,
                              int64_t page_stride_elems, const float* d_k_scale,
                              const float* d_v_scale, float sm_scale, void* d_out, float* d_lse,
                              void* stream);

/*
 * Prefix-tree (multi-level cascade) decode: every request attends the keys of
 * one node per shared level and then its own pages, the states of all parts
 * merged per (request, qo head) (2026 Guide, "Cascade attention for shared
 * prefixes"; README mirror, "Core Features": cascade attention as a
 * hierarchical KV cache).  Each node's keys are read once per kv head for all
 * of its requests (a dense [requests * g, 128] x [128, keys] product on the
 * tensor cores).
 *
 * pkd_plan_tree (host, after pkd_plan, which gives the requests' own pages;
 * not during stream capture) takes num_levels (1..4) shared levels, outermost
 * first.  For level l with h_num_nodes[l] nodes:
 *   h_req_indptr[l]        host int32 [nodes + 1]: node n serves requests
 *                          req_indptr[n] .. req_indptr[n+1]-1; the nodes
 *                          cover the batch in order (req_indptr[nodes] = batch).
 *   h_kv_indptr[l]         host int32 [nodes + 1] into the level's page list.
 *   d_kv_page_indices[l]   device int32 page ids (borrowed until the next plan;
 *                          a captured graph keeps these pointers, as for pkd_plan).
 *   h_kv_last_page_len[l]  host int32 [nodes]: 1..page_size (ignored for a
 *                          node without pages).
 * It cuts each level into key-range pieces (at most max_prefix_splits over all
 * levels; a level needs one), pairs each node's 128-row query tiles (one CTA
 * per pair, piece and kv head; a node's odd last tile is paired with an empty
 * one), writes the work units into the workspace with
 * one cudaMemcpyAsync on `stream` (waiting first for the previous such upload
 * of this plan) and fails with PKD_ERR_CAPACITY_EXCEEDED above the workspace's
 * unit capacity (8 * (max_batch + num_ctas), at least 4096).  f16/bf16 only
 * (q and K/V of one type), group sizes dividing 128, page sizes dividing 128
 * or multiples of 64.
 *
 * pkd_tree_decode enqueues the schedule upload, the requests' own decode
 * (every item writes a partial state), the tree kernel (one launch for all
 * levels) and the merge; arguments as pkd_run.  It fails with PKD_ERR_NO_PLAN
 * unless pkd_plan_tree followed the last pkd_plan.  The launch shapes follow
 * the tree's node and tile counts: a graph captured around it stays valid for
 * re-plans whose trees keep those counts.
 */
pkd_status pkd_plan_tree(pkd_plan_t plan, int num_levels, const int32_t* const* h_req_indptr,
                         const int32_t* const* h_kv_indptr, const int32_t* const* d_kv_page_indices,
                         const int32_t* const* h_kv_last_page_len, const int32_t* h_num_nodes, void* stream);
pkd_status pkd_tree_decode(pkd_plan_t plan, const void* d_q, const void* d_k_cache, const void* d_v_cache,
                           int64_t num_pages, int64_t page_stride_elems, float sm_scale, void* d_out,
                           float* d_lse, void* stream);

/*
 * Paged prefill / append attention (README mirror, "Core Features": prefill
 * and append kernels over a paged KV cache): several query tokens per request.
 * Request r's query tokens are rows h_qo_indptr[r] .. h_qo_indptr[r+1]-1 of
 * d_q [T, num_qo_heads, 128]; its keys are all of its pages (kv_len_r keys,
 * the query tokens' own keys already appended), so its token i sits at
 * position kv_len_r - q_len_r + i and, with `causal`, attends keys 0 .. that
 * position (otherwise all keys); q_len_r <= kv_len_r.
 *
 * pkd_plan_prefill (host; not during stream capture): page table as for
 * pkd_plan (h_kv_indptr, d_kv_page_indices borrowed until the next plan,
 * h_kv_last_page_len), head counts equal to the plan's, f16/bf16 q and K/V of
 * one type, group sizes dividing 128, page sizes dividing 128 or multiples of
 * 64.  One unit per 128-row query tile (128 / g tokens x g heads of a kv
 * head), in pairs of consecutive tiles of a request that one CTA per kv head
 * runs together, each key tile read once for both (a request's odd last tile
 * is paired with an empty one); the pairs are listed longest first and
 * uploaded like pkd_plan_tree's units (PKD_ERR_CAPACITY_EXCEEDED above the
 * unit capacity).
 *
 * pkd_prefill_run: d_out [T, num_qo_heads, 128] in q's dtype, d_lse fp32
 * [T, num_qo_heads] (natural log) or NULL; pools as pkd_run (the plan's
 * layout).  One kernel on `stream` (ordered after everything before it),
 * no allocation, no host sync.
 */
pkd_status pkd_plan_prefill(pkd_plan_t plan, const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                            const int32_t* d_kv_page_indices, const int32_t* h_kv_last_page_len, int batch,
                            int num_qo_heads, int num_kv_heads, int head_dim, int page_size, int q_dtype,
                            int kv_dtype, int causal, void* stream);
pkd_status pkd_prefill_run(pkd_plan_t plan, const void* d_q, const void* d_k_cache, const void* d_v_cache,
                           int64_t num_pages, int64_t page_stride_elems, float sm_scale, void* d_out,
                           float* d_lse, void* stream);

/*
 * Multi-latent attention (MLA) decode over a paged latent cache (deep dive,
 * "Technical Moats": DeepSeek-V2/V3's compressed KV attended without expanding
 * it; "The Code, Annotated": kv_lora_rank 512, q_rope_dim 64).  Every query
 * head of a request attends the request's cached rows, each a latent row ckv
 * (512) and a rotary key kpe (64) shared by all heads:
 *   s_j = sm_scale * (<q_nope[h], ckv_j> + <q_pe[h], kpe_j>),
 *   out[b, h] = sum_j softmax(s)_j ckv_j (512, in the latent space),
 *   lse[b, h] = ln sum_j exp(s_j).
 * q_nope is the no-RoPE query with the key up-projection already applied
 * (512), q_pe the rotary query (64); the value up-projection is the caller's.
 *   d_q_nope   bf16 [batch, num_heads, 512];  d_q_pe bf16 [batch, num_heads, 64].
 *   d_ckv_cache  bf16 pool: page p, slot t, dim d at p * ckv_page_stride_elems + t * 512 + d.
 *   d_kpe_cache  bf16 pool: p * kpe_page_stride_elems + t * 64 + d.
 *   h_kv_indptr, d_kv_page_indices, h_kv_last_page_len: the page table as for pkd_plan.
 *   num_heads 1..128; page_size a divisor of 32 or a multiple of 32.
 *   sm_scale <= 0 selects 1/sqrt(192) (128 no-RoPE + 64 RoPE query-key dims).
 *   d_out bf16 [batch, num_heads, 512]; d_lse fp32 [batch, num_heads] or NULL.
 *   d_workspace  pkd_mla_workspace_bytes(batch, num_heads, num_sms) bytes, 16-byte
 *                aligned; num_sms the device's SM count (work is cut for it).
 * Plans on the host (requests cut into key ranges that fill the SMs about
 * twice; two CTAs per range, one per half of the 512 output dims, each forming
 * the full S on the tensor cores), uploads the units with cudaMemcpyAsync into
 * the workspace (so not capturable), then enqueues the kernel and, when a
 * request was cut, a merge kernel.  Page ids outside [0, num_pages) are read
 * as page 0 and flagged in the workspace's first word (PKD_DEVERR_* bits).
 */
size_t pkd_mla_workspace_bytes(int max_batch, int num_heads, int num_sms);
pkd_status pkd_mla_decode(const void* d_q_nope, const void* d_q_pe, const void* d_ckv_cache,
                          const void* d_kpe_cache, const int32_t* h_kv_indptr, const int32_t* d_kv_page_indices,
                          const int32_t* h_kv_last_page_len, int batch, int num_heads, int page_size,
                          int64_t num_pages, int64_t ckv_page_stride_elems, int64_t kpe_page_stride_elems,
                          float sm_scale, void* d_out, float* d_lse, void* d_workspace, size_t workspace_bytes,
                          int num_sms, void* stream);

/*
 * Append new tokens' keys and values to the paged cache: the write step on
 * either side of each decode step (README mirror, "Core Features": decode,
 * prefill and append kernels over a paged KV cache).  Token i belongs to
 * request d_batch_indices[i] at position d_positions[i] of that request's
 * sequence; its rows, every kv head, go to page
 * d_kv_page_indices[d_kv_indptr[b] + pos / page_size], slot pos % page_size.
 * Pages must already be in the table (allocating them is the caller's); the
 * caller then plans the next decode with the longer lengths.
 *   d_k_new, d_v_new   device [n_tokens, num_kv_heads, 128] in new_dtype (F16 or BF16).
 *   d_batch_indices, d_positions   device int32 [n_tokens].
 *   d_kv_indptr        device int32 [batch + 1]; d_kv_page_indices device int32.
 *   d_k_cache, d_v_cache, num_pages, page_stride_elems   the pools as in pkd_run, kv_dtype;
 *   kv_layout          PKD_LAYOUT_NHD or PKD_LAYOUT_HND (the pools' page layout).
 *   kv_dtype F16/BF16: must equal new_dtype; the values are copied.
 *   kv_dtype E4M3: codes e4m3(x / scale[h]) with the quotient in fp32 (IEEE
 *     division), rounded to nearest even and saturated to +-448;
 *     d_k_scale / d_v_scale fp32 [num_kv_heads] (the scales decode reads).
 *   d_err_word         optional device uint32: a token whose request, position
 *     or page lies outside the table or the pool writes nothing and sets
 *     PKD_DEVERR_PAGE_INDEX here (a plan's workspace start is such a word).
 * Tokens must not target the same (page, slot) twice.  One kernel on `stream`,
 * no allocation, no host sync (capturable).
 */
pkd_status pkd_append_kv(const void* d_k_new, const void* d_v_new, int new_dtype,
                         const int32_t* d_batch_indices, const int32_t* d_positions, int n_tokens,
                         const int32_t* d_kv_indptr, const int32_t* d_kv_page_indices, int batch,
                         int num_kv_heads, int head_dim, int page_size, void* d_k_cache,
                         void* d_v_cache, int kv_dtype, int kv_layout, int64_t num_pages,
                         int64_t page_stride_elems, const float* d_k_scale,
                         const float* d_v_scale, uint32_t* d_err_word, void* stream);

/*
 * Single-request decode with contiguous K/V (the quickstart call):
 *   d_q [num_qo_heads, 128]; d_k, d_v [kv_len, num_kv_heads, 128] (kv_len >= 0);
 *   d_out [num_qo_heads, 128] (q dtype); d_lse fp32 [num_qo_heads] or NULL.
 *   q_dtype / kv_dtype as for pkd_plan; d_k_scale / d_v_scale for E4M3.
 * Plans internally and runs the batched path on it.  The schedule (a few KB
 * for one request) is carried in the parameters of the kernel that writes it
 * into d_workspace, so the call allocates nothing, never touches a copy engine
 * and can be captured in a CUDA graph (the graph replays the kv_len it was
 * captured with); only a schedule above 16 KB (num_kv_heads + num_ctas above
 * ~900) falls back to one cudaMemcpyAsync, which is not capturable.
 * d_workspace must hold pkd_workspace_bytes(1, num_qo_heads, num_kv_heads,
 * 128, num_ctas, 0) bytes.
 */
pkd_status pkd_single_decode(const void* d_q, const void* d_k, const void* d_v, int kv_len,
                             int num_qo_heads, int num_kv_heads, int head_dim, int q_dtype,
                             int kv_dtype, const float* d_k_scale, const float* d_v_scale,
                             float sm_scale, void* d_out, float* d_lse, void* d_workspace,
                             size_t workspace_bytes, void* stream);

/*
 * merge_state: the state over the union of two disjoint key sets
 * (flashinfer.cascade merge_state):
 *   s = logaddexp(s_a, s_b);  v = v_a * exp(s_a - s) + v_b * exp(s_b - s).
 * v_a, v_b, v_out: [n, num_heads, head_dim] in v_dtype (F32, F16 or BF16);
 * s_a, s_b, s_out: fp32 [n, num_heads], natural log.  A state with s = -inf is
 * empty (identity); two empty states give v = 0, s = -inf.  v_out / s_out may
 * alias v_a / s_a.  head_dim: any multiple of 8 up to 1024.
 */
pkd_status pkd_merge_state(const void* d_v_a, const float* d_s_a, const void* d_v_b,
                           const float* d_s_b, void* d_v_out, float* d_s_out, int64_t n,
                           int num_heads, int head_dim, int v_dtype, void* stream);

/*
 * merge_states: merge k states per (index, head):
 *   d_v [n, k, num_heads, head_dim] (v_dtype), d_s fp32 [n, k, num_heads]
 *   -> d_v_out [n, num_heads, head_dim] (v_dtype), d_s_out fp32 [n, num_heads].
 * k = 0 gives empty states.  Same dtype and head_dim rules as pkd_merge_state.
 */
pkd_status pkd_merge_states(const void* d_v, const float* d_s, int64_t n, int k, int num_heads,
                            int head_dim, int v_dtype, void* d_v_out, float* d_s_out,
                            void* stream);

/*
 * Timing hook: when both are non-NULL, pkd_run and pkd_cascade_decode record
 * start_event just before the decode kernel and stop_event just after it, on
 * the call's stream (cudaEvent_t handles passed as void*; the caller owns
 * them).  NULL, NULL turns the hook off.  Lets a caller time the dominant
 * kernel alone with CUDA events.  The stop event is recorded on a side stream
 * of the plan that waits for the decode kernel and rejoins the call's stream
 * at the end of the call, so the kernel after decode keeps its programmatic
 * early launch.  During stream capture the records are made with
 * cudaEventRecordExternal, so a captured graph records them on every replay.
 * The first call that enables the hook creates the side stream and two
 * events (PKD_ERR_CUDA if that fails); pkd_plan_destroy releases them.
 */
pkd_status pkd_plan_set_timing_events(pkd_plan_t plan, void* start_event, void* stop_event);

/*
 * Read and clear the plan's device error word (PKD_DEVERR_* bits), after
 * synchronising `stream`.  Returns PKD_ERR_DEVICE_CHECK when a bit was set.
 */
pkd_status pkd_check_device_errors(pkd_plan_t plan, uint32_t* flags_out, void* stream);

/*
 * Page layout (pkd_kv_layout) of the pools later pkd_run / pkd_cascade_decode
 * calls of this plan read; PKD_LAYOUT_NHD until set.  PKD_ERR_INVALID_ARG for
 * another value.  Host-side only; a graph captured around run keeps the
 * layout it was captured with.
 */
pkd_status pkd_plan_set_kv_layout(pkd_plan_t plan, int kv_layout);

/*
 * Test hook for the pipeline's failure path (the pages have no counterpart).
 * With PKD_DEBUG_STALL_PIPELINE set, the decode kernel of later pkd_run calls
 * issues no copies, so every consumer's first pipeline wait runs out after its
 * time limit (about 2 s): the kernel then leaves with PKD_DEVERR_WAIT_TIMEOUT
 * in the device error word instead of hanging, and its outputs are undefined.
 * 0 turns it off.  Host-side only; no other effect.
 */
#define PKD_DEBUG_STALL_PIPELINE 1
pkd_status pkd_plan_set_debug(pkd_plan_t plan, int flags);

/*
 * Batched paged decode that allocates nothing (the pages have no counterpart:
 * this is a library convenience, not part of the method).
 *
 * For callers that may not allocate device memory when they run attention --
 * a serving loop whose memory is carved out up front by its own pool (a
 * cudaMalloc there can synchronise the device and fragment the pool), a plugin
 * inside a runtime that owns every allocation, or code held to a fixed memory
 * footprint.  It takes the arguments of pkd_plan and pkd_run together and does
 * both, using a scratch area built into the library instead of a caller
 * workspace: PKD_NOALLOC_SCRATCH_BYTES of device memory that every GPU loading
 * this library holds until the process exits.  Calls that need more scratch
 * (roughly: batch * num_kv_heads + 2 * SM count work items, each with
 * g * 128 fp32 partial outputs) return PKD_ERR_CAPACITY_EXCEEDED with a message.
 * No cudaMalloc, cudaFree, pinned-host or other allocating call is made.
 *   - The first call on a device looks up that device's scratch address
 *     (cudaGetSymbolAddress, with the device current); make that first call
 *     before any stream capture on the device.
 *   - The schedule is uploaded from a host buffer of the library that every
 *     call rewrites, with a cudaMemcpyAsync on `stream`; the call returns
 *     PKD_ERR_UNSUPPORTED while `stream` is being captured.
 *   - All calls share the one scratch area per device: calls whose work can
 *     overlap on the GPU (different streams, different threads) race and must
 *     be serialised by the caller.  Each call resets what must start at zero,
 *     the device error word included.
 *   - Device error bits (PKD_DEVERR_*) of the last call are kept in the
 *     scratch area (pkd_noalloc_device_errors reads them); an out-of-range
 *     page id is read as page 0 and sets PKD_DEVERR_PAGE_INDEX.
 *   - Two limits, each reported as PKD_ERR_CAPACITY_EXCEEDED with a message
 *     naming it: the device scratch (PKD_NOALLOC_SCRATCH_BYTES) and the
 *     library's 256 KiB host buffer for the schedule.
 * Arguments as pkd_plan and pkd_run (h_* are host arrays, d_* device);
 * kv_layout is the pools' page layout (pkd_kv_layout).
 */
#define PKD_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
pkd_status pkd_decode_noalloc(const int32_t* h_kv_indptr, const int32_t* d_kv_page_indices,
                              const int32_t* h_kv_last_page_len, int batch, int num_qo_heads,
                              int num_kv_heads, int head_dim, int page_size, int q_dtype,
                              int kv_dtype, int kv_layout, const void* d_q, const void* d_k_cache,
                              const void* d_v_cache, int64_t num_pages, int64_t page_stride_elems,
                              const float* d_k_scale, const float* d_v_scale, float sm_scale,
                              void* d_out, float* d_lse, void* stream);

/*
 * Device error bits (PKD_DEVERR_*) recorded by the last pkd_decode_noalloc
 * call on the current device, read from its scratch area after synchronising
 * `stream` (the next call clears them).  *flags_out gets the bits; returns
 * PKD_ERR_DEVICE_CHECK when a bit was set.  Allocates nothing.
 */
pkd_status pkd_noalloc_device_errors(uint32_t* flags_out, void* stream);

/*
 * The split-KV rule of pkd_plan, run on the host only (no GPU), for
 * inspection and testing.  Outputs (caller-allocated host arrays):
 *   items           int32 [max_items * 4]: (row, chunk_begin, chunk_end, cta) per item,
 *                   row = b * num_kv_heads + h; an item's index is its partial slot.
 *   cta_item_begin  int32 [num_ctas + 1]: items of CTA c are [cta_item_begin[c], cta_item_begin[c+1]).
 *   row_item_begin, row_item_count  int32 [batch * num_kv_heads].
 *   merge_rows      int32 [batch * num_kv_heads]: rows whose item count is not 1, ascending.
 *   counts          int32 [4]: n_items, n_merge_rows, chunk_keys, chunks per CTA (quota).
 * Returns PKD_ERR_CAPACITY_EXCEEDED if more than max_items items result
 * (batch * num_kv_heads + num_ctas always suffices).
 */
pkd_status pkd_plan_host(const int32_t* h_kv_indptr, const int32_t* h_kv_last_page_len, int batch,
                         int num_kv_heads, int page_size, int num_ctas, int32_t* items,
                         int max_items, int32_t* cta_item_begin, int32_t* row_item_begin,
                         int32_t* row_item_count, int32_t* merge_rows, int32_t* counts);

/*
 * The work lists of pkd_plan_prefill and pkd_plan_tree, built on the host only
 * (no GPU, no plan), for inspection and testing.  Each unit is 12 int32 in the
 * order (q0, q_end, page_begin, kv_len, t0, t1, piece, level, diag, 0, 0, 0):
 * query rows (tokens for prefill, requests for the tree) q0 .. min(q0 + 128/g,
 * q_end) - 1 of one 128-row tile, keys of the page list starting at entry
 * page_begin (kv_len of them) in 128-key tiles t0 .. t1 - 1, output piece
 * (-1: final output) of tree level `level`, causal offset diag (token q sees
 * keys 0 .. q + diag; 2^31 - 1: every key).  Units 2j and 2j + 1 form one CTA's
 * pair: the same keys, the second tile's rows following the first's (or
 * q0 = q_end: no rows); pairs are listed longest key range first.
 *   units_out   int32 [max_units * 12]; *n_units_out the number of units (also
 *               when it exceeds max_units, which returns PKD_ERR_CAPACITY_EXCEEDED).
 * pkd_prefill_units_host takes the arguments of pkd_plan_prefill that shape the
 * list (num_qo_heads / num_kv_heads a group size dividing 128).
 * pkd_tree_units_host takes those of pkd_plan_tree plus the plan's batch,
 * head counts, page size, num_ctas (pkd_num_ctas) and max_prefix_splits;
 * *n_pieces_out receives the pieces per request row over all levels.
 * Errors: the statuses pkd_plan_prefill / pkd_plan_tree return for the same
 * arguments.
 */
pkd_status pkd_prefill_units_host(const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                                  const int32_t* h_kv_last_page_len, int batch, int num_qo_heads,
                                  int num_kv_heads, int page_size, int causal, int32_t* units_out, int max_units,
                                  int* n_units_out);
pkd_status pkd_tree_units_host(int num_levels, const int32_t* const* h_req_indptr,
                               const int32_t* const* h_kv_indptr, const int32_t* const* h_kv_last_page_len,
                               const int32_t* h_num_nodes, int batch, int num_qo_heads, int num_kv_heads,
                               int page_size, int num_ctas, int max_prefix_splits, int32_t* units_out,
                               int max_units, int* n_units_out, int* n_pieces_out);

/*
 * The key-range split of pkd_mla_decode, built on the host only (no GPU), for
 * inspection and testing: units of 12 int32 as above with q0 = request,
 * q_end = request + 1, t0 .. t1 - 1 in 32-key tiles, piece (-1: the request is
 * one range, written directly) and level = the half of the 512 output dims
 * (0, 1); the two halves of a range are adjacent, ranges longest first.
 *   req_piece_begin_out  int32 [batch + 1]: a cut request's pieces are
 *                        req_piece_begin[b] .. req_piece_begin[b+1] - 1.
 * Errors: those of pkd_mla_decode for the same page table and num_sms;
 * PKD_ERR_CAPACITY_EXCEEDED (with *n_units_out set) above max_units.
 */
pkd_status pkd_mla_units_host(const int32_t* h_kv_indptr, const int32_t* h_kv_last_page_len, int batch,
                              int page_size, int num_sms, int32_t* units_out, int max_units, int* n_units_out,
                              int32_t* req_piece_begin_out);

#ifdef __cplusplus
}
#endif

#endif /* PKD_H */
