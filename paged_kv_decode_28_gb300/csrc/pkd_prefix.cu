// pkd_prefix.cu -- shared-prefix (cascade level 0) attention on pairs of SMs:
// tcgen05 MMAs of cta_group::2 with TMEM accumulators, for sm_103a.
//
// Cascade decode attends one shared prefix for every request and merges that
// state with each request's own (2026 guide, "Cascade attention for shared
// prefixes"; deep dive, "Why This Design Works": the shared prefix is read once
// but counted as if each request owns it).  For one kv head h the prefix part
// is a dense product: the B * g query rows of the group against the prefix
// keys.  A CTA holds R = floor(128 / g) requests, i.e. R * g query rows (row r
// is qo head h * g + r % g of request b0 + r / g; the rows past R * g are
// zero); the two CTAs of a cluster form a pair and compute a 256-row product:
// the MMA, issued by the even CTA, takes each CTA's 128 query rows and each
// CTA's half of every key tile's K rows (keys 64 c .. 64 c + 63 of CTA c) and
// V columns (head dims 64 c .. 64 c + 63), and leaves each CTA's rows of S and
// of O in that CTA's TMEM.  So every SM receives half of each K/V tile it
// multiplies, and no load is shared between CTAs (no multicast).  A pair takes
// a contiguous range of 128-key tiles of the prefix and writes an fp32 partial
// state (o, base-2 lse) per row; the merge pass folds these into each
// request's suffix state.
//
// Per CTA (384 threads):
//   warp 0      Q (once) and the K ring, page by page: boxes of gcd(P, 64)
//               keys, 128-byte swizzled, K-major.  16-bit pools load straight
//               into the K slots and signal the even CTA's "K full" barrier
//               (cta_group::2 loads), so it fires when both halves landed;
//   warp 2      the V ring, this CTA's 64 head dims of all 128 keys, MN-major,
//               signalled on this CTA's own "V full" barrier.  For e4m3 pools
//               warps 0 and 2 load the codes into a two-slot staging ring and
//               widen them exactly into q's 16-bit type in the slots the MMAs
//               read (every E4M3 value is an f16 and a bf16) while the next
//               tile's codes are in flight; the per-kv-head scales are folded
//               into the score scale and the output;
//   warp 1      allocates the pair's 512 TMEM columns (both CTAs); in the even
//               CTA one thread issues every MMA: S = Q K^T into one of three S
//               buffers two tiles ahead of O += P_hi V + P_lo V, and commits
//               to both CTAs' barriers;
//   warp 3      in the odd CTA, relays its softmax warps' "P written" to the
//               even CTA with one cluster-scope arrival per tile;
//   warps 4..11 softmax, two threads per query row (keys 0..63 / 64..127 of
//               each tile), the 64 scores of a tile read from TMEM once (the
//               next tile's read is issued as soon as P is written): maximum
//               with the row's other half through shared memory, a running
//               reference max (O is rescaled in TMEM only when the tile max
//               exceeds it by more than 8 in log2 units), P = 2^(s * scale - m)
//               written over the scores as two 16-bit parts (P_hi = round(P),
//               P_lo = round(P - P_hi), so P enters the product to ~2^-17);
//               then, once this CTA's V tile has landed (16-bit pools: zeroing
//               V rows past the prefix end), one arrival per warp: the P V
//               product of a tile waits for the softmax of both CTAs.
// TMEM columns: S0 [0,128), S1 [128,256), S2 [256,384), O [384,512).  P of a
// tile's keys 16k .. 16k + 15: P_hi of keys 16k + 2e, 16k + 2e + 1 in column
// 16k + e, P_lo in column 16k + 8 + e (e = 0..7), over the scores of those keys.
#include "pkd_internal.h"
#include "pkd_ptx.cuh"

namespace pkd {
namespace {

constexpr int kRows = 128;      // query rows per CTA (a pair computes 256)
constexpr int kKeys = 128;      // keys per key tile (the S product's N)
constexpr int kHalfKeys = 64;   // keys of a K tile one CTA holds
constexpr int kKStages = 3;     // ring depth of K
constexpr int kVStages = 4;     // ring depth of V (a V slot is freed two tiles after its K slot)
constexpr int kSoftmaxWarps = 8;
constexpr int kStaging = 2;     // e4m3: staging slots of codes per side
constexpr int kCluster = 2;     // one pair
constexpr float kRescaleThreshold = 8.0f;

template <bool FP8>
struct PCfg {
  static constexpr int kThreads = (4 + kSoftmaxWarps) * 32;
  static constexpr int kQHalf = kRows * 128;      // [128 rows][128 B]: 64 of q's dims
  static constexpr int kKHalf = kHalfKeys * 128;  // [64 keys][128 B]: 64 dims of this CTA's keys
  static constexpr int kKStage = 2 * kKHalf;
  static constexpr int kVStage = kKeys * 128;     // [128 keys][128 B]: this CTA's 64 dims
  static constexpr int kVSt = FP8 ? kVStages - 1 : kVStages;  // e4m3: one slot less, for the staging ring
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + 2 * kQHalf;
  static constexpr int kV = kK + kKStages * kKStage;
  // e4m3 codes as loaded: K [64 keys][128 B], V [128 keys][64 B] (this CTA's
  // dims).  A copy's shared-memory destination must be 128-byte aligned, so
  // when the boxes are single keys (odd page sizes) the V rows sit 128 bytes
  // apart: the V slot has room for that.
  static constexpr int kK8Stage = kHalfKeys * 128;
  static constexpr int kV8Stage = kKeys * 128;
  static constexpr int kK8 = kV + kVSt * kVStage;
  static constexpr int kV8 = kK8 + (FP8 ? kStaging * kK8Stage : 0);
  static constexpr int kBars = kV8 + (FP8 ? kStaging * kV8Stage : 0);
  static constexpr int kTmemSlot = kBars + 64 * 8;
  static constexpr int kAbort = kTmemSlot + 8;
  static constexpr int kXchg = kAbort + 8;  // fp32 [buffer][half][row]: the halves' partial maxima / sums
  static constexpr int kTotal = kXchg + 4 * 2 * 2 * kRows;
  static constexpr int kAlloc = kTotal + 1024;
  static_assert(kAlloc <= 227 * 1024, "dynamic shared memory above the 227 KB a CTA may use");
};

enum {
  B_Q = 0,                   // Q of both CTAs landed (even CTA)
  B_KF = 1,                  // K tile of both CTAs ready (even CTA) [kKStages]
  B_KE = B_KF + kKStages,    // K slot free (each CTA) [kKStages]
  B_VF = B_KE + kKStages,    // this CTA's V tile ready [kVStages]
  B_VE = B_VF + kVStages,    // V slot free (each CTA) [kVStages]
  B_SF = B_VE + kVStages,    // S ready (each CTA) [3]
  B_PF = B_SF + 3,           // P of both CTAs written (even CTA) [3]
  B_OD = B_PF + 3,           // P V done (each CTA) [3]
  B_K8F = B_OD + 3,          // e4m3: codes landed in a staging slot [kStaging]
  B_V8F = B_K8F + kStaging,
  B_PL = B_V8F + kStaging,   // odd CTA: its softmax warps' P written [3] (relayed by warp 3)
  B_DRAIN = B_PL + 3,        // even CTA: every MMA done
  kNumBars = B_DRAIN + 1
};
static_assert(kNumBars <= 64, "barrier area");

constexpr uint32_t kColO = 384, kTmemCols = 512;
__device__ __forceinline__ uint32_t col_s(int u) { return static_cast<uint32_t>(u) * 128u; }

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, unsigned* err, volatile int* abort_flag) {
  if (*abort_flag) return false;
  if (ptx::mbar_wait(bar, parity, err)) return true;
  *abort_flag = 1;
  return false;
}

// The same for a barrier that the other CTA of the pair arrives on.
__device__ __forceinline__ bool wait_or_abort_cluster(uint32_t bar, uint32_t parity, unsigned* err,
                                                      volatile int* abort_flag) {
  if (*abort_flag) return false;
  if (ptx::mbar_wait_cluster(bar, parity, err)) return true;
  *abort_flag = 1;
  return false;
}

// The same, for a whole warp: every lane polls, and the result is made
// warp-uniform so that no lane leaves a loop that the others stay in.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, unsigned* err, volatile int* abort_flag) {
  const bool r = wait_or_abort(bar, parity, err, abort_flag);
  return __all_sync(0xffffffffu, r);
}

// Eight E4M3 codes (bytes of w0, w1) -> eight 16-bit values (bf16 when BF,
// else f16) as four packed pairs, exact: every E4M3 value is an f16 and a bf16.
template <bool BF>
__device__ __forceinline__ void widen8(uint32_t w0, uint32_t w1, uint32_t (&o)[4]) {
  const uint32_t w[2] = {w0, w1};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t lo, hi;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w[i]));
    if constexpr (BF) {
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
      lo = ptx::pack2<true>(a.x, a.y);
      hi = ptx::pack2<true>(b.x, b.y);
    }
    o[2 * i] = lo;
    o[2 * i + 1] = hi;
  }
}

template <bool BF, bool FP8>
__global__ void __launch_bounds__(PCfg<FP8>::kThreads, 1)
    prefix_pair_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const PrefixParams p) {
  using C = PCfg<FP8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::kAbort);
  auto bar = [&](int i) { return base + C::kBars + 8u * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int Hq = p.num_kv_heads * G;
  const int R = p.req_per_tile;  // requests per CTA
  // cluster rank c (0 or 1): K keys 64 c .. 64 c + 63 and V dims 64 c ..
  // 64 c + 63 of every tile; rank 0 issues the pair's MMAs
  const uint32_t rank = ptx::cluster_ctarank() & 1u;
  const uint32_t leader = 0;
  const bool lead = rank == 0;
  const uint16_t pair_mask = 3;
  // this pair's unit: kv head h, CTA rows from request b0, prefix keys in
  // tiles t0 .. t0 + n - 1, piece `split`;
  // blockIdx.x = ((h * n_splits + split) * m_groups + mpair) * 2 + rank
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int mpair = pair % p.m_groups;
  const int hs = pair / p.m_groups;
  const int split = hs % p.n_splits;
  const int h = hs / p.n_splits;
  const int b0 = (2 * mpair + static_cast<int>(rank)) * R;  // may pass the batch: the CTA then only loads its halves
  const int kv_len = p.prefix_len;
  const int* pages = p.prefix_pages;
  const int n_tiles_all = (kv_len + kKeys - 1) / kKeys;
  const int t0 = split * p.tiles_per_split;
  const int n = max(min(t0 + p.tiles_per_split, n_tiles_all) - t0, 0);
  const int used_rows = R * G;
  auto tile_of = [&](int i) { return t0 + i; };  // the i-th tile processed

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(B_Q), 1);
    for (int s = 0; s < kKStages; ++s) {
      // 16-bit pools: the even CTA's producer arrives with the pair's bytes;
      // e4m3: the K producer of each CTA arrives once it has widened its half
      ptx::mbar_init(bar(B_KF + s), FP8 ? 2 : 1);
      ptx::mbar_init(bar(B_KE + s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      ptx::mbar_init(bar(B_VF + s), 1);
      ptx::mbar_init(bar(B_VE + s), 1);
    }
    for (int s = 0; s < kStaging; ++s) {
      ptx::mbar_init(bar(B_K8F + s), 1);
      ptx::mbar_init(bar(B_V8F + s), 1);
    }
    for (int u = 0; u < 3; ++u) {
      ptx::mbar_init(bar(B_SF + u), 1);
      // the even CTA's softmax warps, and one relayed arrival for the odd CTA's
      ptx::mbar_init(bar(B_PF + u), kSoftmaxWarps + 1);
      ptx::mbar_init(bar(B_OD + u), 1);
      ptx::mbar_init(bar(B_PL + u), kSoftmaxWarps);
    }
    ptx::mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    // launched programmatically behind the schedule upload, which itself
    // waits for the previous step's merge (a reader of pre_o) and for the
    // kernels that wrote this step's inputs
    ptx::pdl_wait_prior_grid();
  }
  // the odd CTA of the last pair may hold no request at all: it loads no Q
  const bool has_q = b0 < p.batch;
  if (warp == 0 && (used_rows < kRows || !has_q)) {
    // query rows that get no box (past R * g, or all of them) are zero in both column halves
    for (int i = (has_q ? used_rows : 0) * 8 + lane; i < kRows * 8; i += 32) {
      const int r = i >> 3, c = i & 7;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(base_ptr + C::kQ + r * 128 + c * 16) = z;
      *reinterpret_cast<uint4*>(base_ptr + C::kQ + C::kQHalf + r * 128 + c * 16) = z;
    }
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(base + C::kTmemSlot, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  // The suffix decode grid behind this one may start now, on the SMs this grid
  // leaves free: it reads nothing this grid writes, and it ends only after
  // this grid has, so the merge grid behind it finds both done.
  ptx::pdl_launch_dependents();
  ptx::cluster_sync();  // both CTAs' barriers exist (and Q's zero rows are written) before any signal crosses
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base_ptr + C::kTmemSlot);
  const int box = p.box_tok;

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ TMA producers (K: warp 0, V: warp 2)
    const bool kside = warp == 0;
    if (n > 0) {
      if (kside && lane == 0) {
        ptx::prefetch_tensormap(&tmq);
        ptx::prefetch_tensormap(&tmk);
        ptx::prefetch_tensormap(&tmv);
        // q viewed as [B][Hk][g][128]: a box of R requests x g heads of kv head h
        // (the even CTA expects the box bytes of both CTAs that hold requests)
        const uint32_t qbytes = static_cast<uint32_t>(used_rows) * 128u * 2u;
        if (lead)
          ptx::mbar_arrive_expect_tx(bar(B_Q), (has_q ? qbytes : 0u) + (b0 + R < p.batch ? qbytes : 0u));
        if (has_q) {
          const uint32_t lead_q = ptx::mapa(bar(B_Q), leader);  // the even CTA's barrier
          ptx::tma_load_4d_pair(base + C::kQ, &tmq, lead_q, 0, 0, h, b0);
          ptx::tma_load_4d_pair(base + C::kQ + C::kQHalf, &tmq, lead_q, 64, 0, h, b0);
        }
      }
      // this CTA's keys of tile i: K rows key0 + 64 rank .. (kside), or all
      // 128 keys of the tile (V side); boxes of `box` keys never cross a page
      auto span = [&](int i, int& first, int& cnt) {
        const int key0 = tile_of(i) * kKeys;
        if (kside) {
          first = key0 + kHalfKeys * static_cast<int>(rank);
          cnt = min(max(kv_len - first, 0), kHalfKeys);
        } else {
          first = key0;
          cnt = min(kv_len - key0, kKeys);
        }
      };
      const CUtensorMap* map = kside ? &tmk : &tmv;
      const int vst = kside ? kKStages : C::kVSt;  // ring depth of this side
      // page ids and in-page offsets of tile i's boxes that this lane issues
      // (box j = lane + 32 r; at most 128 boxes of a 128-key tile), read two
      // tiles ahead of their use so that the table's latency stays off the loads
      auto fetch = [&](int i, int (&pg)[4], int (&tk)[4]) {
        int first = 0, cnt = 0;
        if (i < n) span(i, first, cnt);
        const int boxes = (cnt + box - 1) / box;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          pg[r] = 0;
          tk[r] = 0;
          const int j = lane + 32 * r;
          if (j < boxes) {
            const int key = first + j * box;
            const int pi = key / p.page_size;
            pg[r] = __ldg(pages + pi);  // checked at use, so the load stays in flight
            tk[r] = key - pi * p.page_size;
          }
        }
      };
      // issue the boxes of tile i into dst0 (rows row_bytes apart), completing on
      // `full`; pair loads (16-bit K) signal the even CTA's barrier
      auto issue = [&](int i, const int (&pg)[4], const int (&tk)[4], uint32_t dst0, uint32_t row_bytes, uint32_t full,
                       int c0, bool pair_load) {
        int first, cnt;
        span(i, first, cnt);
        const int boxes = (cnt + box - 1) / box;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int j = lane + 32 * r;
          if (j < boxes) {
            int page = pg[r];
            if (static_cast<unsigned>(page) >= static_cast<unsigned>(p.num_pages)) {
              atomicOr(p.err, kDevErrPageIndex);
              page = 0;
            }
            // map coordinates (dim, head, key, page) for NHD pages, (dim, key, head, page) for HND
            const int c1 = p.kv_hnd ? tk[r] : h, c2 = p.kv_hnd ? h : tk[r];
            const uint32_t d = dst0 + static_cast<uint32_t>(j * box) * row_bytes;
            if (pair_load) {
              ptx::tma_load_4d_pair(d, map, full, c0, c1, c2, page);
              ptx::tma_load_4d_pair(d + C::kKHalf, map, full, c0 + 64, c1, c2, page);
            } else {
              ptx::tma_load_4d(d, map, full, c0, c1, c2, page);
            }
          }
        }
      };
      // the side's loads of tile i with its fetched page ids; false once a wait gave up
      auto step = [&](int i, const int (&pg)[4], const int (&tk)[4]) -> bool {
        if constexpr (!FP8) {
          // 16-bit pools: straight into the K / V slots
          const int s = i % vst;
          if (!warp_wait(bar((kside ? B_KE : B_VE) + s), ((i / vst) & 1) ^ 1, p.err, abort_flag)) return false;
          int first, cnt;
          span(i, first, cnt);
          const uint32_t bytes_here = static_cast<uint32_t>((cnt + box - 1) / box * box) * 128u;
          if (kside) {
            // the even CTA expects both CTAs' K bytes of this tile (its own
            // keys and the odd CTA's, from key0 + 64 on), two column halves each
            if (lead && lane == 0) {
              const int c1 = min(max(kv_len - (tile_of(i) * kKeys + kHalfKeys), 0), kHalfKeys);
              ptx::mbar_arrive_expect_tx(bar(B_KF + s),
                                         2u * bytes_here + static_cast<uint32_t>((c1 + box - 1) / box * box) * 256u);
            }
            __syncwarp();
            issue(i, pg, tk, base + C::kK + s * C::kKStage, 128u, ptx::mapa(bar(B_KF + s), leader), 0, true);
          } else {
            if (lane == 0) ptx::mbar_arrive_expect_tx(bar(B_VF + s), bytes_here);
            __syncwarp();
            issue(i, pg, tk, base + C::kV + s * C::kVStage, 128u, bar(B_VF + s), 64 * static_cast<int>(rank), false);
          }
          return true;
        } else {
          // e4m3 pools: the codes of tile i go to a two-slot staging ring; this
          // warp then widens tile i - 1 into its K / V slot (V rows past the
          // prefix end as zeros) while tile i's codes are in flight
          const int f8 = kside ? B_K8F : B_V8F;
          const uint32_t stg = base + (kside ? C::kK8 : C::kV8);
          const uint32_t stg_bytes = kside ? C::kK8Stage : C::kV8Stage;
          const uint32_t row_bytes = kside ? 128u : 64u;
          // where the rows land: V rows of single-key boxes 128 bytes apart
          const uint32_t row_stride = kside || box > 1 ? row_bytes : 128u;
          if (i < n) {
            const int s8 = i % kStaging;
            int first, cnt;
            span(i, first, cnt);
            // the widening reads of this slot (tile i - 2) come before the copy into it
            ptx::fence_proxy_async_smem();
            if (lane == 0)
              ptx::mbar_arrive_expect_tx(bar(f8 + s8), static_cast<uint32_t>((cnt + box - 1) / box * box) * row_bytes);
            __syncwarp();
            issue(i, pg, tk, stg + s8 * stg_bytes, row_stride, bar(f8 + s8), kside ? 0 : 64 * static_cast<int>(rank),
                  false);
          }
          if (i == 0) return true;
          const int w = i - 1;  // the tile to widen
          const int s8 = w % kStaging, s = w % vst;
          if (!warp_wait(bar(f8 + s8), (w / kStaging) & 1, p.err, abort_flag)) return false;
          if (!warp_wait(bar((kside ? B_KE : B_VE) + s), ((w / vst) & 1) ^ 1, p.err, abort_flag)) return false;
          const uint8_t* src = base_ptr + (stg - base) + s8 * stg_bytes;
          if (kside) {
            // [64 keys][128 codes] -> [2 halves][64 keys][128 B]
            const uint32_t kb = base + C::kK + s * C::kKStage;
#pragma unroll 4
            for (int item = lane; item < kHalfKeys * 8; item += 32) {
              const int key = item >> 3, c = item & 7;  // 16 codes = head dims 16 c .. 16 c + 15
              const uint4 raw = *reinterpret_cast<const uint4*>(src + key * 128 + c * 16);
              uint32_t a[4], bq[4];
              widen8<BF>(raw.x, raw.y, a);
              widen8<BF>(raw.z, raw.w, bq);
              const uint32_t half = static_cast<uint32_t>(c >> 2), ch = 2u * static_cast<uint32_t>(c & 3);
              ptx::sts128(kb + half * C::kKHalf + ptx::sw128(key, ch), a[0], a[1], a[2], a[3]);
              ptx::sts128(kb + half * C::kKHalf + ptx::sw128(key, ch + 1), bq[0], bq[1], bq[2], bq[3]);
            }
          } else {
            // [128 keys][64 codes] -> [128 keys][128 B]
            const int nv = min(kKeys, kv_len - tile_of(w) * kKeys);
            const uint32_t vb = base + C::kV + s * C::kVStage;
#pragma unroll 4
            for (int item = lane; item < kKeys * 4; item += 32) {
              const int key = item >> 2, c = item & 3;
              uint32_t a[4] = {0u, 0u, 0u, 0u}, bq[4] = {0u, 0u, 0u, 0u};
              if (key < nv) {
                const uint4 raw = *reinterpret_cast<const uint4*>(src + key * row_stride + c * 16);
                widen8<BF>(raw.x, raw.y, a);
                widen8<BF>(raw.z, raw.w, bq);
              }
              ptx::sts128(vb + ptx::sw128(key, 2u * c), a[0], a[1], a[2], a[3]);
              ptx::sts128(vb + ptx::sw128(key, 2u * c + 1u), bq[0], bq[1], bq[2], bq[3]);
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (kside) {
              ptx::mbar_arrive_cluster(ptx::mapa(bar(B_KF + s), leader));  // the pair's K tile: both CTAs' halves
            } else {
              ptx::mbar_arrive(bar(B_VF + s));
            }
          }
          return true;
        }
      };
      // three register sets of page ids in rotation, unrolled so that no set is
      // copied while its loads are in flight: tile i's ids were requested two
      // tiles earlier.  e4m3 pools run one step past the last tile (its widening).
      const int steps = FP8 ? n + 1 : n;
      int pgA[4], tkA[4], pgB[4], tkB[4], pgC[4], tkC[4];
      fetch(0, pgA, tkA);
      fetch(1, pgB, tkB);
      for (int i = 0; i < steps; i += 3) {
        fetch(i + 2, pgC, tkC);
        if (!step(i, pgA, tkA)) break;
        if (i + 1 >= steps) break;
        fetch(i + 3, pgA, tkA);
        if (!step(i + 1, pgB, tkB)) break;
        if (i + 2 >= steps) break;
        fetch(i + 4, pgB, tkB);
        if (!step(i + 2, pgC, tkC)) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lead && lane == 0 && n > 0) {
      constexpr uint32_t idesc_s = ptx::idesc_f16(BF, false, 2 * kRows, kKeys);
      constexpr uint32_t idesc_pv = ptx::idesc_f16(BF, true, 2 * kRows, kHeadDim);
      bool ok = wait_or_abort(bar(B_Q), 0, p.err, abort_flag);
      // O += P_hi V + P_lo V of tile t once both CTAs' softmax has written P
      // and seen its V tile land
      auto pv = [&](int t) -> bool {
        const int u = t % 3;
        const int sv = t % C::kVSt;
        if (!wait_or_abort_cluster(bar(B_PF + u), (t / 3) & 1, p.err, abort_flag)) return false;
        ptx::tc_fence_after();
        const uint32_t pcol = col_s(u);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t bdesc = ptx::smem_desc_sw128(base + C::kV + sv * C::kVStage + k * 2048, C::kVStage, 1024);
          ptx::umma_ts_pair(tmem + kColO, tmem + pcol + 16 * k, bdesc, idesc_pv, (t > 0 || k > 0) ? 1u : 0u);
          ptx::umma_ts_pair(tmem + kColO, tmem + pcol + 16 * k + 8, bdesc, idesc_pv, 1u);
        }
        ptx::tc_commit_pair(bar(B_OD + u), pair_mask);
        if (t + C::kVSt < n) ptx::tc_commit_pair(bar(B_VE + sv), pair_mask);
        return true;
      };
      // S = Q K^T of tile i into S buffer i mod 3 once the pair's K tile has
      // landed and the P V product of tile i - 3 (whose P the buffer holds) is
      // done; the P V product runs two tiles behind
      for (int i = 0; i < n && ok; ++i) {
        const int u = i % 3;
        const int sk = i % kKStages;
        if (!wait_or_abort_cluster(bar(B_KF + sk), (i / kKStages) & 1, p.err, abort_flag)) break;
        if (i >= 3 && !wait_or_abort(bar(B_OD + u), ((i - 3) / 3) & 1, p.err, abort_flag)) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t adesc =
              ptx::smem_desc_sw128(base + C::kQ + (k >> 2) * C::kQHalf + (k & 3) * 32, 16, 1024);
          const uint64_t bdesc =
              ptx::smem_desc_sw128(base + C::kK + sk * C::kKStage + (k >> 2) * C::kKHalf + (k & 3) * 32, 16, 1024);
          ptx::umma_ss_pair(tmem + col_s(u), adesc, bdesc, idesc_s, k > 0 ? 1u : 0u);
        }
        ptx::tc_commit_pair(bar(B_SF + u), pair_mask);
        if (i + kKStages < n) ptx::tc_commit_pair(bar(B_KE + sk), pair_mask);
        if (i >= 2 && !pv(i - 2)) {
          ok = false;
          break;
        }
      }
      if (ok && !*abort_flag && n >= 2) ok = pv(n - 2);
      if (ok && !*abort_flag) pv(n - 1);
      // drain: every MMA issued above has finished before TMEM is released
      ptx::tc_commit_pair_local(bar(B_DRAIN));
      ptx::mbar_wait(bar(B_DRAIN), 0, p.err);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ odd CTA: P-full relay
    // its softmax warps arrive on a local barrier; one cluster-scope arrival
    // per tile reaches the even CTA
    if (!lead && lane == 0) {
      for (int i = 0; i < n; ++i) {
        const int u = i % 3;
        if (!wait_or_abort(bar(B_PL + u), (i / 3) & 1, p.err, abort_flag)) break;
        ptx::mbar_arrive_cluster(ptx::mapa(bar(B_PF + u), leader));
      }
    }
  } else if (warp >= 4 && warp < 4 + kSoftmaxWarps) {
    // ------------------------------------------------------------ softmax
    const int wq = warp & 3;
    const int hf = (warp - 4) >> 2;  // keys [64 hf, 64 hf + 64) of each tile
    const int row = wq * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(wq * 32) << 16;
    const int bar_id = 1 + wq;  // the row's two halves
    float* xchg = reinterpret_cast<float*>(base_ptr + C::kXchg);  // [buffer][half][row]
    const float ksc = FP8 ? __ldg(p.k_scale + h) : 1.f;
    const float sl2 = p.scale_log2 * ksc;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    // this thread's query row: request b, qo head h * G + jj
    const int b = b0 + row / G;
    const int jj = row - (row / G) * G;
    const uint32_t scol_base = tmem + lanes + 64 * hf;
    const uint32_t ocol = tmem + lanes + kColO + 64 * hf;
    const int pf = lead ? B_PF : B_PL;  // where this CTA's "P written" arrivals go
    // this thread's 64 scores of a tile, loaded once; the next tile's load is
    // issued as soon as this tile's P is in TMEM
    uint32_t sr[64];
    if (n > 0) {
      ok = warp_wait(bar(B_SF), 0, p.err, abort_flag);
      if (ok) {
        ptx::tc_fence_after();
        ptx::tmem_ld32(scol_base, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        ptx::tmem_ld32(scol_base + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      }
    }
    // Each iteration passes the row's named barrier exactly once, also after a
    // failed wait (ok false: the rest of the work is skipped, and every later
    // wait returns at once on the abort flag), so the two halves never wait at
    // barriers the other does not reach.
    for (int i = 0; i < n; ++i) {
      const int u = i % 3;
      const uint32_t scol = scol_base + col_s(u);
      const int key0 = tile_of(i) * kKeys;
      const int nv = min(kKeys, kv_len - key0);
      const int vr = min(max(nv - 64 * hf, 0), 64);  // keys before the prefix end in this half
      // the maximum of the raw scores (the scale is positive, so it commutes
      // with max): 8 independent chains, then the other half's
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = -INFINITY;
      if (ok) {
        ptx::tmem_ld_wait();
        ptx::reg_fence32(&sr[0]);
        ptx::reg_fence32(&sr[32]);
        if (vr < 64) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e >= vr) sr[e] = __float_as_uint(-INFINITY);
        }
#pragma unroll
        for (int e = 0; e < 32; ++e)
          m8[e & 7] = ptx::fmax3(m8[e & 7], __uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]));
      }
      const float mh = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      // one barrier per tile: tile i uses buffer i % 2, and a half writes that
      // buffer again (tile i + 2) only after passing tile i + 1's barrier,
      // which its partner reaches after reading tile i's value
      float* xb = xchg + (i & 1) * 2 * kRows;
      xb[hf * kRows + row] = mh;
      ptx::named_bar_sync(bar_id, 64);
      const float mo = xb[(hf ^ 1) * kRows + row];
      if (!ok) continue;
      const float mx = sl2 * fmaxf(mh, mo);
      const bool need = (i > 0) && (mx > m_ref + kRescaleThreshold);
      if (i == 0) m_ref = mx;
      if (__any_sync(0xffffffffu, need)) {
        if (!warp_wait(bar(B_OD + (i - 1) % 3), ((i - 1) / 3) & 1, p.err, abort_flag)) {
          ok = false;
          continue;
        }
        ptx::tc_fence_after();
        const float alpha = need ? ptx::ex2(m_ref - mx) : 1.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(ocol + 32 * c, o);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          ptx::tmem_st32(ocol + 32 * c, o);
        }
        ptx::tmem_st_wait();
        if (need) {
          l *= alpha;
          m_ref = mx;
        }
      }
      // P over the scores, sixteen keys at a time: P_hi of the block's keys
      // in its first 8 columns, P_lo in the last 8; pairs of scores go through
      // the two-wide fp32 instructions (scale and shift, sums, residuals)
      const uint64_t sl2x2 = ptx::f2pack(sl2, sl2), negm = ptx::f2pack(-m_ref, -m_ref);
      uint64_t rs2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) rs2[e] = ptx::f2pack(0.f, 0.f);
#pragma unroll
      for (int bk = 0; bk < 4; bk += 2) {
        uint32_t pp[32];  // blocks bk, bk + 1: P_hi pairs, P_lo pairs, P_hi pairs, P_lo pairs
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint64_t x = ptx::f2fma(ptx::f2pack(__uint_as_float(sr[16 * bk + 2 * e]),
                                                    __uint_as_float(sr[16 * bk + 2 * e + 1])),
                                        sl2x2, negm);
          float x0, x1;
          ptx::f2unpack(x, x0, x1);
          const uint64_t pv = ptx::f2pack(ptx::ex2(x0), ptx::ex2(x1));
          rs2[e & 3] = ptx::f2add(rs2[e & 3], pv);
          const int slot = (e >> 3) * 16 + (e & 7);
          if constexpr (BF) {
            ptx::split2_bf16_packed(pv, pp[slot], pp[slot + 8]);
          } else {
            float q0, q1;
            ptx::f2unpack(pv, q0, q1);
            ptx::split2<false>(q0, q1, pp[slot], pp[slot + 8]);
          }
        }
        ptx::tmem_st32(scol + 16 * bk, pp);
      }
      {
        float a0, a1, b0s, b1s, c0, c1, d0, d1;
        ptx::f2unpack(rs2[0], a0, a1);
        ptx::f2unpack(rs2[1], b0s, b1s);
        ptx::f2unpack(rs2[2], c0, c1);
        ptx::f2unpack(rs2[3], d0, d1);
        l += ((a0 + a1) + (b0s + b1s)) + ((c0 + c1) + (d0 + d1));
      }
      // the next tile's scores (another S buffer) while this tile's tail runs
      if (i + 1 < n) {
        const int un = (i + 1) % 3;
        if (!warp_wait(bar(B_SF + un), ((i + 1) / 3) & 1, p.err, abort_flag)) {
          ok = false;
          continue;
        }
        ptx::tc_fence_after();
        ptx::tmem_ld32(scol_base + col_s(un), *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        ptx::tmem_ld32(scol_base + col_s(un) + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      }
      // this CTA's V tile must have landed before the pair's P V product; keys
      // past the prefix end have P = 0 and their V rows must be finite, so the
      // first half's threads zero them (16-bit pools; the widening warps do it
      // for e4m3 pools)
      const int sv = i % C::kVSt;
      if (!warp_wait(bar(B_VF + sv), (i / C::kVSt) & 1, p.err, abort_flag)) {
        ok = false;
        continue;
      }
      if (!FP8 && hf == 0 && row >= nv) {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        uint8_t* vrow_p = base_ptr + C::kV + sv * C::kVStage + row * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow_p + 16 * c) = z;
        ptx::fence_proxy_async_smem();
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(pf + u));
    }
    if (ok) ptx::tmem_ld_wait();  // no load is left in flight
    // ---- epilogue: o = O / l, lse2 = m_ref + log2(l) into piece `split` as
    // an fp32 partial state; each half writes its 64 columns, the first half
    // the lse
    const bool row_valid = row < used_rows && b < p.batch;
    const size_t orow = static_cast<size_t>(b) * Hq + h * G + jj;
    const size_t sidx = static_cast<size_t>(split) * p.rows_per_piece + orow;
    float* dst = p.pre_o + sidx * kHeadDim + 64 * hf;
    // the row sum is the two halves' partial sums (every thread arrives here,
    // also after a failed wait, so the barrier is always complete)
    float* xe = xchg + (n & 1) * 2 * kRows;  // the buffer a tile n would use
    xe[hf * kRows + row] = l;
    ptx::named_bar_sync(bar_id, 64);
    l += xe[(hf ^ 1) * kRows + row];
    if (n > 0 && ok && warp_wait(bar(B_OD + (n - 1) % 3), ((n - 1) / 3) & 1, p.err, abort_flag)) {
      ptx::tc_fence_after();
      const float inv = (FP8 ? __ldg(p.v_scale + h) : 1.f) / l;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(ocol + 32 * c, o);
        ptx::tmem_ld_wait();
        if (row_valid) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 v = make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                                         __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
            *reinterpret_cast<float4*>(dst + 32 * c + e) = v;
          }
        }
      }
      if (hf == 0 && row_valid) p.pre_lse[sidx] = m_ref + ptx::lg2(l);
    } else if (row_valid) {
      for (int d = 0; d < 64; d += 4) *reinterpret_cast<float4*>(dst + d) = make_float4(0.f, 0.f, 0.f, 0.f);
      if (hf == 0) p.pre_lse[sidx] = -INFINITY;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  // neither CTA leaves (or frees TMEM) while the pair's MMAs or loads may still
  // touch its shared memory or TMEM
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

template <bool BF, bool FP8>
void* kernel_ptr() {
  return reinterpret_cast<void*>(prefix_pair_kernel<BF, FP8>);
}

void* pick(int q_dtype, int kv_dtype) {
  const bool bf = q_dtype == kBF16;
  if (kv_dtype == kE4M3) return bf ? kernel_ptr<true, true>() : kernel_ptr<false, true>();
  return bf ? kernel_ptr<true, false>() : kernel_ptr<false, false>();
}

int smem_of(int kv_dtype) { return kv_dtype == kE4M3 ? PCfg<true>::kAlloc : PCfg<false>::kAlloc; }
int threads_of(int kv_dtype) { return kv_dtype == kE4M3 ? PCfg<true>::kThreads : PCfg<false>::kThreads; }

}  // namespace

int prefix_smem_bytes(int kv_dtype) { return smem_of(kv_dtype); }

int prefix_max_active_clusters(int q_dtype, int kv_dtype) {
  const void* kern = pick(q_dtype, kv_dtype);
  const int smem = smem_of(kv_dtype);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCluster);
  cfg.blockDim = dim3(threads_of(kv_dtype));
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int nclusters = 0;
  if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return nclusters;
}

cudaError_t launch_prefix(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                          const PrefixParams& p, int q_dtype, int kv_dtype, cudaStream_t stream, bool pdl) {
  const int grid = p.num_kv_heads * p.n_splits * p.m_groups * kCluster;
  if (grid <= 0) return cudaSuccess;
  if (!(q_dtype == kBF16 || q_dtype == kF16) || !(kv_dtype == q_dtype || kv_dtype == kE4M3))
    return cudaErrorInvalidValue;
  const void* kern = pick(q_dtype, kv_dtype);
  const int smem = smem_of(kv_dtype);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads_of(kv_dtype));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  void* args[] = {const_cast<CUtensorMap*>(&tmq), const_cast<CUtensorMap*>(&tmk), const_cast<CUtensorMap*>(&tmv),
                  const_cast<PrefixParams*>(&p)};
  e = cudaLaunchKernelExC(&cfg, kern, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pkd
