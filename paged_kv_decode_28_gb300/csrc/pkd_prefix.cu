// pkd_prefix.cu -- tile attention on the sm_103a tensor cores (tcgen05 +
// TMEM): a 128-row query tile of one kv head against a range of 128-key tiles
// of the shared prefix's page list.
//
// Cascade decode attends one shared prefix for every request and merges that
// state with each request's own (2026 guide, "Cascade attention for shared
// prefixes"; deep dive, "Why This Design Works": the shared prefix is read once
// but counted as if each request owns it).  For one kv head h the prefix part
// is a dense product: the B * g query rows of the group (row r = b * g + j is
// qo head h * g + j of request b) against the prefix keys.  One CTA takes a
// 128-row query tile and a contiguous range of 128-key tiles of the prefix and
// writes an fp32 partial state (o, base-2 lse) per row; the merge pass folds
// these partials into each request's suffix states.
//
// (The prefix tree's levels and paged prefill are work lists of query tiles in
// pairs, run by the paired-tile kernel of pkd_tile2.cu.)
//
// CTAs run in clusters of C (1, 2, 4 or 8): the C query tiles of one kv head
// and key range read the same K/V tiles, so each CTA fetches 1/C of every
// tile's TMA boxes and multicasts them to the whole cluster, and a K or V slot
// is reused only after all C CTAs have released it (their tcgen05.commit
// arrives on the slot's "empty" barrier in every CTA).
//
// Per CTA (384 threads, one CTA per SM):
//   warp 0      TMA producer of Q (once) and of the K ring; warp 2 producer of
//               the V ring: key tiles page by page into two 3-stage rings
//               (128-byte swizzled, K-major for K, MN-major for V); a K slot is
//               freed as soon as its S product is done, a V slot when its P V
//               product is done, so K loads run ahead of V;
//   warp 1      allocates 512 TMEM columns and issues the MMAs from one thread:
//               S = Q K^T into one of three S buffers (two tiles ahead of the
//               P V product), then O += P_hi V + P_lo V with both parts of P
//               read from TMEM; tcgen05.commit signals the mbarriers;
//   warps 4..11 softmax, two threads per query row: warps 4 + q and 8 + q
//               share TMEM lanes 32q .. 32q+31 (query rows), the first taking
//               keys 0..63 of each tile and the second keys 64..127.  The two
//               halves of a row swap their partial maxima through shared
//               memory, keep one running reference max (rescaling O in TMEM,
//               each its 64 columns, only when the tile max exceeds it by more
//               than 8 in log2 units, which leaves the result exact), write P
//               as two bf16/f16 parts (P_hi = round(P), P_lo = round(P - P_hi),
//               so P reaches the product to ~2^-17 instead of the 16-bit type's
//               2^-9 / 2^-11) into TMEM and keep partial row sums, added at the
//               end.
// TMEM columns: S0 [0,128), S1 [128,256), S2 [256,384), O [384,512).  Tile
// i uses S (i mod 3): once its scores are in registers, P_hi overwrites its
// columns [0,64) and P_lo [64,128), so S u is rewritten (for tile i + 3) only
// after the P V product of tile i is done.
#include "pkd_internal.h"
#include "pkd_ptx.cuh"

namespace pkd {
namespace {

constexpr int kRows = 128;  // query rows per CTA
constexpr int kKeys = 128;  // keys per tile
constexpr int kThreads = 384;
constexpr int kSoftmaxWarps = 8;
constexpr float kRescaleThreshold = 8.0f;

constexpr int kHalf = 16384;   // one 64-element (128-byte) column half of a 128-row tile
constexpr int kStage = 32768;  // a K (or V) tile: two halves
constexpr int kStages = 3;     // ring depth of K and of V
constexpr int kQ = 0;
constexpr int kK = kQ + kStage;
constexpr int kV = kK + kStages * kStage;
constexpr int kBars = kV + kStages * kStage;
enum {
  B_Q = 0,
  B_KF = 1,                  // K full  [kStages]
  B_KE = B_KF + kStages,     // K empty [kStages]
  B_VF = B_KE + kStages,     // V full  [kStages]
  B_VE = B_VF + kStages,     // V empty [kStages]
  B_SF = B_VE + kStages,     // S full  [3]
  B_PF = B_SF + 3,           // P full  [3]
  B_OD = B_PF + 3,           // P V done [3]
  B_DRAIN = B_OD + 3,
  kNumBars = B_DRAIN + 1
};
constexpr int kTmemSlot = kBars + kNumBars * 8;
constexpr int kAbort = kTmemSlot + 8;
constexpr int kXchg = kAbort + 16;  // fp32 [2 halves][128 rows]: the softmax halves' partial maxima / sums
constexpr int kTotal = kXchg + 4 * 2 * kRows;
constexpr int kAlloc = kTotal + 1024;
static_assert(kAlloc <= 227 * 1024, "dynamic shared memory above the 227 KB a CTA may use");

constexpr uint32_t kColO = 384, kTmemCols = 512;
__device__ __forceinline__ uint32_t col_s(int u) { return static_cast<uint32_t>(u) * 128u; }  // S buffer u

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, unsigned* err, volatile int* abort_flag) {
  if (*abort_flag) return false;
  if (ptx::mbar_wait(bar, parity, err)) return true;
  *abort_flag = 1;
  return false;
}

// The same, for a whole warp: every lane polls, and the result is made
// warp-uniform so that no lane leaves a loop that the others stay in.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, unsigned* err, volatile int* abort_flag) {
  const bool r = wait_or_abort(bar, parity, err, abort_flag);
  return __all_sync(0xffffffffu, r);
}

template <bool BF>
__global__ void __launch_bounds__(kThreads, 1)
    prefix_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const PrefixParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + kAbort);
  auto bar = [&](int i) { return base + kBars + 8u * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int Hq = p.num_kv_heads * G;
  const int C = p.cluster;
  const int rank = static_cast<int>(ptx::cluster_ctarank());
  const uint16_t cta_mask = static_cast<uint16_t>((1u << C) - 1u);
  // this CTA's unit: kv head h, query rows from request b0 (requests past
  // the batch are not written), prefix keys in tiles t0 .. t0+n-1, piece
  // `split`; blockIdx.x = ((h * n_splits + split) * m_groups + mgroup) * C + rank
  const int cl = blockIdx.x / C;
  const int mgroup = cl % p.m_groups;
  const int hs = cl / p.m_groups;
  const int split = hs % p.n_splits;
  const int h = hs / p.n_splits;
  const int mt = mgroup * C + rank;  // may pass m_tiles: such a CTA only helps load
  const int b0 = mt * (kRows / G);
  const int row_end = p.batch;
  const int kv_len = p.prefix_len;
  const int* pages = p.prefix_pages;
  const int n_tiles_all = (kv_len + kKeys - 1) / kKeys;
  const int t0 = split * p.tiles_per_split;
  const int n = max(min(t0 + p.tiles_per_split, n_tiles_all) - t0, 0);
  const int piece = split;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(B_Q), 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar(B_KF + s), 1);
      ptx::mbar_init(bar(B_KE + s), C);
      ptx::mbar_init(bar(B_VF + s), 1);
      ptx::mbar_init(bar(B_VE + s), C);
    }
    for (int s = 0; s < 3; ++s) {
      ptx::mbar_init(bar(B_SF + s), 1);
      ptx::mbar_init(bar(B_PF + s), kSoftmaxWarps * 32);
      ptx::mbar_init(bar(B_OD + s), 1);
    }
    ptx::mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(base + kTmemSlot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // every CTA's barriers exist before any multicast reaches them
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base_ptr + kTmemSlot);

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ TMA producers (K: warp 0, V: warp 2)
    const bool kside = warp == 0;
    if (n > 0) {
      if (kside && lane == 0) {
        ptx::prefetch_tensormap(&tmq);
        ptx::prefetch_tensormap(&tmk);
        ptx::prefetch_tensormap(&tmv);
        ptx::mbar_arrive_expect_tx(bar(B_Q), 2u * kHalf);
        ptx::tma_load_4d(base + kQ, &tmq, bar(B_Q), 0, 0, h, b0);
        ptx::tma_load_4d(base + kQ + kHalf, &tmq, bar(B_Q), 64, 0, h, b0);
      }
      const int box = p.box_tok;
      // this CTA's boxes of a tile are bx = rank + C * (lane + 32 * r); page ids
      // are fetched two tiles ahead of their use
      auto fetch = [&](int i, int (&pg)[4], int (&tk)[4]) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          pg[r] = 0;
          tk[r] = 0;
          if (i >= n) continue;
          const int key0 = (t0 + i) * kKeys;
          const int boxes = (min(kKeys, kv_len - key0) + box - 1) / box;
          const int bx = rank + C * (lane + 32 * r);
          if (bx < boxes) {
            const int key = key0 + bx * box;
            const int pi = key / p.page_size;
            pg[r] = __ldg(pages + pi);  // checked at use, so the load stays in flight
            tk[r] = key - pi * p.page_size;
          }
        }
      };
      const int eb = kside ? B_KE : B_VE;
      const int fb = kside ? B_KF : B_VF;
      const CUtensorMap* map = kside ? &tmk : &tmv;
      const uint32_t ring = kside ? kK : kV;
      auto issue = [&](int i, const int (&pg)[4], const int (&tk)[4]) -> bool {
        const int s = i % kStages;
        const uint32_t par = ((i / kStages) & 1) ^ 1;
        const int key0 = (t0 + i) * kKeys;
        const int boxes = (min(kKeys, kv_len - key0) + box - 1) / box;
        const uint32_t tile_bytes = static_cast<uint32_t>(boxes) * box * 128u * 2u;  // all CTAs' boxes
        if (!warp_wait(bar(eb + s), par, p.err, abort_flag)) return false;
        if (lane == 0) ptx::mbar_arrive_expect_tx(bar(fb + s), tile_bytes);
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int bx = rank + C * (lane + 32 * r);
          if (bx < boxes) {
            int page = pg[r];
            if (static_cast<unsigned>(page) >= static_cast<unsigned>(p.num_pages)) {
              atomicOr(p.err, kDevErrPageIndex);
              page = 0;
            }
            const uint32_t d = base + ring + s * kStage + static_cast<uint32_t>(bx * box) * 128u;
            // map coordinates (dim, head, key, page) for NHD pages, (dim, key, head, page) for HND
            const int c1 = p.kv_hnd ? tk[r] : h, c2 = p.kv_hnd ? h : tk[r];
            ptx::tma_load_4d_mc(d, map, bar(fb + s), 0, c1, c2, page, cta_mask);
            ptx::tma_load_4d_mc(d + kHalf, map, bar(fb + s), 64, c1, c2, page, cta_mask);
          }
        }
        return true;
      };
      // three register sets in rotation, unrolled so that no set is copied
      // while its loads are in flight: tile i's ids were requested two tiles earlier
      int pgA[4], tkA[4], pgB[4], tkB[4], pgC[4], tkC[4];
      fetch(0, pgA, tkA);
      fetch(1, pgB, tkB);
      for (int i = 0; i < n; i += 3) {
        fetch(i + 2, pgC, tkC);
        if (!issue(i, pgA, tkA)) break;
        if (i + 1 >= n) break;
        fetch(i + 3, pgA, tkA);
        if (!issue(i + 1, pgB, tkB)) break;
        if (i + 2 >= n) break;
        fetch(i + 4, pgB, tkB);
        if (!issue(i + 2, pgC, tkC)) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_s = ptx::idesc_f16(BF, false, kRows, kKeys);
      constexpr uint32_t idesc_pv = ptx::idesc_f16(BF, true, kRows, kHeadDim);
      bool ok = wait_or_abort(bar(B_Q), 0, p.err, abort_flag);
      auto pv = [&](int t) -> bool {
        const int u = t % 3;
        const int sv = t % kStages;
        if (!wait_or_abort(bar(B_PF + u), (t / 3) & 1, p.err, abort_flag)) return false;
        if (!wait_or_abort(bar(B_VF + sv), (t / kStages) & 1, p.err, abort_flag)) return false;
        ptx::tc_fence_after();
        const uint32_t pcol = col_s(u);       // P_hi
        const uint32_t lcol = col_s(u) + 64;  // P_lo
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t bdesc = ptx::smem_desc_sw128(base + kV + sv * kStage + k * 2048, kHalf, 1024);
          ptx::umma_ts(tmem + kColO, tmem + pcol + 8 * k, bdesc, idesc_pv, (t > 0 || k > 0) ? 1u : 0u);
          ptx::umma_ts(tmem + kColO, tmem + lcol + 8 * k, bdesc, idesc_pv, 1u);
        }
        ptx::tc_commit(bar(B_OD + u));
        if (t + kStages < n) ptx::tc_commit_mc(bar(B_VE + sv), cta_mask);
        return true;
      };
      for (int i = 0; i < n && ok; ++i) {
        const int u = i % 3;
        const int sk = i % kStages;
        if (!wait_or_abort(bar(B_KF + sk), (i / kStages) & 1, p.err, abort_flag)) break;
        // S u holds P of tile i - 3 until that tile's P V product is done
        // (issued by this thread in the previous iteration)
        if (i >= 3 && !wait_or_abort(bar(B_OD + u), ((i - 3) / 3) & 1, p.err, abort_flag)) break;
        ptx::tc_fence_after();
        const uint32_t scol = col_s(u);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t koff = (k >> 2) * kHalf + (k & 3) * 32;
          const uint64_t adesc = ptx::smem_desc_sw128(base + kQ + koff, 16, 1024);
          const uint64_t bdesc = ptx::smem_desc_sw128(base + kK + sk * kStage + koff, 16, 1024);
          ptx::umma_ss(tmem + scol, adesc, bdesc, idesc_s, k > 0 ? 1u : 0u);
        }
        ptx::tc_commit(bar(B_SF + u));
        if (i + kStages < n) ptx::tc_commit_mc(bar(B_KE + sk), cta_mask);
        // the P V product runs two tiles behind S
        if (i >= 2 && !pv(i - 2)) {
          ok = false;
          break;
        }
      }
      if (ok && !*abort_flag && n >= 2) ok = pv(n - 2);
      if (ok && !*abort_flag) pv(n - 1);
      // drain: every MMA issued above has finished before TMEM is released
      ptx::tc_commit(bar(B_DRAIN));
      ptx::mbar_wait(bar(B_DRAIN), 0, p.err);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int wq = warp & 3;
    const int hf = (warp - 4) >> 2;  // keys [64 hf, 64 hf + 64) of each tile
    const int row = wq * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(wq * 32) << 16;
    float* xchg = reinterpret_cast<float*>(base_ptr + kXchg);  // [half][row]
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    // this thread's query row: request tok, qo head h * G + jj
    const int tok = b0 + row / G;
    const int jj = row - (row / G) * G;
    // Each iteration passes the pair's named barrier exactly twice, also after
    // a failed wait (ok false: the rest of the work is skipped, and every later
    // wait returns at once on the abort flag), so the two halves never wait at
    // barriers the other does not reach.
    for (int i = 0; i < n; ++i) {
      const int u = i % 3;
      ok = ok && warp_wait(bar(B_SF + u), (i / 3) & 1, p.err, abort_flag);
      const uint32_t scol = tmem + lanes + col_s(u);
      uint32_t sr[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) sr[c] = __float_as_uint(-INFINITY);
      if (ok) {
        ptx::tc_fence_after();
        ptx::tmem_ld32(scol + 64 * hf, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        ptx::tmem_ld32(scol + 64 * hf + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        ptx::tmem_ld_wait();
      }
      const int key0 = (t0 + i) * kKeys;
      const int nv = min(kKeys, kv_len - key0);
      // the tile's keys before the prefix's end, counted within this thread's half
      const int vr = min(max(nv - 64 * hf, 0), 64);
      // mask, then a tree max of the raw scores (the scale is positive, so it
      // commutes with max): 8 independent chains, then the other half's
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = -INFINITY;
      if (vr < 64) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= vr) sr[c] = __float_as_uint(-INFINITY);
      }
#pragma unroll
      for (int c = 0; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], __uint_as_float(sr[c]));
      const float mh = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      xchg[hf * kRows + row] = mh;
      // both halves' scores are in registers past this barrier, so P may
      // overwrite any column of S u
      ptx::named_bar_sync(1 + wq, 64);
      const float mo = xchg[(hf ^ 1) * kRows + row];
      ptx::named_bar_sync(1 + wq, 64);  // both have read before the next tile writes
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
          ptx::tmem_ld32(tmem + lanes + kColO + 64 * hf + 32 * c, o);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          ptx::tmem_st32(tmem + lanes + kColO + 64 * hf + 32 * c, o);
        }
        ptx::tmem_st_wait();
        if (need) {
          l *= alpha;
          m_ref = mx;
        }
      }
      // P goes into S u itself: P_hi of keys 2c, 2c + 1 in column c, P_lo in
      // column 64 + c (this half: columns 32 hf .. 32 hf + 31 of each)
      const uint32_t pcol = scol + 32 * hf;
      const uint32_t lcol = scol + 64 + 32 * hf;
      float rs[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) rs[e] = 0.f;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[16], pl[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ptx::ex2(fmaf(__uint_as_float(sr[32 * c + 2 * e]), sl2, -m_ref));
          const float p1 = ptx::ex2(fmaf(__uint_as_float(sr[32 * c + 2 * e + 1]), sl2, -m_ref));
          rs[e & 7] += p0 + p1;
          ptx::split2<BF>(p0, p1, pk[e], pl[e]);
        }
        ptx::tmem_st16(pcol + 16 * c, pk);
        ptx::tmem_st16(lcol + 16 * c, pl);
      }
      l += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
      if (nv < kKeys) {
        // keys past the prefix's end: their P is 0, and their V rows must be
        // finite for the product, so zero them (each half one column half)
        // once the tile's V has landed
        if (!warp_wait(bar(B_VF + i % kStages), (i / kStages) & 1, p.err, abort_flag)) {
          ok = false;
          continue;
        }
      }
      if (nv < kKeys && row >= nv) {
        uint4 z = make_uint4(0u, 0u, 0u, 0u);
        uint8_t* vrow = base_ptr + kV + (i % kStages) * kStage + hf * kHalf + row * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + 16 * c) = z;
        ptx::fence_proxy_async_smem();
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(B_PF + u));
    }
    // ---- epilogue: o = O / l, lse2 = m_ref + log2(l) into piece `piece` as
    // an fp32 partial state; each half writes its 64 columns, the first half
    // the lse
    const bool row_valid = tok < row_end;
    const size_t orow = static_cast<size_t>(tok) * Hq + h * G + jj;
    const size_t sidx = static_cast<size_t>(piece) * p.rows_per_piece + orow;
    float* dst = p.pre_o + sidx * kHeadDim + 64 * hf;
    // the row sum is the two halves' partial sums (every thread arrives here,
    // also after a failed wait, so the barrier is always complete)
    xchg[hf * kRows + row] = l;
    ptx::named_bar_sync(1 + wq, 64);
    l += xchg[(hf ^ 1) * kRows + row];
    if (n > 0 && ok && warp_wait(bar(B_OD + (n - 1) % 3), ((n - 1) / 3) & 1, p.err, abort_flag)) {
      ptx::tc_fence_after();
      const float inv = 1.f / l;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(tmem + lanes + kColO + 64 * hf + 32 * c, o);
        ptx::tmem_ld_wait();
        if (row_valid) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            float4 v = make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
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
  // no CTA leaves while a peer may still deliver into its shared memory
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  // This grid is launched programmatically behind the decode grid and reads
  // nothing it writes; it does not finish before that grid has, so the merge
  // grid behind it, which waits for this one, sees the decode's partials too.
  if (threadIdx.x == 0) ptx::pdl_wait_prior_grid();
}

}  // namespace

int prefix_smem_bytes() { return kAlloc; }

int prefix_max_active_clusters(int cluster) {
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, PrefixParams) = prefix_kernel<true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kAlloc;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_prefix(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                          const PrefixParams& p, int kv_dtype, cudaStream_t stream, bool pdl) {
  const int grid = p.num_kv_heads * p.n_splits * p.m_groups * p.cluster;
  if (grid <= 0) return cudaSuccess;
  if (kv_dtype != kBF16 && kv_dtype != kF16) return cudaErrorInvalidValue;
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, PrefixParams) =
      kv_dtype == kBF16 ? prefix_kernel<true> : prefix_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kern, tmq, tmk, tmv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pkd
