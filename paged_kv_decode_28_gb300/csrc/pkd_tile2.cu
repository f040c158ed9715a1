// pkd_tile2.cu -- paired-tile attention on the sm_103a tensor cores (tcgen05 +
// TMEM): two 128-row query tiles of one kv head against one stream of 128-key
// tiles of one page list.
//
// The units are work-list units (TileWork): the nodes of a prefix tree's
// shared levels (2026 guide, "Cascade attention for shared prefixes"; README
// mirror, "Core Features": hierarchical KV cache), each written as fp32
// partial states per key-range piece, and the query tiles of paged prefill
// (README mirror, "Core Features": prefill and append attention over a paged
// KV cache), causal to the end of the sequence and written as the final
// output.  The host lists them in pairs -- units 2j and 2j + 1 are two query
// tiles with the same keys -- and one CTA takes a pair for one kv head, so
// every K/V byte an SM receives serves 256 query rows instead of 128.  (An SM
// receives TMA data from L2 at a few tens of GB/s, which bounds a CTA that
// serves one tile; here the tensor pipe does twice the work per byte.)  A pair
// whose second tile has no rows (a node's lone last tile) skips that tile.
//
// Per CTA (640 threads, one CTA per SM):
//   warp 0      TMA of both Q tiles (once) and of the K ring; warp 2 the V
//               ring: two stages each, 128-byte swizzle, K-major K and
//               MN-major V, key tiles page by page as boxes of whole pages;
//   warp 1      allocates the 512 TMEM columns and issues every MMA from one
//               thread.  Each tile has one S buffer, rewritten only after the
//               tile's previous P V product is done; the issue order per key
//               tile i is P V(A, i), S(A, i + 1), P V(B, i), S(B, i + 1), so
//               the tensor pipe works on one tile while the other's softmax
//               runs;
//   warps 4..19 softmax: tile t = (warp - 4) / 8, key half hf =
//               ((warp - 4) / 4) % 2, TMEM lane quarter warp % 4; two threads
//               per query row, each reading its 64 scores of a tile from TMEM
//               once and keeping them in registers: first the row maximum
//               (swapped with the row's other half through shared memory),
//               then, sixteen keys at a time and two scores per two-wide fp32
//               instruction, P = 2^(s * scale_log2 - m), written as two 16-bit
//               parts (P_hi = round(P), P_lo = round(P - P_hi)) over the
//               columns read.  O is rescaled in TMEM only when the row
//               maximum grows by more than 8 in log2 units (exact either way).
// TMEM columns: O_A [0,128), O_B [128,256), S_A [256,384), S_B [384,512).
// P of a tile's keys 16k .. 16k + 15 (k = 0..7): P_hi of keys 16k + 2e and
// 16k + 2e + 1 in column 16k + e, P_lo in column 16k + 8 + e (e = 0..7).
#include "pkd_internal.h"
#include "pkd_ptx.cuh"

namespace pkd {
namespace {

constexpr int kRows = 128;  // query rows per tile
constexpr int kKeys = 128;  // keys per key tile
constexpr int kThreads = 640;
constexpr float kRescaleThreshold = 8.0f;

constexpr int kHalf = 16384;   // one 64-element (128-byte) column half of a 128-row tile
constexpr int kStage = 32768;  // a Q, K or V tile: two halves
constexpr int kStages = 2;     // ring depth of K and of V
constexpr int kQA = 0;
constexpr int kQB = kQA + kStage;
constexpr int kK = kQB + kStage;
constexpr int kV = kK + kStages * kStage;
constexpr int kBars = kV + kStages * kStage;
enum {
  B_Q = 0,
  B_KF = 1,               // K full  [kStages]
  B_KE = B_KF + kStages,  // K empty [kStages]
  B_VF = B_KE + kStages,  // V full  [kStages]
  B_VE = B_VF + kStages,  // V empty [kStages]
  B_SF = B_VE + kStages,  // S full  [tile]
  B_PF = B_SF + 2,        // P full  [tile]
  B_OD = B_PF + 2,        // P V done [tile]
  B_DRAIN = B_OD + 2,
  kNumBars = B_DRAIN + 1
};
constexpr int kTmemSlot = kBars + kNumBars * 8;
constexpr int kAbort = kTmemSlot + 8;
constexpr int kXchg = kAbort + 16;  // fp32 [buffer][tile][half][row]: the halves' partial maxima / sums
constexpr int kTotal = kXchg + 4 * 2 * 2 * 2 * kRows;
constexpr int kAlloc = kTotal + 1024;
static_assert(kAlloc <= 227 * 1024, "dynamic shared memory above the 227 KB a CTA may use");

constexpr uint32_t kTmemCols = 512;

// 32 lanes x 16 consecutive 32-bit columns -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
}

// Registers just written by tcgen05.ld, redefined after tcgen05.wait::ld so
// that no use of them is scheduled before the wait.
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
#pragma unroll
  for (int i = 0; i < 16; i += 8)
    asm volatile("" : "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]),
                 "+r"(r[i + 6]), "+r"(r[i + 7]));
}
__device__ __forceinline__ uint32_t col_o(int t) { return static_cast<uint32_t>(t) * 128u; }
__device__ __forceinline__ uint32_t col_s(int t) { return 256u + static_cast<uint32_t>(t) * 128u; }

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
    tile2_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
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
  const int Hk = p.num_kv_heads;
  const int Hq = Hk * G;
  // blockIdx.x = pair * Hk + h: the list's pairs in list order, the kv heads
  // of a pair side by side
  const int h = static_cast<int>(blockIdx.x % static_cast<unsigned>(Hk));
  const int pair = static_cast<int>(blockIdx.x / static_cast<unsigned>(Hk));
  const int4* wp = reinterpret_cast<const int4*>(p.work + 2 * pair);
  const int4 wa = __ldg(wp), wb = __ldg(wp + 1), wc = __ldg(wp + 2);
  const int4 xa = __ldg(wp + 3);  // the second unit's query range
  // both tiles: keys of `pages` (kv_len of them) in tiles t0 .. t0 + n - 1,
  // output piece (or -1: final output), causal offset; tile A's rows start at
  // token (or request) b0A, tile B's at b0B, rows at or past the end are not written
  const int b0A = wa.x, endA = wa.y, b0B = xa.x, endB = xa.y;
  const bool hasB = b0B < endB;
  const int kv_len = wa.w;
  const int lv = wb.w;
  const int* pages = (lv == 0 ? p.level_pages[0] : lv == 1 ? p.level_pages[1] : lv == 2 ? p.level_pages[2]
                                                                                      : p.level_pages[3]) + wa.z;
  const int t0 = wb.x;
  const int n = max(min(wb.y, (kv_len + kKeys - 1) / kKeys) - t0, 0);
  const int piece = wb.z;
  const int diag = wc.x;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(B_Q), 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar(B_KF + s), 1);
      ptx::mbar_init(bar(B_KE + s), 1);
      ptx::mbar_init(bar(B_VF + s), 1);
      ptx::mbar_init(bar(B_VE + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(bar(B_SF + t), 1);
      ptx::mbar_init(bar(B_PF + t), 8 * 32);
      ptx::mbar_init(bar(B_OD + t), 1);
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
        ptx::mbar_arrive_expect_tx(bar(B_Q), (hasB ? 4u : 2u) * kHalf);
        ptx::tma_load_4d(base + kQA, &tmq, bar(B_Q), 0, 0, h, b0A);
        ptx::tma_load_4d(base + kQA + kHalf, &tmq, bar(B_Q), 64, 0, h, b0A);
        if (hasB) {
          ptx::tma_load_4d(base + kQB, &tmq, bar(B_Q), 0, 0, h, b0B);
          ptx::tma_load_4d(base + kQB + kHalf, &tmq, bar(B_Q), 64, 0, h, b0B);
        }
      }
      const int box = p.box_tok;
      // the boxes of a tile are bx = lane + 32 * r; page ids are fetched two
      // tiles ahead of their use
      auto fetch = [&](int i, int (&pg)[4], int (&tk)[4]) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          pg[r] = 0;
          tk[r] = 0;
          if (i >= n) continue;
          const int key0 = (t0 + i) * kKeys;
          const int boxes = (min(kKeys, kv_len - key0) + box - 1) / box;
          const int bx = lane + 32 * r;
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
        const uint32_t tile_bytes = static_cast<uint32_t>(boxes) * box * 128u * 2u;
        if (!warp_wait(bar(eb + s), par, p.err, abort_flag)) return false;
        if (lane == 0) ptx::mbar_arrive_expect_tx(bar(fb + s), tile_bytes);
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int bx = lane + 32 * r;
          if (bx < boxes) {
            int page = pg[r];
            if (static_cast<unsigned>(page) >= static_cast<unsigned>(p.num_pages)) {
              atomicOr(p.err, kDevErrPageIndex);
              page = 0;
            }
            const uint32_t d = base + ring + s * kStage + static_cast<uint32_t>(bx * box) * 128u;
            // map coordinates (dim, head, key, page) for NHD pages, (dim, key, head, page) for HND
            const int c1 = p.kv_hnd ? tk[r] : h, c2 = p.kv_hnd ? h : tk[r];
            ptx::tma_load_4d(d, map, bar(fb + s), 0, c1, c2, page);
            ptx::tma_load_4d(d + kHalf, map, bar(fb + s), 64, c1, c2, page);
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
      // S_t = Q_t K_i^T into tile t's S buffer
      auto s_mma = [&](int t, int i) {
        const int sk = i % kStages;
        const uint32_t q = base + (t ? kQB : kQA);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t koff = (k >> 2) * kHalf + (k & 3) * 32;
          const uint64_t adesc = ptx::smem_desc_sw128(q + koff, 16, 1024);
          const uint64_t bdesc = ptx::smem_desc_sw128(base + kK + sk * kStage + koff, 16, 1024);
          ptx::umma_ss(tmem + col_s(t), adesc, bdesc, idesc_s, k > 0 ? 1u : 0u);
        }
        ptx::tc_commit(bar(B_SF + t));
      };
      // O_t += P_hi V_i + P_lo V_i, sixteen keys per product
      auto pv_mma = [&](int t, int i) {
        const int sv = i % kStages;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t bdesc = ptx::smem_desc_sw128(base + kV + sv * kStage + k * 2048, kHalf, 1024);
          const uint32_t pc = col_s(t) + 16u * k;
          ptx::umma_ts(tmem + col_o(t), tmem + pc, bdesc, idesc_pv, (i > 0 || k > 0) ? 1u : 0u);
          ptx::umma_ts(tmem + col_o(t), tmem + pc + 8, bdesc, idesc_pv, 1u);
        }
        ptx::tc_commit(bar(B_OD + t));
      };
      bool ok = wait_or_abort(bar(B_Q), 0, p.err, abort_flag) && wait_or_abort(bar(B_KF), 0, p.err, abort_flag);
      if (ok) {
        ptx::tc_fence_after();
        s_mma(0, 0);
        if (hasB) s_mma(1, 0);
        if (kStages < n) ptx::tc_commit(bar(B_KE));
      }
      for (int i = 0; i < n && ok; ++i) {
        const int sv = i % kStages;
        const bool next = i + 1 < n;
        const int sk = (i + 1) % kStages;
        ok = wait_or_abort(bar(B_PF + 0), i & 1, p.err, abort_flag) &&
             wait_or_abort(bar(B_VF + sv), (i / kStages) & 1, p.err, abort_flag);
        if (!ok) break;
        ptx::tc_fence_after();
        pv_mma(0, i);
        if (next) {
          // S_A is free once the P V product just issued has read P_A
          ok = wait_or_abort(bar(B_KF + sk), ((i + 1) / kStages) & 1, p.err, abort_flag) &&
               wait_or_abort(bar(B_OD + 0), i & 1, p.err, abort_flag);
          if (!ok) break;
          ptx::tc_fence_after();
          s_mma(0, i + 1);
        }
        if (hasB) {
          ok = wait_or_abort(bar(B_PF + 1), i & 1, p.err, abort_flag);
          if (!ok) break;
          ptx::tc_fence_after();
          pv_mma(1, i);
        }
        if (i + kStages < n) ptx::tc_commit(bar(B_VE + sv));
        if (next) {
          if (hasB) {
            ok = wait_or_abort(bar(B_OD + 1), i & 1, p.err, abort_flag);
            if (!ok) break;
            ptx::tc_fence_after();
            s_mma(1, i + 1);
          }
          if (i + 1 + kStages < n) ptx::tc_commit(bar(B_KE + sk));
        }
      }
      // drain: every MMA issued above has finished before TMEM is released
      ptx::tc_commit(bar(B_DRAIN));
      ptx::mbar_wait(bar(B_DRAIN), 0, p.err);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 3;
    const int hf = ((warp - 4) >> 2) & 1;  // keys [64 hf, 64 hf + 64) of each key tile
    const int wq = warp & 3;
    if (t == 0 || hasB) {
      const int row = wq * 32 + lane;
      const uint32_t lanes = static_cast<uint32_t>(wq * 32) << 16;
      const int bar_id = 1 + t * 4 + wq;  // the row's two halves
      float* xchg = reinterpret_cast<float*>(base_ptr + kXchg) + t * 2 * kRows;  // [buffer][tile][half][row]
      const float sl2 = p.scale_log2;
      const int b0 = t ? b0B : b0A;
      const int row_end = t ? endB : endA;
      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      // this thread's query row: token (or request) tok, qo head h * G + jj
      const int tok = b0 + row / G;
      const int jj = row - (row / G) * G;
      const uint32_t scol = tmem + lanes + col_s(t) + 64 * hf;  // this half's 64 columns
      const uint32_t ocol = tmem + lanes + col_o(t) + 64 * hf;
      // Each iteration passes the row's named barrier exactly twice, also after
      // a failed wait (ok false: the rest of the work is skipped, and every later
      // wait returns at once on the abort flag), so the two halves never wait at
      // barriers the other does not reach.
      for (int i = 0; i < n; ++i) {
        ok = ok && warp_wait(bar(B_SF + t), i & 1, p.err, abort_flag);
        const int key0 = (t0 + i) * kKeys;
        const int nv = min(kKeys, kv_len - key0);
        // keys this row sees: those before the list's end and, for a causal
        // unit, at or before the row's position tok + diag (units that mask
        // start at key 0, so every row of theirs sees key 0 in its first tile);
        // vr counts them within this thread's half
        const int vrow = diag == kNoCausal ? nv : max(0, min(nv, tok + diag + 1 - key0));
        const int vr = min(max(vrow - 64 * hf, 0), 64);
        // the maximum of the raw scores (the scale is positive, so it commutes
        // with max): 4 independent chains of three-way maxima, then the other half's
        float m4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) m4[e] = -INFINITY;
        uint32_t sr[64];  // this half's 64 scores, both chunks in one round trip, kept for P
        if (ok) {
          ptx::tc_fence_after();
          ptx::tmem_ld32(scol, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
          ptx::tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
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
            m4[e & 3] = ptx::fmax3(m4[e & 3], __uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]));
        }
        const float mh = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        // one barrier per tile: tile i uses buffer i % 2, and a half writes
        // that buffer again (tile i + 2) only after passing tile i + 1's
        // barrier, which its partner reaches after reading tile i's value
        float* xb = xchg + (i & 1) * 4 * kRows;
        xb[hf * kRows + row] = mh;
        ptx::named_bar_sync(bar_id, 64);
        const float mo = xb[(hf ^ 1) * kRows + row];
        if (!ok) continue;
        const float mx = sl2 * fmaxf(mh, mo);
        const bool need = (i > 0) && (mx > m_ref + kRescaleThreshold);
        if (i == 0) m_ref = mx;
        if (__any_sync(0xffffffffu, need)) {
          if (!warp_wait(bar(B_OD + t), (i - 1) & 1, p.err, abort_flag)) {
            ok = false;
            continue;
          }
          ptx::tc_fence_after();
          const float alpha = need ? ptx::ex2(m_ref - mx) : 1.f;
          // sixteen columns at a time: the scores stay in registers meanwhile
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[16];
            tmem_ld16(ocol + 16 * c, o);
            ptx::tmem_ld_wait();
            reg_fence16(o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            ptx::tmem_st16(ocol + 16 * c, o);
          }
          ptx::tmem_st_wait();
          if (need) {
            l *= alpha;
            m_ref = mx;
          }
        }
        // P over the scores, sixteen keys at a time: P_hi of the block's keys
        // in its first 8 columns, P_lo in the last 8; pairs of scores go
        // through the two-wide fp32 instructions (scale and shift, sums,
        // residuals)
        const uint64_t sl2x2 = ptx::f2pack(sl2, sl2), negm = ptx::f2pack(-m_ref, -m_ref);
        uint64_t rs2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) rs2[e] = ptx::f2pack(0.f, 0.f);
#pragma unroll
        for (int bk = 0; bk < 4; ++bk) {
          uint32_t pp[16];  // P_hi pairs, then P_lo pairs
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint64_t x = ptx::f2fma(ptx::f2pack(__uint_as_float(sr[16 * bk + 2 * e]),
                                                      __uint_as_float(sr[16 * bk + 2 * e + 1])),
                                          sl2x2, negm);
            float x0, x1;
            ptx::f2unpack(x, x0, x1);
            const uint64_t pv = ptx::f2pack(ptx::ex2(x0), ptx::ex2(x1));
            rs2[e & 1] = ptx::f2add(rs2[e & 1], pv);
            if constexpr (BF) {
              ptx::split2_bf16_packed(pv, pp[e], pp[8 + e]);
            } else {
              float q0, q1;
              ptx::f2unpack(pv, q0, q1);
              ptx::split2<false>(q0, q1, pp[e], pp[8 + e]);
            }
          }
          ptx::tmem_st16(scol + 16 * bk, pp);
        }
        {
          float a0, a1, b0s, b1s;
          ptx::f2unpack(rs2[0], a0, a1);
          ptx::f2unpack(rs2[1], b0s, b1s);
          l += (a0 + a1) + (b0s + b1s);
        }
        if (t == 0 && nv < kKeys) {
          // keys past the list's end: their P is 0, and their V rows must be
          // finite for both tiles' products, so tile A's threads zero them
          // (each half one column half) once the tile's V has landed; tile B's
          // product is issued after tile A's, which waits for this
          if (!warp_wait(bar(B_VF + i % kStages), (i / kStages) & 1, p.err, abort_flag)) {
            ok = false;
            continue;
          }
          if (row >= nv) {
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            uint8_t* vrow_p = base_ptr + kV + (i % kStages) * kStage + hf * kHalf + row * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow_p + 16 * c) = z;
            ptx::fence_proxy_async_smem();
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(B_PF + t));
      }
      // ---- epilogue: o = O / l, lse2 = m_ref + log2(l); into piece `piece`
      // as an fp32 partial state, or (piece < 0) as the final out / lse; each
      // half writes its 64 columns, the first half the lse
      const bool row_valid = tok < row_end;
      const size_t orow = static_cast<size_t>(tok) * Hq + h * G + jj;
      const size_t sidx = static_cast<size_t>(piece < 0 ? 0 : piece) * p.rows_per_piece + orow;
      float* dst = p.pre_o + sidx * kHeadDim + 64 * hf;
      uint16_t* fdst = static_cast<uint16_t*>(p.out) + orow * kHeadDim + 64 * hf;
      // the row sum is the two halves' partial sums (every thread arrives here,
      // also after a failed wait, so the barrier is always complete)
      float* xe = xchg + (n & 1) * 4 * kRows;  // the buffer a tile n would use
      xe[hf * kRows + row] = l;
      ptx::named_bar_sync(bar_id, 64);
      l += xe[(hf ^ 1) * kRows + row];
      if (n > 0 && ok && warp_wait(bar(B_OD + t), (n - 1) & 1, p.err, abort_flag)) {
        ptx::tc_fence_after();
        const float inv = 1.f / l;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(ocol + 32 * c, o);
          ptx::tmem_ld_wait();
          if (row_valid && piece >= 0) {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              float4 v = make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                                     __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
              *reinterpret_cast<float4*>(dst + 32 * c + e) = v;
            }
          } else if (row_valid) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 v;
              v.x = ptx::pack2<BF>(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
              v.y = ptx::pack2<BF>(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
              v.z = ptx::pack2<BF>(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
              v.w = ptx::pack2<BF>(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
              *reinterpret_cast<uint4*>(fdst + 32 * c + e) = v;
            }
          }
        }
        if (hf == 0 && row_valid && piece >= 0) p.pre_lse[sidx] = m_ref + ptx::lg2(l);
        if (hf == 0 && row_valid && piece < 0 && p.lse) p.lse[orow] = (m_ref + ptx::lg2(l)) * 0.6931471805599453f;
      } else if (row_valid && piece >= 0) {
        for (int d = 0; d < 64; d += 4) *reinterpret_cast<float4*>(dst + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (hf == 0) p.pre_lse[sidx] = -INFINITY;
      } else if (row_valid) {
        for (int d = 0; d < 64; d += 8) *reinterpret_cast<uint4*>(fdst + d) = make_uint4(0u, 0u, 0u, 0u);
        if (hf == 0 && p.lse) p.lse[orow] = -INFINITY;
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  // Launched programmatically behind the decode grid (prefix tree), this grid
  // reads nothing that grid writes; it does not finish before that grid has,
  // so the merge grid behind it, which waits for this one, sees the decode's
  // partials too.
  if (threadIdx.x == 0) ptx::pdl_wait_prior_grid();
}

}  // namespace

cudaError_t launch_tile2(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                         const PrefixParams& p, int kv_dtype, cudaStream_t stream, bool pdl) {
  if (p.work == nullptr || (p.n_work & 1) != 0) return cudaErrorInvalidValue;
  const int64_t grid = static_cast<int64_t>(p.num_kv_heads) * (p.n_work / 2);
  if (grid <= 0) return cudaSuccess;
  if (grid > INT32_MAX) return cudaErrorInvalidValue;
  if (kv_dtype != kBF16 && kv_dtype != kF16) return cudaErrorInvalidValue;
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, PrefixParams) =
      kv_dtype == kBF16 ? tile2_kernel<true> : tile2_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, tmq, tmk, tmv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int tile2_smem_bytes() { return kAlloc; }

}  // namespace pkd
