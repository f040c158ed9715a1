// pkd_mla.cu -- multi-latent attention (MLA) decode over a paged latent cache,
// on the sm_103a tensor cores (tcgen05 + TMEM).
//
// The pages' other decode variant (deep dive, "Technical Moats": the latent KV
// of DeepSeek-V2/V3 attended without expanding it to full K and V; "The Code,
// Annotated" and "It In Action": kv_lora_rank 512, q_rope_dim 64, page 16,
// bf16, 128 query heads).  Every query head attends the same cached rows: per
// key a latent row ckv (512) and a rotary key kpe (64).  With the key
// up-projection already folded into the query (q_nope, 512) and the rotary
// query q_pe (64), s = sm_scale (<q_nope, ckv> + <q_pe, kpe>), and the output
// is the softmax-weighted sum of the ckv rows (512, still in the latent space).
//
// For one request the heads are the M dimension of dense products: S = Q K^T
// with Q [H <= 128 heads][576] and K the tile's rows [keys][576], then O += P V
// with V the tile's ckv rows.  O for 128 heads x 512 dims would fill all of
// TMEM, so a CTA owns one half of the 512 output dimensions (its unit's
// `level` field): the two halves of a request run as two CTAs that each form
// the whole S (the dot products need all 576 dimensions) and each accumulate
// P V for their 256 dimensions.
//
// Q is 144 KB for 128 heads; its first five 64-dim chunks stay in shared
// memory and the other four (latent dims 320..511 and the rotary part) go to
// TMEM, so that shared memory holds a 4-stage ring of key tiles and the loads
// run ahead of the MMAs.  S takes 36 single-thread MMA issues per tile, so it
// is issued by two threads into two accumulators that the softmax adds.
//
// The two CTAs of a key range form a cluster: each issues half of every
// tile's TMA boxes with multicast to both, and a stage is refilled once both
// have finished its P V product (their commits arrive on both CTAs' "empty"
// barriers).
//
// Per CTA (256 threads, one CTA per SM):
//   warp 0      TMA producer: Q chunks 0..4 once (64 dims x H heads each), then
//               its half of the boxes of key tiles of 32 keys (9 boxes of 64
//               dims x 32 keys per page, 36 KB a tile) into a 4-stage ring,
//               multicast to the pair;
//   warp 1      allocates 512 TMEM columns; one thread issues S_a = Q K^T over
//               chunks 0..2 (12 MMAs of N = 32, A from shared memory) into one
//               of two buffers and, one tile behind, O += P_hi V + P_lo V
//               (4 MMAs of N = 256);
//   warp 3      one thread issues S_b over chunks 3..8 (24 MMAs, A = Q from
//               shared memory for 3..4 and from TMEM for 5..8) into its own two
//               buffers, so the two threads issue about equal work;
//   warps 4..7  first write Q chunks 5..8 of their head row into TMEM, then the
//               softmax, thread r = head row r (TMEM lane r): S = S_a + S_b, a
//               running reference max with lazy rescaling of O, P written over
//               S_a's buffer as two 16-bit parts (P_hi = round(p), P_lo =
//               round(p - P_hi)), the row sum in a register.
// TMEM columns: O [0,256), S_a u [256 + 32u, 288 + 32u), S_b u [320 + 32u,
// 352 + 32u) for u = 0, 1, Q chunks 5..8 [384, 512) (two bf16 per column, K
// order).
#include "pkd_internal.h"
#include "pkd_ptx.cuh"

namespace pkd {
namespace {

constexpr int kMlaThreads = 256;
constexpr int kMlaRows = 128;      // head rows of the M dimension
constexpr int kMlaKeys = 32;       // keys per tile
constexpr int kChunks = 9;         // 64-dim chunks of a 576-dim row (8 latent + 1 rotary)
constexpr int kQBox = 16384;       // one chunk of Q: 128 rows x 128 bytes
constexpr int kKBox = 4096;        // one chunk of a key tile: 32 rows x 128 bytes
constexpr int kTile = kChunks * kKBox;
constexpr int kSplitA = 3;         // S chunks of the first issuer (it also issues P V); the rest are the second's
constexpr int kMlaStages = 4;
constexpr int kQSmem = 5;          // Q chunks in shared memory (the rest in TMEM)
constexpr int kMQ = 0;
constexpr int kMK = kMQ + kQSmem * kQBox;
constexpr int kMBars = kMK + kMlaStages * kTile;
enum {
  MB_Q = 0,
  MB_F = 1,                    // tile full  [kMlaStages]
  MB_E = MB_F + kMlaStages,     // tile empty [kMlaStages]
  MB_SF = MB_E + kMlaStages,    // S_a full [2]
  MB_SB = MB_SF + 2,            // S_b full [2]
  MB_PF = MB_SB + 2,            // P full (S_a and S_b read) [2]
  MB_OD = MB_PF + 2,            // P V done [2]
  MB_QT = MB_OD + 2,            // Q chunks in TMEM written
  MB_DRAIN = MB_QT + 1,
  MB_DRAINB = MB_DRAIN + 1,
  kMNumBars = MB_DRAINB + 1
};
constexpr int kMTmemSlot = kMBars + kMNumBars * 8;
constexpr int kMAbort = kMTmemSlot + 8;
constexpr int kMTotal = kMAbort + 16;
constexpr int kMAlloc = kMTotal + 1024;
static_assert(kMAlloc <= 227 * 1024, "dynamic shared memory above the 227 KB a CTA may use");
constexpr uint32_t kMColO = 0, kMColQ = 384, kMTmemCols = 512;
constexpr float kMRescale = 8.0f;
__device__ __forceinline__ uint32_t mcol_s(int u) { return 256u + 32u * static_cast<uint32_t>(u); }   // S_a u
__device__ __forceinline__ uint32_t mcol_sb(int u) { return 320u + 32u * static_cast<uint32_t>(u); }  // S_b u

__device__ __forceinline__ bool mwait(uint32_t bar, uint32_t parity, unsigned* err, volatile int* abort_flag) {
  if (*abort_flag) return false;
  if (ptx::mbar_wait(bar, parity, err)) return true;
  *abort_flag = 1;
  return false;
}

__device__ __forceinline__ bool mwarp_wait(uint32_t bar, uint32_t parity, unsigned* err, volatile int* abort_flag) {
  const bool r = mwait(bar, parity, err, abort_flag);
  return __all_sync(0xffffffffu, r);
}

__global__ void __launch_bounds__(kMlaThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap tq_nope, const __grid_constant__ CUtensorMap tq_pe,
               const __grid_constant__ CUtensorMap tckv, const __grid_constant__ CUtensorMap tkpe,
               const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + kMAbort);
  auto bar = [&](int i) { return base + kMBars + 8u * i; };
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = p.num_heads;

  // this CTA's unit: request b, output half hv, key tiles t0 .. t0 + n - 1
  const int4* wp = reinterpret_cast<const int4*>(p.work + blockIdx.x);
  const int4 wa = __ldg(wp), wb = __ldg(wp + 1);
  const int b = wa.x;
  const int page_begin = wa.z;
  const int kv_len = wa.w;
  const int t0 = wb.x;
  const int n = max(min(wb.y, (kv_len + kMlaKeys - 1) / kMlaKeys) - t0, 0);
  const int piece = wb.z;
  const int hv = wb.w;  // equals the cluster rank: the pair's units are adjacent, first half first
  const uint32_t rank = ptx::cluster_ctarank();
  constexpr uint16_t kPair = 0x3;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(MB_Q), 1);
    for (int s = 0; s < kMlaStages; ++s) {
      ptx::mbar_init(bar(MB_F + s), 1);
      ptx::mbar_init(bar(MB_E + s), 2);  // both CTAs' P V products of the tile
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(bar(MB_SF + s), 1);
      ptx::mbar_init(bar(MB_SB + s), 1);
      ptx::mbar_init(bar(MB_PF + s), kMlaRows);
      ptx::mbar_init(bar(MB_OD + s), 1);
    }
    ptx::mbar_init(bar(MB_QT), kMlaRows);
    ptx::mbar_init(bar(MB_DRAIN), 1);
    ptx::mbar_init(bar(MB_DRAINB), 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(base + kMTmemSlot, kMTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers exist before any multicast reaches them
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base_ptr + kMTmemSlot);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (n > 0) {
      if (lane == 0) {
        ptx::prefetch_tensormap(&tq_nope);
        ptx::prefetch_tensormap(&tq_pe);
        ptx::prefetch_tensormap(&tckv);
        ptx::prefetch_tensormap(&tkpe);
        ptx::mbar_arrive_expect_tx(bar(MB_Q), static_cast<uint32_t>(kQSmem) * H * 128u);
        for (int c = 0; c < kQSmem; ++c) ptx::tma_load_4d(base + kMQ + c * kQBox, &tq_nope, bar(MB_Q), 0, c, 0, b);
      }
      const int P = p.page_size;
      const int box = p.box_tok;  // keys per box: min(P, 32)
      for (int i = 0; i < n; ++i) {
        const int s = i % kMlaStages;
        const uint32_t par = ((i / kMlaStages) & 1) ^ 1;
        const int key0 = (t0 + i) * kMlaKeys;
        const int nv = min(kMlaKeys, kv_len - key0);
        const int boxes = (nv + box - 1) / box;
        if (!mwarp_wait(bar(MB_E + s), par, p.err, abort_flag)) break;
        if (lane == 0) ptx::mbar_arrive_expect_tx(bar(MB_F + s), static_cast<uint32_t>(boxes) * box * 128u * kChunks);
        __syncwarp();
        for (int j = lane; j < boxes; j += 32) {
          const int key = key0 + j * box;
          const int pi = key / P;
          int page = __ldg(p.page_indices + page_begin + pi);
          if (static_cast<unsigned>(page) >= static_cast<unsigned>(p.num_pages)) {
            atomicOr(p.err, kDevErrPageIndex);
            page = 0;
          }
          const int tok = key - pi * P;
          const uint32_t d = base + kMK + s * kTile + static_cast<uint32_t>(j * box) * 128u;
          // this CTA's half of the page's nine boxes, delivered to both CTAs
          for (int c = 0; c < 8; ++c)
            if (((c + j) & 1) == static_cast<int>(rank))
              ptx::tma_load_4d_mc(d + c * kKBox, &tckv, bar(MB_F + s), 0, c, tok, page, kPair);
          if (((8 + j) & 1) == static_cast<int>(rank))
            ptx::tma_load_4d_mc(d + 8 * kKBox, &tkpe, bar(MB_F + s), 0, tok, page, 0, kPair);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_s = ptx::idesc_f16(true, false, kMlaRows, kMlaKeys);
      constexpr uint32_t idesc_pv = ptx::idesc_f16(true, true, kMlaRows, 256);
      bool ok = mwait(bar(MB_Q), 0, p.err, abort_flag);
      auto pv = [&](int t) -> bool {
        const int u = t & 1;
        const int s = t % kMlaStages;
        if (!mwait(bar(MB_PF + u), (t >> 1) & 1, p.err, abort_flag)) return false;
        ptx::tc_fence_after();
        const uint32_t scol = mcol_s(u);
#pragma unroll
        for (int k = 0; k < kMlaKeys / 16; ++k) {
          // V = the tile's ckv chunks 4 hv .. 4 hv + 3 (this CTA's 256 dims), MN-major
          const uint64_t bdesc = ptx::smem_desc_sw128(base + kMK + s * kTile + 4 * hv * kKBox + k * 2048, kKBox, 1024);
          ptx::umma_ts(tmem + kMColO, tmem + scol + 8 * k, bdesc, idesc_pv, (t > 0 || k > 0) ? 1u : 0u);
          ptx::umma_ts(tmem + kMColO, tmem + scol + 16 + 8 * k, bdesc, idesc_pv, 1u);
        }
        ptx::tc_commit(bar(MB_OD + u));
        ptx::tc_commit_mc(bar(MB_E + s), kPair);  // both CTAs' stage s: this CTA is done with the tile
        return true;
      };
      for (int i = 0; i < n && ok; ++i) {
        const int u = i & 1;
        const int s = i % kMlaStages;
        if (!mwait(bar(MB_F + s), (i / kMlaStages) & 1, p.err, abort_flag)) break;
        // S_a u holds P of tile i - 2 until that tile's P V product is done
        // (issued by this thread in the previous iteration)
        if (i >= 2 && !mwait(bar(MB_OD + u), ((i - 2) >> 1) & 1, p.err, abort_flag)) break;
        ptx::tc_fence_after();
        // descriptors of the first chunk; a byte offset adds offset / 16 to
        // the start-address field (addresses stay below 256 KB)
        const uint64_t a0 = ptx::smem_desc_sw128(base + kMQ, 16, 1024);
        const uint64_t b0 = ptx::smem_desc_sw128(base + kMK + s * kTile, 16, 1024);
        const uint32_t dcol = tmem + mcol_s(u);
#pragma unroll
        for (int k = 0; k < kSplitA * 4; ++k) {
          const uint32_t c = static_cast<uint32_t>(k >> 2), sub = static_cast<uint32_t>(k & 3) * 32u;
          ptx::umma_ss(dcol, a0 + ((c * kQBox + sub) >> 4), b0 + ((c * kKBox + sub) >> 4), idesc_s, k > 0 ? 1u : 0u);
        }
        ptx::tc_commit(bar(MB_SF + u));
        if (i >= 1 && !pv(i - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && !*abort_flag) pv(n - 1);
      ptx::tc_commit(bar(MB_DRAIN));
      ptx::mbar_wait(bar(MB_DRAIN), 0, p.err);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ second S issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_s = ptx::idesc_f16(true, false, kMlaRows, kMlaKeys);
      bool ok = mwait(bar(MB_Q), 0, p.err, abort_flag) && mwait(bar(MB_QT), 0, p.err, abort_flag);
      for (int i = 0; i < n && ok; ++i) {
        const int u = i & 1;
        const int s = i % kMlaStages;
        if (!mwait(bar(MB_F + s), (i / kMlaStages) & 1, p.err, abort_flag)) break;
        // S_b u was read by the softmax of tile i - 2 (before its P arrived)
        if (i >= 2 && !mwait(bar(MB_PF + u), ((i - 2) >> 1) & 1, p.err, abort_flag)) break;
        ptx::tc_fence_after();
        const uint64_t a0 = ptx::smem_desc_sw128(base + kMQ, 16, 1024);
        const uint64_t b0 = ptx::smem_desc_sw128(base + kMK + s * kTile, 16, 1024);
        const uint32_t dcol = tmem + mcol_sb(u);
#pragma unroll
        for (int k = kSplitA * 4; k < kQSmem * 4; ++k) {  // A = Q from shared memory
          const uint32_t c = static_cast<uint32_t>(k >> 2), sub = static_cast<uint32_t>(k & 3) * 32u;
          ptx::umma_ss(dcol, a0 + ((c * kQBox + sub) >> 4), b0 + ((c * kKBox + sub) >> 4), idesc_s,
                       k > kSplitA * 4 ? 1u : 0u);
        }
#pragma unroll
        for (int k = kQSmem * 4; k < kChunks * 4; ++k) {  // A = Q from TMEM
          const uint32_t c = static_cast<uint32_t>(k >> 2), sub = static_cast<uint32_t>(k & 3);
          ptx::umma_ts(dcol, tmem + kMColQ + 32u * (c - kQSmem) + 8u * sub, b0 + ((c * kKBox + sub * 32u) >> 4),
                       idesc_s, 1u);
        }
        ptx::tc_commit(bar(MB_SB + u));
      }
      // every MMA this thread issued has finished before TMEM is released
      ptx::tc_commit(bar(MB_DRAINB));
      ptx::mbar_wait(bar(MB_DRAINB), 0, p.err);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    if (n > 0) {
      // Q chunks 4..8 of this head row into TMEM (zeros for rows past H)
      const uint4* qn = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q_nope) +
                                                       (static_cast<size_t>(b) * H + row) * 512 + 64 * kQSmem);
      const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q_pe) +
                                                       (static_cast<size_t>(b) * H + row) * 64);
#pragma unroll 1
      for (int c = 0; c < kChunks - kQSmem; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4 x = make_uint4(0u, 0u, 0u, 0u);
          if (row < H) x = __ldg(c < kChunks - kQSmem - 1 ? qn + 8 * c + q : qp + q);
          v[4 * q] = x.x;
          v[4 * q + 1] = x.y;
          v[4 * q + 2] = x.z;
          v[4 * q + 3] = x.w;
        }
        ptx::tmem_st32(tmem + lanes + kMColQ + 32 * c, v);
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(MB_QT));
    }
    for (int i = 0; i < n; ++i) {
      const int u = i & 1;
      if (!mwarp_wait(bar(MB_SF + u), (i >> 1) & 1, p.err, abort_flag) ||
          !mwarp_wait(bar(MB_SB + u), (i >> 1) & 1, p.err, abort_flag)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t scol = tmem + lanes + mcol_s(u);
      uint32_t sr[32], sb[32];
      ptx::tmem_ld32(scol, sr);
      ptx::tmem_ld32(tmem + lanes + mcol_sb(u), sb);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 32; ++c) sr[c] = __float_as_uint(__uint_as_float(sr[c]) + __uint_as_float(sb[c]));
      const int key0 = (t0 + i) * kMlaKeys;
      const int nv = min(kMlaKeys, kv_len - key0);
      if (nv < kMlaKeys) {
#pragma unroll
        for (int c = 0; c < kMlaKeys; ++c)
          if (c >= nv) sr[c] = __float_as_uint(-INFINITY);
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < kMlaKeys; ++c) m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(sr[c]));
      const float mx = sl2 * fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      const bool need = (i > 0) && (mx > m_ref + kMRescale);
      if (i == 0) m_ref = mx;
      if (__any_sync(0xffffffffu, need)) {
        // O holds the products of tiles up to i - 1
        if (!mwarp_wait(bar(MB_OD + ((i - 1) & 1)), ((i - 1) >> 1) & 1, p.err, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const float alpha = need ? ptx::ex2(m_ref - mx) : 1.f;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(tmem + lanes + kMColO + 32 * c, o);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          ptx::tmem_st32(tmem + lanes + kMColO + 32 * c, o);
        }
        ptx::tmem_st_wait();
        if (need) {
          l *= alpha;
          m_ref = mx;
        }
      }
      // P over S u: P_hi of keys 2c, 2c + 1 in column c, P_lo in column 16 + c
      uint32_t pk[16], pl[16];
      float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float p0 = ptx::ex2(fmaf(__uint_as_float(sr[2 * e]), sl2, -m_ref));
        const float p1 = ptx::ex2(fmaf(__uint_as_float(sr[2 * e + 1]), sl2, -m_ref));
        rs[e & 3] += p0 + p1;
        ptx::split2<true>(p0, p1, pk[e], pl[e]);
      }
      ptx::tmem_st16(scol, pk);
      ptx::tmem_st16(scol + 16, pl);
      l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
      if (nv < kMlaKeys && row < kMlaKeys && row >= nv) {
        // a key past the end: its P is 0, and its V row must be finite for
        // the product, so zero this CTA's four V chunks of it
        uint8_t* vrow = base_ptr + kMK + (i % kMlaStages) * kTile + 4 * hv * kKBox + row * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(vrow + c * kKBox + 16 * q) = make_uint4(0u, 0u, 0u, 0u);
        }
        ptx::fence_proxy_async_smem();
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(MB_PF + u));
    }
    // ---- epilogue: this CTA's 256 dims of o = O / l and lse, for heads < H
    const bool row_valid = row < H;
    const size_t orow = static_cast<size_t>(b) * H + row;
    if (n > 0 && ok && mwarp_wait(bar(MB_OD + ((n - 1) & 1)), ((n - 1) >> 1) & 1, p.err, abort_flag)) {
      ptx::tc_fence_after();
      const float inv = 1.f / l;
      const float lse2 = m_ref + ptx::lg2(l);
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(tmem + lanes + kMColO + 32 * c, o);
        ptx::tmem_ld_wait();
        if (!row_valid) continue;
        const int d0 = 256 * hv + 32 * c;
        if (piece >= 0) {
          float* dst = p.part_o + (static_cast<size_t>(piece) * H + row) * 512 + d0;
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + e) =
                make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                            __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
        } else {
          uint16_t* dst = static_cast<uint16_t*>(p.out) + orow * 512 + d0;
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 v;
            v.x = ptx::pack2<true>(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
            v.y = ptx::pack2<true>(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
            v.z = ptx::pack2<true>(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
            v.w = ptx::pack2<true>(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + e) = v;
          }
        }
      }
      if (row_valid && hv == 0) {
        if (piece >= 0) {
          p.part_lse[static_cast<size_t>(piece) * H + row] = lse2;
        } else if (p.lse) {
          p.lse[orow] = lse2 * 0.6931471805599453f;
        }
      }
    } else if (row_valid) {
      // no keys (or a failed wait): the empty state
      const int d0 = 256 * hv;
      if (piece >= 0) {
        float* dst = p.part_o + (static_cast<size_t>(piece) * H + row) * 512 + d0;
        for (int d = 0; d < 256; d += 4) *reinterpret_cast<float4*>(dst + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (hv == 0) p.part_lse[static_cast<size_t>(piece) * H + row] = -INFINITY;
      } else {
        uint16_t* dst = static_cast<uint16_t*>(p.out) + orow * 512 + d0;
        for (int d = 0; d < 256; d += 8) *reinterpret_cast<uint4*>(dst + d) = make_uint4(0u, 0u, 0u, 0u);
        if (hv == 0 && p.lse) p.lse[orow] = -INFINITY;
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  // no CTA leaves while its peer may still deliver into its shared memory or
  // arrive on its barriers
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kMTmemCols);
  }
}

// Merge of the split requests' pieces: one warp per (request, head), lane l
// owning dims 16 l .. 16 l + 15; pieces folded in order, out in bf16 and lse
// in natural log.  Requests with one piece were written by mla_kernel.
__global__ void __launch_bounds__(256) mla_merge_kernel(const MlaParams p) {
  const int gw = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int H = p.num_heads;
  if (gw >= p.batch * H) return;
  const int b = gw / H, h = gw - (gw / H) * H;
  const int beg = p.req_piece_begin[b], end = p.req_piece_begin[b + 1];
  if (end - beg <= 1) return;
  float m = -INFINITY;
  for (int j = beg; j < end; ++j) m = fmaxf(m, p.part_lse[static_cast<size_t>(j) * H + h]);
  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  float tot = 0.f;
  if (m != -INFINITY) {
    for (int j = beg; j < end; ++j) {
      const float s = p.part_lse[static_cast<size_t>(j) * H + h];
      const float w = (s == -INFINITY) ? 0.f : ptx::ex2(s - m);
      tot += w;
      const float4* src = reinterpret_cast<const float4*>(p.part_o + (static_cast<size_t>(j) * H + h) * 512 + 16 * lane);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = __ldcg(src + q);
        acc[4 * q] += w * v.x;
        acc[4 * q + 1] += w * v.y;
        acc[4 * q + 2] += w * v.z;
        acc[4 * q + 3] += w * v.w;
      }
    }
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  uint16_t* dst = static_cast<uint16_t*>(p.out) + (static_cast<size_t>(b) * H + h) * 512 + 16 * lane;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint4 v;
    v.x = ptx::pack2<true>(acc[8 * q] * inv, acc[8 * q + 1] * inv);
    v.y = ptx::pack2<true>(acc[8 * q + 2] * inv, acc[8 * q + 3] * inv);
    v.z = ptx::pack2<true>(acc[8 * q + 4] * inv, acc[8 * q + 5] * inv);
    v.w = ptx::pack2<true>(acc[8 * q + 6] * inv, acc[8 * q + 7] * inv);
    *reinterpret_cast<uint4*>(dst + 8 * q) = v;
  }
  if (lane == 0 && p.lse) p.lse[static_cast<size_t>(b) * H + h] = m == -INFINITY ? -INFINITY : (m + ptx::lg2(tot)) * 0.6931471805599453f;
}

}  // namespace

int mla_smem_bytes() { return kMAlloc; }

cudaError_t launch_mla(const CUtensorMap& tq_nope, const CUtensorMap& tq_pe, const CUtensorMap& tckv,
                       const CUtensorMap& tkpe, const MlaParams& p, cudaStream_t stream) {
  if (p.n_work <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_work);
  cfg.blockDim = dim3(kMlaThreads);
  cfg.dynamicSmemBytes = kMAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;  // the two output halves of a key range
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mla_kernel, tq_nope, tq_pe, tckv, tkpe, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || !p.any_split) return e;
  const int warps = p.batch * p.num_heads;
  mla_merge_kernel<<<(warps + 7) / 8, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pkd
