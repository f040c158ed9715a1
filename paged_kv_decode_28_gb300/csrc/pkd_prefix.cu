// pkd_prefix.cu -- shared-prefix attention (cascade level 0) on the sm_103a
// tensor cores (tcgen05 + TMEM).
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
// Per CTA (256 threads, one CTA per SM):
//   warp 0      TMA producer: the Q tile once, then K and V key tiles page by
//               page into two 3-stage rings (128-byte swizzled, K-major for K,
//               MN-major for V); a K slot is freed as soon as its S product is
//               done, a V slot when its P V product is done;
//   warp 1      allocates 512 TMEM columns and issues the MMAs from one thread:
//               S = Q K^T into one of two S buffers, then O += P V with P read
//               from TMEM; tcgen05.commit signals the mbarriers;
//   warps 4..7  softmax: thread r owns query row r (TMEM lane r), loads its 128
//               scores, keeps a running reference max (rescaling O in TMEM only
//               when the tile max exceeds it by more than 8 in log2 units, which
//               leaves the result exact), writes P as bf16/f16 into TMEM and
//               accumulates its row sum in a register.
// TMEM columns: S0 [0,128), S1 [128,256), O [256,384), P0 [384,448), P1 [448,512).
#include "pkd_internal.h"
#include "pkd_ptx.cuh"

namespace pkd {
namespace {

constexpr int kRows = 128;  // query rows per CTA
constexpr int kKeys = 128;  // keys per tile
constexpr int kThreads = 256;
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
  B_SF = B_VE + kStages,     // S full  [2]
  B_SFREE = B_SF + 2,        // S read  [2]
  B_PF = B_SFREE + 2,        // P full  [2]
  B_OD = B_PF + 2,           // P V done [2]
  B_DRAIN = B_OD + 2,
  kNumBars = B_DRAIN + 1
};
constexpr int kTmemSlot = kBars + kNumBars * 8;
constexpr int kAbort = kTmemSlot + 8;
constexpr int kTotal = kAbort + 16;
constexpr int kAlloc = kTotal + 1024;

constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP0 = 384, kColP1 = 448, kTmemCols = 512;

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
  const int per_head = p.m_tiles * p.n_splits;
  const int h = blockIdx.x / per_head;
  const int rem = blockIdx.x - h * per_head;
  const int mt = rem / p.n_splits;
  const int split = rem - mt * p.n_splits;
  const int n_tiles_all = (p.prefix_len + kKeys - 1) / kKeys;
  const int t0 = split * p.tiles_per_split;
  const int t1 = min(t0 + p.tiles_per_split, n_tiles_all);
  const int n = max(t1 - t0, 0);

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(B_Q), 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar(B_KF + s), 1);
      ptx::mbar_init(bar(B_KE + s), 1);
      ptx::mbar_init(bar(B_VF + s), 1);
      ptx::mbar_init(bar(B_VE + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(bar(B_SF + s), 1);
      ptx::mbar_init(bar(B_SFREE + s), kRows);
      ptx::mbar_init(bar(B_PF + s), kRows);
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
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base_ptr + kTmemSlot);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (n > 0) {
      if (lane == 0) {
        ptx::prefetch_tensormap(&tmq);
        ptx::prefetch_tensormap(&tmk);
        ptx::prefetch_tensormap(&tmv);
        ptx::mbar_arrive_expect_tx(bar(B_Q), 2u * kHalf);
        const int b0 = mt * (kRows / G);
        ptx::tma_load_4d(base + kQ, &tmq, bar(B_Q), 0, 0, h, b0);
        ptx::tma_load_4d(base + kQ + kHalf, &tmq, bar(B_Q), 64, 0, h, b0);
      }
      const uint64_t policy = ptx::policy_evict_last();  // the prefix is re-read by every query tile
      const int box = p.box_tok;
      for (int i = 0; i < n; ++i) {
        const int s = i % kStages;
        const uint32_t par = ((i / kStages) & 1) ^ 1;
        const int key0 = (t0 + i) * kKeys;
        const int nv = min(kKeys, p.prefix_len - key0);
        const int boxes = (nv + box - 1) / box;
        const uint32_t tile_bytes = static_cast<uint32_t>(boxes) * box * 128u * 2u;
        // page ids of this lane's boxes (at most 4 per lane: 128 keys / box >= 1 key)
        int pages[4], toks[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int bx = lane + 32 * r;
          pages[r] = 0;
          toks[r] = 0;
          if (bx < boxes) {
            const int key = key0 + bx * box;
            const int pi = key / p.page_size;
            int page = __ldg(p.prefix_pages + pi);
            if (static_cast<unsigned>(page) >= static_cast<unsigned>(p.num_pages)) {
              atomicOr(p.err, kDevErrPageIndex);
              page = 0;
            }
            pages[r] = page;
            toks[r] = key - pi * p.page_size;
          }
        }
        if (!warp_wait(bar(B_KE + s), par, p.err, abort_flag)) break;
        if (lane == 0) ptx::mbar_arrive_expect_tx(bar(B_KF + s), tile_bytes);
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int bx = lane + 32 * r;
          if (bx < boxes) {
            const uint32_t kd = base + kK + s * kStage + static_cast<uint32_t>(bx * box) * 128u;
            ptx::tma_load_4d_hint(kd, &tmk, bar(B_KF + s), 0, h, toks[r], pages[r], policy);
            ptx::tma_load_4d_hint(kd + kHalf, &tmk, bar(B_KF + s), 64, h, toks[r], pages[r], policy);
          }
        }
        if (!warp_wait(bar(B_VE + s), par, p.err, abort_flag)) break;
        if (lane == 0) ptx::mbar_arrive_expect_tx(bar(B_VF + s), tile_bytes);
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int bx = lane + 32 * r;
          if (bx < boxes) {
            const uint32_t vd = base + kV + s * kStage + static_cast<uint32_t>(bx * box) * 128u;
            ptx::tma_load_4d_hint(vd, &tmv, bar(B_VF + s), 0, h, toks[r], pages[r], policy);
            ptx::tma_load_4d_hint(vd + kHalf, &tmv, bar(B_VF + s), 64, h, toks[r], pages[r], policy);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_s = ptx::idesc_f16(BF, false, kRows, kKeys);
      constexpr uint32_t idesc_pv = ptx::idesc_f16(BF, true, kRows, kHeadDim);
      bool ok = wait_or_abort(bar(B_Q), 0, p.err, abort_flag);
      auto pv = [&](int t) -> bool {
        const int u = t & 1;
        const int sv = t % kStages;
        if (!wait_or_abort(bar(B_PF + u), (t >> 1) & 1, p.err, abort_flag)) return false;
        if (!wait_or_abort(bar(B_VF + sv), (t / kStages) & 1, p.err, abort_flag)) return false;
        ptx::tc_fence_after();
        const uint32_t pcol = u ? kColP1 : kColP0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t bdesc = ptx::smem_desc_sw128(base + kV + sv * kStage + k * 2048, kHalf, 1024);
          ptx::umma_ts(tmem + kColO, tmem + pcol + 8 * k, bdesc, idesc_pv, (t > 0 || k > 0) ? 1u : 0u);
        }
        ptx::tc_commit(bar(B_OD + u));
        ptx::tc_commit(bar(B_VE + sv));
        return true;
      };
      for (int i = 0; i < n && ok; ++i) {
        const int u = i & 1;
        const int sk = i % kStages;
        if (!wait_or_abort(bar(B_KF + sk), (i / kStages) & 1, p.err, abort_flag)) break;
        if (i >= 2 && !wait_or_abort(bar(B_SFREE + u), ((i - 2) >> 1) & 1, p.err, abort_flag)) break;
        ptx::tc_fence_after();
        const uint32_t scol = u ? kColS1 : kColS0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t koff = (k >> 2) * kHalf + (k & 3) * 32;
          const uint64_t adesc = ptx::smem_desc_sw128(base + kQ + koff, 16, 1024);
          const uint64_t bdesc = ptx::smem_desc_sw128(base + kK + sk * kStage + koff, 16, 1024);
          ptx::umma_ss(tmem + scol, adesc, bdesc, idesc_s, k > 0 ? 1u : 0u);
        }
        ptx::tc_commit(bar(B_SF + u));
        ptx::tc_commit(bar(B_KE + sk));
        if (i >= 1 && !pv(i - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && !*abort_flag) pv(n - 1);
      // drain: every MMA issued above has finished before TMEM is released
      ptx::tc_commit(bar(B_DRAIN));
      ptx::mbar_wait(bar(B_DRAIN), 0, p.err);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int u = i & 1;
      if (!warp_wait(bar(B_SF + u), (i >> 1) & 1, p.err, abort_flag)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t scol = tmem + lanes + (u ? kColS1 : kColS0);
      uint32_t sr[128];
      ptx::tmem_ld32(scol + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      ptx::tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      ptx::tmem_ld32(scol + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
      ptx::tmem_ld32(scol + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(B_SFREE + u));
      const int nv = min(kKeys, p.prefix_len - (t0 + i) * kKeys);
      // scale (and, on a ragged last tile, mask), then a tree max: 8 independent chains
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = -INFINITY;
      if (nv == kKeys) {
#pragma unroll
        for (int c = 0; c < kKeys; ++c) {
          const float x = __uint_as_float(sr[c]) * sl2;
          sr[c] = __float_as_uint(x);
          m8[c & 7] = fmaxf(m8[c & 7], x);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kKeys; ++c) {
          const float x = (c < nv) ? __uint_as_float(sr[c]) * sl2 : -INFINITY;
          sr[c] = __float_as_uint(x);
          m8[c & 7] = fmaxf(m8[c & 7], x);
        }
      }
      const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      const bool need = (i > 0) && (mx > m_ref + kRescaleThreshold);
      if (i == 0) m_ref = mx;
      if (__any_sync(0xffffffffu, need)) {
        if (!warp_wait(bar(B_OD + ((i - 1) & 1)), ((i - 1) >> 1) & 1, p.err, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const float alpha = need ? ptx::ex2(m_ref - mx) : 1.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(tmem + lanes + kColO + 32 * c, o);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          ptx::tmem_st32(tmem + lanes + kColO + 32 * c, o);
        }
        ptx::tmem_st_wait();
        if (need) {
          l *= alpha;
          m_ref = mx;
        }
      }
      // P buffer u was last read by the P V product of tile i - 2
      if (i >= 2 && !warp_wait(bar(B_OD + u), ((i - 2) >> 1) & 1, p.err, abort_flag)) {
        ok = false;
        break;
      }
      const uint32_t pcol = tmem + lanes + (u ? kColP1 : kColP0);
      float rs[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) rs[e] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ptx::ex2(__uint_as_float(sr[32 * c + 2 * e]) - m_ref);
          const float p1 = ptx::ex2(__uint_as_float(sr[32 * c + 2 * e + 1]) - m_ref);
          rs[e & 7] += p0 + p1;
          pk[e] = ptx::pack2<BF>(p0, p1);
        }
        ptx::tmem_st16(pcol + 16 * c, pk);
      }
      l += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
      if (nv < kKeys) {
        // keys past the prefix end: their P is 0, and their V rows must be
        // finite for the product, so zero them (both column halves) once the
        // tile's V has landed
        if (!warp_wait(bar(B_VF + i % kStages), (i / kStages) & 1, p.err, abort_flag)) {
          ok = false;
          break;
        }
      }
      if (nv < kKeys && row >= nv) {
        uint4 z = make_uint4(0u, 0u, 0u, 0u);
        uint8_t* vrow = base_ptr + kV + (i % kStages) * kStage + row * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(vrow + 16 * c) = z;
          *reinterpret_cast<uint4*>(vrow + kHalf + 16 * c) = z;
        }
        ptx::fence_proxy_async_smem();
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(B_PF + u));
    }
    // ---- epilogue: o = O / l, lse2 = m_ref + log2(l)
    const int grow = mt * kRows + row;
    const bool row_valid = grow < p.batch * G;
    float* dst = nullptr;
    size_t sidx = 0;
    if (row_valid) {
      const int b = grow / G;
      const int jj = grow - b * G;
      sidx = static_cast<size_t>(split) * p.batch * Hq + static_cast<size_t>(b) * Hq + h * G + jj;
      dst = p.pre_o + sidx * kHeadDim;
    }
    if (n > 0 && ok && warp_wait(bar(B_OD + ((n - 1) & 1)), ((n - 1) >> 1) & 1, p.err, abort_flag)) {
      ptx::tc_fence_after();
      const float inv = 1.f / l;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(tmem + lanes + kColO + 32 * c, o);
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
      if (row_valid) p.pre_lse[sidx] = m_ref + ptx::lg2(l);
    } else if (row_valid) {
      for (int d = 0; d < kHeadDim; d += 4) *reinterpret_cast<float4*>(dst + d) = make_float4(0.f, 0.f, 0.f, 0.f);
      p.pre_lse[sidx] = -INFINITY;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int prefix_smem_bytes() { return kAlloc; }

cudaError_t launch_prefix(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                          const PrefixParams& p, int kv_dtype, cudaStream_t stream) {
  const int grid = p.num_kv_heads * p.m_tiles * p.n_splits;
  if (grid <= 0) return cudaSuccess;
  if (kv_dtype == kBF16) {
    auto kern = prefix_kernel<true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, kAlloc, stream>>>(tmq, tmk, tmv, p);
  } else if (kv_dtype == kF16) {
    auto kern = prefix_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, kAlloc, stream>>>(tmq, tmk, tmv, p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace pkd
