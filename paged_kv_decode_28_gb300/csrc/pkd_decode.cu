// pkd_decode.cu -- split-KV paged decode attention for sm_103a.
//
// One persistent CTA per plan slot (the plan hands CTA c the contiguous run of
// work items cta_begin[c] .. cta_begin[c+1]).  Warp 4 is the producer: for every
// 64-key chunk of an item it reads the chunk's physical page ids from the CSR
// page table and issues TMA tensor loads (cp.async.bulk.tensor) of the K and V
// rows of those pages for the item's kv head into a ring of shared-memory
// stages, completing on an mbarrier (page-table gather of the deep dive's
// paged pool, "The Code, Annotated", snippet one).  Warps 0..3 are consumers:
// each owns 16 keys of every stage and keeps its own online-softmax state for
// all g query heads of the kv head (the GQA group is the M dimension of a
// warp-level tensor-core MMA, so every KV byte is read from HBM once).  At the
// end of an item the four states are combined in shared memory and written
// either as the final (out, lse) or, for a row split across CTAs, as an fp32
// partial state that the merge pass combines (merge_state of the 2026 guide,
// "Cascade attention for shared prefixes").
//
// Scores are fp32; the softmax runs in base 2 with sm_scale * log2(e) applied
// to the fp32 dot product; partial states carry a base-2 log-sum-exp.
#include "pkd_internal.h"
#include "pkd_ptx.cuh"

namespace pkd {
namespace {

constexpr int kConsumerWarps = 4;
// row stride (floats) of the shared buffer the consumer warps combine their
// states through: 8 floats of padding put the float2 accesses of a half-warp
// (4 head rows x 4 column pairs) on distinct banks
constexpr int kCombStride = kHeadDim + 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr float kLn2 = 0.693147180559945309f;
// a split row of at most this many items is merged with one round trip of loads
constexpr int kFewStates = 8;

template <int KVT>
struct Cfg {
  // bytes of one key (or value) row of one kv head
  static constexpr int kRowBytes = (KVT == kE4M3) ? kHeadDim : 2 * kHeadDim;
  // fp8: consumers hold two stages per step, so the ring runs three ahead
  static constexpr int kStages = (KVT == kE4M3) ? 5 : 3;
  static constexpr bool kMmaBf16 = (KVT == kBF16);
  // one 64-key tile of K (or V): 16-bit -> two [64][128 B] halves (d 0..63, 64..127)
  static constexpr int kTensorBytes = kChunkKeys * kRowBytes;
  static constexpr int kStageBytes = 2 * kTensorBytes;
  // fp8: each consumer warp's 16 value rows of a stage converted to f16,
  // [2 halves][16][128 B] per warp
  static constexpr int kV16Bytes = (KVT == kE4M3) ? 4 * 4096 : 0;
  static constexpr int kV16 = kStages * kStageBytes;
  static constexpr int kCombO = kV16 + kV16Bytes;                               // f32 [3][8][kCombStride]
  static constexpr int kCombML = kCombO + 3 * kMaxGroup * kCombStride * 4;      // f32 [3][8][2]
  static constexpr int kBars = kCombML + 3 * kMaxGroup * 2 * 4;                 // u64 [2][stages]
  static constexpr int kAbort = kBars + 2 * kStages * 8;                        // int
  static constexpr int kTotal = kAbort + 16;
  static constexpr int kAlloc = kTotal + 1024;  // slack for the 1024-byte alignment of stages
  // two CTAs per SM: 228 KB of shared memory, 1 KB of it reserved per CTA
  static_assert(kCtasPerSm * (kAlloc + 1024) <= 228 * 1024, "two CTAs per SM");
};

__device__ __forceinline__ int load_page(const DecodeParams& p, int idx) {
  int v = __ldg(p.page_indices + idx);
  if (static_cast<unsigned>(v) >= static_cast<unsigned>(p.num_pages)) {
    atomicOr(p.err, kDevErrPageIndex);
    v = 0;
  }
  return v;
}

// Bounded wait that also gives up at once when another warp already did.
__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t parity, unsigned* err,
                                           volatile int* abort_flag) {
  if (*abort_flag) return false;
  if (ptx::mbar_wait(bar, parity, err)) return true;
  *abort_flag = 1;
  return false;
}

// Query fragments (A operand rows = heads of the group, padded to 16 with zeros).
// 16-bit KV: k-step j covers d = 16j .. 16j+15 in natural order.
// fp8 KV:   k-step j, thread t covers d = 32t + 4j + {0,1} (a0) and {2,3} (a2):
//           the same permutation is applied to K, so the dot product is unchanged.
template <int QT, int KVT>
__device__ __forceinline__ void load_q(const DecodeParams& p, int b, int qo, bool hv, int t,
                                       uint32_t (&qa0)[8], uint32_t (&qa2)[8]) {
  const int Hq = p.num_kv_heads * p.group;
  const uint16_t* qrow = static_cast<const uint16_t*>(p.q) + (static_cast<size_t>(b) * Hq + qo) * kHeadDim;
  if constexpr (KVT != kE4M3) {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qrow);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      qa0[j] = hv ? __ldg(q32 + (16 * j + 2 * t) / 2) : 0u;
      qa2[j] = hv ? __ldg(q32 + (16 * j + 8 + 2 * t) / 2) : 0u;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (!hv) {
        qa0[j] = qa2[j] = 0u;
        continue;
      }
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(qrow + 32 * t + 4 * j));
      float f[4];
      const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint16_t bits = static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
        if constexpr (QT == kBF16) {
          f[e] = __uint_as_float(static_cast<uint32_t>(bits) << 16);
        } else {
          __half_raw hr;
          hr.x = bits;
          f[e] = __half2float(__half(hr));
        }
      }
      qa0[j] = ptx::pack2<false>(f[0], f[1]);
      qa2[j] = ptx::pack2<false>(f[2], f[3]);
    }
  }
}

// Scale the output accumulators (both the hi rows 0..7 and the lo rows 8..15)
// by the row's rescale factor; skipped when no row of the warp changed its max.
__device__ __forceinline__ void rescale_o(float (&o)[16][4], float alpha) {
  if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
      for (int i = 0; i < 4; ++i) o[nt][i] *= alpha;
    }
  }
}

// Online-softmax update for one 16-key sub-tile given the raw scores.
// x[] = (n-tile 0: keys 2t, 2t+1; n-tile 1: keys 8+2t, 9+2t) of head row gid.
// P leaves as hi/lo 16-bit pairs: the P V product puts hi in A rows 0..7
// (the group's heads) and lo in the otherwise empty rows 8..15, so the
// accumulator rows gid and gid + 8 sum to P V with P carried to ~2^-17.
template <bool PBF16>
__device__ __forceinline__ void softmax_step(const float (&sacc)[2][4], int t, int valid, float sl2,
                                             float& m_run, float& l_run, float (&o)[16][4],
                                             uint32_t& pa0, uint32_t& pa2, uint32_t& pl0, uint32_t& pl2) {
  float x[4];
  x[0] = (2 * t < valid) ? sacc[0][0] * sl2 : -INFINITY;
  x[1] = (2 * t + 1 < valid) ? sacc[0][1] * sl2 : -INFINITY;
  x[2] = (2 * t + 8 < valid) ? sacc[1][0] * sl2 : -INFINITY;
  x[3] = (2 * t + 9 < valid) ? sacc[1][1] * sl2 : -INFINITY;
  float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  // key 0 of the sub-tile is always valid, so m_new is finite
  const float m_new = fmaxf(m_run, mx);
  const float alpha = ptx::ex2(m_run - m_new);
  float pr[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) pr[i] = ptx::ex2(x[i] - m_new);
  l_run = l_run * alpha + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
  m_run = m_new;
  rescale_o(o, alpha);
  ptx::split2<PBF16>(pr[0], pr[1], pa0, pl0);
  ptx::split2<PBF16>(pr[2], pr[3], pa2, pl2);
}

// 16 keys of a 16-bit stage: S = Q K^T (ldmatrix), softmax, O += P V (ldmatrix.trans).
template <bool BF>
__device__ __forceinline__ void tile16_16bit(uint32_t kb, uint32_t vb, int w, int lane, int valid,
                                             const uint32_t (&qa0)[8], const uint32_t (&qa2)[8],
                                             float sl2, float& m_run, float& l_run,
                                             float (&o)[16][4]) {
  const int t = lane & 3;
  float sacc[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) sacc[nt][i] = 0.f;
#pragma unroll
  for (int kp = 0; kp < 4; ++kp) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint32_t tok = 16 * w + 8 * nt + (lane & 7);
      const uint32_t dch = 4 * kp + (lane >> 3);  // 16-byte chunk of the 256-byte row
      const uint32_t addr = kb + (dch >> 3) * (kChunkKeys * 128u) + ptx::sw128(tok, dch & 7u);
      uint32_t r0, r1, r2, r3;
      ptx::ldsm_x4(addr, r0, r1, r2, r3);
      ptx::mma_16816<BF>(sacc[nt], qa0[2 * kp], 0u, qa2[2 * kp], 0u, r0, r1);
      ptx::mma_16816<BF>(sacc[nt], qa0[2 * kp + 1], 0u, qa2[2 * kp + 1], 0u, r2, r3);
    }
  }
  uint32_t pa0, pa2, pl0, pl2;
  softmax_step<BF>(sacc, t, valid, sl2, m_run, l_run, o, pa0, pa2, pl0, pl2);
  // values of keys past the valid count are zeroed (their P is 0, but the
  // shared-memory rows may hold stale or non-finite bits)
  const uint32_t mlo = (2 * t < valid ? 0x0000ffffu : 0u) | (2 * t + 1 < valid ? 0xffff0000u : 0u);
  const uint32_t mhi = (2 * t + 8 < valid ? 0x0000ffffu : 0u) | (2 * t + 9 < valid ? 0xffff0000u : 0u);
#pragma unroll
  for (int dp = 0; dp < 8; ++dp) {
    const uint32_t tok = 16 * w + (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t dch = 2 * dp + (lane >> 4);
    const uint32_t addr = vb + (dch >> 3) * (kChunkKeys * 128u) + ptx::sw128(tok, dch & 7u);
    uint32_t r0, r1, r2, r3;
    ptx::ldsm_x4_trans(addr, r0, r1, r2, r3);
    r0 &= mlo;
    r1 &= mhi;
    r2 &= mlo;
    r3 &= mhi;
    ptx::mma_16816<BF>(o[2 * dp], pa0, pl0, pa2, pl2, r0, r1);
    ptx::mma_16816<BF>(o[2 * dp + 1], pa0, pl0, pa2, pl2, r2, r3);
  }
}

// Four E4M3 codes (bytes 0..3 of w) -> two f16x2 (lo: bytes 0,1; hi: bytes 2,3), exact.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Offset of 16-byte chunk c of row r, column half hf, in a [2 halves][16][128 B]
// f16 buffer: the chunk is XOR-swizzled by (r + 4 hf) mod 8, so both the
// row-wise writes (two halves at once) and the 8-row ldmatrix reads are free of
// bank conflicts.
__device__ __forceinline__ uint32_t v16_off(uint32_t r, uint32_t hf, uint32_t c) {
  return hf * (16 * 128u) + r * 128u + ((c ^ ((r + 4 * hf) & 7u)) << 4);
}

// The warp's 16 value rows of an fp8 stage -> f16.  Lane l converts row l / 2,
// head-dim half l % 2.
__device__ __forceinline__ void convert_v16(uint32_t vb, uint32_t v16, int w, int lane) {
  const uint32_t vr = lane >> 1, hf = lane & 1;
  const uint32_t tok = 16 * w + vr;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 raw = ptx::lds128(vb + ptx::sw128(tok, 4 * hf + c));  // codes d = 64 hf + 16 c ..
    uint32_t f[8];
    e4m3x4_to_f16x2x2(raw.x, f[0], f[1]);
    e4m3x4_to_f16x2x2(raw.y, f[2], f[3]);
    e4m3x4_to_f16x2x2(raw.z, f[4], f[5]);
    e4m3x4_to_f16x2x2(raw.w, f[6], f[7]);
    ptx::sts128(v16 + v16_off(vr, hf, 2 * c), f[0], f[1], f[2], f[3]);
    ptx::sts128(v16 + v16_off(vr, hf, 2 * c + 1), f[4], f[5], f[6], f[7]);
  }
}

// S = Q K^T for the warp's 16 keys of an fp8 stage (two n-tiles): the thread's
// 32 bytes of key row gid, converted e4m3x2 -> f16x2 in registers (head
// dimension permuted as in load_q).
__device__ __forceinline__ void qk_e4m3(uint32_t kb, int w, int lane, const uint32_t (&qa0)[8],
                                        const uint32_t (&qa2)[8], float (&sacc)[2][4]) {
  const int gid = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) sacc[nt][i] = 0.f;
    const uint32_t tok = 16 * w + 8 * nt + gid;
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {  // the row's 16-byte chunks 2t and 2t + 1, one at a time
      const uint4 c = ptx::lds128(kb + ptx::sw128(tok, 2 * t + hc));
      const uint32_t wd[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t b0, b1;
        e4m3x4_to_f16x2x2(wd[j], b0, b1);
        ptx::mma_16816<false>(sacc[nt], qa0[4 * hc + j], 0u, qa2[4 * hc + j], 0u, b0, b1);
      }
    }
  }
}

// O += P V for 16 keys whose values are f16 in a [2][16][128 B] buffer; keys
// past `valid` contribute zero whatever the buffer holds.  P as hi/lo pairs
// (A rows 0..7 and 8..15).
__device__ __forceinline__ void pv_f16buf(uint32_t v16, int lane, int valid, uint32_t pa0, uint32_t pa2,
                                          uint32_t pl0, uint32_t pl2, float (&o)[16][4]) {
  const int t = lane & 3;
  const uint32_t mlo = (2 * t < valid ? 0x0000ffffu : 0u) | (2 * t + 1 < valid ? 0xffff0000u : 0u);
  const uint32_t mhi = (2 * t + 8 < valid ? 0x0000ffffu : 0u) | (2 * t + 9 < valid ? 0xffff0000u : 0u);
#pragma unroll
  for (int dp = 0; dp < 8; ++dp) {
    const uint32_t tok = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t dch = 2 * dp + (lane >> 4);
    const uint32_t addr = v16 + v16_off(tok, dch >> 3, dch & 7u);
    uint32_t r0, r1, r2, r3;
    ptx::ldsm_x4_trans(addr, r0, r1, r2, r3);
    r0 &= mlo;
    r1 &= mhi;
    r2 &= mlo;
    r3 &= mhi;
    ptx::mma_16816<false>(o[2 * dp], pa0, pl0, pa2, pl2, r0, r1);
    ptx::mma_16816<false>(o[2 * dp + 1], pa0, pl0, pa2, pl2, r2, r3);
  }
}

// 16 keys of an fp8 stage.
__device__ __forceinline__ void tile16_e4m3(uint32_t kb, uint32_t vb, uint32_t v16, int w, int lane, int valid,
                                            const uint32_t (&qa0)[8], const uint32_t (&qa2)[8],
                                            float sl2, float& m_run, float& l_run,
                                            float (&o)[16][4]) {
  convert_v16(vb, v16, w, lane);
  float sacc[2][4];
  qk_e4m3(kb, w, lane, qa0, qa2, sacc);
  uint32_t pa0, pa2, pl0, pl2;
  softmax_step<false>(sacc, lane & 3, valid, sl2, m_run, l_run, o, pa0, pa2, pl0, pl2);
  __syncwarp();  // the f16 value rows are written by other lanes of this warp
  pv_f16buf(v16, lane, valid, pa0, pa2, pl0, pl2, o);
  __syncwarp();  // the buffer is rewritten by the next tile
}

// 32 keys: the warp's 16 keys of two consecutive fp8 stages (A, B).  The two
// S products are independent work for the scheduler, and the softmax state is
// updated once for the 32 keys; the values of A and then of B pass through
// the warp's one f16 buffer.
__device__ __forceinline__ void tile32_e4m3(uint32_t kbA, uint32_t vbA, int validA, uint32_t kbB, uint32_t vbB,
                                            int validB, uint32_t v16, int w, int lane,
                                            const uint32_t (&qa0)[8], const uint32_t (&qa2)[8], float sl2,
                                            float& m_run, float& l_run, float (&o)[16][4]) {
  const int t = lane & 3;
  convert_v16(vbA, v16, w, lane);
  // the scaled scores of A's and then B's keys (each S product's accumulators
  // are dead once its four scores of this thread's head row are taken)
  float x[8];
  {
    float sA[2][4];
    qk_e4m3(kbA, w, lane, qa0, qa2, sA);
    x[0] = (2 * t < validA) ? sA[0][0] * sl2 : -INFINITY;
    x[1] = (2 * t + 1 < validA) ? sA[0][1] * sl2 : -INFINITY;
    x[2] = (2 * t + 8 < validA) ? sA[1][0] * sl2 : -INFINITY;
    x[3] = (2 * t + 9 < validA) ? sA[1][1] * sl2 : -INFINITY;
  }
  {
    float sB[2][4];
    qk_e4m3(kbB, w, lane, qa0, qa2, sB);
    x[4] = (2 * t < validB) ? sB[0][0] * sl2 : -INFINITY;
    x[5] = (2 * t + 1 < validB) ? sB[0][1] * sl2 : -INFINITY;
    x[6] = (2 * t + 8 < validB) ? sB[1][0] * sl2 : -INFINITY;
    x[7] = (2 * t + 9 < validB) ? sB[1][1] * sl2 : -INFINITY;
  }
  float mx = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])), fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  // the caller guarantees a valid key in A or B, so m_new is finite
  const float m_new = fmaxf(m_run, mx);
  const float alpha = ptx::ex2(m_run - m_new);
  float pr[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) pr[i] = ptx::ex2(x[i] - m_new);
  l_run = l_run * alpha + (((pr[0] + pr[1]) + (pr[2] + pr[3])) + ((pr[4] + pr[5]) + (pr[6] + pr[7])));
  m_run = m_new;
  rescale_o(o, alpha);
  {
    uint32_t h0, h1, l0, l1;
    ptx::split2<false>(pr[0], pr[1], h0, l0);
    ptx::split2<false>(pr[2], pr[3], h1, l1);
    __syncwarp();  // the f16 value rows are written by other lanes of this warp
    pv_f16buf(v16, lane, validA, h0, h1, l0, l1, o);
  }
  __syncwarp();  // every lane has read A's rows
  convert_v16(vbB, v16, w, lane);
  {
    uint32_t h0, h1, l0, l1;
    ptx::split2<false>(pr[4], pr[5], h0, l0);
    ptx::split2<false>(pr[6], pr[7], h1, l1);
    __syncwarp();
    pv_f16buf(v16, lane, validB, h0, h1, l0, l1, o);
  }
  __syncwarp();  // the buffer is rewritten by the next step
}

// Head dimension index of accumulator o[nt][e] held by thread t.
template <int KVT>
__device__ __forceinline__ int o_dim(int nt, int e, int t) {
  return 8 * nt + 2 * t + e;
}

template <int QT>
__device__ __forceinline__ void store_out(void* out, size_t idx, float v) {
  if constexpr (QT == kBF16) {
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  } else {
    static_cast<__half*>(out)[idx] = __float2half_rn(v);
  }
}

template <int QT>
__device__ __forceinline__ void store_out4(void* out, size_t idx, float4 v) {
  uint2 u;
  u.x = ptx::pack2<QT == kBF16>(v.x, v.y);
  u.y = ptx::pack2<QT == kBF16>(v.z, v.w);
  *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + idx) = u;
}

// Merge of split row `row` for qo head j of its group by one warp (lane l: dims
// 4l..4l+3): its items' partial states (slots beg .. beg + cnt - 1) folded in
// slot order, out in q dtype and lse in natural log.  The partials were written
// by other CTAs; the caller has ordered them before these loads.
template <int QT>
__device__ __forceinline__ void merge_split_row(const DecodeParams& p, int row, int j, int lane) {
  const int Hk = p.num_kv_heads, G = p.group, Hq = Hk * G;
  const int b = row / Hk, h = row - b * Hk;
  const int beg = p.row_item_begin[row], cnt = p.row_item_count[row];
  auto lse_of = [&](int s) { return __ldcg(p.part_lse + static_cast<size_t>(beg + s) * G + j); };
  auto o_of = [&](int s) {
    return __ldcg(reinterpret_cast<const float4*>(p.part_o + (static_cast<size_t>(beg + s) * G + j) * kHeadDim) + lane);
  };
  float M = -INFINITY;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (cnt <= kFewStates) {
    // every state's lse and o requested at once: one memory round trip
    float4 ov[kFewStates];
#pragma unroll
    for (int s = 0; s < kFewStates; ++s) ov[s] = s < cnt ? o_of(s) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float x = lane < cnt ? lse_of(lane) : -INFINITY;
    M = x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M != -INFINITY) {
      const float wgt = (x == -INFINITY) ? 0.f : ptx::ex2(x - M);
      L = wgt;
#pragma unroll
      for (int s = 0; s < kFewStates; ++s) {
        const float w = __shfl_sync(0xffffffffu, wgt, s);
        if (s < cnt) {
          acc.x += w * ov[s].x;
          acc.y += w * ov[s].y;
          acc.z += w * ov[s].z;
          acc.w += w * ov[s].w;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
      const float inv = 1.f / L;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
    }
  } else {
    for (int s0 = 0; s0 < cnt; s0 += 32) M = fmaxf(M, (s0 + lane < cnt) ? lse_of(s0 + lane) : -INFINITY);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M != -INFINITY) {
      for (int s0 = 0; s0 < cnt; s0 += 32) {
        const int ns = min(32, cnt - s0);
        const float x = (lane < ns) ? lse_of(s0 + lane) : -INFINITY;
        const float wgt = (x == -INFINITY) ? 0.f : ptx::ex2(x - M);
        L += wgt;
        int s = 0;
        for (; s + 2 <= ns; s += 2) {
          const float w0 = __shfl_sync(0xffffffffu, wgt, s), w1 = __shfl_sync(0xffffffffu, wgt, s + 1);
          const float4 a = o_of(s0 + s), c = o_of(s0 + s + 1);
          acc.x += w0 * a.x + w1 * c.x;
          acc.y += w0 * a.y + w1 * c.y;
          acc.z += w0 * a.z + w1 * c.z;
          acc.w += w0 * a.w + w1 * c.w;
        }
        if (s < ns) {
          const float w0 = __shfl_sync(0xffffffffu, wgt, s);
          const float4 a = o_of(s0 + s);
          acc.x += w0 * a.x;
          acc.y += w0 * a.y;
          acc.z += w0 * a.z;
          acc.w += w0 * a.w;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
      const float inv = 1.f / L;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
    }
  }
  const size_t bq = static_cast<size_t>(b) * Hq + h * G + j;
  store_out4<QT>(p.out, bq * kHeadDim + 4 * lane, acc);
  if (lane == 0 && p.lse) p.lse[bq] = (M == -INFINITY) ? -INFINITY : (M + ptx::lg2(L)) * kLn2;
}

template <int QT, int KVT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeParams p) {
  using C = Cfg<KVT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t bar_full = base + C::kBars;
  const uint32_t bar_empty = bar_full + 8 * C::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::kAbort);
  float* comb_o = reinterpret_cast<float*>(base_ptr + C::kCombO);
  float* comb_ml = reinterpret_cast<float*>(base_ptr + C::kCombML);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(bar_full + 8 * s, 1);
      ptx::mbar_init(bar_empty + 8 * s, kConsumerWarps);
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();

  // This grid may have been launched before the schedule upload finished.  A
  // grid launched behind the cascade's prefix kernel is launched only once
  // every CTA of that kernel has waited for the upload, so the schedule and
  // the caller's inputs were complete before its launch; it reads nothing the
  // prefix kernel writes, and must not wait for that kernel to end: it waits
  // for it at its own end instead, so that the grid behind it finds both done.
  if (!p.behind_prefix) ptx::pdl_wait_prior_grid();
  // the next grid (the merge, or the prefix kernel of a prefix tree) may be
  // scheduled now: everything enqueued before this step is complete, so it may
  // read the step's inputs; it waits for this grid before reading its output
  ptx::pdl_launch_dependents();
  const int it0 = p.cta_begin[blockIdx.x];
  const int it1 = p.cta_begin[blockIdx.x + 1];
  const int Hk = p.num_kv_heads;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (p.debug_stall) return;  // test hook: no copy is issued, so the consumers' waits run out
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmk);
      ptx::prefetch_tensormap(&tmv);
    }
    const uint64_t policy = ptx::policy_evict_first();
    const uint32_t box_bytes = static_cast<uint32_t>(p.box_tok) * 128u;
    const uint32_t per_page = (C::kRowBytes == 256 ? 4u : 2u) * box_bytes;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
#pragma unroll 1
    for (int it = it0; it < it1 && ok; ++it) {
      const int4 item = p.items[it];
      const int b = item.x / Hk;
      const int h = item.x - b * Hk;
      const int L = p.kv_len[b];
      const int pb = p.page_begin[b];
#pragma unroll 1
      for (int k = item.y; k < item.z; ++k) {
        int npg, first, tok_off;
        if (p.pages_per_chunk > 0) {
          first = k * p.pages_per_chunk;
          const int row_pages = (L + p.page_size - 1) / p.page_size;
          npg = min(p.pages_per_chunk, row_pages - first);
          tok_off = 0;
        } else {
          npg = 1;
          first = (k * kChunkKeys) / p.page_size;
          tok_off = (k * kChunkKeys) - first * p.page_size;
        }
        int pid0 = 0, pid1 = 0;
        if (lane < npg) pid0 = load_page(p, pb + first + lane);
        if (lane + 32 < npg) pid1 = load_page(p, pb + first + lane + 32);
        if (!stage_wait(bar_empty + 8 * s, ph ^ 1u, p.err, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t fb = bar_full + 8 * s;
        if (lane == 0) ptx::mbar_arrive_expect_tx(fb, static_cast<uint32_t>(npg) * per_page);
        __syncwarp();
        const uint32_t kdst = base + s * C::kStageBytes;
        const uint32_t vdst = kdst + C::kTensorBytes;
        // tensor-map coordinates (dim, head, key, page) for NHD pages, (dim, key, head, page) for HND
        const int c1 = p.kv_hnd ? tok_off : h, c2 = p.kv_hnd ? h : tok_off;
#pragma unroll 1
        for (int j = lane; j < npg; j += 32) {
          const int pid = (j < 32) ? pid0 : pid1;
          const uint32_t off = static_cast<uint32_t>(j) * box_bytes;
          if constexpr (C::kRowBytes == 256) {
            constexpr uint32_t kHalf = kChunkKeys * 128u;
            ptx::tma_load_4d_hint(kdst + off, &tmk, fb, 0, c1, c2, pid, policy);
            ptx::tma_load_4d_hint(kdst + kHalf + off, &tmk, fb, 64, c1, c2, pid, policy);
            ptx::tma_load_4d_hint(vdst + off, &tmv, fb, 0, c1, c2, pid, policy);
            ptx::tma_load_4d_hint(vdst + kHalf + off, &tmv, fb, 64, c1, c2, pid, policy);
          } else {
            ptx::tma_load_4d_hint(kdst + off, &tmk, fb, 0, c1, c2, pid, policy);
            ptx::tma_load_4d_hint(vdst + off, &tmv, fb, 0, c1, c2, pid, policy);
          }
        }
        if (++s == C::kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int w = warp;
  const int gid = lane >> 2;
  const int t = lane & 3;
  const int G = p.group;
  const int Hq = Hk * G;
  volatile int* merge_flag = abort_flag + 1;
  if (p.fused_merge) {
    // rows without items: o = 0, lse = -inf (one warp per row, while the
    // producer fills the first stages)
    const int n_empty = p.header->n_empty_rows;
    for (int i = blockIdx.x * kConsumerWarps + w; i < n_empty; i += gridDim.x * kConsumerWarps) {
      const int row = p.empty_rows[i];
      const int b = row / Hk, h = row - b * Hk;
      for (int j = 0; j < G; ++j) {
        const size_t bq = static_cast<size_t>(b) * Hq + h * G + j;
        *(reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + bq * kHeadDim) + lane) = make_uint2(0u, 0u);
        if (lane == 0 && p.lse) p.lse[bq] = -INFINITY;
      }
    }
  }
  int s = 0;
  uint32_t ph = 0;
#pragma unroll 1
  for (int it = it0; it < it1; ++it) {
    const int4 item = p.items[it];
    const int b = item.x / Hk;
    const int h = item.x - b * Hk;
    const int L = p.kv_len[b];
    const bool hv = gid < G;
    const int qo = h * G + gid;
    uint32_t qa0[8], qa2[8];
    load_q<QT, KVT>(p, b, qo, hv, t, qa0, qa2);
    const float sl2 = p.scale_log2 * (p.k_scale ? __ldg(p.k_scale + h) : 1.f);
    float m_run = -INFINITY, l_run = 0.f;
    float o[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[nt][i] = 0.f;

#pragma unroll 1
    for (int k = item.y; k < item.z; ++k) {
      if constexpr (KVT == kE4M3) {
        if (k + 1 < item.z) {
          // two stages at once (32 keys per warp)
          const int s2 = (s + 1 == C::kStages) ? 0 : s + 1;
          const uint32_t ph2 = (s + 1 == C::kStages) ? (ph ^ 1u) : ph;
          const int validA = min(p.chunk_keys, L - k * p.chunk_keys) - 16 * w;
          const int validB = min(p.chunk_keys, L - (k + 1) * p.chunk_keys) - 16 * w;
          const bool okA = stage_wait(bar_full + 8 * s, ph, p.err, abort_flag);
          const bool okB = stage_wait(bar_full + 8 * s2, ph2, p.err, abort_flag);
          if (okA && okB && (validA > 0 || validB > 0)) {
            const uint32_t kbA = base + s * C::kStageBytes, kbB = base + s2 * C::kStageBytes;
            tile32_e4m3(kbA, kbA + C::kTensorBytes, validA, kbB, kbB + C::kTensorBytes, validB,
                        base + C::kV16 + w * 4096u, w, lane, qa0, qa2, sl2, m_run, l_run, o);
          }
          __syncwarp();
          if (lane == 0) {
            ptx::mbar_arrive(bar_empty + 8 * s);
            ptx::mbar_arrive(bar_empty + 8 * s2);
          }
          s = s2 + 1;
          ph = ph2;
          if (s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
          ++k;  // the loop's increment takes the second chunk
          continue;
        }
      }
      const int n_valid = min(p.chunk_keys, L - k * p.chunk_keys);
      const bool ok = stage_wait(bar_full + 8 * s, ph, p.err, abort_flag);
      const int valid = n_valid - 16 * w;
      if (ok && valid > 0) {
        const uint32_t kb = base + s * C::kStageBytes;
        const uint32_t vb = kb + C::kTensorBytes;
        if constexpr (KVT == kE4M3) {
          tile16_e4m3(kb, vb, base + C::kV16 + w * 4096u, w, lane, valid, qa0, qa2, sl2, m_run, l_run, o);
        } else {
          tile16_16bit<C::kMmaBf16>(kb, vb, w, lane, valid, qa0, qa2, sl2, m_run, l_run, o);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * s);
      if (++s == C::kStages) {
        s = 0;
        ph ^= 1u;
      }
    }

    // ---- combine the four warps' states and write
    // the lo rows (P's low parts) join the hi rows
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[nt][0] += o[nt][2];
      o[nt][1] += o[nt][3];
    }
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    ptx::named_bar_sync(1, kConsumerWarps * 32);
    if (w > 0 && hv) {
      float* dst = comb_o + ((w - 1) * kMaxGroup + gid) * kCombStride;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
        *reinterpret_cast<float2*>(dst + o_dim<KVT>(nt, 0, t)) = make_float2(o[nt][0], o[nt][1]);
      if (t == 0) {
        comb_ml[((w - 1) * kMaxGroup + gid) * 2 + 0] = m_run;
        comb_ml[((w - 1) * kMaxGroup + gid) * 2 + 1] = l_run;
      }
    }
    ptx::named_bar_sync(1, kConsumerWarps * 32);
    if (w == 0 && hv) {
      float mw[4], lw[4];
      mw[0] = m_run;
      lw[0] = l_run;
#pragma unroll
      for (int i = 1; i < 4; ++i) {
        mw[i] = comb_ml[((i - 1) * kMaxGroup + gid) * 2 + 0];
        lw[i] = comb_ml[((i - 1) * kMaxGroup + gid) * 2 + 1];
      }
      const float M = fmaxf(fmaxf(mw[0], mw[1]), fmaxf(mw[2], mw[3]));
      float sc[4];
      float Ls = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sc[i] = (mw[i] == -INFINITY) ? 0.f : ptx::ex2(mw[i] - M);
        Ls += lw[i] * sc[i];
      }
      const float inv = 1.f / Ls;
      const float vsc = p.v_scale ? __ldg(p.v_scale + h) : 1.f;
      const float lse2 = M + ptx::lg2(Ls);
      const bool partial = (item.w & kItemSplit) || p.force_partial;
      const float* c1 = comb_o + (0 * kMaxGroup + gid) * kCombStride;
      const float* c2 = comb_o + (1 * kMaxGroup + gid) * kCombStride;
      const float* c3 = comb_o + (2 * kMaxGroup + gid) * kCombStride;
      // this thread's two columns 8 nt + 2t, 8 nt + 2t + 1 of the combined row
      auto comb2 = [&](int nt) {
        const int d = o_dim<KVT>(nt, 0, t);
        const float2 a = *reinterpret_cast<const float2*>(c1 + d);
        const float2 bb = *reinterpret_cast<const float2*>(c2 + d);
        const float2 c = *reinterpret_cast<const float2*>(c3 + d);
        return make_float2((o[nt][0] * sc[0] + a.x * sc[1] + bb.x * sc[2] + c.x * sc[3]) * inv * vsc,
                           (o[nt][1] * sc[0] + a.y * sc[1] + bb.y * sc[2] + c.y * sc[3]) * inv * vsc);
      };
      if (partial) {
        float* po = p.part_o + (static_cast<size_t>(it) * G + gid) * kHeadDim;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) *reinterpret_cast<float2*>(po + o_dim<KVT>(nt, 0, t)) = comb2(nt);
        if (t == 0) p.part_lse[static_cast<size_t>(it) * G + gid] = lse2;
      } else {
        const size_t orow = (static_cast<size_t>(b) * Hq + qo) * kHeadDim;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          const float2 v = comb2(nt);
          *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + orow + o_dim<KVT>(nt, 0, t)) =
              ptx::pack2<QT == kBF16>(v.x, v.y);
        }
        if (t == 0 && p.lse) p.lse[static_cast<size_t>(b) * Hq + qo] = lse2 * kLn2;
      }
    }
    if (p.fused_merge && (item.w & kItemSplit)) {
      // Publish this item's partial state (the fence orders its stores before
      // the count); the item that completes the row merges it, its consumer
      // warps taking the row's qo heads in turn.
      if (w == 0) {
        __threadfence();
        __syncwarp();
        if (lane == 0) *merge_flag = (atomicAdd(p.row_done + item.x, 1) + 1 == p.row_item_count[item.x]) ? 1 : 0;
      }
      ptx::named_bar_sync(1, kConsumerWarps * 32);
      if (*merge_flag) {
        __threadfence();  // the other items' partial states are visible after the count
        for (int j = w; j < G; j += kConsumerWarps) merge_split_row<QT>(p, item.x, j, lane);
      }
    }
  }
  // see the top: the grid does not end before the prefix kernel ahead of it
  if (p.behind_prefix && threadIdx.x == 0) ptx::pdl_wait_prior_grid();
}

template <int QT, int KVT>
cudaError_t launch_t(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p, int grid,
                     cudaStream_t stream) {
  auto kern = decode_kernel<QT, KVT>;
  const int smem = Cfg<KVT>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the grid may start while the kernel before
  // it (the schedule upload) finishes; it waits in griddepcontrol.wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, tmk, tmv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int decode_smem_bytes(int kv_dtype) {
  return kv_dtype == kE4M3 ? Cfg<kE4M3>::kAlloc : Cfg<kBF16>::kAlloc;
}

cudaError_t launch_decode(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p,
                          int q_dtype, int kv_dtype, int grid, cudaStream_t stream) {
  if (q_dtype == kF16 && kv_dtype == kF16) return launch_t<kF16, kF16>(tmk, tmv, p, grid, stream);
  if (q_dtype == kBF16 && kv_dtype == kBF16) return launch_t<kBF16, kBF16>(tmk, tmv, p, grid, stream);
  if (q_dtype == kBF16 && kv_dtype == kE4M3) return launch_t<kBF16, kE4M3>(tmk, tmv, p, grid, stream);
  if (q_dtype == kF16 && kv_dtype == kE4M3) return launch_t<kF16, kE4M3>(tmk, tmv, p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkd
