// pkd_append.cu -- writing new tokens' keys and values into the paged cache.
//
// The step on either side of each decode step (README mirror, "Core Features":
// decode, prefill and append over a paged KV cache; deep dive, "The Code,
// Annotated", snippet one: request b owns pages indices[indptr[b]:indptr[b+1]],
// page_size slots each, NHD layout): token i of the new ones, of request
// batch_indices[i] at position positions[i], goes to page
// indices[indptr[b] + pos / page_size], slot pos % page_size, every kv head.
// 16-bit pools store the values as they are; e4m3 pools store
// e4m3(x / scale[h]), the quotient in fp32 (IEEE division), rounded to nearest
// even and saturated to +-448.
//
// One warp per token (the grid one wave of resident blocks, warps striding over
// the tokens): after one page lookup the warp moves the token's Hk * 256
// bytes of K and of V with independent 16-byte loads and stores (8-byte stores
// of codes for e4m3).  The token's rows are contiguous in the new-token tensor
// ([Hk, 128]); in an NHD page they are contiguous too ((slot * Hk + h) * 128),
// in an HND page ([Hk, P, 128]) head h's row sits at (h * P + slot) * 128.  A
// decode step's append is a few hundred KB, bound by launch latency; a bulk
// append is bound by HBM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "pkd_internal.h"
#include "pkd_ptx.cuh"

namespace pkd {
namespace {

constexpr int kAppendWarps = 8;
static_assert(kHeadDim == 128, "a head row is sixteen 16-byte chunks of 16-bit source");

// Two fp32 -> two E4M3 codes (round to nearest even, saturating): the low
// byte holds `lo`.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight 16-bit values (one uint4) -> fp32.
template <int NT>
__device__ __forceinline__ void unpack8(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 t;
    if constexpr (NT == kBF16) {
      t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
    } else {
      t = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
    }
    f[2 * k] = t.x;
    f[2 * k + 1] = t.y;
  }
}

// Eight values of head h -> eight E4M3 codes of x / scale (IEEE division).
__device__ __forceinline__ uint2 quantise8(const float (&f)[8], float scale) {
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) c[k] = e4m3x2(__fdiv_rn(f[2 * k], scale), __fdiv_rn(f[2 * k + 1], scale));
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

template <int NT, int KVT>
__global__ void __launch_bounds__(kAppendWarps * 32, 6) append_kv_kernel(const AppendParams p) {
  const int lane = threadIdx.x & 31;
  const int Hk = p.num_kv_heads;
  const int chunks = Hk * (kHeadDim / 8);  // 16-byte chunks of 16-bit source per token
  const int warps = gridDim.x * kAppendWarps;
#pragma unroll 1
  for (int i = blockIdx.x * kAppendWarps + (threadIdx.x >> 5); i < p.n_tokens; i += warps) {
    const int b = p.batch_indices[i];
    const int pos = p.positions[i];
    int page = -1;
    if (static_cast<unsigned>(b) < static_cast<unsigned>(p.batch) && pos >= 0) {
      const int beg = p.kv_indptr[b], end = p.kv_indptr[b + 1];
      const int pi = pos / p.page_size;
      if (pi < end - beg) {
        const int pg = p.page_indices[beg + pi];
        if (static_cast<unsigned>(pg) < static_cast<unsigned>(p.num_pages)) page = pg;
      }
    }
    if (page < 0) {  // outside the table or the pool: nothing is written
      if (lane == 0 && p.err) atomicOr(p.err, kDevErrPageIndex);
      continue;
    }
    const int slot = pos - (pos / p.page_size) * p.page_size;
    // element offsets of the token's first row (head 0) and of 16-byte chunk c
    // of its 16-bit source (eight elements, never straddling two heads)
    const size_t src = static_cast<size_t>(i) * Hk * kHeadDim;
    const size_t dst = static_cast<size_t>(page) * p.page_stride +
                       static_cast<size_t>(slot) * (p.kv_hnd ? kHeadDim : Hk * kHeadDim);
    // within the page: head h's row starts h * P * 128 (HND) or h * 128 (NHD)
    // elements after head 0's (a page holds under 2^31 elements)
    const uint32_t head_step = p.kv_hnd ? static_cast<uint32_t>(p.page_size) * kHeadDim : kHeadDim;
    auto chunk_off = [&](int c) -> uint32_t { return (c >> 4) * head_step + (c & 15) * 8; };
    const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.k_new) + src);
    const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.v_new) + src);
    if constexpr (KVT == kE4M3) {
      uint8_t* kd = static_cast<uint8_t*>(p.k_cache) + dst;
      uint8_t* vd = static_cast<uint8_t*>(p.v_cache) + dst;
      // two chunks in flight per lane and K, then V, quantised in turn: 40
      // registers (a few bytes of spill) for six blocks per SM, whose warps
      // hide the latency that the divisions leave exposed
#pragma unroll 2
      for (int c = lane; c < chunks; c += 32) {
        const int h = c >> 4;
        const uint4 ku = __ldg(ks + c), vu = __ldg(vs + c);
        const float ksc = __ldg(p.k_scale + h), vsc = __ldg(p.v_scale + h);
        const uint32_t o = chunk_off(c);
        {
          float f[8];
          unpack8<NT>(ku, f);
          *reinterpret_cast<uint2*>(kd + o) = quantise8(f, ksc);
        }
        {
          float f[8];
          unpack8<NT>(vu, f);
          *reinterpret_cast<uint2*>(vd + o) = quantise8(f, vsc);
        }
      }
    } else {
      uint16_t* kd = static_cast<uint16_t*>(p.k_cache) + dst;
      uint16_t* vd = static_cast<uint16_t*>(p.v_cache) + dst;
#pragma unroll 4
      for (int c = lane; c < chunks; c += 32) {
        const uint4 ku = __ldg(ks + c), vu = __ldg(vs + c);
        const uint32_t o = chunk_off(c);
        *reinterpret_cast<uint4*>(kd + o) = ku;
        *reinterpret_cast<uint4*>(vd + o) = vu;
      }
    }
  }
}

template <int NT, int KVT>
cudaError_t launch_t(const AppendParams& p, cudaStream_t stream) {
  // one wave of resident blocks (SM count x occupancy), warps striding over
  // the tokens: no block launches past the first wave
  // (queried once per device and instantiation; a failed query falls back
  // to a fixed grid)
  static std::atomic<int> cached[64];
  int64_t grid = (static_cast<int64_t>(p.n_tokens) + kAppendWarps - 1) / kAppendWarps;
  int64_t cap = 8192;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
    int c = cached[dev].load(std::memory_order_relaxed);
    if (c == 0) {
      int sms = 0, per_sm = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, append_kv_kernel<NT, KVT>, kAppendWarps * 32, 0) ==
              cudaSuccess &&
          sms > 0 && per_sm > 0) {
        c = sms * per_sm;
      } else {
        cudaGetLastError();
        c = -1;
      }
      cached[dev].store(c, std::memory_order_relaxed);
    }
    if (c > 0) cap = c;
  }
  grid = grid < 1 ? 1 : (grid > cap ? cap : grid);
  append_kv_kernel<NT, KVT><<<static_cast<int>(grid), kAppendWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append_kv(const AppendParams& p, int new_dtype, int kv_dtype, cudaStream_t stream) {
  if (p.n_tokens <= 0) return cudaSuccess;
  if (kv_dtype == kE4M3) {
    if (new_dtype == kBF16) return launch_t<kBF16, kE4M3>(p, stream);
    if (new_dtype == kF16) return launch_t<kF16, kE4M3>(p, stream);
    return cudaErrorInvalidValue;
  }
  if (new_dtype != kv_dtype) return cudaErrorInvalidValue;
  if (kv_dtype == kBF16) return launch_t<kBF16, kBF16>(p, stream);
  if (kv_dtype == kF16) return launch_t<kF16, kF16>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkd
