// pkd_merge.cu -- attention-state merges for sm_103a.
//
// A state over a key set is (o, lse): the normalised output and the log of the
// softmax denominator.  The state over the union of disjoint key sets is
//   lse = log sum_i exp(lse_i),   o = sum_i exp(lse_i - lse) o_i
// (merge_state / merge_states of flashinfer.cascade, 2026 guide, "Cascade
// attention for shared prefixes").  Three kernels use it:
//   merge_rows_kernel   the second pass of split-KV decode (and of cascade
//                       decode): per (request, kv head) row it merges the
//                       row's partial states, in slot order, for its g heads;
//   merge_state_kernel  the user-facing pairwise merge;
//   merge_states_kernel the user-facing k-way merge.
// Merges are deterministic: a fixed order, no atomics.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "pkd_internal.h"
#include "pkd_ptx.cuh"

namespace pkd {
namespace {

constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLog2e = 1.442695040888963407f;

__device__ __forceinline__ void store_elem(void* out, size_t idx, float v, int dtype) {
  if (dtype == kBF16) {
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  } else if (dtype == kF16) {
    static_cast<__half*>(out)[idx] = __float2half_rn(v);
  } else {
    static_cast<float*>(out)[idx] = v;
  }
}

__device__ __forceinline__ float load_elem(const void* in, size_t idx, int dtype) {
  if (dtype == kBF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(in)[idx]);
  if (dtype == kF16) return __half2float(static_cast<const __half*>(in)[idx]);
  return static_cast<const float*>(in)[idx];
}

// One warp per (request, qo head) output row; lane i owns head dimensions
// 4i .. 4i+3.  The row's states are the cascade prefix pieces (if any) and
// then its split-KV items, in slot order.  Lanes first load up to 32 state
// log-sum-exps at once (the max and the normaliser are warp reductions), then
// stream the states' fp32 partial outputs as float4.  Partial log-sum-exps are
// base 2 (the decode kernels' convention); the output lse is natural log.
constexpr int kMergeWarps = 8;
constexpr int kFewStates = 8;  // rows with at most this many states take the single-round-trip path

__device__ __forceinline__ void store4(void* out, size_t idx, float4 v, int dtype) {
  if (dtype == kBF16) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + idx) = u;
  } else if (dtype == kF16) {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(static_cast<__half*>(out) + idx) = u;
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + idx) = v;
  }
}

__global__ void __launch_bounds__(kMergeWarps * 32) merge_rows_kernel(const MergeParams p) {
  ptx::pdl_wait_prior_grid();  // the partials of the grids before this one are complete and visible
  const int batch = p.header->batch;
  const int Hk = p.num_kv_heads;
  const int G = p.group;
  const int Hq = Hk * G;
  const int n_rows = p.all_rows ? batch * Hk : p.header->n_merge_rows;
  const int lane = threadIdx.x & 31;
  const size_t pre_stride = static_cast<size_t>(batch) * Hq;
  const int n_pre = p.n_pre_splits;
  const int64_t n_units = static_cast<int64_t>(n_rows) * G;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * kMergeWarps;
#pragma unroll 1
  for (int64_t unit = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5); unit < n_units;
       unit += warps) {
    const int i = static_cast<int>(unit / G);
    const int j = static_cast<int>(unit - static_cast<int64_t>(i) * G);
    const int row = p.all_rows ? i : p.merge_rows[i];
    const int b = row / Hk;
    const int h = row - b * Hk;
    const int beg = p.row_item_begin[row];
    const int cnt = p.row_item_count[row];
    const size_t bq = static_cast<size_t>(b) * Hq + h * G + j;
    const int n_states = n_pre + cnt;
    // state s: prefix piece s (s < n_pre) or item beg + s - n_pre
    auto lse_of = [&](int s) -> float {
      return s < n_pre ? p.pre_lse[s * pre_stride + bq] : p.part_lse[static_cast<size_t>(beg + s - n_pre) * G + j];
    };
    auto o_of = [&](int s) -> const float4* {
      const float* base = s < n_pre ? p.pre_o + (s * pre_stride + bq) * kHeadDim
                                    : p.part_o + (static_cast<size_t>(beg + s - n_pre) * G + j) * kHeadDim;
      return reinterpret_cast<const float4*>(base) + lane;
    };
    float M = -INFINITY;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (n_states <= kFewStates) {
      // few states (a cascade row: the prefix pieces and one or two items):
      // every load is issued before any result is used, so the row costs one
      // memory round trip; the states are folded in the same slot order
      const float x = (lane < n_states) ? lse_of(lane) : -INFINITY;
      float4 o[kFewStates];
#pragma unroll
      for (int s = 0; s < kFewStates; ++s) o[s] = (s < n_states) ? *o_of(s) : make_float4(0.f, 0.f, 0.f, 0.f);
      M = x;
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, k));
      if (M != -INFINITY) {
        const float w = (x == -INFINITY) ? 0.f : ptx::ex2(x - M);
        L = w;
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) L += __shfl_xor_sync(0xffffffffu, L, k);
#pragma unroll
        for (int s = 0; s < kFewStates; ++s) {
          const float ws = __shfl_sync(0xffffffffu, w, s);
          if (s < n_states) {
            acc.x += ws * o[s].x;
            acc.y += ws * o[s].y;
            acc.z += ws * o[s].z;
            acc.w += ws * o[s].w;
          }
        }
        const float inv = 1.f / L;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
      }
      store4(p.out, bq * kHeadDim + 4 * lane, acc, p.out_dtype);
      if (lane == 0 && p.lse) p.lse[bq] = (M == -INFINITY) ? -INFINITY : (M + ptx::lg2(L)) * kLn2;
      continue;
    }
    for (int s0 = 0; s0 < n_states; s0 += 32) {
      const float x = (s0 + lane < n_states) ? lse_of(s0 + lane) : -INFINITY;
      M = fmaxf(M, x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M != -INFINITY) {
      for (int s0 = 0; s0 < n_states; s0 += 32) {
        const int ns = min(32, n_states - s0);
        const float x = (lane < ns) ? lse_of(s0 + lane) : -INFINITY;
        const float w = (x == -INFINITY) ? 0.f : ptx::ex2(x - M);
        L += w;
        int s = 0;
        for (; s + 2 <= ns; s += 2) {
          const float w0 = __shfl_sync(0xffffffffu, w, s), w1 = __shfl_sync(0xffffffffu, w, s + 1);
          const float4 a = *o_of(s0 + s), c = *o_of(s0 + s + 1);
          acc.x += w0 * a.x + w1 * c.x;
          acc.y += w0 * a.y + w1 * c.y;
          acc.z += w0 * a.z + w1 * c.z;
          acc.w += w0 * a.w + w1 * c.w;
        }
        if (s < ns) {
          const float w0 = __shfl_sync(0xffffffffu, w, s);
          const float4 a = *o_of(s0 + s);
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
    store4(p.out, bq * kHeadDim + 4 * lane, acc, p.out_dtype);
    if (lane == 0 && p.lse) p.lse[bq] = (M == -INFINITY) ? -INFINITY : (M + ptx::lg2(L)) * kLn2;
  }
}

// Weights of two states of log-sum-exps a, b (natural log) and the merged one.
__device__ __forceinline__ void pair_weights(float a, float b, float& wa, float& wb, float& s) {
  const float M = fmaxf(a, b);
  wa = 0.f;
  wb = 0.f;
  s = -INFINITY;
  if (M != -INFINITY) {
    const float ea = (a == -INFINITY) ? 0.f : ptx::ex2((a - M) * kLog2e);
    const float eb = (b == -INFINITY) ? 0.f : ptx::ex2((b - M) * kLog2e);
    const float tot = ea + eb;
    wa = ea / tot;
    wb = eb / tot;
    s = M + ptx::lg2(tot) * kLn2;
  }
}

// 16 bytes of values (8 16-bit or 4 fp32 elements) as fp32, and back.
struct Chunk {
  float f[8];
};

__device__ __forceinline__ uint4 load_raw(const void* in, size_t idx, int dtype) {
  return *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(in) + idx * (dtype == kF32 ? 4 : 2));
}

__device__ __forceinline__ Chunk to_chunk(const uint4& u, int dtype) {
  Chunk c;
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  if (dtype == kF32) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      c.f[e] = __uint_as_float(w[e]);
      c.f[4 + e] = 0.f;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 v = dtype == kBF16 ? __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]))
                                      : __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
      c.f[2 * e] = v.x;
      c.f[2 * e + 1] = v.y;
    }
  }
  return c;
}

__device__ __forceinline__ Chunk load_chunk(const void* in, size_t idx, int dtype) {
  return to_chunk(load_raw(in, idx, dtype), dtype);
}

__device__ __forceinline__ void store_chunk(void* out, size_t idx, const Chunk& c, int dtype) {
  uint4 u;
  uint32_t* w = reinterpret_cast<uint32_t*>(&u);
  if (dtype == kF32) {
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = __float_as_uint(c.f[e]);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = dtype == kBF16 ? ptx::pack2<true>(c.f[2 * e], c.f[2 * e + 1])
                                                      : ptx::pack2<false>(c.f[2 * e], c.f[2 * e + 1]);
  }
  *reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + idx * (dtype == kF32 ? 4 : 2)) = u;
}

// The flat pairwise merge with chunk indices of type I (32-bit when the
// chunk count allows: the index arithmetic is most of the instructions).
template <typename I>
__device__ __forceinline__ void merge_state_flat(const void* va, const float* sa, const void* vb, const float* sb,
                                                 void* vo, float* so, int64_t rows, int dim, int dtype) {
  const int ce = dtype == kF32 ? 4 : 8;  // elements per chunk
  const int per_row = dim / ce;
  const I chunks = static_cast<I>(rows) * per_row;
  const I stride = static_cast<I>(gridDim.x) * blockDim.x;
  // one chunk per iteration, its four loads issued first; the grid is one wave
  // of resident blocks, so the latency is covered by the many threads
  for (I j = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x; j < chunks; j += stride) {
    const I r = j / per_row;
    const uint4 xa = load_raw(va, static_cast<size_t>(j) * ce, dtype);
    const uint4 xb = load_raw(vb, static_cast<size_t>(j) * ce, dtype);
    const float la = __ldg(sa + r), lb = __ldg(sb + r);
    const Chunk x = to_chunk(xa, dtype), y = to_chunk(xb, dtype);
    float wa, wb, st;
    pair_weights(la, lb, wa, wb, st);
    Chunk o;
#pragma unroll
    for (int e = 0; e < 8; ++e) o.f[e] = x.f[e] * wa + y.f[e] * wb;
    store_chunk(vo, static_cast<size_t>(j) * ce, o, dtype);
    if (j - r * per_row == 0) so[r] = st;
  }
}

// Pairwise merge.  flat: one thread per 16-byte chunk of the values (dim a
// multiple of the chunk, 16-byte aligned arrays, s_out not one of the inputs),
// each thread taking its row's weights from the (cached) log-sum-exps; else
// one warp per (index, head) row, lanes striding over head_dim (the order that
// lets s_out overwrite an input in place).

__global__ void merge_state_kernel(const void* va, const float* sa, const void* vb, const float* sb,
                                   void* vo, float* so, int64_t rows, int dim, int dtype, int flat) {
  if (flat) {
    if (flat == 2) {
      merge_state_flat<uint32_t>(va, sa, vb, sb, vo, so, rows, dim, dtype);
    } else {
      merge_state_flat<int64_t>(va, sa, vb, sb, vo, so, rows, dim, dtype);
    }
    return;
  }
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
#pragma unroll 1
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    float wa, wb, s;
    pair_weights(sa[r], sb[r], wa, wb, s);
    __syncwarp();  // every lane has read sa/sb before lane 0 may overwrite them
#pragma unroll 1
    for (int c = lane; c < dim; c += 32) {
      const size_t idx = static_cast<size_t>(r) * dim + c;
      const float x = load_elem(va, idx, dtype) * wa + load_elem(vb, idx, dtype) * wb;
      store_elem(vo, idx, x, dtype);
    }
    if (lane == 0) so[r] = s;
  }
}

// The flat k-way merge with chunk indices of type I (see merge_state_flat).
template <typename I>
__device__ __forceinline__ void merge_states_flat(const void* v, const float* s, int64_t rows, int k, int heads,
                                                  int dim, int dtype, void* vo, float* so) {
  const int ce = dtype == kF32 ? 4 : 8;
  const int esz = dtype == kF32 ? 4 : 2;
  const int per_row = dim / ce;
  const I chunks = static_cast<I>(rows) * per_row;
  const I stride = static_cast<I>(gridDim.x) * blockDim.x;
  // bytes from one state's values to the next state's (the log-sum-exps are
  // `heads` floats apart)
  const size_t vstep = static_cast<size_t>(heads) * dim * esz;
  const uint8_t* vbytes = static_cast<const uint8_t*>(v);
  // one output chunk per iteration (more resident threads beat more chunks per
  // thread here): the first four states' chunks and log-sum-exps are
  // requested before any is used
  for (I j = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x; j < chunks; j += stride) {
    const I r = j / per_row;
    const I i = r / static_cast<I>(heads);
    const I hh = r - i * static_cast<I>(heads);
    const I c = j - r * per_row;
    // state 0 of (index i, head hh): this thread's chunk and the lse
    const size_t row0 = static_cast<size_t>(i) * k * heads + hh;
    const uint8_t* vp = vbytes + (row0 * dim + static_cast<size_t>(c) * ce) * esz;
    const float* sp = s + row0;
    uint4 x[4];
    float sc[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (e < k) {
        x[e] = *reinterpret_cast<const uint4*>(vp + e * vstep);
        sc[e] = __ldg(sp + static_cast<size_t>(e) * heads);
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < k) M = fmaxf(M, sc[e]);
    for (int e = 4; e < k; ++e) M = fmaxf(M, __ldg(sp + static_cast<size_t>(e) * heads));
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (e < k) {
          const float w = (sc[e] == -INFINITY) ? 0.f : ptx::ex2((sc[e] - M) * kLog2e);
          const Chunk ch = to_chunk(x[e], dtype);
          L += w;
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] += w * ch.f[q];
        }
      }
      // states past the fourth, in order
      for (int e = 4; e < k; ++e) {
        const float sce = __ldg(sp + static_cast<size_t>(e) * heads);
        const float w = (sce == -INFINITY) ? 0.f : ptx::ex2((sce - M) * kLog2e);
        const Chunk ch = to_chunk(*reinterpret_cast<const uint4*>(vp + e * vstep), dtype);
        L += w;
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] += w * ch.f[q];
      }
    }
    const float inv = M != -INFINITY ? 1.f / L : 0.f;
    Chunk o;
#pragma unroll
    for (int q = 0; q < 8; ++q) o.f[q] = acc[q] * inv;
    store_chunk(vo, static_cast<size_t>(j) * ce, o, dtype);
    if (c == 0) so[r] = (M == -INFINITY) ? -INFINITY : M + ptx::lg2(L) * kLn2;
  }
}

// k-way merge, states folded in order.  flat (as above, values 16-byte
// aligned, dim a multiple of the chunk): one thread per 16-byte chunk of the
// output, up to four states' chunks loaded before they are used; else one
// warp per (index, head) row.

__global__ void merge_states_kernel(const void* v, const float* s, int64_t n, int k, int heads,
                                    int dim, int dtype, void* vo, float* so, int flat) {
  const int64_t rows = n * heads;
  if (flat) {
    if (flat == 2) {
      merge_states_flat<uint32_t>(v, s, rows, k, heads, dim, dtype, vo, so);
    } else {
      merge_states_flat<int64_t>(v, s, rows, k, heads, dim, dtype, vo, so);
    }
    return;
  }
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
#pragma unroll 1
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const int64_t i = r / heads;
    const int hh = static_cast<int>(r - i * heads);
    float M = -INFINITY;
    for (int c = 0; c < k; ++c) M = fmaxf(M, s[(i * k + c) * heads + hh]);
    float L = 0.f;
    if (M != -INFINITY) {
      for (int c = 0; c < k; ++c) {
        const float x = s[(i * k + c) * heads + hh];
        L += (x == -INFINITY) ? 0.f : ptx::ex2((x - M) * kLog2e);
      }
    }
#pragma unroll 1
    for (int cd = lane; cd < dim; cd += 32) {
      float acc = 0.f;
      if (M != -INFINITY) {
        for (int c = 0; c < k; ++c) {
          const float x = s[(i * k + c) * heads + hh];
          const float w = (x == -INFINITY) ? 0.f : ptx::ex2((x - M) * kLog2e);
          acc += w * load_elem(v, ((i * k + c) * heads + hh) * static_cast<int64_t>(dim) + cd, dtype);
        }
        acc /= L;
      }
      store_elem(vo, static_cast<size_t>(r) * dim + cd, acc, dtype);
    }
    if (lane == 0) so[r] = (M == -INFINITY) ? -INFINITY : M + ptx::lg2(L) * kLn2;
  }
}

// Copies the plan's schedule from pinned host memory (read through its
// device mapping) into the workspace: for a few tens of KB a kernel reaches
// the data sooner than a DMA copy.  The decode grid behind it may be
// scheduled at once; it waits for this grid in griddepcontrol.wait.  This grid
// is itself launched programmatically: it may become resident while the
// previous step's merge drains, and waits for that grid before it overwrites
// the schedule the merge reads.
// The reads of the first four words per thread are issued before the wait, so
// that their latency (the staging buffer is host memory) overlaps the tail of
// the previous grid.
__global__ void copy_words_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, int64_t n16) {
  ptx::pdl_launch_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  uint4 w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (i0 + e * stride < n16) w[e] = src[i0 + e * stride];
  ptx::pdl_wait_prior_grid();
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (i0 + e * stride < n16) dst[i0 + e * stride] = w[e];
  for (int64_t i = i0 + 4 * stride; i < n16; i += stride) dst[i] = src[i];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Blocks of `threads` threads of `kernel` resident on the whole GPU at once
// (SM count x occupancy), for a grid-stride kernel sized to run in one wave;
// `cache` holds the answer per device (0: not asked yet, -1: the query
// failed, and a fixed grid is used).
int64_t resident_blocks(const void* kernel, int threads, std::atomic<int> (&cache)[64]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 8192;
  }
  int c = cache[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) == cudaSuccess && sms > 0 &&
        per_sm > 0) {
      c = sms * per_sm;
    } else {
      cudaGetLastError();
      c = -1;
    }
    cache[dev].store(c, std::memory_order_relaxed);
  }
  return c > 0 ? c : 8192;
}

int grid_for_rows(int64_t rows) {
  const int64_t per_block = 8;  // warps per 256-thread block
  int64_t g = (rows + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > 4096) g = 4096;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_merge_rows(const MergeParams& p, int grid, cudaStream_t stream) {
  // programmatic dependent launch: scheduled while the grid before it (the
  // cascade's prefix kernel, or the decode grid of the no-alloc path) runs, it
  // waits in griddepcontrol.wait for that grid to complete
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, merge_rows_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_copy16(void* dst, const void* src, int64_t bytes, cudaStream_t stream) {
  const int64_t n16 = bytes / 16;
  if (n16 <= 0) return cudaSuccess;
  int grid = static_cast<int>((n16 + 255) / 256);
  grid = grid > 64 ? 64 : grid;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, copy_words_kernel, static_cast<uint4*>(dst), static_cast<const uint4*>(src), n16);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_merge_state(const void* va, const float* sa, const void* vb, const float* sb,
                               void* vo, float* so, int64_t n, int heads, int dim, int dtype,
                               cudaStream_t stream) {
  const int64_t rows = n * heads;
  if (rows == 0) return cudaSuccess;
  const int ce = dtype == kF32 ? 4 : 8;
  const bool flat = dim % ce == 0 && aligned16(va) && aligned16(vb) && aligned16(vo) && so != sa && so != sb;
  if (flat) {
    const int64_t chunks = rows * (dim / ce);
    const int64_t blocks = (chunks + 255) / 256;
    static std::atomic<int> cache[64];
    const int64_t cap = resident_blocks(reinterpret_cast<const void*>(merge_state_kernel), 256, cache);
    merge_state_kernel<<<static_cast<int>(blocks < cap ? blocks : cap), 256, 0, stream>>>(
        va, sa, vb, sb, vo, so, rows, dim, dtype, chunks < (int64_t(1) << 31) ? 2 : 1);
  } else {
    merge_state_kernel<<<grid_for_rows(rows), 256, 0, stream>>>(va, sa, vb, sb, vo, so, rows, dim, dtype, 0);
  }
  return cudaGetLastError();
}

cudaError_t launch_merge_states(const void* v, const float* s, int64_t n, int k, int heads, int dim,
                                int dtype, void* vo, float* so, cudaStream_t stream) {
  const int64_t rows = n * heads;
  if (rows == 0) return cudaSuccess;
  const int ce = dtype == kF32 ? 4 : 8;
  const bool flat = dim % ce == 0 && aligned16(v) && aligned16(vo);
  if (flat) {
    const int64_t chunks = rows * (dim / ce);
    const int64_t blocks = (chunks + 255) / 256;
    static std::atomic<int> cache[64];
    const int64_t cap = resident_blocks(reinterpret_cast<const void*>(merge_states_kernel), 256, cache);
    merge_states_kernel<<<static_cast<int>(blocks < cap ? blocks : cap), 256, 0, stream>>>(
        v, s, n, k, heads, dim, dtype, vo, so, chunks < (int64_t(1) << 31) ? 2 : 1);
  } else {
    merge_states_kernel<<<grid_for_rows(rows), 256, 0, stream>>>(v, s, n, k, heads, dim, dtype, vo, so, 0);
  }
  return cudaGetLastError();
}

}  // namespace pkd
