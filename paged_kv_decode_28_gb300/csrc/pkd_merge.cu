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

// One CTA of 128 threads per row; thread d owns head dimension d.  Partial
// log-sum-exps are base 2 (the decode kernels' convention); the output lse is
// natural log.
__global__ void __launch_bounds__(kHeadDim) merge_rows_kernel(const MergeParams p) {
  const int batch = p.header->batch;
  const int Hk = p.num_kv_heads;
  const int G = p.group;
  const int Hq = Hk * G;
  const int n_rows = p.all_rows ? batch * Hk : p.header->n_merge_rows;
  const int d = threadIdx.x;
  const size_t pre_stride = static_cast<size_t>(batch) * Hq;
#pragma unroll 1
  for (int i = blockIdx.x; i < n_rows; i += gridDim.x) {
    const int row = p.all_rows ? i : p.merge_rows[i];
    const int b = row / Hk;
    const int h = row - b * Hk;
    const int beg = p.row_item_begin[row];
    const int cnt = p.row_item_count[row];
#pragma unroll 1
    for (int j = 0; j < G; ++j) {
      const int qo = h * G + j;
      const size_t bq = static_cast<size_t>(b) * Hq + qo;
      float M = -INFINITY;
      for (int s = 0; s < p.n_pre_splits; ++s) M = fmaxf(M, p.pre_lse[s * pre_stride + bq]);
      for (int c = 0; c < cnt; ++c) M = fmaxf(M, p.part_lse[static_cast<size_t>(beg + c) * G + j]);
      float acc = 0.f, L = 0.f;
      if (M != -INFINITY) {
        for (int s = 0; s < p.n_pre_splits; ++s) {
          const float ls = p.pre_lse[s * pre_stride + bq];
          const float w = (ls == -INFINITY) ? 0.f : ptx::ex2(ls - M);
          L += w;
          acc += w * p.pre_o[(s * pre_stride + bq) * kHeadDim + d];
        }
        for (int c = 0; c < cnt; ++c) {
          const size_t slot = static_cast<size_t>(beg + c) * G + j;
          const float ls = p.part_lse[slot];
          const float w = (ls == -INFINITY) ? 0.f : ptx::ex2(ls - M);
          L += w;
          acc += w * p.part_o[slot * kHeadDim + d];
        }
      }
      const float v = (M == -INFINITY) ? 0.f : acc / L;
      store_elem(p.out, bq * kHeadDim + d, v, p.out_dtype);
      if (d == 0 && p.lse) p.lse[bq] = (M == -INFINITY) ? -INFINITY : (M + ptx::lg2(L)) * kLn2;
    }
  }
}

// One warp per (index, head) row; lanes stride over head_dim.
__global__ void merge_state_kernel(const void* va, const float* sa, const void* vb, const float* sb,
                                   void* vo, float* so, int64_t rows, int dim, int dtype) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
#pragma unroll 1
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const float a = sa[r], b = sb[r];
    const float M = fmaxf(a, b);
    float wa = 0.f, wb = 0.f, s = -INFINITY;
    if (M != -INFINITY) {
      const float ea = (a == -INFINITY) ? 0.f : ptx::ex2((a - M) * kLog2e);
      const float eb = (b == -INFINITY) ? 0.f : ptx::ex2((b - M) * kLog2e);
      const float tot = ea + eb;
      wa = ea / tot;
      wb = eb / tot;
      s = M + ptx::lg2(tot) * kLn2;
    }
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

// One warp per (index, head): merges k states in order.
__global__ void merge_states_kernel(const void* v, const float* s, int64_t n, int k, int heads,
                                    int dim, int dtype, void* vo, float* so) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = n * heads;
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

int grid_for_rows(int64_t rows) {
  const int64_t per_block = 8;  // warps per 256-thread block
  int64_t g = (rows + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > 4096) g = 4096;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_merge_rows(const MergeParams& p, int grid, cudaStream_t stream) {
  merge_rows_kernel<<<grid, kHeadDim, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_merge_state(const void* va, const float* sa, const void* vb, const float* sb,
                               void* vo, float* so, int64_t n, int heads, int dim, int dtype,
                               cudaStream_t stream) {
  const int64_t rows = n * heads;
  if (rows == 0) return cudaSuccess;
  merge_state_kernel<<<grid_for_rows(rows), 256, 0, stream>>>(va, sa, vb, sb, vo, so, rows, dim, dtype);
  return cudaGetLastError();
}

cudaError_t launch_merge_states(const void* v, const float* s, int64_t n, int k, int heads, int dim,
                                int dtype, void* vo, float* so, cudaStream_t stream) {
  const int64_t rows = n * heads;
  if (rows == 0) return cudaSuccess;
  merge_states_kernel<<<grid_for_rows(rows), 256, 0, stream>>>(v, s, n, k, heads, dim, dtype, vo, so);
  return cudaGetLastError();
}

}  // namespace pkd
