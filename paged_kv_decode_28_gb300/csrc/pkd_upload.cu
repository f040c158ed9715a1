// pkd_upload.cu -- the schedule upload of one-shot plans (see pkd_upload.h).
#include "pkd_upload.h"

#include <cstring>

#include "pkd_ptx.cuh"

namespace pkd {
namespace {

struct Blob {
  uint4 w[kBlobBytes / 16];
};

// The schedule of a one-shot plan, carried in the launch itself.  The grid
// after it (decode) may be scheduled at once; it waits for this one in
// griddepcontrol.wait.
__global__ void copy_blob_kernel(uint4* __restrict__ dst, int n16, const __grid_constant__ Blob b) {
  ptx::pdl_launch_dependents();
  for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = b.w[i];
}

}  // namespace

cudaError_t launch_copy_blob(void* dst, const void* host_src, int64_t bytes, cudaStream_t stream) {
  if (bytes <= 0) return cudaSuccess;
  if (bytes > kBlobBytes || (bytes & 15) != 0 || (reinterpret_cast<uintptr_t>(dst) & 15u) != 0)
    return cudaErrorInvalidValue;
  static thread_local Blob b;  // 16 KB: off the stack
  memcpy(b.w, host_src, static_cast<size_t>(bytes));
  copy_blob_kernel<<<1, 256, 0, stream>>>(static_cast<uint4*>(dst), static_cast<int>(bytes / 16), b);
  return cudaGetLastError();
}

}  // namespace pkd
