// pkd_upload.h -- the schedule upload of one-shot plans (single-request decode).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace pkd {

// Up to kBlobBytes of host data written to dst by a kernel that receives them
// as its parameter: no copy engine and no host memory read at run time (the
// bytes are part of the launch, so a captured graph replays them).  dst
// 16-byte aligned, bytes a multiple of 16.
constexpr int64_t kBlobBytes = 16384;
cudaError_t launch_copy_blob(void* dst, const void* host_src, int64_t bytes, cudaStream_t stream);

}  // namespace pkd
