// pkd_host.h -- host-side helpers shared by the C-ABI translation units:
// status messages, alignment rules and the driver's tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>

#include "pkd.h"

namespace pkd {

// The calling thread's last error message (pkd_last_error), defined in pkd_capi.cu.
void set_last_error(const char* msg);

namespace host {

// Record a formatted message for pkd_last_error and return `st`.
pkd_status fail(pkd_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));

inline pkd_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKD_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int elem_bytes(int dt) { return dt == PKD_E4M3 ? 1 : (dt == PKD_F32 ? 4 : 2); }

// cuTensorMapEncodeTiled from the driver (looked up once), or nullptr.
PFN_cuTensorMapEncodeTiled_v12000 get_encode();

}  // namespace host
}  // namespace pkd
