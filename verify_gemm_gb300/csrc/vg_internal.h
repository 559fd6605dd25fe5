// vg_internal.h -- host-side helpers shared by the library's translation
// units: argument validation and CUDA error capture.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/vgemm.h"

namespace vg {

// Last CUDA error message (per host thread), surfaced by vg_last_cuda_error.
void set_cuda_error(cudaError_t e);

inline cudaStream_t as_cuda(vg_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kMaxElems = int64_t(1) << 40;

inline vg_status check_mk(int64_t M, int64_t K) {
  if (M < 1 || K < 16 || K % 16 != 0) return VG_ERR_INVALID_ARG;
  if (M > kMaxElems / K || M >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
    return VG_ERR_UNSUPPORTED;
  return VG_OK;
}

#define VG_CUDA(call)                     \
  do {                                    \
    cudaError_t e_ = (call);              \
    if (e_ != cudaSuccess) {              \
      ::vg::set_cuda_error(e_);           \
      return VG_ERR_CUDA;                 \
    }                                     \
  } while (0)

#define VG_LAUNCH_CHECK()                        \
  do {                                           \
    cudaError_t e_ = cudaGetLastError();         \
    if (e_ != cudaSuccess) {                     \
      ::vg::set_cuda_error(e_);                  \
      return VG_ERR_CUDA;                        \
    }                                            \
  } while (0)

}  // namespace vg
