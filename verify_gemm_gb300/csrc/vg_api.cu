// vg_api.cu -- status strings, version and CUDA error capture of the C ABI.
#include <cuda_runtime.h>

#include <cstdio>

#include "vg_internal.h"

namespace vg {
namespace {
thread_local char g_last_error[256] = "";
}

void set_cuda_error(cudaError_t e) {
  const char *name = cudaGetErrorName(e);
  const char *msg = cudaGetErrorString(e);
  std::snprintf(g_last_error, sizeof g_last_error, "%s: %s", name ? name : "?", msg ? msg : "?");
}
}  // namespace vg

extern "C" const char *vg_status_string(vg_status s) {
  switch (s) {
    case VG_OK: return "ok";
    case VG_ERR_INVALID_ARG: return "invalid argument";
    case VG_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case VG_ERR_UNSUPPORTED: return "unsupported device or size";
    case VG_ERR_CUDA: return "CUDA error";
    case VG_ERR_TIMEOUT: return "device-side wait timed out";
    case VG_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

extern "C" int vg_version(void) { return 100; }

extern "C" const char *vg_last_cuda_error(void) { return vg::g_last_error; }
