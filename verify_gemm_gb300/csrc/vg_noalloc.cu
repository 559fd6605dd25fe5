// vg_noalloc.cu -- vg_gemv_nvfp4_noalloc: the NVFP4 GEMV for callers that
// cannot allocate device memory, and vg_gemv_nvfp4_noalloc_check, which
// reports whether its bounded device-side waits ran out.
//
// vg_gemv_nvfp4 needs a workspace (a few header words and FP32 partial
// sums for row blocks whose K range is split between thread blocks), and
// expects the caller to allocate it.  Some callers cannot:
// code that runs inside a host application which owns all device memory
// and only lends out the input and output buffers (a plugin or an engine
// adapter), code that must not call cudaMalloc because it can synchronise
// the whole device and stall other work, and code that runs under a memory
// budget that a hidden allocation would break.  For them this file keeps
// one fixed scratch array in device memory and runs the unchanged GEMV with
// that array as its workspace.  The array is created on each device when
// the library's module is first used there (CUDA loads modules lazily) and
// is held until the process exits.
#include <cuda_runtime.h>

#include <cstdint>

#include "vg_internal.h"

namespace {

// Largest workspace this entry point can serve: 4 MiB, enough for one
// thread block per SM (16 KiB of partial sums each) on devices of up to 255
// SMs, whatever the matrix size.
constexpr size_t kScratchBytes = VG_NOALLOC_SCRATCH_BYTES;

// The workspace lives here.  In host code this name is only a stand-in for
// the device array, never a usable address: the device address is looked
// up with cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

// Device address of g_scratch on the current device.  It is looked up on
// every call rather than cached: after a device reset, or once the primary
// context has been torn down and created again, the module is loaded anew
// and the array may sit elsewhere.  The first lookup on a device is what
// loads the module there, which is why the first call on a device must come
// before any stream capture; later lookups only read the module's table.
vg_status scratch_address(void **out) {
  void *p = nullptr;
  VG_CUDA(cudaGetSymbolAddress(&p, g_scratch));
  *out = p;
  return VG_OK;
}

}  // namespace

extern "C" vg_status vg_gemv_nvfp4_noalloc(const void *w, const void *scales, float gscale,
                                           const uint16_t *x, int N, int64_t M, int64_t K,
                                           uint16_t *y, vg_stream_t stream) {
  // Arguments are checked by vg_gemv_nvfp4 below; the size check needs M, K.
  if (vg_status s = vg::check_mk(M, K)) return s;
  size_t need = 0;
  if (N < 1 || N > 32) return VG_ERR_INVALID_ARG;
  if (vg_status s = vg_gemv_workspace_size_n(M, K, VG_FMT_NVFP4, N, &need)) return s;
  if (need > kScratchBytes) return VG_ERR_UNSUPPORTED;   // beyond the fixed maximum
  void *scratch = nullptr;
  if (vg_status s = scratch_address(&scratch)) return s;
  // The array starts zeroed and every call leaves it consistent for the
  // next one (finished-block count back at zero, pass epoch advanced), except
  // for the error word: a call whose wait ran out leaves it set (read it with
  // vg_gemv_nvfp4_noalloc_check), and a set error word makes the kernel's
  // waits give up early.  So each call starts by clearing it (4 bytes).
  VG_CUDA(cudaMemsetAsync(scratch, 0, sizeof(int), vg::as_cuda(stream)));
  return vg_gemv_nvfp4(w, scales, gscale, x, N, M, K, y, scratch, kScratchBytes, stream);
}

extern "C" vg_status vg_gemv_nvfp4_noalloc_check(int *device_error, vg_stream_t stream) {
  if (!device_error) return VG_ERR_INVALID_ARG;
  void *scratch = nullptr;
  if (vg_status s = scratch_address(&scratch)) return s;
  // vg_gemv_workspace_check reads the word into host memory (a plain
  // stack variable: no pinned staging buffer is allocated) and, if it is
  // set, zero-fills the whole array with cudaMemsetAsync.
  return vg_gemv_workspace_check(scratch, kScratchBytes, device_error, stream);
}
