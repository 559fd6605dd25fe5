// vg_probe.cu -- read-only HBM bandwidth probe.
//
// The verify GEMV is bound by weight reads (mtp7-device-confidence engine
// card, Measured section: 19.26 GB read per verify pass, its floor set by
// the card's read rate; crit README, Eval: limits derived from the measured
// memory bandwidth).  This probe measures the practical read ceiling of the
// device with the two access styles the library could use, so that the
// GEMV can be judged against what the hardware actually delivers:
//   mode 0: every thread streams 16-byte vector loads (grid-stride);
//   mode 1: every warp streams `chunk`-byte 1-D bulk copies into a private
//           ring of shared-memory slots, like the GEMV kernel does.
// The bytes read are folded into one word per block so nothing is elided.
#include <cuda_runtime.h>

#include <cstdint>

#include "vg_device.cuh"
#include "vg_internal.h"

namespace vg {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeWarps = kProbeThreads / 32;
constexpr int kProbeRingBytes = 192 * 1024;

__global__ void __launch_bounds__(kProbeThreads) probe_ldg(const uint4 *__restrict__ p, int64_t n,
                                                           uint32_t *sink) {
  uint32_t acc = 0;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = ldg128(p + i), b = ldg128(p + i + stride);
    const uint4 c = ldg128(p + i + 2 * stride), d = ldg128(p + i + 3 * stride);
    acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^
           d.z ^ d.w;
  }
  for (; i < n; i += stride) {
    const uint4 a = ldg128(p + i);
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
  acc = __reduce_xor_sync(0xFFFFFFFFu, acc);
  if ((threadIdx.x & 31) == 0) atomicXor(sink + blockIdx.x, acc);
}

// Each warp owns kProbeRingBytes / kProbeWarps bytes of slots.  Pattern 0:
// chunks are assigned to (block, warp) round-robin over the whole device, so
// all warps read neighbouring chunks at the same time.  Pattern 1: each block
// streams its own contiguous range (warps take neighbouring chunks of it),
// the order the GEMV's split of work produces.
__global__ void __launch_bounds__(kProbeThreads, 1) probe_bulk(const uint8_t *__restrict__ p,
                                                               int64_t nchunks, int chunk,
                                                               int slots, int pattern,
                                                               uint32_t *sink,
                                                               uint64_t timeout_ns) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kProbeRingBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ring = smem_addr(smem + warp * (kProbeRingBytes / kProbeWarps));
  const uint32_t bar0 = smem_addr(bars + warp * 16);
  if (lane == 0)
    for (int s = 0; s < slots; ++s) mbar_init(bar0 + 8 * s, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();
  // pattern 2: like pattern 1, plus a second copy of chunk/8 bytes per slot
  // from the upper eighth of the buffer (the block scales next to the codes)
  const int side = pattern == 2 ? chunk / 8 : 0;
  const uint8_t *sp = p + (nchunks * int64_t(chunk)) / 9 * 8;
  if (pattern == 2) nchunks = nchunks / 9 * 8;
  int64_t workers = int64_t(gridDim.x) * kProbeWarps;
  int64_t next = int64_t(warp) * gridDim.x + blockIdx.x;
  if (pattern >= 1) {
    const int64_t per = nchunks / gridDim.x / kProbeWarps * kProbeWarps;
    workers = kProbeWarps;
    next = blockIdx.x * per + warp;
    nchunks = blockIdx.x * per + per;
  }
  const uint64_t policy = policy_evict_first();
  int64_t issued = 0, done = 0;
  uint32_t acc = 0;
  const int stride = chunk + side;
  for (int s = 0; s < slots && next < nchunks; ++s, next += workers, ++issued)
    if (lane == 0) {
      mbar_arrive_expect_tx(bar0 + 8 * s, uint32_t(chunk + side));
      bulk_g2s(ring + s * stride, p + next * chunk, uint32_t(chunk), bar0 + 8 * s, policy);
      if (side)
        bulk_g2s(ring + s * stride + chunk, sp + next * side, uint32_t(side), bar0 + 8 * s, policy);
    }
  while (done < issued) {
    const int s = int(done % slots);
    if (!mbar_wait(bar0 + 8 * s, uint32_t(done / slots) & 1u, globaltimer() + timeout_ns)) break;
    acc ^= lds64(ring + s * stride + lane * 8).x;
    __syncwarp();
    if (next < nchunks) {
      if (lane == 0) {
        fence_proxy_async();
        mbar_arrive_expect_tx(bar0 + 8 * s, uint32_t(chunk + side));
        bulk_g2s(ring + s * stride, p + next * chunk, uint32_t(chunk), bar0 + 8 * s, policy);
        if (side)
          bulk_g2s(ring + s * stride + chunk, sp + next * side, uint32_t(side), bar0 + 8 * s,
                   policy);
      }
      next += workers;
      ++issued;
    }
    ++done;
  }
  // wait for anything still in flight (only after a timeout)
  for (int64_t k = done; k < issued; ++k)
    mbar_wait(bar0 + 8 * int(k % slots), uint32_t(k / slots) & 1u, globaltimer() + timeout_ns);
  acc = __reduce_xor_sync(0xFFFFFFFFu, acc);
  if (lane == 0) atomicXor(sink + blockIdx.x, acc);
}

}  // namespace
}  // namespace vg

using namespace vg;

extern "C" vg_status vg_hbm_read_probe(const void *buf, size_t bytes, int mode, int chunk,
                                       int slots, uint32_t *sink, int sink_words,
                                       vg_stream_t stream) {
  if (!buf || !sink || bytes < 4096 || mode < 0 || mode > 3) return VG_ERR_INVALID_ARG;
  if (!aligned16(buf) || !aligned16(sink)) return VG_ERR_ALIGNMENT;
  int dev = 0, sms = 0;
  VG_CUDA(cudaGetDevice(&dev));
  VG_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  cudaStream_t st = as_cuda(stream);
  if (mode == 0) {
    int per_sm = 0;
    VG_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, probe_ldg, kProbeThreads, 0));
    const int grid = sms * (per_sm > 0 ? per_sm : 1);
    if (sink_words < grid) return VG_ERR_INVALID_ARG;
    probe_ldg<<<grid, kProbeThreads, 0, st>>>(static_cast<const uint4 *>(buf),
                                              int64_t(bytes / 16), sink);
  } else {
    if (chunk < 256 || chunk % 256 || slots < 1 || slots > 16 ||
        int64_t(chunk + (mode == 3 ? chunk / 8 : 0)) * slots > kProbeRingBytes / kProbeWarps)
      return VG_ERR_INVALID_ARG;
    if (sink_words < sms) return VG_ERR_INVALID_ARG;
    const int smem = kProbeRingBytes + kProbeWarps * 16 * 8;
    VG_CUDA(cudaFuncSetAttribute(probe_bulk, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    probe_bulk<<<sms, kProbeThreads, smem, st>>>(static_cast<const uint8_t *>(buf),
                                                 int64_t(bytes / size_t(chunk)), chunk, slots,
                                                 mode - 1, sink, 2000000000ull);
  }
  VG_LAUNCH_CHECK();
  return VG_OK;
}
