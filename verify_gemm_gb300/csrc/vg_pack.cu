// vg_pack.cu -- load-time kernels: NVFP4, row-scaled FP8, MXFP8 and
// groupwise-INT4 round-to-nearest quantisation into the packed layout (and
// gate/up pairs packed as one matrix), unpack to the canonical layout, and
// canonical -> packed conversion.
//
// The re-encoding of stored weights at load is what the crit landing page's
// "Models" paragraph (round-to-nearest post-training quantisation to FP8 or
// NVFP4) and the mtp7-device-confidence engine card's Model section (draft
// layer re-encoded as row-scaled FP8, head as NVFP4) describe.  Every FP32
// step is one IEEE operation (explicit _rn intrinsics, no contraction), so
// the codes are bit-identical to any other correct implementation of the
// same recipe.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "vg_device.cuh"
#include "vg_internal.h"

namespace vg {
namespace {

// ---------------------------------------------------------- conversions

// E4M3 value of a byte 0x00..0x7E (exact in FP32).
__device__ __forceinline__ float e4m3_to_float(uint32_t c) {
  const int e = (c >> 3) & 15, f = c & 7;
  return e ? ldexpf(1.0f + f * 0.125f, e - 7) : ldexpf(float(f), -9);
}

// Round to nearest even with saturation to +-448 (PTX cvt.rn.satfinite).
__device__ __forceinline__ uint32_t e4m3_rn_sat(float s) {
  unsigned short h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(h) : "f"(s), "f"(0.0f));
  return h & 0xFFu;
}

// Round to nearest even with saturation to +-6; the sign is kept, so a
// negative value that rounds to zero gives 0x8.
__device__ __forceinline__ uint32_t e2m1_rn_sat(float q) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %2, %1; cvt.u32.u8 %0, t; }"
      : "=r"(r)
      : "f"(q), "f"(0.0f));
  return r & 0xFu;
}

__device__ __forceinline__ uint32_t abs_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }

// Position of the code of (row half ri, column ii of an MMA step) in the
// packed NVFP4 word: register R and 16-bit half.
__device__ __forceinline__ uint32_t nv_place(uint32_t code, int ri, int ii) {
  const int r = ri == 0 ? (ii < 2 ? 0 : 2) : (ii < 2 ? 1 : 3);
  const int half = (ii & 1) * 16;
  uint32_t w = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) w |= ((code >> b) & 1u) << (nv_bitpos(r, b) + half);
  return w;
}

__device__ __forceinline__ uint32_t nv_extract(uint32_t word, int ri, int ii) {
  const int r = ri == 0 ? (ii < 2 ? 0 : 2) : (ii < 2 ? 1 : 3);
  const int half = (ii & 1) * 16;
  uint32_t c = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) c |= ((word >> (nv_bitpos(r, b) + half)) & 1u) << b;
  return c;
}

// Byte offset, inside a lane's 32 FP8 bytes of a unit, of (row half ri,
// column 4j + ii of the lane's 16 columns).
__device__ __forceinline__ int f8_byte(int ri, int j, int ii) {
  return 4 * (2 * j + (ii >> 1)) + 2 * (ii & 1) + ri;
}

// Geometry of a packed matrix; rt: row tiles per row block (layout_rt).
struct Geom {
  int64_t M, K, MT, KU, KC, rt;
};

inline Geom geom(int64_t M, int64_t K, int cu) {
  Geom g;
  g.M = M;
  g.K = K;
  g.MT = ceil_div(M, kTileRows);
  g.KU = ceil_div(K, kUnitK);
  g.KC = ceil_div(g.KU, cu);
  g.rt = layout_rt(M, K, cu);
  return g;
}
inline Geom nv_geom(int64_t M, int64_t K) { return geom(M, K, kNvChunkUnits); }
inline Geom f8_geom(int64_t M, int64_t K) { return geom(M, K, kF8ChunkUnits); }

// ----------------------------------------------------------- amax kernels

__global__ void amax_kernel(const float *__restrict__ W, int64_t n, uint32_t *out) {
  uint32_t m = 0;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    m = max(m, abs_bits(W[i]));
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if ((threadIdx.x & 31) == 0) atomicMax(out, m);
}

// One warp per row: rowscale = rowamax / 448 (NaN/Inf propagate).
__global__ void f8_rowscale_kernel(const float *__restrict__ W, int64_t M, int64_t K,
                                   float *__restrict__ rs) {
  const int64_t row = int64_t(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  if (row >= M) return;
  const int lane = threadIdx.x & 31;
  uint32_t m = 0;
  for (int64_t k = lane; k < K; k += 32) m = max(m, abs_bits(W[row * K + k]));
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if (lane == 0) rs[row] = __fdiv_rn(__uint_as_float(m), 448.0f);
}

// --------------------------------------------------------- NVFP4 packing
// One thread per (tile, unit, lane): the lane's 16 columns of rows g, g+8.
// With W2 set the matrix is a gated pair of M = 2I rows: tile row g comes
// from row 8*mt + g of W (gate, tensor scale gs) and tile row g + 8 from the
// same row of W2 (up, tensor scale gs2).

__global__ void nv_pack_kernel(const float *__restrict__ W, Geom G, float gs,
                               uint8_t *__restrict__ w_out, uint8_t *__restrict__ sc_out,
                               const float *__restrict__ W2 = nullptr, float gs2 = 0.0f) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= G.MT * G.KU * 32) return;
  const int lane = int(idx & 31);
  const int64_t u = (idx >> 5) % G.KU, mt = (idx >> 5) / G.KU;
  const int g = lane >> 2, t = lane & 3;
  const int64_t k0 = u * kUnitK + 16 * t;
  uint32_t words[4] = {0, 0, 0, 0};
  for (int ri = 0; ri < 2; ++ri) {
    const int64_t row = mt * kTileRows + g + 8 * ri;
    const int64_t srow = W2 ? mt * 8 + g : row;          // row of the source matrix
    const float *Ws = W2 && ri ? W2 : W;
    const float gsr = W2 && ri ? gs2 : gs;
    uint32_t code = 0;
    if (row < G.M && k0 < G.K) {
      const float *w = Ws + srow * G.K + k0;
      float v[16];
      uint32_t bm = 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        v[j] = w[j];
        bm = max(bm, abs_bits(v[j]));
      }
      const float bamax = __uint_as_float(bm);
      if (gsr != 0.0f) code = e4m3_rn_sat(__fdiv_rn(__fdiv_rn(bamax, gsr), 6.0f));
      const float d = __fmul_rn(e4m3_to_float(code), gsr);
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const uint32_t c = d == 0.0f ? 0u : e2m1_rn_sat(__fdiv_rn(v[kk], d));
        words[kk >> 2] |= nv_place(c, ri, kk & 3);
      }
    }
    sc_out[scale_offset(mt, u / kNvChunkUnits, G.MT, G.KC, G.rt) + lane * kNvScaleLaneBytes +
           (u % kNvChunkUnits) * 2 + ri] = uint8_t(scale_code_from_e4m3(code));
  }
  *reinterpret_cast<uint4 *>(w_out + code_offset(mt, u, G.MT, G.KU, kNvChunkUnits, kNvUnitBytes, G.rt) +
                             lane * 16) =
      make_uint4(words[0], words[1], words[2], words[3]);
}

__global__ void nv_unpack_kernel(const uint8_t *__restrict__ w, const uint8_t *__restrict__ sc,
                                 Geom G, uint8_t *__restrict__ nib, uint8_t *__restrict__ scc) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= G.MT * G.KU * 32) return;
  const int lane = int(idx & 31);
  const int64_t u = (idx >> 5) % G.KU, mt = (idx >> 5) / G.KU;
  const int g = lane >> 2, t = lane & 3;
  const int64_t k0 = u * kUnitK + 16 * t;
  if (k0 >= G.K) return;
  const uint4 v = *reinterpret_cast<const uint4 *>(
      w + code_offset(mt, u, G.MT, G.KU, kNvChunkUnits, kNvUnitBytes, G.rt) + lane * 16);
  const uint32_t words[4] = {v.x, v.y, v.z, v.w};
  for (int ri = 0; ri < 2; ++ri) {
    const int64_t row = mt * kTileRows + g + 8 * ri;
    if (row >= G.M) continue;
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const uint32_t c = nv_extract(words[kk >> 2], ri, kk & 3);
      if (kk < 8)
        lo |= c << (4 * kk);
      else
        hi |= c << (4 * (kk - 8));
    }
    *reinterpret_cast<uint2 *>(nib + row * (G.K / 2) + k0 / 2) = make_uint2(lo, hi);
    const uint8_t d = sc[scale_offset(mt, u / kNvChunkUnits, G.MT, G.KC, G.rt) + lane * kNvScaleLaneBytes +
                         (u % kNvChunkUnits) * 2 + ri];
    scc[row * (G.K / 16) + k0 / 16] = uint8_t(e4m3_from_scale_code(d));
  }
}

__global__ void nv_check_canonical_kernel(const uint8_t *__restrict__ sc, int64_t n,
                                          uint32_t *bad) {
  uint32_t cnt = 0;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint32_t b = sc[i];
    cnt += (b & 0x80u) || b == 0x7Fu;
  }
  cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
  if ((threadIdx.x & 31) == 0 && cnt) atomicAdd(bad, cnt);
}

__global__ void nv_from_canonical_kernel(const uint8_t *__restrict__ nib,
                                         const uint8_t *__restrict__ scc, Geom G,
                                         uint8_t *__restrict__ w_out,
                                         uint8_t *__restrict__ sc_out) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= G.MT * G.KU * 32) return;
  const int lane = int(idx & 31);
  const int64_t u = (idx >> 5) % G.KU, mt = (idx >> 5) / G.KU;
  const int g = lane >> 2, t = lane & 3;
  const int64_t k0 = u * kUnitK + 16 * t;
  uint32_t words[4] = {0, 0, 0, 0};
  for (int ri = 0; ri < 2; ++ri) {
    const int64_t row = mt * kTileRows + g + 8 * ri;
    uint32_t code = 0;
    if (row < G.M && k0 < G.K) {
      code = scc[row * (G.K / 16) + k0 / 16];
      if (code != 0) {
        const uint2 c2 = *reinterpret_cast<const uint2 *>(nib + row * (G.K / 2) + k0 / 2);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint32_t c = ((kk < 8 ? c2.x : c2.y) >> (4 * (kk & 7))) & 15u;
          words[kk >> 2] |= nv_place(c, ri, kk & 3);
        }
      }
    }
    sc_out[scale_offset(mt, u / kNvChunkUnits, G.MT, G.KC, G.rt) + lane * kNvScaleLaneBytes +
           (u % kNvChunkUnits) * 2 + ri] = uint8_t(scale_code_from_e4m3(code));
  }
  *reinterpret_cast<uint4 *>(w_out + code_offset(mt, u, G.MT, G.KU, kNvChunkUnits, kNvUnitBytes, G.rt) +
                             lane * 16) =
      make_uint4(words[0], words[1], words[2], words[3]);
}

// ------------------------------------------------------------ FP8 packing

// With W2 set, a gated pair as in nv_pack_kernel: tile row g + 8 comes from
// W2 with row scales rs2.
__global__ void f8_pack_kernel(const float *__restrict__ W, const float *__restrict__ rs, Geom G,
                               uint8_t *__restrict__ w_out, const float *__restrict__ W2 = nullptr,
                               const float *__restrict__ rs2 = nullptr) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= G.MT * G.KU * 32) return;
  const int lane = int(idx & 31);
  const int64_t u = (idx >> 5) % G.KU, mt = (idx >> 5) / G.KU;
  const int g = lane >> 2, t = lane & 3;
  const int64_t k0 = u * kUnitK + 16 * t;
  uint8_t out[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) out[i] = 0;
  for (int ri = 0; ri < 2; ++ri) {
    const int64_t row = mt * kTileRows + g + 8 * ri;
    if (row >= G.M || k0 >= G.K) continue;
    const int64_t srow = W2 ? mt * 8 + g : row;
    const float s = (W2 && ri ? rs2 : rs)[srow];
    const float *w = (W2 && ri ? W2 : W) + srow * G.K + k0;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const uint32_t c = s == 0.0f ? 0u : e4m3_rn_sat(__fdiv_rn(w[kk], s));
      out[f8_byte(ri, kk >> 2, kk & 3)] = uint8_t(c);
    }
  }
  uint4 *dst = reinterpret_cast<uint4 *>(
      w_out + code_offset(mt, u, G.MT, G.KU, kF8ChunkUnits, kF8UnitBytes, G.rt) + lane * 32);
  dst[0] = *reinterpret_cast<const uint4 *>(out);
  dst[1] = *reinterpret_cast<const uint4 *>(out + 16);
}

__global__ void f8_unpack_kernel(const uint8_t *__restrict__ w, Geom G, uint8_t *__restrict__ q) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= G.MT * G.KU * 32) return;
  const int lane = int(idx & 31);
  const int64_t u = (idx >> 5) % G.KU, mt = (idx >> 5) / G.KU;
  const int g = lane >> 2, t = lane & 3;
  const int64_t k0 = u * kUnitK + 16 * t;
  if (k0 >= G.K) return;
  uint8_t in[32];
  const uint4 *src = reinterpret_cast<const uint4 *>(
      w + code_offset(mt, u, G.MT, G.KU, kF8ChunkUnits, kF8UnitBytes, G.rt) + lane * 32);
  *reinterpret_cast<uint4 *>(in) = src[0];
  *reinterpret_cast<uint4 *>(in + 16) = src[1];
  for (int ri = 0; ri < 2; ++ri) {
    const int64_t row = mt * kTileRows + g + 8 * ri;
    if (row >= G.M) continue;
    uint8_t o[16];
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) o[kk] = in[f8_byte(ri, kk >> 2, kk & 3)];
    *reinterpret_cast<uint4 *>(q + row * G.K + k0) = *reinterpret_cast<const uint4 *>(o);
  }
}

__global__ void f8_check_canonical_kernel(const uint8_t *__restrict__ q, int64_t n, uint32_t *bad) {
  uint32_t cnt = 0;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    cnt += (q[i] & 0x7Fu) == 0x7Fu;
  cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
  if ((threadIdx.x & 31) == 0 && cnt) atomicAdd(bad, cnt);
}

__global__ void f8_from_canonical_kernel(const uint8_t *__restrict__ q, Geom G,
                                         uint8_t *__restrict__ w_out) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= G.MT * G.KU * 32) return;
  const int lane = int(idx & 31);
  const int64_t u = (idx >> 5) % G.KU, mt = (idx >> 5) / G.KU;
  const int g = lane >> 2, t = lane & 3;
  const int64_t k0 = u * kUnitK + 16 * t;
  uint8_t out[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) out[i] = 0;
  for (int ri = 0; ri < 2; ++ri) {
    const int64_t row = mt * kTileRows + g + 8 * ri;
    if (row >= G.M || k0 >= G.K) continue;
    uint8_t in[16];
    *reinterpret_cast<uint4 *>(in) = *reinterpret_cast<const uint4 *>(q + row * G.K + k0);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) out[f8_byte(ri, kk >> 2, kk & 3)] = in[kk];
  }
  uint4 *dst = reinterpret_cast<uint4 *>(
      w_out + code_offset(mt, u, G.MT, G.KU, kF8ChunkUnits, kF8UnitBytes, G.rt) + lane * 32);
  dst[0] = *reinterpret_cast<const uint4 *>(out);
  dst[1] = *reinterpret_cast<const uint4 *>(out + 16);
}

// ------------------------------------------- MXFP8 and groupwise INT4
// One thread per (tile, unit, lane), as above.  MXFP8 codes sit in the FP8
// layout; a lane with even t also writes the E8M0 bytes of the 32-block its
// 16 columns belong to (rows g and g + 8).  INT4 codes sit in NVFP4 units
// at i4_bitpos (padding codes are 8, the zero); the lane with t == 0 of an
// even unit writes the group's BF16 scales.

// Byte of the MXFP8 scale of (row half ri) for lane (g, t) in unit u of a
// tile-chunk whose scales start at `base`.
__device__ __forceinline__ int64_t mx_scale_at(int64_t base, int g, int t, int64_t u, int ri) {
  return base + (g * 2 + (t >> 1)) * 8 + (u % kF8ChunkUnits) * 2 + ri;
}
// Byte of the INT4 group scale (2 bytes, BF16) of (row half ri) for row
// group g in unit u of a tile-chunk whose scales start at `base`.
__device__ __forceinline__ int64_t i4_scale_at(int64_t base, int g, int64_t u, int ri) {
  return base + g * 16 + ((u % kNvChunkUnits) / 2) * 4 + ri * 2;
}

// floor(log2(amax)) - 8 + 127 from the FP32 exponent field, limited to the
// supported scale bytes; a zero block gets 127.
__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
  if (amax == 0.0f) return 127u;
  const int E = int((__float_as_uint(amax) >> 23) & 0xFFu);   // 0 for subnormal amax
  const int e = E == 0 ? kMxScaleMin : E - 8;
  return uint32_t(min(max(e, kMxScaleMin), kMxScaleMax));
}

__global__ void mx_pack_kernel(const float *__restrict__ W, Geom G, uint8_t *__restrict__ w_out,
                               uint8_t *__restrict__ sc_out) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= G.MT * G.KU * 32) return;
  const int lane = int(idx & 31);
  const int64_t u = (idx >> 5) % G.KU, mt = (idx >> 5) / G.KU;
  const int g = lane >> 2, t = lane & 3;
  const int64_t k0 = u * kUnitK + 16 * t;
  const int64_t sbase = scale_offset(mt, u / kF8ChunkUnits, G.MT, G.KC, G.rt, kMxScaleChunkBytes);
  uint8_t out[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) out[i] = 0;
  for (int ri = 0; ri < 2; ++ri) {
    const int64_t row = mt * kTileRows + g + 8 * ri;
    if (row >= G.M || k0 >= G.K) continue;
    const float *blk = W + row * G.K + (k0 & ~int64_t(31));
    uint32_t bm = 0;
    for (int j = 0; j < 32; ++j) bm = max(bm, abs_bits(blk[j]));
    const uint32_t e = mx_scale_byte(__uint_as_float(bm));
    const float X = __uint_as_float(e << 23);                // 2^(e - 127), exact
    const float *w = W + row * G.K + k0;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk)
      out[f8_byte(ri, kk >> 2, kk & 3)] = uint8_t(e4m3_rn_sat(__fdiv_rn(w[kk], X)));
    if ((t & 1) == 0) sc_out[mx_scale_at(sbase, g, t, u, ri)] = uint8_t(e);
  }
  uint4 *dst = reinterpret_cast<uint4 *>(
      w_out + code_offset(mt, u, G.MT, G.KU, kF8ChunkUnits, kF8UnitBytes, G.rt) + lane * 32);
  dst[0] = *reinterpret_cast<const uint4 *>(out);
  dst[1] = *reinterpret_cast<const uint4 *>(out + 16);
}

__global__ void mx_unpack_kernel(const uint8_t *__restrict__ w, const uint8_t *__restrict__ sc,
                                 Geom G, uint8_t *__restrict__ q, uint8_t *__restrict__ scc) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= G.MT * G.KU * 32) return;
  const int lane = int(idx & 31);
  const int64_t u = (idx >> 5) % G.KU, mt = (idx >> 5) / G.KU;
  const int g = lane >> 2, t = lane & 3;
  const int64_t k0 = u * kUnitK + 16 * t;
  if (k0 >= G.K) return;
  const int64_t sbase = scale_offset(mt, u / kF8ChunkUnits, G.MT, G.KC, G.rt, kMxScaleChunkBytes);
  uint8_t in[32];
  const uint4 *src = reinterpret_cast<const uint4 *>(
      w + code_offset(mt, u, G.MT, G.KU, kF8ChunkUnits, kF8UnitBytes, G.rt) + lane * 32);
  *reinterpret_cast<uint4 *>(in) = src[0];
  *reinterpret_cast<uint4 *>(in + 16) = src[1];
  for (int ri = 0; ri < 2; ++ri) {
    const int64_t row = mt * kTileRows + g + 8 * ri;
    if (row >= G.M) continue;
    uint8_t o[16];
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) o[kk] = in[f8_byte(ri, kk >> 2, kk & 3)];
    *reinterpret_cast<uint4 *>(q + row * G.K + k0) = *reinterpret_cast<const uint4 *>(o);
    if ((t & 1) == 0) scc[row * (G.K / 32) + k0 / 32] = sc[mx_scale_at(sbase, g, t, u, ri)];
  }
}

__global__ void mx_from_canonical_kernel(const uint8_t *__restrict__ q,
                                         const uint8_t *__restrict__ scc, Geom G,
                                         uint8_t *__restrict__ w_out,
                                         uint8_t *__restrict__ sc_out) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= G.MT * G.KU * 32) return;
  const int lane = int(idx & 31);
  const int64_t u = (idx >> 5) % G.KU, mt = (idx >> 5) / G.KU;
  const int g = lane >> 2, t = lane & 3;
  const int64_t k0 = u * kUnitK + 16 * t;
  const int64_t sbase = scale_offset(mt, u / kF8ChunkUnits, G.MT, G.KC, G.rt, kMxScaleChunkBytes);
  uint8_t out[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) out[i] = 0;
  for (int ri = 0; ri < 2; ++ri) {
    const int64_t row = mt * kTileRows + g + 8 * ri;
    if (row >= G.M || k0 >= G.K) continue;
    uint8_t in[16];
    *reinterpret_cast<uint4 *>(in) = *reinterpret_cast<const uint4 *>(q + row * G.K + k0);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) out[f8_byte(ri, kk >> 2, kk & 3)] = in[kk];
    if ((t & 1) == 0) sc_out[mx_scale_at(sbase, g, t, u, ri)] = scc[row * (G.K / 32) + k0 / 32];
  }
  uint4 *dst = reinterpret_cast<uint4 *>(
      w_out + code_offset(mt, u, G.MT, G.KU, kF8ChunkUnits, kF8UnitBytes, G.rt) + lane * 32);
  dst[0] = *reinterpret_cast<const uint4 *>(out);
  dst[1] = *reinterpret_cast<const uint4 *>(out + 16);
}

// Counts E8M0 bytes outside the supported range (in *bad) and NaN codes
// (in bad[1]).
__global__ void mx_check_canonical_kernel(const uint8_t *__restrict__ q, int64_t nq,
                                          const uint8_t *__restrict__ sc, int64_t ns,
                                          uint32_t *bad) {
  uint32_t bs = 0, bq = 0;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < ns; i += stride)
    bs += sc[i] < kMxScaleMin || sc[i] > kMxScaleMax;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < nq; i += stride)
    bq += (q[i] & 0x7Fu) == 0x7Fu;
  bs = __reduce_add_sync(0xFFFFFFFFu, bs);
  bq = __reduce_add_sync(0xFFFFFFFFu, bq);
  if ((threadIdx.x & 31) == 0) {
    if (bs) atomicAdd(bad, bs);
    if (bq) atomicAdd(bad + 1, bq);
  }
}

__global__ void i4_pack_kernel(const float *__restrict__ W, Geom G, uint8_t *__restrict__ w_out,
                               uint8_t *__restrict__ sc_out) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= G.MT * G.KU * 32) return;
  const int lane = int(idx & 31);
  const int64_t u = (idx >> 5) % G.KU, mt = (idx >> 5) / G.KU;
  const int g = lane >> 2, t = lane & 3;
  const int64_t k0 = u * kUnitK + 16 * t;
  const int64_t sbase = scale_offset(mt, u / kNvChunkUnits, G.MT, G.KC, G.rt, kI4ScaleChunkBytes);
  uint32_t words[4] = {0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u};
  for (int ri = 0; ri < 2; ++ri) {
    const int64_t row = mt * kTileRows + g + 8 * ri;
    if (row >= G.M || k0 >= G.K) continue;
    const float *grp = W + row * G.K + (k0 & ~int64_t(kI4GroupK - 1));
    uint32_t bm = 0;
    for (int j = 0; j < kI4GroupK; ++j) bm = max(bm, abs_bits(grp[j]));
    const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(__uint_as_float(bm), 7.0f));
    const float sv = __bfloat162float(sb);
    const float *w = W + row * G.K + k0;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      uint32_t c = 8u;
      if (sv != 0.0f) c = uint32_t(int(fminf(fmaxf(rintf(__fdiv_rn(w[kk], sv)), -8.0f), 7.0f)) + 8);
      const int pos = i4_bitpos(ri, kk & 3);
      words[kk >> 2] = (words[kk >> 2] & ~(0xFu << pos)) | (c << pos);
    }
    if (t == 0 && (u & 1) == 0)
      *reinterpret_cast<__nv_bfloat16 *>(sc_out + i4_scale_at(sbase, g, u, ri)) = sb;
  }
  *reinterpret_cast<uint4 *>(w_out + code_offset(mt, u, G.MT, G.KU, kNvChunkUnits, kNvUnitBytes, G.rt) +
                             lane * 16) = make_uint4(words[0], words[1], words[2], words[3]);
}

__global__ void i4_unpack_kernel(const uint8_t *__restrict__ w, const uint8_t *__restrict__ sc,
                                 Geom G, uint8_t *__restrict__ nib, uint16_t *__restrict__ scc) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= G.MT * G.KU * 32) return;
  const int lane = int(idx & 31);
  const int64_t u = (idx >> 5) % G.KU, mt = (idx >> 5) / G.KU;
  const int g = lane >> 2, t = lane & 3;
  const int64_t k0 = u * kUnitK + 16 * t;
  if (k0 >= G.K) return;
  const int64_t sbase = scale_offset(mt, u / kNvChunkUnits, G.MT, G.KC, G.rt, kI4ScaleChunkBytes);
  const uint4 v = *reinterpret_cast<const uint4 *>(
      w + code_offset(mt, u, G.MT, G.KU, kNvChunkUnits, kNvUnitBytes, G.rt) + lane * 16);
  const uint32_t words[4] = {v.x, v.y, v.z, v.w};
  for (int ri = 0; ri < 2; ++ri) {
    const int64_t row = mt * kTileRows + g + 8 * ri;
    if (row >= G.M) continue;
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const uint32_t c = (words[kk >> 2] >> i4_bitpos(ri, kk & 3)) & 15u;
      if (kk < 8)
        lo |= c << (4 * kk);
      else
        hi |= c << (4 * (kk - 8));
    }
    *reinterpret_cast<uint2 *>(nib + row * (G.K / 2) + k0 / 2) = make_uint2(lo, hi);
    if (t == 0 && (u & 1) == 0)
      scc[row * (G.K / kI4GroupK) + k0 / kI4GroupK] =
          *reinterpret_cast<const uint16_t *>(sc + i4_scale_at(sbase, g, u, ri));
  }
}

__global__ void i4_from_canonical_kernel(const uint8_t *__restrict__ nib,
                                         const uint16_t *__restrict__ scc, Geom G,
                                         uint8_t *__restrict__ w_out,
                                         uint8_t *__restrict__ sc_out) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= G.MT * G.KU * 32) return;
  const int lane = int(idx & 31);
  const int64_t u = (idx >> 5) % G.KU, mt = (idx >> 5) / G.KU;
  const int g = lane >> 2, t = lane & 3;
  const int64_t k0 = u * kUnitK + 16 * t;
  const int64_t sbase = scale_offset(mt, u / kNvChunkUnits, G.MT, G.KC, G.rt, kI4ScaleChunkBytes);
  uint32_t words[4] = {0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u};
  for (int ri = 0; ri < 2; ++ri) {
    const int64_t row = mt * kTileRows + g + 8 * ri;
    if (row >= G.M || k0 >= G.K) continue;
    const uint2 c2 = *reinterpret_cast<const uint2 *>(nib + row * (G.K / 2) + k0 / 2);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const uint32_t c = ((kk < 8 ? c2.x : c2.y) >> (4 * (kk & 7))) & 15u;
      const int pos = i4_bitpos(ri, kk & 3);
      words[kk >> 2] = (words[kk >> 2] & ~(0xFu << pos)) | (c << pos);
    }
    if (t == 0 && (u & 1) == 0)
      *reinterpret_cast<uint16_t *>(sc_out + i4_scale_at(sbase, g, u, ri)) =
          scc[row * (G.K / kI4GroupK) + k0 / kI4GroupK];
  }
  *reinterpret_cast<uint4 *>(w_out + code_offset(mt, u, G.MT, G.KU, kNvChunkUnits, kNvUnitBytes, G.rt) +
                             lane * 16) = make_uint4(words[0], words[1], words[2], words[3]);
}

// Counts BF16 scales that are Inf or NaN.
__global__ void i4_check_canonical_kernel(const uint16_t *__restrict__ sc, int64_t n,
                                          uint32_t *bad) {
  uint32_t cnt = 0;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    cnt += (sc[i] & 0x7F80u) == 0x7F80u;
  cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
  if ((threadIdx.x & 31) == 0 && cnt) atomicAdd(bad, cnt);
}

inline unsigned blocks_for(int64_t threads, int per_block) {
  return unsigned(ceil_div(threads, per_block));
}

// Grid of a grid-stride reduction: enough blocks to fill the device.
inline unsigned reduce_blocks(int64_t n) {
  return unsigned(n / 256 < 4096 ? (n / 256 > 0 ? n / 256 : 1) : 4096);
}

}  // namespace
}  // namespace vg

using namespace vg;

// ===================================================================== ABI

extern "C" vg_status vg_nvfp4_sizes(int64_t M, int64_t K, size_t *w_bytes, size_t *scale_bytes) {
  if (vg_status s = check_mk(M, K)) return s;
  const Geom G = nv_geom(M, K);
  if (w_bytes) *w_bytes = size_t(G.MT * G.KU * kNvUnitBytes);
  if (scale_bytes) *scale_bytes = size_t(G.MT * G.KC * kNvScaleChunkBytes);
  return VG_OK;
}

extern "C" vg_status vg_fp8_sizes(int64_t M, int64_t K, size_t *w_bytes) {
  if (vg_status s = check_mk(M, K)) return s;
  const Geom G = f8_geom(M, K);
  if (w_bytes) *w_bytes = size_t(G.MT * G.KU * kF8UnitBytes);
  return VG_OK;
}

extern "C" vg_status vg_nvfp4_pack(const float *W, int64_t M, int64_t K, void *w_out,
                                   void *scales_out, float *gscale_out, vg_stream_t stream) {
  if (vg_status s = check_mk(M, K)) return s;
  if (!W || !w_out || !scales_out || !gscale_out) return VG_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(w_out) || !aligned16(scales_out)) return VG_ERR_ALIGNMENT;
  cudaStream_t st = as_cuda(stream);
  const Geom G = nv_geom(M, K);
  uint32_t *amax_dev = static_cast<uint32_t *>(scales_out);   // scratch, rewritten below
  VG_CUDA(cudaMemsetAsync(amax_dev, 0, sizeof(uint32_t), st));
  amax_kernel<<<reduce_blocks(M * K), 256, 0, st>>>(W, M * K, amax_dev);
  VG_LAUNCH_CHECK();
  uint32_t amax_bits = 0;
  VG_CUDA(cudaMemcpyAsync(&amax_bits, amax_dev, sizeof amax_bits, cudaMemcpyDeviceToHost, st));
  VG_CUDA(cudaStreamSynchronize(st));
  if (amax_bits >= 0x7F800000u) return VG_ERR_INVALID_ARG;
  float amax;
  std::memcpy(&amax, &amax_bits, sizeof amax);
  const float gs = amax / 2688.0f;                     // 6 * 448, IEEE division
  VG_CUDA(cudaMemsetAsync(scales_out, 0, size_t(G.MT * G.KC * kNvScaleChunkBytes), st));
  const int64_t threads = G.MT * G.KU * 32;
  nv_pack_kernel<<<blocks_for(threads, 256), 256, 0, st>>>(
      W, G, gs, static_cast<uint8_t *>(w_out), static_cast<uint8_t *>(scales_out));
  VG_LAUNCH_CHECK();
  *gscale_out = gs;
  return VG_OK;
}

extern "C" vg_status vg_fp8_pack(const float *W, int64_t M, int64_t K, void *w_out,
                                 float *rowscale_out, vg_stream_t stream) {
  if (vg_status s = check_mk(M, K)) return s;
  if (!W || !w_out || !rowscale_out) return VG_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(w_out) || !aligned16(rowscale_out)) return VG_ERR_ALIGNMENT;
  cudaStream_t st = as_cuda(stream);
  const Geom G = f8_geom(M, K);
  f8_rowscale_kernel<<<blocks_for(M, 8), 256, 0, st>>>(W, M, K, rowscale_out);
  VG_LAUNCH_CHECK();
  std::vector<float> rs(static_cast<size_t>(M));
  VG_CUDA(cudaMemcpyAsync(rs.data(), rowscale_out, sizeof(float) * size_t(M),
                          cudaMemcpyDeviceToHost, st));
  VG_CUDA(cudaStreamSynchronize(st));
  for (float v : rs)
    if (!(v <= 3.4028234663852886e38f)) return VG_ERR_INVALID_ARG;   // NaN or Inf
  const int64_t threads = G.MT * G.KU * 32;
  f8_pack_kernel<<<blocks_for(threads, 256), 256, 0, st>>>(W, rowscale_out, G,
                                                           static_cast<uint8_t *>(w_out));
  VG_LAUNCH_CHECK();
  return VG_OK;
}

extern "C" vg_status vg_nvfp4_unpack(const void *w, const void *scales, int64_t M, int64_t K,
                                     uint8_t *nib_out, uint8_t *sc_out, vg_stream_t stream) {
  if (vg_status s = check_mk(M, K)) return s;
  if (!w || !scales || !nib_out || !sc_out) return VG_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(scales) || !aligned16(nib_out) || !aligned16(sc_out))
    return VG_ERR_ALIGNMENT;
  const Geom G = nv_geom(M, K);
  const int64_t threads = G.MT * G.KU * 32;
  nv_unpack_kernel<<<blocks_for(threads, 256), 256, 0, as_cuda(stream)>>>(
      static_cast<const uint8_t *>(w), static_cast<const uint8_t *>(scales), G, nib_out, sc_out);
  VG_LAUNCH_CHECK();
  return VG_OK;
}

extern "C" vg_status vg_fp8_unpack(const void *w, int64_t M, int64_t K, uint8_t *q_out,
                                   vg_stream_t stream) {
  if (vg_status s = check_mk(M, K)) return s;
  if (!w || !q_out) return VG_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(q_out)) return VG_ERR_ALIGNMENT;
  const Geom G = f8_geom(M, K);
  const int64_t threads = G.MT * G.KU * 32;
  f8_unpack_kernel<<<blocks_for(threads, 256), 256, 0, as_cuda(stream)>>>(
      static_cast<const uint8_t *>(w), G, q_out);
  VG_LAUNCH_CHECK();
  return VG_OK;
}

extern "C" vg_status vg_nvfp4_from_canonical(const uint8_t *nib, const uint8_t *sc, int64_t M,
                                             int64_t K, void *w_out, void *scales_out,
                                             vg_stream_t stream) {
  if (vg_status s = check_mk(M, K)) return s;
  if (!nib || !sc || !w_out || !scales_out) return VG_ERR_INVALID_ARG;
  if (!aligned16(nib) || !aligned16(sc) || !aligned16(w_out) || !aligned16(scales_out))
    return VG_ERR_ALIGNMENT;
  cudaStream_t st = as_cuda(stream);
  const Geom G = nv_geom(M, K);
  uint32_t *bad_dev = static_cast<uint32_t *>(scales_out);   // scratch, rewritten below
  VG_CUDA(cudaMemsetAsync(bad_dev, 0, sizeof(uint32_t), st));
  nv_check_canonical_kernel<<<reduce_blocks(M * K / 16), 256, 0, st>>>(sc, M * (K / 16), bad_dev);
  VG_LAUNCH_CHECK();
  uint32_t bad = 0;
  VG_CUDA(cudaMemcpyAsync(&bad, bad_dev, sizeof bad, cudaMemcpyDeviceToHost, st));
  VG_CUDA(cudaStreamSynchronize(st));
  if (bad) return VG_ERR_INVALID_ARG;
  VG_CUDA(cudaMemsetAsync(scales_out, 0, size_t(G.MT * G.KC * kNvScaleChunkBytes), st));
  const int64_t threads = G.MT * G.KU * 32;
  nv_from_canonical_kernel<<<blocks_for(threads, 256), 256, 0, st>>>(
      nib, sc, G, static_cast<uint8_t *>(w_out), static_cast<uint8_t *>(scales_out));
  VG_LAUNCH_CHECK();
  return VG_OK;
}

extern "C" vg_status vg_fp8_from_canonical(const uint8_t *q, int64_t M, int64_t K, void *w_out,
                                           vg_stream_t stream) {
  if (vg_status s = check_mk(M, K)) return s;
  if (!q || !w_out) return VG_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(w_out)) return VG_ERR_ALIGNMENT;
  cudaStream_t st = as_cuda(stream);
  const Geom G = f8_geom(M, K);
  uint32_t *bad_dev = static_cast<uint32_t *>(w_out);   // scratch, rewritten below
  VG_CUDA(cudaMemsetAsync(bad_dev, 0, sizeof(uint32_t), st));
  f8_check_canonical_kernel<<<reduce_blocks(M * K), 256, 0, st>>>(q, M * K, bad_dev);
  VG_LAUNCH_CHECK();
  uint32_t bad = 0;
  VG_CUDA(cudaMemcpyAsync(&bad, bad_dev, sizeof bad, cudaMemcpyDeviceToHost, st));
  VG_CUDA(cudaStreamSynchronize(st));
  if (bad) return VG_ERR_INVALID_ARG;
  const int64_t threads = G.MT * G.KU * 32;
  f8_from_canonical_kernel<<<blocks_for(threads, 256), 256, 0, st>>>(
      q, G, static_cast<uint8_t *>(w_out));
  VG_LAUNCH_CHECK();
  return VG_OK;
}

// The row-scaled FP8 quantiser and its unpack under the names the boundary
// lists for them (the format is FP8-E4M3 with one FP32 scale per row);
// vg_fp8_pack / vg_fp8_unpack are the same functions.
extern "C" vg_status vg_fp8_rowscale_pack(const float *W, int64_t M, int64_t K, void *w_out,
                                          float *rowscale_out, vg_stream_t stream) {
  return vg_fp8_pack(W, M, K, w_out, rowscale_out, stream);
}

extern "C" vg_status vg_fp8_rowscale_unpack(const void *w, int64_t M, int64_t K, uint8_t *q_out,
                                            vg_stream_t stream) {
  return vg_fp8_unpack(w, M, K, q_out, stream);
}

// ------------------------------------------------------------ gated pairs

namespace {
// Tensor scale of one FP32 matrix (amax / 2688), through a word of device
// scratch; synchronises.
vg_status nv_tensor_scale(const float *W, int64_t n, uint32_t *scratch, cudaStream_t st,
                          float *gs) {
  VG_CUDA(cudaMemsetAsync(scratch, 0, sizeof(uint32_t), st));
  amax_kernel<<<reduce_blocks(n), 256, 0, st>>>(W, n, scratch);
  VG_LAUNCH_CHECK();
  uint32_t bits = 0;
  VG_CUDA(cudaMemcpyAsync(&bits, scratch, sizeof bits, cudaMemcpyDeviceToHost, st));
  VG_CUDA(cudaStreamSynchronize(st));
  if (bits >= 0x7F800000u) return VG_ERR_INVALID_ARG;
  float amax;
  std::memcpy(&amax, &bits, sizeof amax);
  *gs = amax / 2688.0f;
  return VG_OK;
}
}  // namespace

extern "C" vg_status vg_nvfp4_pack_gated(const float *Wgate, const float *Wup, int64_t I,
                                         int64_t K, void *w_out, void *scales_out,
                                         float *gscales_out, vg_stream_t stream) {
  if (I % 8 != 0) return VG_ERR_INVALID_ARG;
  if (vg_status s = check_mk(2 * I, K)) return s;
  if (!Wgate || !Wup || !w_out || !scales_out || !gscales_out) return VG_ERR_INVALID_ARG;
  if (!aligned16(Wgate) || !aligned16(Wup) || !aligned16(w_out) || !aligned16(scales_out))
    return VG_ERR_ALIGNMENT;
  cudaStream_t st = as_cuda(stream);
  const Geom G = nv_geom(2 * I, K);
  uint32_t *scratch = static_cast<uint32_t *>(scales_out);   // rewritten below
  float gs[2];
  if (vg_status s = nv_tensor_scale(Wgate, I * K, scratch, st, &gs[0])) return s;
  if (vg_status s = nv_tensor_scale(Wup, I * K, scratch, st, &gs[1])) return s;
  VG_CUDA(cudaMemsetAsync(scales_out, 0, size_t(G.MT * G.KC * kNvScaleChunkBytes), st));
  const int64_t threads = G.MT * G.KU * 32;
  nv_pack_kernel<<<blocks_for(threads, 256), 256, 0, st>>>(
      Wgate, G, gs[0], static_cast<uint8_t *>(w_out), static_cast<uint8_t *>(scales_out), Wup,
      gs[1]);
  VG_LAUNCH_CHECK();
  gscales_out[0] = gs[0];
  gscales_out[1] = gs[1];
  return VG_OK;
}

extern "C" vg_status vg_fp8_pack_gated(const float *Wgate, const float *Wup, int64_t I, int64_t K,
                                       void *w_out, float *rs_gate_out, float *rs_up_out,
                                       vg_stream_t stream) {
  if (I % 8 != 0) return VG_ERR_INVALID_ARG;
  if (vg_status s = check_mk(2 * I, K)) return s;
  if (!Wgate || !Wup || !w_out || !rs_gate_out || !rs_up_out) return VG_ERR_INVALID_ARG;
  if (!aligned16(Wgate) || !aligned16(Wup) || !aligned16(w_out) || !aligned16(rs_gate_out) ||
      !aligned16(rs_up_out))
    return VG_ERR_ALIGNMENT;
  cudaStream_t st = as_cuda(stream);
  const Geom G = f8_geom(2 * I, K);
  f8_rowscale_kernel<<<blocks_for(I, 8), 256, 0, st>>>(Wgate, I, K, rs_gate_out);
  VG_LAUNCH_CHECK();
  f8_rowscale_kernel<<<blocks_for(I, 8), 256, 0, st>>>(Wup, I, K, rs_up_out);
  VG_LAUNCH_CHECK();
  std::vector<float> rs(static_cast<size_t>(2 * I));
  VG_CUDA(cudaMemcpyAsync(rs.data(), rs_gate_out, sizeof(float) * size_t(I),
                          cudaMemcpyDeviceToHost, st));
  VG_CUDA(cudaMemcpyAsync(rs.data() + I, rs_up_out, sizeof(float) * size_t(I),
                          cudaMemcpyDeviceToHost, st));
  VG_CUDA(cudaStreamSynchronize(st));
  for (float v : rs)
    if (!(v <= 3.4028234663852886e38f)) return VG_ERR_INVALID_ARG;   // NaN or Inf
  const int64_t threads = G.MT * G.KU * 32;
  f8_pack_kernel<<<blocks_for(threads, 256), 256, 0, st>>>(
      Wgate, rs_gate_out, G, static_cast<uint8_t *>(w_out), Wup, rs_up_out);
  VG_LAUNCH_CHECK();
  return VG_OK;
}

// ------------------------------------------- MXFP8 and groupwise INT4

namespace {
inline Geom block_geom(int fmt, int64_t M, int64_t K) {
  return fmt == VG_FMT_MXFP8 ? f8_geom(M, K) : nv_geom(M, K);
}
inline size_t block_scale_bytes(const Geom &G) { return size_t(G.MT * G.KC * 128); }

vg_status block_args(int fmt, int64_t M, int64_t K, const void *a, const void *b, const void *c,
                     const void *d) {
  if (vg_status s = check_mk(M, K)) return s;
  if (!a || !b || !c || !d) return VG_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || !aligned16(c) || !aligned16(d)) return VG_ERR_ALIGNMENT;
  if (fmt == VG_FMT_MXFP8 && K % (kF8ChunkUnits * kUnitK) != 0) return VG_ERR_UNSUPPORTED;
  if (fmt == VG_FMT_INT4G && K % (kNvChunkUnits * kUnitK) != 0) return VG_ERR_UNSUPPORTED;
  return VG_OK;
}

// Largest |W| through a word of device scratch; NaN/Inf -> VG_ERR_INVALID_ARG.
vg_status check_finite(const float *W, int64_t n, uint32_t *scratch, cudaStream_t st) {
  VG_CUDA(cudaMemsetAsync(scratch, 0, sizeof(uint32_t), st));
  amax_kernel<<<reduce_blocks(n), 256, 0, st>>>(W, n, scratch);
  VG_LAUNCH_CHECK();
  uint32_t bits = 0;
  VG_CUDA(cudaMemcpyAsync(&bits, scratch, sizeof bits, cudaMemcpyDeviceToHost, st));
  VG_CUDA(cudaStreamSynchronize(st));
  return bits >= 0x7F800000u ? VG_ERR_INVALID_ARG : VG_OK;
}

vg_status block_pack(int fmt, const float *W, int64_t M, int64_t K, void *w_out, void *scales_out,
                     vg_stream_t stream) {
  if (vg_status s = block_args(fmt, M, K, W, w_out, scales_out, W)) return s;
  cudaStream_t st = as_cuda(stream);
  const Geom G = block_geom(fmt, M, K);
  if (vg_status s = check_finite(W, M * K, static_cast<uint32_t *>(scales_out), st)) return s;
  VG_CUDA(cudaMemsetAsync(scales_out, 0, block_scale_bytes(G), st));
  const int64_t threads = G.MT * G.KU * 32;
  if (fmt == VG_FMT_MXFP8)
    mx_pack_kernel<<<blocks_for(threads, 256), 256, 0, st>>>(
        W, G, static_cast<uint8_t *>(w_out), static_cast<uint8_t *>(scales_out));
  else
    i4_pack_kernel<<<blocks_for(threads, 256), 256, 0, st>>>(
        W, G, static_cast<uint8_t *>(w_out), static_cast<uint8_t *>(scales_out));
  VG_LAUNCH_CHECK();
  return VG_OK;
}
}  // namespace

extern "C" vg_status vg_weight_sizes(int format, int64_t M, int64_t K, size_t *w_bytes,
                                     size_t *scale_bytes) {
  if (vg_status s = check_mk(M, K)) return s;
  size_t w = 0, sc = 0;
  switch (format) {
    case VG_FMT_NVFP4: {
      const Geom G = nv_geom(M, K);
      w = size_t(G.MT * G.KU * kNvUnitBytes);
      sc = size_t(G.MT * G.KC * kNvScaleChunkBytes);
      break;
    }
    case VG_FMT_FP8_ROWSCALE: {
      const Geom G = f8_geom(M, K);
      w = size_t(G.MT * G.KU * kF8UnitBytes);
      break;
    }
    case VG_FMT_MXFP8: {
      const Geom G = f8_geom(M, K);
      w = size_t(G.MT * G.KU * kF8UnitBytes);
      sc = block_scale_bytes(G);
      break;
    }
    case VG_FMT_INT4G: {
      const Geom G = nv_geom(M, K);
      w = size_t(G.MT * G.KU * kNvUnitBytes);
      sc = block_scale_bytes(G);
      break;
    }
    default:
      return VG_ERR_INVALID_ARG;
  }
  if (w_bytes) *w_bytes = w;
  if (scale_bytes) *scale_bytes = sc;
  return VG_OK;
}

extern "C" vg_status vg_mxfp8_pack(const float *W, int64_t M, int64_t K, void *w_out,
                                   void *scales_out, vg_stream_t stream) {
  return block_pack(VG_FMT_MXFP8, W, M, K, w_out, scales_out, stream);
}

extern "C" vg_status vg_int4g_pack(const float *W, int64_t M, int64_t K, void *w_out,
                                   void *scales_out, vg_stream_t stream) {
  return block_pack(VG_FMT_INT4G, W, M, K, w_out, scales_out, stream);
}

extern "C" vg_status vg_mxfp8_unpack(const void *w, const void *scales, int64_t M, int64_t K,
                                     uint8_t *q_out, uint8_t *sc_out, vg_stream_t stream) {
  if (vg_status s = block_args(VG_FMT_MXFP8, M, K, w, scales, q_out, sc_out)) return s;
  const Geom G = f8_geom(M, K);
  const int64_t threads = G.MT * G.KU * 32;
  mx_unpack_kernel<<<blocks_for(threads, 256), 256, 0, as_cuda(stream)>>>(
      static_cast<const uint8_t *>(w), static_cast<const uint8_t *>(scales), G, q_out, sc_out);
  VG_LAUNCH_CHECK();
  return VG_OK;
}

extern "C" vg_status vg_int4g_unpack(const void *w, const void *scales, int64_t M, int64_t K,
                                     uint8_t *nib_out, uint16_t *sc_out, vg_stream_t stream) {
  if (vg_status s = block_args(VG_FMT_INT4G, M, K, w, scales, nib_out, sc_out)) return s;
  const Geom G = nv_geom(M, K);
  const int64_t threads = G.MT * G.KU * 32;
  i4_unpack_kernel<<<blocks_for(threads, 256), 256, 0, as_cuda(stream)>>>(
      static_cast<const uint8_t *>(w), static_cast<const uint8_t *>(scales), G, nib_out, sc_out);
  VG_LAUNCH_CHECK();
  return VG_OK;
}

extern "C" vg_status vg_mxfp8_from_canonical(const uint8_t *q, const uint8_t *sc, int64_t M,
                                             int64_t K, void *w_out, void *scales_out,
                                             vg_stream_t stream) {
  if (vg_status s = block_args(VG_FMT_MXFP8, M, K, q, sc, w_out, scales_out)) return s;
  cudaStream_t st = as_cuda(stream);
  const Geom G = f8_geom(M, K);
  uint32_t *bad = static_cast<uint32_t *>(scales_out);   // scratch, rewritten below
  VG_CUDA(cudaMemsetAsync(bad, 0, 2 * sizeof(uint32_t), st));
  mx_check_canonical_kernel<<<reduce_blocks(M * K), 256, 0, st>>>(q, M * K, sc, M * (K / 32), bad);
  VG_LAUNCH_CHECK();
  uint32_t nbad[2] = {0, 0};
  VG_CUDA(cudaMemcpyAsync(nbad, bad, sizeof nbad, cudaMemcpyDeviceToHost, st));
  VG_CUDA(cudaStreamSynchronize(st));
  if (nbad[1]) return VG_ERR_INVALID_ARG;
  if (nbad[0]) return VG_ERR_UNSUPPORTED;
  VG_CUDA(cudaMemsetAsync(scales_out, 0, block_scale_bytes(G), st));
  const int64_t threads = G.MT * G.KU * 32;
  mx_from_canonical_kernel<<<blocks_for(threads, 256), 256, 0, st>>>(
      q, sc, G, static_cast<uint8_t *>(w_out), static_cast<uint8_t *>(scales_out));
  VG_LAUNCH_CHECK();
  return VG_OK;
}

extern "C" vg_status vg_int4g_from_canonical(const uint8_t *nib, const uint16_t *sc, int64_t M,
                                             int64_t K, void *w_out, void *scales_out,
                                             vg_stream_t stream) {
  if (vg_status s = block_args(VG_FMT_INT4G, M, K, nib, sc, w_out, scales_out)) return s;
  cudaStream_t st = as_cuda(stream);
  const Geom G = nv_geom(M, K);
  uint32_t *bad = static_cast<uint32_t *>(scales_out);   // scratch, rewritten below
  VG_CUDA(cudaMemsetAsync(bad, 0, sizeof(uint32_t), st));
  i4_check_canonical_kernel<<<reduce_blocks(M * (K / kI4GroupK)), 256, 0, st>>>(
      sc, M * (K / kI4GroupK), bad);
  VG_LAUNCH_CHECK();
  uint32_t nbad = 0;
  VG_CUDA(cudaMemcpyAsync(&nbad, bad, sizeof nbad, cudaMemcpyDeviceToHost, st));
  VG_CUDA(cudaStreamSynchronize(st));
  if (nbad) return VG_ERR_INVALID_ARG;
  VG_CUDA(cudaMemsetAsync(scales_out, 0, block_scale_bytes(G), st));
  const int64_t threads = G.MT * G.KU * 32;
  i4_from_canonical_kernel<<<blocks_for(threads, 256), 256, 0, st>>>(
      nib, sc, G, static_cast<uint8_t *>(w_out), static_cast<uint8_t *>(scales_out));
  VG_LAUNCH_CHECK();
  return VG_OK;
}
