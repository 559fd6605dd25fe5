// vg_device.cuh -- device-side building blocks shared by the pack and GEMV
// kernels: packed-layout constants, inline PTX for mbarriers, bulk copies,
// BF16 tensor-core MMA and BF16x2 multiplies, and the in-register decode of
// the packed NVFP4, FP8, MXFP8 and INT4 codes.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace vg {

// ---------------------------------------------------------------- layout
// A row tile is 16 rows (the M of one m16n8k16 MMA).  A unit is 64 columns
// of one row tile: 32 lanes x 16 bytes of NVFP4 codes (512 B) or 32 lanes x
// 32 bytes of FP8 codes (1024 B).  Lane l = 4*g + t holds rows g and g+8 of
// the tile at columns 64u + 16t .. 64u + 16t + 15, i.e. exactly one NVFP4
// scale block of each of its two rows.
constexpr int kTileRows = 16;
constexpr int kUnitK = 64;
constexpr int kNvUnitBytes = 512;
constexpr int kF8UnitBytes = 1024;
// A chunk is 8 NVFP4 units (512 columns, 4096 bytes per tile) or 4 FP8
// units (256 columns, 4096 bytes).  NVFP4 block scales: per tile per chunk,
// 32 lanes x 16 bytes: [unit 0..7][row g, row g+8].
#ifndef VG_NV_CHUNK
#define VG_NV_CHUNK 8
#endif
constexpr int kNvChunkUnits = VG_NV_CHUNK;
static_assert(kNvChunkUnits == 4 || kNvChunkUnits == 8, "4- or 8-unit chunks");
constexpr int kNvScaleLaneBytes = 2 * kNvChunkUnits;                    // 16
constexpr int kNvScaleChunkBytes = 32 * kNvScaleLaneBytes;              // 512
constexpr int kF8ChunkUnits = kNvChunkUnits / 2;

// A work item is 16 tile-chunks, one per consumer warp, arranged as rt row
// tiles x (16 / rt) consecutive chunks of each; a row block is rt tiles.
// rt = 16 (one chunk of 16 tiles) suits matrices with many rows.  For
// matrices with few rows, a smaller rt gives more, shorter row blocks, so
// that fewer thread blocks share one row block's K range and its partial
// sums are added in fewer rounds (layout_rt below).  Items stream through a
// ring of kSlots shared-memory slots; one slot holds a whole item: the 16
// tile-chunks' codes (contiguous in the packed buffer), their block scales,
// and the x slice (N rows of the item's columns).
#ifndef VG_WARPS
#define VG_WARPS 16
#endif
#ifndef VG_SLOTS
#define VG_SLOTS 2
#endif
constexpr int kBlockTiles = 16;
constexpr int kWarps = VG_WARPS;
static_assert(kWarps == kBlockTiles, "one tile of the row block per warp");
constexpr int kSlots = VG_SLOTS;
constexpr int kSlotCodeBytes = kNvChunkUnits * kNvUnitBytes;          // 4096: one tile's chunk
constexpr int kThreads = kWarps * 32;
// One x row of a chunk (512 BF16 columns) plus 16 bytes of padding, so that
// the 8 rows read by a quarter warp fall in different banks.  Row-copied x
// only serves items of one chunk (rt = 16).
constexpr int kXRowBytes = kNvChunkUnits * kUnitK * 2 + 16;             // 1040
// Units (64 columns each) of x one item may span: the tensor-copied slice is
// 8 rows x 128 bytes per unit, 32 KB at most.
constexpr int kMaxItemUnits = 32;
// An item slot: codes of 16 tile-chunks, then their scales, then the x
// slice: 8 rows, either padded rows of kXRowBytes (copied row by row) or one
// tensor copy in the 128-byte-swizzled layout [unit][row][128 B], which
// needs 1024-byte alignment (slots are multiples of 1024 bytes).
constexpr int kItemScaleOff = kBlockTiles * kSlotCodeBytes;            // 65536
constexpr int kItemXOff = kItemScaleOff + kBlockTiles * kNvScaleChunkBytes;  // 73728
constexpr int kItemXBytes =
    kMaxItemUnits * 1024 > 8 * kXRowBytes ? kMaxItemUnits * 1024 : 8 * kXRowBytes;
constexpr int kItemSlotBytes = (kItemXOff + kItemXBytes + 1023) / 1024 * 1024;  // 106496
static_assert(kItemXOff % 1024 == 0, "the swizzled x slice starts 1024-byte aligned");

static_assert(kF8ChunkUnits * kF8UnitBytes == kSlotCodeBytes,
              "an FP8 chunk has the bytes of an NVFP4 chunk");

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Row tiles per row block of an M x K matrix with cu units per chunk.  The
// work of one verify group is split over all SMs in contiguous item ranges,
// so a row block of KC / (16 / rt) items is shared by about
// rt * SMs / MT thread blocks.  The largest rt (fewest pieces per block) that
// keeps that at 3 or less is taken; if none does, the smallest allowed.  An
// rt below 16 is allowed only when every item is whole: K a multiple of the
// chunk, the item's chunks dividing KC, and its x slice within
// kMaxItemUnits.  The choice depends on (M, K, cu) alone, so the packers and
// the GEMV agree on it; kLayoutSMs is the SM count it is tuned for (any
// device runs any layout).
constexpr int kLayoutSMs = 152;
__host__ __device__ inline int layout_rt(int64_t M, int64_t K, int cu) {
  const int64_t chunk_cols = int64_t(cu) * kUnitK;
  if (K % chunk_cols != 0) return kBlockTiles;
  const int64_t KC = K / chunk_cols, MT = ceil_div(M, kTileRows);
  int smallest = kBlockTiles;
  for (int rt = kBlockTiles; rt >= 2; rt /= 2) {
    const int cpi = kBlockTiles / rt;
    if (KC % cpi != 0 || cpi * cu > kMaxItemUnits) continue;
    if (int64_t(rt) * kLayoutSMs <= 3 * MT) return rt;
    smallest = rt;
  }
  return smallest;
}

// Item-contiguous order of the packed buffers.  Codes are grouped by row
// block (rt tiles), then by item (16 / rt consecutive chunks of cu units),
// then by tile-chunk (tile-major: tile, then chunk), then by unit, so that
// one work item is one contiguous run of bytes and consecutive items of a
// row block follow each other.  Only the last row block may have fewer than
// rt tiles and, with rt = 16, only the last chunk fewer than cu units;
// nothing is padded.
__host__ __device__ inline int64_t code_offset(int64_t mt, int64_t u, int64_t MT, int64_t KU,
                                               int64_t cu, int64_t ub, int64_t rt) {
  const int64_t cpi = kBlockTiles / rt, iu = cpi * cu;   // chunks, units per item
  const int64_t rb = mt / rt, tl = mt % rt, c = u / cu, uu = u % cu, ci = c / cpi, cc = c % cpi;
  const int64_t tiles = (MT - rb * rt) < rt ? (MT - rb * rt) : rt;
  const int64_t nui = (KU - ci * iu) < iu ? (KU - ci * iu) : iu;  // a tail only when cpi == 1
  return rb * rt * KU * ub + ci * tiles * iu * ub + (tl * cpi + cc) * (nui / cpi) * ub + uu * ub;
}
// Byte offset of the scales of chunk c of tile mt (same grouping; every
// tile-chunk has scb bytes of scales, also a K tail).
__host__ __device__ inline int64_t scale_offset(int64_t mt, int64_t c, int64_t MT, int64_t KC,
                                                int64_t rt, int64_t scb = kNvScaleChunkBytes) {
  const int64_t cpi = kBlockTiles / rt;
  const int64_t rb = mt / rt, tl = mt % rt, ci = c / cpi, cc = c % cpi;
  const int64_t tiles = (MT - rb * rt) < rt ? (MT - rb * rt) : rt;
  return (rb * rt * KC + ci * tiles * cpi + tl * cpi + cc) * scb;
}

// ------------------------------------------------ MXFP8 and groupwise INT4
// MXFP8 codes use the FP8 units and chunks; its E8M0 scales (one per 32
// columns) take 128 bytes per tile-chunk: for each (g, t / 2) eight bytes
// [unit 0..3][row g, row g + 8], the block that lane (g, t) covers in
// each unit.  Groupwise INT4 codes use the NVFP4 units and chunks (4 bits
// per weight) with their own bit placement; its BF16 scales (one per 128
// columns = 2 units) take 128 bytes per tile-chunk: for each g sixteen
// bytes [group 0..3][row g, row g + 8].
constexpr int kMxScaleChunkBytes = 128;
constexpr int kI4ScaleChunkBytes = 128;
constexpr int kI4GroupK = 128;
// MXFP8 scale bytes that give normal BF16 weights in one multiply: the
// decode multiplies the placed FP8 bits (e4m3 * 2^-120) by the BF16 value
// 2^(e - 7), whose exponent field e + 120 must stay below 255.
constexpr int kMxScaleMin = 10, kMxScaleMax = 134;
// INT4 nibble of (row half ri, column ii of an MMA step) in a packed word:
// register r = ri + 2 * (ii >> 1) holds it at bit 4 r of its ii & 1 half.
__host__ __device__ constexpr int i4_bitpos(int ri, int ii) {
  return 4 * (ri + 2 * (ii >> 1)) + 16 * (ii & 1);
}

// ------------------------------------------------------ decode constants
// NVFP4 code bit positions inside a packed 32-bit word.  A word holds the 8
// codes of one MMA (k16 step) for one lane: four BF16x2 A-fragment
// registers R0..R3 (rows g, g+8, g, g+8 x column pairs (0,1), (0,1), (2,3),
// (2,3)); the low half of each register is the first column of its pair.
// Target BF16 bits of a code (m, e0, e1, s) are 6, 7, 8, 15: the value of
// those bits alone is e2m1 * 2^-126 (exponent 0 covers the 0.5 code as a
// BF16 subnormal).  R0 sits at the target bits, R1 three bits lower, R2 six
// bits lower; R3 fills the rest (m 13, e0 14, e1 10, s 11) and is moved by
// one multiply that adds shifted copies without carries.
constexpr uint32_t kNvMask = 0x81C081C0u;
constexpr uint32_t kNvR3Pick = 0x00D800D8u;  // bits 3,4,6,7 (+16) after >> 7
constexpr uint32_t kNvR3Spread = 0x821u;     // x1 (m, e0), x32 (e1), x2048 (s)
// Bit position (low half) of code bit b in {m, e0, e1, s} for register r.
__host__ __device__ constexpr int nv_bitpos(int r, int b) {
  return r == 0 ? (b == 3 ? 15 : 6 + b)
       : r == 1 ? (b == 3 ? 12 : 3 + b)
       : r == 2 ? (b == 3 ? 9 : 0 + b)
       : (b == 0 ? 13 : b == 1 ? 14 : b == 2 ? 10 : 11);
}

// Packed scale code: an 8-bit float with 5 exponent bits and 3 mantissa
// bits whose exponent is the E4M3 exponent + 3, so E4M3 subnormal scales
// become normal numbers.  BF16 bits of (code << 4) + kScaleBias decode to
// scale * 2^118; multiplied by the code bits above (e2m1 * 2^-126) this
// gives e2m1 * scale * 2^-8 exactly.  The epilogue multiplies by 2^8 * gs.
constexpr uint32_t kScaleBias = 235u << 7;   // 0x7580 per half
constexpr uint32_t kScaleBias2 = (kScaleBias << 16) | kScaleBias;
constexpr float kNvEpilogueScale = 256.0f;
// FP8 codes placed into BF16 bits ((b & 0x7f) << 4 | sign << 15) are worth
// e4m3 * 2^-120; one multiply by 2^120 (BF16 0x7B80) restores them.
constexpr uint32_t kF8Restore2 = 0x7B807B80u;

// E4M3 byte (0x00..0x7E) -> packed scale code, and back.
__host__ __device__ inline uint32_t scale_code_from_e4m3(uint32_t b) {
  const uint32_t e = b >> 3, f = b & 7;
  if (e != 0) return b + 24;
  // subnormal f * 2^-9 as exponent-5 codes: f=1..7 -> (1,0) (2,0) (2,4) (3,0) (3,2) (3,4) (3,6)
  constexpr uint8_t sub[8] = {0, 8, 16, 20, 24, 26, 28, 30};
  return sub[f];
}
__host__ __device__ inline uint32_t e4m3_from_scale_code(uint32_t d) {
  if (d >= 32) return d - 24;
  switch (d) {
    case 8: return 1;
    case 16: return 2;
    case 20: return 3;
    case 24: return 4;
    case 26: return 5;
    case 28: return 6;
    case 30: return 7;
    default: return 0;
  }
}

#ifdef __CUDACC__
// ------------------------------------------------------------ small PTX
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// BF16x2 product a*b as a fused multiply-add with a -0 addend (native
// HFMA2 on BF16).  Every product formed here is exact in BF16, and adding
// -0 keeps both the value and the sign of a zero product.
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(0x80008000u));
  return d;
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

// Non-blocking test of a phase (never suspends the thread): for polling
// loops whose lanes diverge, where a suspended lane would hold back others.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: true when the phase with `parity` completed, false when
// `deadline` (globaltimer ns) passed first.
// try_wait that may suspend the thread in hardware until the phase completes
// or about hint_ns nanoseconds pass, issuing nothing meanwhile.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t deadline) {
  if (mbar_try_wait(bar, parity)) return true;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() > deadline) return false;
  }
}

// 1-D bulk copy global -> shared, completing on an mbarrier (tx bytes).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Tensor copy of a 3-D box at coordinates (c0, c1, c2) described by the
// tensor map at `tmap` (param, const or global memory) into shared memory,
// completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_tensor_3d(uint32_t dst, const void *tmap, int c0, int c1,
                                               int c2, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
      : "memory");
}

// Bring `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Read-only 16-byte global load (the HBM probe's vector-load mode).
__device__ __forceinline__ uint4 ldg128(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier generic-proxy accesses of global memory
// (an acquire of data other blocks wrote) before its later async-proxy
// (bulk or tensor copy) accesses of the same memory, and the converse.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// GPU-scope accesses for the cross-block protocol.
__device__ __forceinline__ void red_add_release(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_relaxed(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.relaxed.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Two 64-bit words, each a single-copy-atomic access at GPU scope (a vector
// access is a set of independent scalar accesses, one per element).  Used
// for partial sums that carry their own validity tag in the upper half, so
// that no fence is needed between the data and a flag.
__device__ __forceinline__ void st_relaxed_v2u64(uint64_t *p, uint64_t a, uint64_t b) {
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void ld_relaxed_v2u64(const uint64_t *p, uint64_t &a, uint64_t &b) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ----------------------------------------------------- in-register decode
// Four BF16x2 A-fragment registers of one NVFP4 word, each multiplied by
// the packed scale of its row (fg for rows g, fg8 for rows g+8).  The left
// shifts by 3 and 6 are written as multiplies by m8 = 8 and m64 = 64 held in
// registers, so that they run on the FMA pipe next to the integer logic.
__device__ __forceinline__ uint32_t umul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.lo.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ void nv_decode(uint32_t w, uint32_t fg, uint32_t fg8, uint32_t m8,
                                          uint32_t m64, uint32_t &a0, uint32_t &a1,
                                          uint32_t &a2, uint32_t &a3) {
  const uint32_t r0 = w & kNvMask;
  const uint32_t r1 = umul(w, m8) & kNvMask;
  const uint32_t r2 = umul(w, m64) & kNvMask;
  const uint32_t r3 = umul((w >> 7) & kNvR3Pick, kNvR3Spread) & kNvMask;
  a0 = bmul2(r0, fg);
  a1 = bmul2(r1, fg8);
  a2 = bmul2(r2, fg);
  a3 = bmul2(r3, fg8);
}

// BF16x2 {F, F} of the packed scale byte number `byte` (0..3) of `word`.
__device__ __forceinline__ uint32_t nv_scale_pair(uint32_t word, uint32_t byte) {
  const uint32_t dup = prmt(word, 0u, 0x4040u | (byte * 0x0101u));
  return dup * 16u + kScaleBias2;
}

// BF16x2 {2^(e-7), 2^(e-7)} of the MXFP8 scale byte e number `byte` of
// `word`: exponent field e + 120.
__device__ __forceinline__ uint32_t mx_scale_pair(uint32_t word, uint32_t byte) {
  const uint32_t dup = prmt(word, 0u, 0x4040u | (byte * 0x0101u));
  return dup * 128u + 0x3C003C00u;
}

// Two BF16x2 registers of one MXFP8 word: the FP8 placement, multiplied by
// the block scale of row g (sg) and of row g + 8 (sg8); exact.
__device__ __forceinline__ void mx_decode(uint32_t w, uint32_t sg, uint32_t sg8, uint32_t &ra,
                                          uint32_t &rb) {
  const uint32_t pa = ((w << 4) & 0x07F007F0u) | ((w << 8) & 0x80008000u);
  const uint32_t pb = ((w >> 4) & 0x07F007F0u) | (w & 0x80008000u);
  ra = bmul2(pa, sg);
  rb = bmul2(pb, sg8);
}

// (a + b) on BF16x2 as a fused multiply-add by 1.0 (exact here).
__device__ __forceinline__ uint32_t badd2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(0x3F803F80u), "r"(b));
  return d;
}

// Four BF16x2 A registers of one INT4 word: the nibbles of register r sit at
// bits 4 r and 4 r + 16; OR-ed into 0x4300 (the BF16 128) they give 128 + q,
// and adding -136 gives q - 8, exactly.
__device__ __forceinline__ void i4_decode(uint32_t w, uint32_t &a0, uint32_t &a1, uint32_t &a2,
                                          uint32_t &a3) {
  constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u, kMinus136 = 0xC308C308u;
  a0 = badd2((w & kMask) | kMagic, kMinus136);
  a1 = badd2(((w >> 4) & kMask) | kMagic, kMinus136);
  a2 = badd2(((w >> 8) & kMask) | kMagic, kMinus136);
  a3 = badd2(((w >> 12) & kMask) | kMagic, kMinus136);
}

// Two BF16x2 registers of one FP8 word (bytes 0,2 -> ra; bytes 1,3 -> rb).
__device__ __forceinline__ void f8_decode(uint32_t w, uint32_t &ra, uint32_t &rb) {
  const uint32_t pa = ((w << 4) & 0x07F007F0u) | ((w << 8) & 0x80008000u);
  const uint32_t pb = ((w >> 4) & 0x07F007F0u) | (w & 0x80008000u);
  ra = bmul2(pa, kF8Restore2);
  rb = bmul2(pb, kF8Restore2);
}
#endif  // __CUDACC__

}  // namespace vg
