// vg_gemv.cu -- the weight-streaming GEMV over NVFP4, row-scaled FP8,
// MXFP8 or groupwise-INT4 weights, for N = 1..8 BF16 columns
// (stream_kernel) or 9..32 (stream_kernel_wide), as a single product and as
// a fused, ordered verify pass over a layer stack.  The fused instantiation
// also runs RMS norms, the SiLU-gated epilogue of a gate/up pair and x
// written earlier in the same pass.
//
// What it computes: y[N,M] = x[N,K] . dequant(W)[M,K]^T with FP32
// accumulation (mtp7-device-confidence engine card, Design table, "GEMVs"
// row; the verify pass of the Decode row runs it for 2-8 columns, a draft
// step for one).  Why it is the hot path: a verify pass reads every weight
// once (card, Measured section: 19.26 GB per pass, its time set by the read
// rate), so the kernel is built to stream bytes at HBM speed.
//
// Design (sm_103a):
//  * Persistent thread blocks, one per SM: 16 consumer warps + 2 producer
//    warps.  The producers (one lane each; in a verify pass one per slot,
//    in a single product the first alone) keep a 2-slot ring of shared
//    memory full, one whole work item per slot, guarded by full/empty
//    mbarriers:
//    one bulk copy of the item's codes and one of its scales (contiguous in
//    the packed buffers; L2 evict-first) and one TMA tensor copy of its x
//    slice (128-byte swizzle; L2 evict-last).  The weights never pass through
//    registers of the producer.
//  * A work item is 16 tile-chunks (a chunk is 512 columns NVFP4 and INT4,
//    256 FP8 and MXFP8):
//    one chunk of a row block of 16 tiles, or, for matrices with few rows,
//    16 / rt consecutive chunks of a row block of rt tiles.  Consumer warp w
//    owns tile-chunk w.  It decodes the codes in registers to BF16 A
//    fragments (bit placement + one BF16x2 multiply by the block scale,
//    exact) and runs mma.m16n8k16 with x from the slot as the B fragment,
//    accumulating FP32; the warps that share a tile add their sums in
//    shared memory at the end of a row block's piece.
//  * Items are split between thread blocks stream-K style (contiguous item
//    ranges of equal length), so every SM streams the same number of bytes.
//    A row block whose K range is split between blocks is summed by the
//    block holding its first item (it reaches that piece last) from the
//    others' FP32 partial sums, in block order (deterministic).  Each
//    partial sum travels with a tag of the pass and phase in the same 64-bit
//    word, so a contributor publishes it with plain stores and moves on: no
//    fence, counter or barrier on its path.
//  * Verify pass: matrices are grouped; in ordered mode the consumers of
//    group g wait (bounded) until group g-1 has completed every row block,
//    while the producer keeps filling the ring with group g's items and
//    brings a few more into L2.  All waits are bounded by a timeout on
//    %globaltimer and report an error word instead of hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "vg_device.cuh"
#include "vg_internal.h"

namespace vg {

struct MatDev {
  const uint8_t *w;
  const uint8_t *sc;
  const float *rowscale;
  const uint16_t *x;
  uint16_t *y;
  float mult;        // epilogue multiplier (NVFP4: 256 * gscale)
  int fmt;
  // fused neighbours: flags read at the end of every piece, so kept in the
  // same cache line as the fields read there
  int op;            // VG_OP_GEMV, VG_OP_SWIGLU or VG_OP_RMSNORM (then fmt is kFmtNorm)
  int x_after;       // x is written by the previous phase: copy it after that phase completes
  int y_async;       // y is read by a later phase through copies: fence before releasing it
  int M, K, MT, KU, KC, RB;
  int cu, ub;        // units per chunk, bytes per unit
  int rt, cpi;       // tiles per row block, chunks per item (16 / rt)
  int iu, KI;        // units per item (cpi * cu), items per row block
  int kfull;         // items wholly inside K
  int scb;           // block-scale bytes per tile-chunk (0: none)
  int64_t rb_bytes;  // code bytes of a full row block (rt tiles x KU units)
  int item0;         // first item of this matrix within its phase
  const CUtensorMap *xmap;  // x as [K/64 units][N rows][64 columns], or nullptr
  int Mo;            // rows of y (M, or M / 2 for a gated pair)
  float mult2;       // SWIGLU, NVFP4: epilogue multiplier of the up rows
  const float *rowscale2;  // SWIGLU, FP8: row scales of the up rows
  const uint16_t *gamma;   // RMSNORM weights
  float eps;
};
// Internal format of an RMS-norm item (no weights; one item, no copies).
constexpr int kFmtNorm = 7;

// Item counts fit 32 bits: a matrix has fewer than 2^40 / (256 x 512) items
// and a plan's phase is checked on the host.
struct PhaseDev {
  int items;
  int rbs;
  int mat_begin, mat_end;
};

struct Params {
  CUtensorMap xmap0;        // the single product's x tensor map (if x0_tensor)
  const MatDev *mats;       // nullptr: use mat0 / phase0
  const PhaseDev *phases;
  int nphases;
  int N;                    // columns of x and y (the most a width word may ask for)
  const int *width;         // device word read at launch: the pass's width 1..N (or nullptr)
  int ordered;
  int hold_phase;
  int grid;
  uint64_t timeout_ns;
  int *error;               // first failed wait's code, else 0
  uint32_t *ctas_done;      // blocks finished in this pass (left at 0)
  uint32_t *epoch;          // pass counter: tags partial sums
  uint32_t *done;           // per-phase completed row blocks (ordered only)
  uint64_t *partials;       // [grid][nb * kPartialWords]: tagged FP32 partial sums
  int64_t clear_words;      // 64-bit words cleared when the pass counter wraps: every slot
                            // that any call sharing this workspace may have written
  // (host) column blocks of 8: 1, 2 or 4 (N up to 8, 16, 32).  Kept here: placed
  // where it would pad the descriptors below, it changed the register
  // allocation of the kernels (more spills, slower passes).
  int nb;
  uint32_t m8, m64;         // 8 and 64: shift multipliers kept in registers
  int x0_tensor;
  int fused;                // (host) the pass has fused operations or dependent x
  MatDev mat0;
  PhaseDev phase0;
};

// One block's partial-sum slot: the 128 FP32 sums of each of up to 16 tiles,
// each in a 64-bit word whose upper half is the tag of the pass and phase
// that wrote it.
constexpr int kPartialWords = kBlockTiles * 32 * 4;
// Shared memory: the item ring, one zero x row (read for columns >= N), the
// mbarriers (full, then empty, per slot), a few flags, and the scratch in
// which the warps sharing a tile hand their sums to the first of them.
constexpr int kRingBytes = kSlots * kItemSlotBytes;
// The zero row starts 16 bytes past a 128-byte line, like x row 1 of a slot,
// so that lanes reading it and lanes reading row 0 use different banks.
constexpr int kZeroRowOff = kRingBytes + 16;
constexpr int kBarOff = kZeroRowOff + kXRowBytes;
constexpr int kBarBytes = 2 * kSlots * 8;
constexpr int kRedOff = kBarOff + kBarBytes + 64;
constexpr int kRedBytes = kWarps * 32 * 16;             // 4 FP32 sums per consumer thread
constexpr int kSmemUsed = kRedOff + kRedBytes;
constexpr int kSmemBytes = kSmemUsed + 1024;   // room to align the base to 1024 bytes
static_assert(kBarOff % 8 == 0, "mbarriers are 8-byte aligned");
static_assert(kRedOff % 16 == 0, "the sum scratch is read as 16-byte vectors");
static_assert(kItemSlotBytes % 128 == 0 && kItemXOff % 128 == 0, "x rows start 128-byte aligned");
static_assert(kSmemBytes <= 227 * 1024, "fits one block per SM");
constexpr int kConsumers = kWarps * 32;
// + two producer warps (sub-partitions 0 and 1): in a verify pass each fills
// one ring slot, every other item; a single product uses the first alone
constexpr int kProducers = 2;
// each producer owns whole slots (items of one slot in order): a slot's parity
// waits would alias if two producers took turns on it
static_assert(kSlots % kProducers == 0, "every producer owns its own ring slots");
constexpr int kKernelThreads = kConsumers + 32 * kProducers;
constexpr int kErrFullWait = 1, kErrEmptyWait = 2, kErrDepWait = 3, kErrPartialWait = 4;
constexpr int kErrWidth = 5;   // the width word held a value outside 1..N
// Header words of a workspace (GEMV) or plan state: error, finished blocks,
// pass epoch; then, 256 bytes in, the per-phase counters (plans) and the
// partial-sum slots.
constexpr size_t kWsHead = 256;

__host__ __device__ inline int64_t i64min(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ inline int64_t i64max(int64_t a, int64_t b) { return a > b ? a : b; }

__host__ __device__ inline int item_begin(int T, int G, int b) {
  return int(int64_t(T) * b / G);
}
// Block that owns item i of a phase of T items split over G blocks.
__device__ inline int owner(int T, int G, int i) { return int((int64_t(i + 1) * G - 1) / T); }

__device__ inline void set_error(int *error, int code) { atomicCAS(error, 0, code); }

// Bounded wait with the clock read only after a first miss.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, uint64_t timeout) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait(bar, parity, globaltimer() + timeout);
}

// The items one thread block processes, in order, across all phases: for
// each phase with items for this block, its contiguous range [i, i1).  The
// position inside the current matrix (row block rb, item c) advances
// incrementally; the only divisions happen when a phase starts.  The tables
// and the grid come from the caller, so the sequencer holds only the
// position (it is live across the streaming loops).
struct Seq {
  int ph, mi;
  int rb, c, KI, RB;   // row block, item within it; items per row block, row blocks
  int i, i1, items, G; // item, end of the block's range; the phase's items and blocks
  bool valid;

  __device__ void init(const MatDev *mats, const PhaseDev *phases, const Params &p) {
    ph = -1;
    next_phase(mats, phases, p);
  }
  __device__ void next_phase(const MatDev *mats, const PhaseDev *phases, const Params &p) {
    const int b = int(blockIdx.x);
    for (++ph; ph < p.nphases; ++ph) {
      items = phases[ph].items;
      // as few blocks as keep the largest per-block item count: fewer
      // blocks then share each row block (shorter reductions)
      const int per = (items + p.grid - 1) / p.grid;
      G = (items + per - 1) / per;
      if (b < G) {
        i = item_begin(items, G, b);
        i1 = item_begin(items, G, b + 1);
        mi = phases[ph].mat_begin;
        const int mend = phases[ph].mat_end;
        while (mi + 1 < mend && i >= mats[mi].item0 + mats[mi].RB * mats[mi].KI) ++mi;
        KI = mats[mi].KI;
        RB = mats[mi].RB;
        const int rel = i - mats[mi].item0;
        rb = rel / KI;
        c = rel - rb * KI;
        valid = true;
        return;
      }
    }
    valid = false;
  }
  // Skip the n items left in the current row block's piece (never past the
  // row block's end).
  __device__ __forceinline__ void skip(int n, const MatDev *mats, const PhaseDev *phases,
                                       const Params &p) {
    i += n;
    if (i == i1) {
      next_phase(mats, phases, p);
      return;
    }
    c += n;
    if (c == KI) {
      c = 0;
      if (++rb == RB) {
        rb = 0;
        ++mi;
        KI = mats[mi].KI;
        RB = mats[mi].RB;
      }
    }
  }
  __device__ __forceinline__ void advance(const MatDev *mats, const PhaseDev *phases,
                                          const Params &p) {
    skip(1, mats, phases, p);
  }
};

// MMA steps j = 0..3 of a unit accumulate into acc[j % kAcc]: with kAcc
// accumulators the dependent MMA chains are kAcc times shorter.
#ifndef VG_NACC
#define VG_NACC 1   // one chain measured fastest: 16 warps hide the MMA latency
#endif
constexpr int kAcc = VG_NACC;

// One NVFP4 unit of one tile: 4 MMAs (k16 steps).
__device__ __forceinline__ void nv_unit(const uint4 wv, uint32_t fg, uint32_t fg8, const uint4 xa,
                                        const uint4 xb, uint32_t m8, uint32_t m64,
                                        float (&acc)[kAcc][4]) {
  uint32_t a0, a1, a2, a3;
  nv_decode(wv.x, fg, fg8, m8, m64, a0, a1, a2, a3);
  mma_bf16(acc[0], a0, a1, a2, a3, xa.x, xa.y);
  nv_decode(wv.y, fg, fg8, m8, m64, a0, a1, a2, a3);
  mma_bf16(acc[1 % kAcc], a0, a1, a2, a3, xa.z, xa.w);
  nv_decode(wv.z, fg, fg8, m8, m64, a0, a1, a2, a3);
  mma_bf16(acc[2 % kAcc], a0, a1, a2, a3, xb.x, xb.y);
  nv_decode(wv.w, fg, fg8, m8, m64, a0, a1, a2, a3);
  mma_bf16(acc[3 % kAcc], a0, a1, a2, a3, xb.z, xb.w);
}

__device__ __forceinline__ void f8_unit(const uint4 w0, const uint4 w1, const uint4 xa,
                                        const uint4 xb, float (&acc)[kAcc][4]) {
  uint32_t a0, a1, a2, a3;
  f8_decode(w0.x, a0, a1);
  f8_decode(w0.y, a2, a3);
  mma_bf16(acc[0], a0, a1, a2, a3, xa.x, xa.y);
  f8_decode(w0.z, a0, a1);
  f8_decode(w0.w, a2, a3);
  mma_bf16(acc[1 % kAcc], a0, a1, a2, a3, xa.z, xa.w);
  f8_decode(w1.x, a0, a1);
  f8_decode(w1.y, a2, a3);
  mma_bf16(acc[2 % kAcc], a0, a1, a2, a3, xb.x, xb.y);
  f8_decode(w1.z, a0, a1);
  f8_decode(w1.w, a2, a3);
  mma_bf16(acc[3 % kAcc], a0, a1, a2, a3, xb.z, xb.w);
}

// x fragment of one unit for lane (g, t): its 16 columns from the shared x
// slot (two 16-byte loads at xs), or zeros when `on` is false (column g >= N
// or columns past K, whose slot bytes are stale).
__device__ __forceinline__ void load_x(uint32_t xs, int xd, bool on, uint4 &xa, uint4 &xb) {
  if (on) {
    xa = lds128(xs);
    xb = lds128(xs + xd);
  } else {
    xa = make_uint4(0, 0, 0, 0);
    xb = xa;
  }
}

// The lane's scale words of a chunk: two units (rows g, g+8 each) per word.
__device__ __forceinline__ void load_scale_words(uint32_t a, uint32_t (&w)[kNvChunkUnits / 2]) {
  if constexpr (kNvChunkUnits == 8) {
    const uint4 v = lds128(a);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  } else {
    const uint2 v = lds64(a);
    w[0] = v.x;
    w[1] = v.y;
  }
}

// A whole NVFP4 chunk (8 units) of this lane's tile: scale pairs from one
// 16-byte load, codes and x for two units at a time, the next pair loaded
// before the current one is multiplied.  slot, scl: shared-memory addresses
// of the tile's codes and scales in the item slot; xs: the lane's first 16
// x columns of unit 0 in the slot (or in a zero row for a column >= N).
// kTensorX: the slice is tensor-copied (units 1024 bytes apart, the next 16
// columns at xd_t = +-16), else row-copied (units 128 bytes apart, +16).
// empty: if nonzero, the slot's empty mbarrier, arrived on (lane 0, after a
// warp sync) as soon as the last two units are in registers, so the slot is
// refilled while the warp computes them.
template <bool kTensorX>
__device__ __forceinline__ void nv_chunk_full(uint32_t slot, uint32_t scl, int lane, uint32_t xs,
                                              int xd_t, uint32_t m8, uint32_t m64,
                                              float (&acc)[kAcc][4], uint32_t empty = 0) {
  constexpr int kXUnit = kTensorX ? 1024 : kUnitK * 2;
  const int xd = kTensorX ? xd_t : 16;
  uint32_t scw[kNvChunkUnits / 2];
  load_scale_words(scl + lane * kNvScaleLaneBytes, scw);
  uint4 w0 = lds128(slot + lane * 16), w1 = lds128(slot + kNvUnitBytes + lane * 16);
  uint4 x0a = lds128(xs), x0b = lds128(xs + xd);
  uint4 x1a = lds128(xs + kXUnit), x1b = lds128(xs + kXUnit + xd);
#pragma unroll
  for (int h = 0; h < kNvChunkUnits / 2; ++h) {
    uint4 nw0, nw1, nx0a, nx0b, nx1a, nx1b;
    if (h + 1 < kNvChunkUnits / 2) {
      nw0 = lds128(slot + (2 * h + 2) * kNvUnitBytes + lane * 16);
      nw1 = lds128(slot + (2 * h + 3) * kNvUnitBytes + lane * 16);
      nx0a = lds128(xs + (2 * h + 2) * kXUnit);
      nx0b = lds128(xs + (2 * h + 2) * kXUnit + xd);
      nx1a = lds128(xs + (2 * h + 3) * kXUnit);
      nx1b = lds128(xs + (2 * h + 3) * kXUnit + xd);
    }
    if (h + 1 == kNvChunkUnits / 2 && empty != 0) {
      // every read of the slot is done (the arrive releases them)
      __syncwarp();
      if (lane == 0) mbar_arrive(empty);
    }
    // unit 2h uses scale bytes 0,1 of word h; unit 2h+1 bytes 2,3
    nv_unit(w0, nv_scale_pair(scw[h], 0), nv_scale_pair(scw[h], 1), x0a, x0b, m8, m64, acc);
    nv_unit(w1, nv_scale_pair(scw[h], 2), nv_scale_pair(scw[h], 3), x1a, x1b, m8, m64, acc);
    if (h + 1 < kNvChunkUnits / 2) {
      w0 = nw0;
      w1 = nw1;
      x0a = nx0a;
      x0b = nx0b;
      x1a = nx1a;
      x1b = nx1b;
    }
  }
}

// A partial NVFP4 chunk (the K tail): nu units, columns checked against K.
__device__ __forceinline__ void nv_chunk_tail(uint32_t slot, uint32_t scl, int lane, uint32_t xs,
                                              int xu, int xd, bool on, int nu, int kleft,
                                              uint32_t m8, uint32_t m64, float (&acc)[kAcc][4]) {
  uint32_t scw[kNvChunkUnits / 2];
  load_scale_words(scl + lane * kNvScaleLaneBytes, scw);
  for (int u = 0; u < nu; ++u) {
    const uint4 wv = lds128(slot + u * kNvUnitBytes + lane * 16);
    uint4 xa, xb;
    load_x(xs + u * xu, xd, on && u * kUnitK < kleft, xa, xb);
    // select without a runtime-indexed array (that would go to local memory)
    uint32_t word = scw[0];
#pragma unroll
    for (int q = 1; q < kNvChunkUnits / 2; ++q) word = (u >> 1) == q ? scw[q] : word;
    const uint32_t b = uint32_t(u & 1) * 2u;
    nv_unit(wv, nv_scale_pair(word, b), nv_scale_pair(word, b + 1), xa, xb, m8, m64, acc);
  }
}

// An FP8 chunk: nu (<= kF8ChunkUnits) units of 1024 bytes.  `full`: all units
// lie inside K, so x loads need no per-unit condition (xs then points at a
// zero row for a column >= N, or at the zero-filled rows of a tensor copy).
template <bool kTensorX>
__device__ __forceinline__ void f8_chunk(uint32_t slot, int lane, uint32_t xs, int xd_t, bool on,
                                         bool full, int nu, int kleft, float (&acc)[kAcc][4]) {
  constexpr int XU = kTensorX ? 1024 : kUnitK * 2;
  const int xd = kTensorX ? xd_t : 16;
#pragma unroll
  for (int u = 0; u < kF8ChunkUnits; ++u) {
    if (full || u < nu) {
      const uint4 w0 = lds128(slot + u * kF8UnitBytes + lane * 32);
      const uint4 w1 = lds128(slot + u * kF8UnitBytes + lane * 32 + 16);
      uint4 xa, xb;
      if (full) {
        xa = lds128(xs + u * XU);
        xb = lds128(xs + u * XU + xd);
      } else {
        load_x(xs + u * XU, xd, on && u * kUnitK < kleft, xa, xb);
      }
      f8_unit(w0, w1, xa, xb, acc);
    }
  }
}

// A whole MXFP8 chunk (4 units of 1024 bytes, tensor-copied x) of this
// lane's tile: the FP8 decode with each unit's block scales of rows g and
// g + 8 in place of the FP8 restore constant.  scl: the lane's 8 scale bytes
// [unit][row g, row g + 8].
__device__ __forceinline__ void mx_chunk(uint32_t slot, uint32_t scl, int lane, uint32_t xs,
                                         int xd, float (&acc)[kAcc][4]) {
  const uint2 sw = lds64(scl);
#pragma unroll
  for (int u = 0; u < kF8ChunkUnits; ++u) {
    const uint32_t word = u < 2 ? sw.x : sw.y;
    const uint32_t sg = mx_scale_pair(word, uint32_t(u & 1) * 2u);
    const uint32_t sg8 = mx_scale_pair(word, uint32_t(u & 1) * 2u + 1u);
    const uint4 w0 = lds128(slot + u * kF8UnitBytes + lane * 32);
    const uint4 w1 = lds128(slot + u * kF8UnitBytes + lane * 32 + 16);
    const uint4 xa = lds128(xs + u * 1024), xb = lds128(xs + u * 1024 + xd);
    uint32_t a0, a1, a2, a3;
    mx_decode(w0.x, sg, sg8, a0, a1);
    mx_decode(w0.y, sg, sg8, a2, a3);
    mma_bf16(acc[0], a0, a1, a2, a3, xa.x, xa.y);
    mx_decode(w0.z, sg, sg8, a0, a1);
    mx_decode(w0.w, sg, sg8, a2, a3);
    mma_bf16(acc[1 % kAcc], a0, a1, a2, a3, xa.z, xa.w);
    mx_decode(w1.x, sg, sg8, a0, a1);
    mx_decode(w1.y, sg, sg8, a2, a3);
    mma_bf16(acc[2 % kAcc], a0, a1, a2, a3, xb.x, xb.y);
    mx_decode(w1.z, sg, sg8, a0, a1);
    mx_decode(w1.w, sg, sg8, a2, a3);
    mma_bf16(acc[3 % kAcc], a0, a1, a2, a3, xb.z, xb.w);
  }
}

// A whole groupwise-INT4 chunk (8 units = 4 groups of 128 columns,
// tensor-copied x): per group the 8 MMAs of its two units run on integer
// weights q - 8 (exact in BF16) into a fresh FP32 sum, which is then scaled
// by the group's BF16 scales of rows g and g + 8 and added in.  scl: the
// lane's 16 scale bytes [group][row g, row g + 8].  The next unit's codes
// and x are loaded before the current one is decoded, and the slot is
// released (empty: its empty mbarrier, if nonzero) before the last unit is
// computed, as in nv_chunk_full.
__device__ __forceinline__ void i4_chunk(uint32_t slot, uint32_t scl, int lane, uint32_t xs,
                                         int xd, float (&acc)[kAcc][4], uint32_t empty = 0) {
  const uint4 sv = lds128(scl);
  const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
  uint4 wv = lds128(slot + lane * 16);
  uint4 xa = lds128(xs), xb = lds128(xs + xd);
#pragma unroll
  for (int grp = 0; grp < kNvChunkUnits / 2; ++grp) {
    float t4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int u = 2 * grp + h;
      uint4 nwv, nxa, nxb;
      if (u + 1 < kNvChunkUnits) {
        nwv = lds128(slot + (u + 1) * kNvUnitBytes + lane * 16);
        nxa = lds128(xs + (u + 1) * 1024);
        nxb = lds128(xs + (u + 1) * 1024 + xd);
      }
      if (u + 1 == kNvChunkUnits && empty != 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty);
      }
      uint32_t a0, a1, a2, a3;
      i4_decode(wv.x, a0, a1, a2, a3);
      mma_bf16(t4, a0, a1, a2, a3, xa.x, xa.y);
      i4_decode(wv.y, a0, a1, a2, a3);
      mma_bf16(t4, a0, a1, a2, a3, xa.z, xa.w);
      i4_decode(wv.z, a0, a1, a2, a3);
      mma_bf16(t4, a0, a1, a2, a3, xb.x, xb.y);
      i4_decode(wv.w, a0, a1, a2, a3);
      mma_bf16(t4, a0, a1, a2, a3, xb.z, xb.w);
      if (u + 1 < kNvChunkUnits) {
        wv = nwv;
        xa = nxa;
        xb = nxb;
      }
    }
    const float sg = __uint_as_float(sw[grp] << 16), sg8 = __uint_as_float(sw[grp] & 0xFFFF0000u);
    acc[0][0] = fmaf(sg, t4[0], acc[0][0]);
    acc[0][1] = fmaf(sg, t4[1], acc[0][1]);
    acc[0][2] = fmaf(sg8, t4[2], acc[0][2]);
    acc[0][3] = fmaf(sg8, t4[3], acc[0][3]);
  }
}

// Byte offsets of item (rb, ci)'s codes and scales in m (of `tiles` tiles);
// its tile-chunks follow one another in warp order.
__device__ __forceinline__ int64_t item_code_off(const MatDev &m, int rb, int ci, int tiles) {
  return int64_t(rb) * m.rb_bytes + int64_t(ci) * tiles * m.iu * m.ub;
}
__device__ __forceinline__ int64_t item_scale_off(const MatDev &m, int rb, int ci, int tiles) {
  return (int64_t(rb) * m.rt * m.KC + int64_t(ci) * tiles * m.cpi) * m.scb;
}

// Items beyond the ring that the producer brings into L2 while the consumers
// wait on a group dependency (the ring is full and DRAM would sit idle).
#ifndef VG_BPF
#define VG_BPF 4
#endif
constexpr int kBoundaryPf = VG_BPF;

// The producer (one lane): fill the item ring, one whole item per slot, as
// soon as all 16 consumer warps have released the slot.  An item's codes are
// one contiguous range of the packed buffer and its scales another, so an
// item is two bulk copies (L2 evict-first: read once) plus the x slice (x is
// read by every block: evict-last), one tensor copy or one copy per x row.
// Columns past K are zero-filled or not copied; the consumers mask them.
// The time from a slot's release to its refill adds to every item, so the
// next item's addresses and sizes are worked out before the wait (the
// current matrix's fields kept in registers), and the wait parks the lane in
// hardware (mbarrier try_wait with a time hint) instead of spinning on the
// sub-partition it shares with four consumer warps.  While the consumers
// wait on a group dependency it polls instead and brings items beyond the
// ring into L2.
//
// A verify pass runs two producers (np = 2), each owning one ring slot and
// so every other item: the refill work, which slows the consumer warps that
// share its sub-partition (and every slot release waits for the slowest
// warp), is split over two sub-partitions.  A single product, a short
// launch, runs one producer over both slots (np = 1): there the second
// measured 1-2 us slower per launch.  `which` is the producer's index.
// A producer's wait for the previous phase before it copies an x that phase
// writes (bounded), bringing its next items into L2 meanwhile; then the
// acquire is ordered before the x copies.  Returns
// false if the wait ran out or another block failed.
__device__ __forceinline__ bool producer_dep_wait(const Params &p, const MatDev *mats,
                                               const PhaseDev *phases, const Seq &q, int np) {
  const uint32_t *d = p.done + (q.ph - 1);
  const uint32_t target = uint32_t(phases[q.ph - 1].rbs);
  if (ld_acquire(d) < target) {
    const uint64_t deadline = globaltimer() + p.timeout_ns;
    Seq f = q;
    int ahead = 0;
    uint32_t it = 0;
    while (ld_acquire(d) < target) {
      if (ahead < kBoundaryPf && f.valid) {
        const MatDev &fm = mats[f.mi];
        if (fm.fmt != kFmtNorm) {
          const int ft = min(fm.rt, fm.MT - f.rb * fm.rt);
          const int fu = min(fm.iu, fm.KU - f.c * fm.iu);
          bulk_prefetch_l2(fm.w + item_code_off(fm, f.rb, f.c, ft), uint32_t(ft * fu * fm.ub));
          if (fm.scb)
            bulk_prefetch_l2(fm.sc + item_scale_off(fm, f.rb, f.c, ft),
                             uint32_t(ft * fm.cpi * fm.scb));
        }
        for (int k = 0; k < np && f.valid; ++k) f.advance(mats, phases, p);
        ++ahead;
      }
      if ((++it & 7u) == 0) {
        if (globaltimer() > deadline) {
          set_error(p.error, kErrDepWait);
          return false;
        }
        if (ld_relaxed(reinterpret_cast<const uint32_t *>(p.error)) != 0) return false;
      }
      __nanosleep(32);
    }
  }
  fence_proxy_async_global();
  return true;
}

#ifndef VG_PARK_NS
#define VG_PARK_NS 2000
#endif
template <bool kFused, int NB = 1>
__device__ void producer(const Params &p, const MatDev *mats, const PhaseDev *phases,
                         uint32_t ring, uint32_t full0, uint32_t empty0,
                         const volatile int *dep_waiting, int which, int np, int N) {
  const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
  Seq q;
  q.init(mats, phases, p);
  if (which && q.valid) q.advance(mats, phases, p);
  int s = which;
  uint32_t used = 0, last_par = 0;   // per slot (bit s): issued into, its last parity
  uint32_t par = 0;
  Seq pf = q;       // next item to bring into L2 during a dependency wait
  int pf_ahead = 0; // items between q and pf (pf is stale while 0)
  // the current matrix's fields, cached while the matrix does not change
  int cur_mi = -1, is_norm = 0, xdep = 0, dep_ok = -1;
  const uint8_t *w = nullptr, *sc = nullptr;
  const uint16_t *xg = nullptr;
  const CUtensorMap *tmap = nullptr;
  int rt = 0, MT = 0, KU = 0, K = 0, iu = 0, tile_item_bytes = 0, rb_scale_chunks = 0, cpi = 0, ub = 0;
  int scb = 0;
  int64_t rb_bytes = 0;
  while (q.valid) {
    // ---- the item's copies, worked out before its slot is free
    if (q.mi != cur_mi) {
      const MatDev &m = mats[q.mi];
      cur_mi = q.mi;
      is_norm = m.fmt == kFmtNorm;
      xdep = kFused && m.x_after && p.done && q.ph > 0;
      w = m.w;
      sc = m.scb ? m.sc : nullptr;
      scb = m.scb;
      xg = m.x;
      tmap = p.mats ? m.xmap : (p.x0_tensor ? &p.xmap0 : nullptr);
      rt = m.rt;
      MT = m.MT;
      KU = m.KU;
      K = m.K;
      iu = m.iu;
      tile_item_bytes = m.iu * m.ub;
      rb_bytes = m.rb_bytes;
      rb_scale_chunks = m.rt * m.KC;
      cpi = m.cpi;
      ub = m.ub;
    }
    const int tiles = min(rt, MT - q.rb * rt);
    const int nu = min(iu, KU - q.c * iu);   // units per tile in this item
    const uint32_t code_bytes = uint32_t(tiles * nu * ub);
    const uint32_t scale_bytes = sc ? uint32_t(tiles * cpi * scb) : 0u;
    const int k0 = q.c * iu * kUnitK;
    // x: one tensor copy of 8 rows x the item's units (rows >= N and units
    // past K read as zeros), else one bulk copy per row (one-chunk items)
    const uint32_t x_bytes = tmap ? uint32_t(8 * NB * iu * kUnitK * 2)
                                  : uint32_t(min(iu * kUnitK, K - k0) * 2 * N);
    const uint8_t *code_src = w + int64_t(q.rb) * rb_bytes + int64_t(q.c) * tiles * tile_item_bytes;
    const uint8_t *scale_src =
        sc ? sc + (int64_t(q.rb) * rb_scale_chunks + q.c * tiles * cpi) * scb : nullptr;
    const uint32_t slot = ring + s * kItemSlotBytes, full = full0 + 8 * s;

    // ---- an x that the previous phase of this pass writes: its copy waits
    // (bounded) until that phase has completed, after the item's weight
    // copies have been issued (below); the wait brings this producer's next
    // items into L2 and orders the acquire before the x copies
    const bool need_dep = kFused && xdep && dep_ok != q.ph;

    // ---- wait for the slot
    if (!mbar_test_wait(empty0 + 8 * s, par ^ 1u)) {
      const uint64_t deadline = globaltimer() + p.timeout_ns;
      bool ok = false;
      for (;;) {
        if (kBoundaryPf > 0 && which == 0 && *dep_waiting && pf_ahead < kBoundaryPf) {
          if (pf_ahead == 0) pf = q;   // start at the item waiting for this slot
          if (pf.valid) {
            const MatDev &fm = mats[pf.mi];
            // an RMS-norm item has no weights to bring in (only fused passes have them)
            if (!(kFused && fm.fmt == kFmtNorm)) {
              const int ft = min(fm.rt, fm.MT - pf.rb * fm.rt);
              const int fu = min(fm.iu, fm.KU - pf.c * fm.iu);
              bulk_prefetch_l2(fm.w + item_code_off(fm, pf.rb, pf.c, ft), uint32_t(ft * fu * fm.ub));
              if (fm.scb)
                bulk_prefetch_l2(fm.sc + item_scale_off(fm, pf.rb, pf.c, ft),
                                 uint32_t(ft * fm.cpi * fm.scb));
            }
            pf.advance(mats, phases, p);
            ++pf_ahead;
          }
          if ((ok = mbar_test_wait(empty0 + 8 * s, par ^ 1u))) break;
        } else if ((ok = mbar_try_wait_hint(empty0 + 8 * s, par ^ 1u, VG_PARK_NS))) {
          break;
        }
        if (globaltimer() > deadline) break;
      }
      if (!ok) {
        set_error(p.error, kErrEmptyWait);
        break;
      }
    }

    // ---- issue (an RMS-norm item has no weights: its slot takes the rows
    // of x, or nothing)
    if (is_norm) {
      // the rows of x, when they fit the slot (else the consumers read them
      // from global memory), copied once the phase that writes them is done
      const uint64_t xb = uint64_t(N) * uint64_t(K) * 2u;
      if (kFused && xb <= uint64_t(kItemSlotBytes)) {
        mbar_arrive_expect_tx(full, uint32_t(xb));
        if (need_dep) {
          if (!producer_dep_wait(p, mats, phases, q, np)) break;
          dep_ok = q.ph;
        }
        bulk_g2s(slot, reinterpret_cast<const uint8_t *>(xg), uint32_t(xb), full, pol_x);
      } else {
        mbar_arrive_expect_tx(full, 0u);
      }
    } else {
    mbar_arrive_expect_tx(full, code_bytes + scale_bytes + x_bytes);
    bulk_g2s(slot, code_src, code_bytes, full, pol_w);
    if (sc) bulk_g2s(slot + kItemScaleOff, scale_src, scale_bytes, full, pol_w);
    if (kFused && need_dep) {
      // the weights stream in meanwhile; the slot completes once x lands
      if (!producer_dep_wait(p, mats, phases, q, np)) break;
      dep_ok = q.ph;
    }
    if (tmap) {
      bulk_tensor_3d(slot + kItemXOff, tmap, 0, 0, q.c * iu, full, pol_x);
    } else {
      const uint32_t row_bytes = x_bytes / uint32_t(N);
      for (int n = 0; n < N; ++n)
        bulk_g2s(slot + kItemXOff + n * kXRowBytes, xg + int64_t(n) * K + k0, row_bytes, full,
                 pol_x);
    }
    }
    used |= 1u << s;
    last_par = (last_par & ~(1u << s)) | (par << s);
    for (int k = 0; k < np && q.valid; ++k) q.advance(mats, phases, p);
    pf_ahead = pf_ahead > np ? pf_ahead - np : 0;
    s += np;
    if (s >= kSlots) {
      s -= kSlots;
      par ^= 1u;
    }
  }
  // Never leave while a bulk copy may still be writing shared memory.
  for (int k = 0; k < kSlots; ++k)
    if ((used >> k) & 1u) mbar_wait_for(full0 + 8 * k, (last_par >> k) & 1u, p.timeout_ns);
}

// The reducer of a split row block adds the partial sums of the other
// contributors, blocks b0..bl, in block order.  Each thread reads only its
// own four words of every slot; a word counts once its tag matches `tag`, so
// no fence is needed on either side.  One round of loads covers kCollectW
// contributors; while some are not yet published, only their words are read
// again.  Each round costs an L2 round trip (about 1 us on GB300), but wider
// rounds need more than the 96 registers a thread gets with 18 warps per SM
// and spill, which costs more than the rounds they save.
// Returns false if the wait ran out or another block has already failed.
constexpr int kCollectW = 2;

__device__ __forceinline__ bool tags_match(const uint64_t (&v)[4], uint32_t tag) {
  return uint32_t(v[0] >> 32) == tag && uint32_t(v[1] >> 32) == tag &&
         uint32_t(v[2] >> 32) == tag && uint32_t(v[3] >> 32) == tag;
}

__device__ __forceinline__ bool collect(const Params &p, int b0, int bl, uint32_t tag, int at,
                                        float (&accs)[4]) {
  uint64_t deadline = 0;
  uint32_t polls = 0;
  for (int bb = b0; bb <= bl; bb += kCollectW) {
    uint64_t v[kCollectW][4];
    uint32_t pending = 0;
#pragma unroll
    for (int j = 0; j < kCollectW; ++j) {
      if (bb + j <= bl) {
        const uint64_t *src = p.partials + int64_t(bb + j) * kPartialWords + at;
        ld_relaxed_v2u64(src, v[j][0], v[j][1]);
        ld_relaxed_v2u64(src + 64, v[j][2], v[j][3]);
        pending |= 1u << j;
      }
    }
    for (;;) {
#pragma unroll
      for (int j = 0; j < kCollectW; ++j)
        if (((pending >> j) & 1u) && tags_match(v[j], tag)) pending &= ~(1u << j);
      if (pending == 0) break;
      if ((++polls & 7u) == 0) {   // clock and error word every 8th poll
        const uint64_t now = globaltimer();
        if (deadline == 0) {
          deadline = now + p.timeout_ns;
        } else if (now > deadline) {
          set_error(p.error, kErrPartialWait);
          return false;
        }
        if (ld_relaxed(reinterpret_cast<const uint32_t *>(p.error)) != 0) return false;
      }
#pragma unroll
      for (int j = 0; j < kCollectW; ++j) {
        if ((pending >> j) & 1u) {
          const uint64_t *src = p.partials + int64_t(bb + j) * kPartialWords + at;
          ld_relaxed_v2u64(src, v[j][0], v[j][1]);
          ld_relaxed_v2u64(src + 64, v[j][2], v[j][3]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kCollectW; ++j)
      if (bb + j <= bl)
#pragma unroll
        for (int e = 0; e < 4; ++e) accs[e] += __uint_as_float(uint32_t(v[j][e]));
  }
  return true;
}

// collect() for slots of NB column blocks (slot_words 64-bit words each).
template <int NB>
__device__ __forceinline__ bool collect_wide(const Params &p, int b0, int bl, uint32_t tag, int at,
                                             float (&accs)[4]) {
  constexpr int64_t slot_words = int64_t(NB) * kPartialWords;
  uint64_t deadline = 0;
  uint32_t polls = 0;
  for (int bb = b0; bb <= bl; bb += kCollectW) {
    uint64_t v[kCollectW][4];
    uint32_t pending = 0;
#pragma unroll
    for (int j = 0; j < kCollectW; ++j) {
      if (bb + j <= bl) {
        const uint64_t *src = p.partials + int64_t(bb + j) * slot_words + at;
        ld_relaxed_v2u64(src, v[j][0], v[j][1]);
        ld_relaxed_v2u64(src + 64, v[j][2], v[j][3]);
        pending |= 1u << j;
      }
    }
    for (;;) {
#pragma unroll
      for (int j = 0; j < kCollectW; ++j)
        if (((pending >> j) & 1u) && tags_match(v[j], tag)) pending &= ~(1u << j);
      if (pending == 0) break;
      if ((++polls & 7u) == 0) {   // clock and error word every 8th poll
        const uint64_t now = globaltimer();
        if (deadline == 0) {
          deadline = now + p.timeout_ns;
        } else if (now > deadline) {
          set_error(p.error, kErrPartialWait);
          return false;
        }
        if (ld_relaxed(reinterpret_cast<const uint32_t *>(p.error)) != 0) return false;
      }
#pragma unroll
      for (int j = 0; j < kCollectW; ++j) {
        if ((pending >> j) & 1u) {
          const uint64_t *src = p.partials + int64_t(bb + j) * slot_words + at;
          ld_relaxed_v2u64(src, v[j][0], v[j][1]);
          ld_relaxed_v2u64(src + 64, v[j][2], v[j][3]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kCollectW; ++j)
      if (bb + j <= bl)
#pragma unroll
        for (int e = 0; e < 4; ++e) accs[e] += __uint_as_float(uint32_t(v[j][e]));
  }
  return true;
}

// Epilogue of a gated pair: rows g (gate) and g + 8 (up) of tile mt are
// gate and up row 8 mt + g; y = SiLU(gate) * up from the FP32 sums, rounded
// once to BF16.  Only the fused instantiation compiles it, and there it is
// inlined: out of line, the call cost the gated pair's piece ends more than
// the code costs the fused kernel's registers.
__device__ __forceinline__ void swiglu_epilogue(const MatDev &m, int mt, int g, int t, int N,
                                             const float (&accs)[4]) {
  const int gi = mt * 8 + g;
  if (gi >= m.Mo) return;
  const bool nv = m.fmt == VG_FMT_NVFP4;
  const float mg = nv ? m.mult : __ldg(m.rowscale + gi);
  const float mu = nv ? m.mult2 : __ldg(m.rowscale2 + gi);
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int nn = 2 * t + e;
    if (nn < N) {
      const float gate = accs[e] * mg, up = accs[2 + e] * mu;
      const float h = gate / (1.0f + expf(-gate)) * up;
      const __nv_bfloat16 v = __float2bfloat16_rn(h);
      m.y[int64_t(nn) * m.Mo + gi] = *reinterpret_cast<const uint16_t *>(&v);
    }
  }
}

// End of a row-block piece.  With several chunks per item (cpi > 1) the
// warps that share a tile first hand their sums to its first warp (cc == 0)
// through shared memory, added in chunk order; only that warp goes on.
// Then a block that covered the whole row block writes y.  Otherwise the
// row block is split: the block holding its first item (the reducer) adds
// the other contributors' partial sums to its own and writes y; every other
// contributor publishes its partial sums in its slot, tagged, and moves on
// without waiting.  In ordered mode the completed row block is counted for
// its phase.  It runs once per piece, outside the per-item loops.  Returns
// false if the wait for partial sums failed.
template <bool kFused>
__device__ __forceinline__ bool finish_piece(const Params &p, const MatDev &m, int T, int G,
                                          int piece_start, bool full_piece, int rb, int ph,
                                          uint32_t tag, bool aborted, int tl, int cc,
                                          uint32_t red, int N, float a0, float a1, float a2,
                                          float a3) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int mt = rb * m.rt + tl;
  const int at = ((warp * 2) * 32 + lane) * 2;    // this thread's words in a slot
  float accs[4] = {a0, a1, a2, a3};
  if (m.cpi > 1) {
    // barriers of the tile's warps only (ids 3.., one per tile of the block)
    if (cc != 0) sts128(red + uint32_t(warp * 32 + lane) * 16u, accs[0], accs[1], accs[2], accs[3]);
    named_bar(3 + tl, m.cpi * 32);
    if (cc == 0) {
      for (int j = 1; j < m.cpi; ++j) {
        const uint4 q = lds128(red + uint32_t((warp + j) * 32 + lane) * 16u);
        accs[0] += __uint_as_float(q.x);
        accs[1] += __uint_as_float(q.y);
        accs[2] += __uint_as_float(q.z);
        accs[3] += __uint_as_float(q.w);
      }
    }
    named_bar(3 + tl, m.cpi * 32);   // the scratch is free again
  }
  const bool lead = cc == 0;
  bool ok = true;
  if (!full_piece) {
    const int first = m.item0 + rb * m.KI;
    if (piece_start != first) {
      if (!aborted && lead) {
        uint64_t *dst = p.partials + int64_t(blockIdx.x) * kPartialWords + at;
        const uint64_t hi = uint64_t(tag) << 32;
        st_relaxed_v2u64(dst, hi | __float_as_uint(accs[0]), hi | __float_as_uint(accs[1]));
        st_relaxed_v2u64(dst + 64, hi | __float_as_uint(accs[2]), hi | __float_as_uint(accs[3]));
      }
      return true;
    }
    if (!aborted && lead)
      ok = collect(p, int(blockIdx.x) + 1, owner(T, G, first + m.KI - 1), tag, at, accs);
    // mma.sync needs whole warps: a failure anywhere in the warp stops it all
    ok = __all_sync(0xFFFFFFFFu, ok);
  }
  if (kFused && ok && !aborted && lead && mt < m.MT && m.op == VG_OP_SWIGLU) {
    swiglu_epilogue(m, mt, g, t, N, accs);
  } else if (ok && !aborted && lead && mt < m.MT) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = mt * kTileRows + g + 8 * h;
      if (row >= m.M) continue;
      const float mult = m.fmt == VG_FMT_FP8_ROWSCALE ? __ldg(m.rowscale + row) : m.mult;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int nn = 2 * t + e;
        if (nn < N) {
          const __nv_bfloat16 v = __float2bfloat16_rn(accs[2 * h + e] * mult);
          m.y[int64_t(nn) * m.M + row] = *reinterpret_cast<const uint16_t *>(&v);
        }
      }
    }
  }
  // y that a later phase copies in: order these stores before those copies
  if (kFused && m.y_async && lead) fence_proxy_async_global();
  if (p.done) {
    named_bar(1, kConsumers);
    // releases the row block's y (written before the barrier)
    if (tid == 0 && ok && !aborted && ph != p.hold_phase) red_add_release(p.done + ph, 1u);
  }
  return ok;
}

// --------------------------------------------------------- wider passes
// N = 9..32 columns: NB blocks of 8 (NB = 2 or 4).  The item's x slice is
// one tensor copy of 8 NB rows per unit, [unit][8 NB rows][128 B] with the
// same 128-byte swizzle (rows 8b + g read like rows g), so column block b of
// unit u sits at u * 1024 NB + b * 1024.  Every decoded A fragment feeds NB
// MMAs.  Only whole chunks and tensor-copied x take this path.

// Wide units: per half unit (k16 steps 0-1, then 2-3) every column block's
// x fragment is loaded (one 16-byte load per block), then each step's A
// fragment is decoded once and fed to the NB MMAs, so that at most NB x
// fragments and one A fragment are live.
template <int NB>
__device__ __forceinline__ void mma_wide(float (&acc)[NB][4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, const uint4 (&x)[NB], bool hi) {
#pragma unroll
  for (int b = 0; b < NB; ++b)
    mma_bf16(acc[b], a0, a1, a2, a3, hi ? x[b].z : x[b].x, hi ? x[b].w : x[b].y);
}

template <int NB>
__device__ __forceinline__ void load_x_half(uint32_t xs, uint4 (&x)[NB]) {
#pragma unroll
  for (int b = 0; b < NB; ++b) x[b] = lds128(xs + b * 1024);
}

template <int NB>
__device__ __forceinline__ void nv_chunk_wide(uint32_t slot, uint32_t scl, int lane, uint32_t xs,
                                              int xd, uint32_t m8, uint32_t m64,
                                              float (&acc)[NB][4]) {
  uint32_t scw[kNvChunkUnits / 2];
  load_scale_words(scl + lane * kNvScaleLaneBytes, scw);
#pragma unroll
  for (int u = 0; u < kNvChunkUnits; ++u) {
    const uint4 wv = lds128(slot + u * kNvUnitBytes + lane * 16);
    const uint32_t fg = nv_scale_pair(scw[u >> 1], uint32_t(u & 1) * 2u);
    const uint32_t fg8 = nv_scale_pair(scw[u >> 1], uint32_t(u & 1) * 2u + 1u);
    const uint32_t xu = xs + u * 1024 * NB;
    uint4 xv[NB];
    uint32_t a0, a1, a2, a3;
    load_x_half<NB>(xu, xv);
    nv_decode(wv.x, fg, fg8, m8, m64, a0, a1, a2, a3);
    mma_wide<NB>(acc, a0, a1, a2, a3, xv, false);
    nv_decode(wv.y, fg, fg8, m8, m64, a0, a1, a2, a3);
    mma_wide<NB>(acc, a0, a1, a2, a3, xv, true);
    load_x_half<NB>(xu + xd, xv);
    nv_decode(wv.z, fg, fg8, m8, m64, a0, a1, a2, a3);
    mma_wide<NB>(acc, a0, a1, a2, a3, xv, false);
    nv_decode(wv.w, fg, fg8, m8, m64, a0, a1, a2, a3);
    mma_wide<NB>(acc, a0, a1, a2, a3, xv, true);
  }
}

// FP8 (kMx false: the row scale comes in the epilogue) or MXFP8 (kMx: the
// lane's 8 block-scale bytes at scl).
template <int NB, bool kMx>
__device__ __forceinline__ void f8_chunk_wide(uint32_t slot, uint32_t scl, int lane, uint32_t xs,
                                              int xd, float (&acc)[NB][4]) {
  uint2 sw = make_uint2(0u, 0u);
  if (kMx) sw = lds64(scl);
#pragma unroll
  for (int u = 0; u < kF8ChunkUnits; ++u) {
    const uint4 w0 = lds128(slot + u * kF8UnitBytes + lane * 32);
    const uint4 w1 = lds128(slot + u * kF8UnitBytes + lane * 32 + 16);
    const uint32_t word = u < 2 ? sw.x : sw.y;
    const uint32_t sg = kMx ? mx_scale_pair(word, uint32_t(u & 1) * 2u) : kF8Restore2;
    const uint32_t sg8 = kMx ? mx_scale_pair(word, uint32_t(u & 1) * 2u + 1u) : kF8Restore2;
    const uint32_t xu = xs + u * 1024 * NB;
    uint4 xv[NB];
    uint32_t a0, a1, a2, a3;
    load_x_half<NB>(xu, xv);
    mx_decode(w0.x, sg, sg8, a0, a1);
    mx_decode(w0.y, sg, sg8, a2, a3);
    mma_wide<NB>(acc, a0, a1, a2, a3, xv, false);
    mx_decode(w0.z, sg, sg8, a0, a1);
    mx_decode(w0.w, sg, sg8, a2, a3);
    mma_wide<NB>(acc, a0, a1, a2, a3, xv, true);
    load_x_half<NB>(xu + xd, xv);
    mx_decode(w1.x, sg, sg8, a0, a1);
    mx_decode(w1.y, sg, sg8, a2, a3);
    mma_wide<NB>(acc, a0, a1, a2, a3, xv, false);
    mx_decode(w1.z, sg, sg8, a0, a1);
    mx_decode(w1.w, sg, sg8, a2, a3);
    mma_wide<NB>(acc, a0, a1, a2, a3, xv, true);
  }
}

template <int NB>
__device__ __forceinline__ void i4_chunk_wide(uint32_t slot, uint32_t scl, int lane, uint32_t xs,
                                              int xd, float (&acc)[NB][4]) {
  const uint4 sv = lds128(scl);
  const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
  for (int grp = 0; grp < kNvChunkUnits / 2; ++grp) {
    float t4[NB][4];
#pragma unroll
    for (int b = 0; b < NB; ++b) t4[b][0] = t4[b][1] = t4[b][2] = t4[b][3] = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int u = 2 * grp + h;
      const uint4 wv = lds128(slot + u * kNvUnitBytes + lane * 16);
      const uint32_t xu = xs + u * 1024 * NB;
      uint4 xv[NB];
      uint32_t a0, a1, a2, a3;
      load_x_half<NB>(xu, xv);
      i4_decode(wv.x, a0, a1, a2, a3);
      mma_wide<NB>(t4, a0, a1, a2, a3, xv, false);
      i4_decode(wv.y, a0, a1, a2, a3);
      mma_wide<NB>(t4, a0, a1, a2, a3, xv, true);
      load_x_half<NB>(xu + xd, xv);
      i4_decode(wv.z, a0, a1, a2, a3);
      mma_wide<NB>(t4, a0, a1, a2, a3, xv, false);
      i4_decode(wv.w, a0, a1, a2, a3);
      mma_wide<NB>(t4, a0, a1, a2, a3, xv, true);
    }
    const float sg = __uint_as_float(sw[grp] << 16), sg8 = __uint_as_float(sw[grp] & 0xFFFF0000u);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      acc[b][0] = fmaf(sg, t4[b][0], acc[b][0]);
      acc[b][1] = fmaf(sg, t4[b][1], acc[b][1]);
      acc[b][2] = fmaf(sg8, t4[b][2], acc[b][2]);
      acc[b][3] = fmaf(sg8, t4[b][3], acc[b][3]);
    }
  }
}

// finish_piece for NB column blocks: the tile-sum hand-off and the
// partial-sum collection run once per block of 8 columns; a thread block's
// partial-sum slot holds NB blocks' words.
template <int NB>
__device__ __forceinline__ bool finish_piece_wide(const Params &p, const MatDev &m, int T, int G,
                                                  int piece_start, bool full_piece, int rb, int ph,
                                                  uint32_t tag, bool aborted, int tl, int cc,
                                                  uint32_t red, int N, float (&acc)[NB][4]) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int mt = rb * m.rt + tl;
  const int at = ((warp * 2) * 32 + lane) * 2;
  constexpr int64_t kSlot = int64_t(NB) * kPartialWords;
  if (m.cpi > 1) {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (cc != 0) sts128(red + uint32_t(warp * 32 + lane) * 16u, acc[b][0], acc[b][1], acc[b][2],
                          acc[b][3]);
      named_bar(3 + tl, m.cpi * 32);
      if (cc == 0) {
        for (int j = 1; j < m.cpi; ++j) {
          const uint4 q = lds128(red + uint32_t((warp + j) * 32 + lane) * 16u);
          acc[b][0] += __uint_as_float(q.x);
          acc[b][1] += __uint_as_float(q.y);
          acc[b][2] += __uint_as_float(q.z);
          acc[b][3] += __uint_as_float(q.w);
        }
      }
      named_bar(3 + tl, m.cpi * 32);
    }
  }
  const bool lead = cc == 0;
  bool ok = true;
  if (!full_piece) {
    const int first = m.item0 + rb * m.KI;
    if (piece_start != first) {
      if (!aborted && lead) {
        const uint64_t hi = uint64_t(tag) << 32;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          uint64_t *dst = p.partials + int64_t(blockIdx.x) * kSlot + b * kPartialWords + at;
          st_relaxed_v2u64(dst, hi | __float_as_uint(acc[b][0]), hi | __float_as_uint(acc[b][1]));
          st_relaxed_v2u64(dst + 64, hi | __float_as_uint(acc[b][2]), hi | __float_as_uint(acc[b][3]));
        }
      }
      return true;
    }
    if (!aborted && lead) {
#pragma unroll
      for (int b = 0; b < NB; ++b)
        if (ok) ok = collect_wide<NB>(p, int(blockIdx.x) + 1, owner(T, G, first + m.KI - 1), tag,
                                      at + b * kPartialWords, acc[b]);
    }
    ok = __all_sync(0xFFFFFFFFu, ok);
  }
  if (ok && !aborted && lead && mt < m.MT) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = mt * kTileRows + g + 8 * h;
      if (row >= m.M) continue;
      const float mult = m.fmt == VG_FMT_FP8_ROWSCALE ? __ldg(m.rowscale + row) : m.mult;
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int nn = 8 * b + 2 * t + e;
          if (nn < N) {
            const __nv_bfloat16 v = __float2bfloat16_rn(acc[b][2 * h + e] * mult);
            m.y[int64_t(nn) * m.M + row] = *reinterpret_cast<const uint16_t *>(&v);
          }
        }
    }
  }
  if (p.done) {
    named_bar(1, kConsumers);
    if (tid == 0 && ok && !aborted && ph != p.hold_phase) red_add_release(p.done + ph, 1u);
  }
  return ok;
}

// An RMS-norm item, run by all consumer threads of one block:
//   y[n][k] = bf16( x[n][k] * inv[n] * gamma[k] ),
//   inv[n] = 1 / sqrt(sum_k x[n][k]^2 / K + eps),
// sums in FP32 (per thread, then per warp, then across warps in `red`).
// The norm is split into m.RB items, one per thread block: each computes
// the whole rows' sums and writes its slice `slice` of the 8-element vectors
// of y, one (row, vector) pair per thread.  When the N rows fit an item slot
// (N K 2 bytes, 80 KB at N = 8, K = 5120) the producer has copied them into
// the item's slot (xs), so every read is from shared memory; otherwise they
// are read from L2.  Every thread reaches every barrier; `active` false
// skips the work.  Kept out of line: inlined, it costs the streaming loops
// registers.
__device__ __noinline__ void rms_norm_item(const MatDev &m, int N, float *red, bool active,
                                           int slice, uint32_t xs) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K8 = m.K / 8;
  if (xs != 0u) {
    // the rows are in the item's slot (row n at xs + 16 K8 n): all rows at
    // once, so that their sums and shuffle reductions overlap
    float ss[8];
#pragma unroll
    for (int n = 0; n < 8; ++n) ss[n] = 0.f;
    if (active) {
      for (int k = tid; k < K8; k += kConsumers) {
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          if (n < N) {
            const uint4 v = lds128(xs + uint32_t(n * K8 + k) * 16u);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float lo = __uint_as_float(wv[j] << 16), hi = __uint_as_float(wv[j] & 0xFFFF0000u);
              ss[n] = fmaf(lo, lo, ss[n]);
              ss[n] = fmaf(hi, hi, ss[n]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int n = 0; n < 8; ++n)
        if (n < N) ss[n] += __shfl_xor_sync(0xFFFFFFFFu, ss[n], o);
    if (lane == 0)
#pragma unroll
      for (int n = 0; n < 8; ++n)
        if (n < N) red[n * kWarps + warp] = ss[n];
  } else {
    // the rows from global memory (L2: the previous phase wrote them); the
    // same sums in the same order
    for (int n = 0; n < N; ++n) {
      float ss = 0.f;
      if (active) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(m.x + int64_t(n) * m.K);
        for (int k = tid; k < K8; k += kConsumers) {
          const uint4 v = xr[k];
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(wv[j] << 16), hi = __uint_as_float(wv[j] & 0xFFFF0000u);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
      if (lane == 0) red[n * kWarps + warp] = ss;
    }
  }
  named_bar(1, kConsumers);
  if (tid < N) {
    float tot = 0.f;
    for (int w = 0; w < kWarps; ++w) tot += red[tid * kWarps + w];
    red[8 * kWarps + tid] = 1.0f / sqrtf(tot / float(m.K) + m.eps);
  }
  named_bar(1, kConsumers);
  if (active) {
    // this block's slice of every row: one 8-element group per thread,
    // (row, group) pairs spread over all threads
    const uint4 *gr = reinterpret_cast<const uint4 *>(m.gamma);
    const int k0 = int(int64_t(K8) * slice / m.RB), k1 = int(int64_t(K8) * (slice + 1) / m.RB);
    const int L = k1 - k0;
    for (int i = tid; i < N * L; i += kConsumers) {
      const int n = i / L, k = k0 + (i - n * L);
      const float inv = red[8 * kWarps + n];
      const uint4 v = xs != 0u ? lds128(xs + uint32_t(n * K8 + k) * 16u)
                               : reinterpret_cast<const uint4 *>(m.x + int64_t(n) * m.K)[k];
      const uint4 gv = __ldg(gr + k);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float x0 = __uint_as_float(wv[j] << 16), x1 = __uint_as_float(wv[j] & 0xFFFF0000u);
        const float g0 = __uint_as_float(gw[j] << 16), g1 = __uint_as_float(gw[j] & 0xFFFF0000u);
        const __nv_bfloat162 r = __floats2bfloat162_rn(x0 * inv * g0, x1 * inv * g1);
        o[j] = *reinterpret_cast<const uint32_t *>(&r);
      }
      reinterpret_cast<uint4 *>(m.y + int64_t(n) * m.K)[k] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    // a later phase copies y in through the async proxy
    fence_proxy_async_global();
  }
  named_bar(1, kConsumers);
}

// Two instantiations: kFused = false for passes of plain products (single
// GEMVs and verify passes without fused operations or dependent x), which
// then carry none of that code; kFused = true for the rest.
template <bool kFused>
__global__ void __launch_bounds__(kKernelThreads, 1) stream_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the swizzled tensor copies need 1024-byte alignment in shared memory
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kBarOff);
  volatile int *sflag = reinterpret_cast<volatile int *>(smem + kBarOff + kBarBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const MatDev *mats = p.mats ? p.mats : &p.mat0;
  const PhaseDev *phases = p.mats ? p.phases : &p.phase0;

  if (tid * 16 < kXRowBytes)
    *reinterpret_cast<uint4 *>(smem + kZeroRowOff + tid * 16) = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_addr(bars + i), 1);                       // full: the slot's producer
      mbar_init(smem_addr(bars + kSlots + i), kWarps);         // empty: every consumer warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sflag[0] = 0;
    sflag[1] = int(ld_relaxed(p.epoch));
    sflag[2] = 0;
    sflag[3] = 0;   // consumers waiting on a group dependency
    // the pass's width: fixed, or read from the width word at launch
    int n = p.N;
    if (p.width) {
      n = ld_relaxed(reinterpret_cast<const uint32_t *>(p.width));
      if (n < 1 || n > p.N) {
        if (blockIdx.x == 0) set_error(p.error, kErrWidth);
        n = 0;   // no work: every block goes straight to the end of the pass
      }
    }
    sflag[4] = n;
  }
  __syncthreads();
  const uint32_t epoch = uint32_t(sflag[1]);
  const int N = sflag[4];

  if (N == 0) {
    // invalid width: nothing is read or written
  } else if (warp >= kWarps) {
    // ================================================================ producer
    const int np = p.mats ? kProducers : 1;
    if (lane == 0 && warp - kWarps < np)
      producer<kFused>(p, mats, phases, smem_addr(smem), smem_addr(bars), smem_addr(bars + kSlots),
               sflag + 3, warp - kWarps, np, N);

  } else {
    // =============================================================== consumers
    const int g = lane >> 2, t = lane & 3;
    const bool on = g < N;
    const uint32_t ring = smem_addr(smem);
    const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + kSlots);
    // This lane's x columns inside an item slot.  Tensor-copied slices are
    // [unit][row][128 B] with the 16-byte chunks of row r at chunk ^ (r % 8)
    // (128-byte swizzle), so a unit is 1024 bytes and the lane's two chunks
    // 2t, 2t+1 of row g sit at (2t ^ g) and next to it.  Row-copied slices
    // are padded rows of kXRowBytes, and a column g >= N reads a zero row.
    const uint32_t xoff_t0 = uint32_t(kItemXOff + g * 128 + ((2 * t) ^ g) * 16);
    const int xd_t = (g & 1) ? -16 : 16;
    const uint32_t xoff_r = uint32_t(kItemXOff + g * kXRowBytes + t * 32);
    const uint32_t xzero = smem_addr(smem + kZeroRowOff) + t * 32;
    Seq cons;
    cons.init(mats, phases, p);
    bool aborted = false;
    int s = 0;                     // ring slot of the current item
    uint32_t par = 0;              // parity of that slot's current phase
    int cur_ph = -1, cur_mi = -1;
    uint32_t tag = 0;              // tag of this pass and phase
    float acc[kAcc][4];
    // matrix fields cached while the matrix does not change
    int K = 0, KU = 0, MT = 0, fmt = 0, rt = kBlockTiles, kfull = 0, iu = 0;
    int tl = warp, cc = 0;         // this warp's tile and chunk within an item
    uint32_t xoff_t = xoff_t0;     // ... and its x columns (tensor-copied x)
    bool xt = false;               // the matrix's x slice is tensor-copied
    const uint32_t red = smem_addr(smem + kRedOff);   // tile-sum scratch
    while (cons.valid) {
      const int ph = cons.ph;
      // -------------------------------------- ordered: wait for group ph-1
      if (ph != cur_ph) {
        if (p.ordered && ph > 0) {
          if (tid == 0) {
            int ok = 1;
            if (!aborted) {
              const uint32_t *d = p.done + (ph - 1);
              sflag[3] = 1;
              const uint32_t target = uint32_t(phases[ph - 1].rbs);
              if (ld_acquire(d) < target) {
                const uint64_t deadline = globaltimer() + p.timeout_ns;
                uint32_t it = 0;
                // one L2 round trip per poll: the clock and the error word
                // are looked at every 8th poll only
                while (ld_acquire(d) < target) {
                  if ((++it & 7u) == 0) {
                    if (globaltimer() > deadline) {
                      ok = 0;
                      set_error(p.error, kErrDepWait);
                      break;
                    }
                    if (ld_relaxed(reinterpret_cast<const uint32_t *>(p.error)) != 0) {
                      ok = 0;   // another block has failed: results are void
                      break;
                    }
                  }
                  __nanosleep(32);
                }
              }
            }
            sflag[3] = 0;
            sflag[0] = ok ? 0 : 1;
          }
          named_bar(1, kConsumers);
          if (sflag[0]) aborted = true;
          named_bar(1, kConsumers);
        }
        cur_ph = ph;
        tag = epoch * uint32_t(p.nphases) + uint32_t(ph) + 1u;
      }
      if (cons.mi != cur_mi) {
        const MatDev &mm = mats[cons.mi];
        cur_mi = cons.mi;
        K = mm.K;
        KU = mm.KU;
        MT = mm.MT;
        fmt = mm.fmt;
        rt = mm.rt;
        iu = mm.iu;
        kfull = mm.kfull;
        tl = warp / mm.cpi;
        cc = warp - tl * mm.cpi;
        // the warp's chunk starts cc chunks into the item's x slice
        xoff_t = xoff_t0 + uint32_t(cc * mm.cu * 1024);
        xt = p.mats ? mm.xmap != nullptr : p.x0_tensor != 0;
      }
      if (kFused && fmt == kFmtNorm) {
        // an RMS-norm item: its slot carries the rows of x when they fit
        // (else nothing), this block's consumers normalise x into y, give
        // the slot back, and the item completes its phase
        if (!aborted) {
          const bool ready = mbar_wait_for(full0 + 8 * s, par, p.timeout_ns);
          if (!__all_sync(0xFFFFFFFFu, ready)) {
            if (lane == 0) set_error(p.error, kErrFullWait);
            aborted = true;
          }
        }
        const bool x_in_slot = uint64_t(N) * uint64_t(K) * 2u <= uint64_t(kItemSlotBytes);
        rms_norm_item(mats[cons.mi], N, reinterpret_cast<float *>(smem + kRedOff), !aborted,
                      cons.rb, x_in_slot ? ring + s * kItemSlotBytes : 0u);
        // rms_norm_item ends on a barrier of all consumers: the slot is read
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        if (++s == kSlots) {
          s = 0;
          par ^= 1u;
        }
        if (tid == 0 && !aborted && ph != p.hold_phase) red_add_release(p.done + ph, 1u);
        cons.skip(1, mats, phases, p);
        continue;
      }
      // ------------------------------------------------- one row-block piece
      // the block's contiguous items of one row block: set up once, then a
      // tight loop over its chunks
      const int rb = cons.rb, c0 = cons.c;
      const int len = min(cons.KI - c0, cons.i1 - cons.i);
      const int piece_start = cons.i;
#pragma unroll
      for (int a = 0; a < kAcc; ++a)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[a][e] = 0.f;
      const int mt = rb * rt + tl;
      const bool work = mt < MT;
      int c = c0;
      const int c_end = c0 + len;
      // Fast loop: the common case (tensor-copied x, chunks wholly inside K,
      // the warp's tile inside M) with nothing decided per item but the wait.
      if (!aborted && work && xt) {
        const uint32_t scl0 = kItemScaleOff + warp * kNvScaleChunkBytes;
        const uint32_t code0 = warp * kSlotCodeBytes;
        const int c_full = min(c_end, kfull);
        if (fmt == VG_FMT_NVFP4) {
          for (; c < c_full; ++c) {
            const uint32_t item = ring + s * kItemSlotBytes;
            if (!__all_sync(0xFFFFFFFFu, mbar_try_wait(full0 + 8 * s, par)) &&
                !__all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8 * s, par, globaltimer() + p.timeout_ns)))
              break;   // the general loop below records the failure
            // releases the slot itself, before computing its last two units
            nv_chunk_full<true>(item + code0, item + scl0, lane, item + xoff_t, xd_t, p.m8, p.m64,
                                acc, empty0 + 8 * s);
            if (++s == kSlots) {
              s = 0;
              par ^= 1u;
            }
          }
        } else if (fmt == VG_FMT_MXFP8 || fmt == VG_FMT_INT4G) {
          // these formats take whole chunks and tensor-copied x only, so
          // this loop does all of their work
          const bool mx = fmt == VG_FMT_MXFP8;
          const uint32_t scl_l = kItemScaleOff + warp * kMxScaleChunkBytes +
                                 (mx ? uint32_t(g * 2 + (t >> 1)) * 8u : uint32_t(g) * 16u);
          for (; c < c_full; ++c) {
            const uint32_t item = ring + s * kItemSlotBytes;
            if (!__all_sync(0xFFFFFFFFu, mbar_try_wait(full0 + 8 * s, par)) &&
                !__all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8 * s, par, globaltimer() + p.timeout_ns)))
              break;
            if (mx)
              mx_chunk(item + code0, item + scl_l, lane, item + xoff_t, xd_t, acc);
            else
              i4_chunk(item + code0, item + scl_l, lane, item + xoff_t, xd_t, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
            if (++s == kSlots) {
              s = 0;
              par ^= 1u;
            }
          }
          if (c < c_full) {          // a wait ran out: nothing else computes them
            if (lane == 0) set_error(p.error, kErrFullWait);
            aborted = true;
          }
        } else {
          for (; c < c_full; ++c) {
            const uint32_t item = ring + s * kItemSlotBytes;
            if (!__all_sync(0xFFFFFFFFu, mbar_try_wait(full0 + 8 * s, par)) &&
                !__all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8 * s, par, globaltimer() + p.timeout_ns)))
              break;
            f8_chunk<true>(item + code0, lane, item + xoff_t, xd_t, true, true, kF8ChunkUnits, 0,
                           acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
            if (++s == kSlots) {
              s = 0;
              par ^= 1u;
            }
          }
        }
      }
      // General loop: the rest of the piece (K tails, row-copied x, tiles past
      // M, a failed wait).
      for (; c < c_end; ++c) {
        const uint32_t item = ring + s * kItemSlotBytes;
        if (!aborted) {
          // every lane polls; a lane whose wait ran out stops the whole
          // warp, since mma.sync needs all of it
          const bool ready = mbar_wait_for(full0 + 8 * s, par, p.timeout_ns);
          if (!__all_sync(0xFFFFFFFFu, ready)) {
            if (lane == 0) set_error(p.error, kErrFullWait);
            aborted = true;
          }
        }
        if (!aborted && work && fmt <= VG_FMT_FP8_ROWSCALE) {
          const uint32_t xs = xt ? item + xoff_t : (on ? item + xoff_r : xzero);
          const int xd = xt ? xd_t : 16, xu = xt ? 1024 : kUnitK * 2;
          // item c's first column; items past kfull (a K tail) have one chunk
          const int kc = c * iu * kUnitK;
          if (fmt == VG_FMT_NVFP4) {
            const uint32_t scl = item + kItemScaleOff + warp * kNvScaleChunkBytes;
            // warp-uniform test (mma.sync needs the whole warp): the item's
            // whole column range lies inside K
            if (c < kfull) {
              const uint32_t code = item + warp * kSlotCodeBytes;
              if (xt)
                nv_chunk_full<true>(code, scl, lane, xs, xd, p.m8, p.m64, acc);
              else
                nv_chunk_full<false>(code, scl, lane, xs, xd, p.m8, p.m64, acc);
            } else {
              const int nu = min(kNvChunkUnits, KU - c * kNvChunkUnits);
              nv_chunk_tail(item + warp * nu * kNvUnitBytes, scl, lane, xs, xu, xd, on, nu,
                            K - kc - 16 * t, p.m8, p.m64, acc);
            }
          } else {
            const bool full = c < kfull;
            const int nu = full ? kF8ChunkUnits : min(kF8ChunkUnits, KU - c * kF8ChunkUnits);
            const uint32_t code = item + warp * nu * kF8UnitBytes;
            if (xt)
              f8_chunk<true>(code, lane, xs, xd, on, full, nu, K - kc - 16 * t, acc);
            else
              f8_chunk<false>(code, lane, xs, xd, on, full, nu, K - kc - 16 * t, acc);
          }
        }
        // release the slot to the producer once every warp has read it
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        if (++s == kSlots) {
          s = 0;
          par ^= 1u;
        }
      }

      // ---------------------------------------------- end of the piece
      float accs[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        accs[e] = acc[0][e];
#pragma unroll
        for (int a = 1; a < kAcc; ++a) accs[e] += acc[a][e];
      }
      if (!finish_piece<kFused>(p, mats[cons.mi], cons.items, cons.G, piece_start,
                        c0 == 0 && len == cons.KI, rb, ph, tag, aborted, tl, cc, red, N,
                        accs[0], accs[1], accs[2], accs[3]))
        aborted = true;
      cons.skip(len, mats, phases, p);
    }
  }

  // The last block out resets the per-phase completion counters and
  // advances the pass epoch, so that the next pass's partial sums carry new
  // tags.  Before the tags would overflow 32 bits the epoch restarts at 0
  // and every slot that a call sharing this workspace may have written is
  // cleared (tag 0 never matches): a slot written by an earlier call with a
  // larger grid would otherwise carry a tag that becomes valid again.
  __syncthreads();
  if (tid == 0) sflag[2] = atom_add_relaxed(p.ctas_done, 1u) == uint32_t(p.grid - 1) ? 1 : 0;
  __syncthreads();
  if (sflag[2]) {
    if (tid == 0) {
      fence_acq_rel_gpu();    // every other block has finished with the state
      if (p.done)
        for (int ph = 0; ph < p.nphases; ++ph) p.done[ph] = 0u;
      const bool wrap = (uint64_t(epoch) + 2u) * uint64_t(p.nphases) > 0xFFFFFFFFull;
      *p.epoch = wrap ? 0u : epoch + 1u;
      *p.ctas_done = 0u;
      sflag[0] = wrap ? 1 : 0;
    }
    __syncthreads();
    if (sflag[0]) {
      uint4 *dst = reinterpret_cast<uint4 *>(p.partials);
      const int64_t n = p.clear_words / 2;
      for (int64_t k = tid; k < n; k += kKernelThreads) dst[k] = make_uint4(0, 0, 0, 0);
    }
  }
}

// Passes of 9..32 columns (NB = 2 or 4 blocks of 8): the kernel above with
// wider accumulators and x slices, for plain products whose items are whole
// in K and take x by tensor copy, so that the streaming loop does all of the
// work.  A kernel of its own: folding it into the one above changes how that
// one's registers are allocated, which costs the 8-column passes measurably.
template <int NB>
__global__ void __launch_bounds__(kKernelThreads, 1) stream_kernel_wide(const __grid_constant__ Params p) {
  static_assert(NB > 1 && kAcc == 1, "wide passes: one accumulator chain per column block");
  constexpr bool kFused = false;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the swizzled tensor copies need 1024-byte alignment in shared memory
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kBarOff);
  volatile int *sflag = reinterpret_cast<volatile int *>(smem + kBarOff + kBarBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const MatDev *mats = p.mats ? p.mats : &p.mat0;
  const PhaseDev *phases = p.mats ? p.phases : &p.phase0;

  if (tid * 16 < kXRowBytes)
    *reinterpret_cast<uint4 *>(smem + kZeroRowOff + tid * 16) = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_addr(bars + i), 1);                       // full: the slot's producer
      mbar_init(smem_addr(bars + kSlots + i), kWarps);         // empty: every consumer warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sflag[0] = 0;
    sflag[1] = int(ld_relaxed(p.epoch));
    sflag[2] = 0;
    sflag[3] = 0;   // consumers waiting on a group dependency
    // the pass's width: fixed, or read from the width word at launch
    int n = p.N;
    if (p.width) {
      n = ld_relaxed(reinterpret_cast<const uint32_t *>(p.width));
      if (n < 1 || n > p.N) {
        if (blockIdx.x == 0) set_error(p.error, kErrWidth);
        n = 0;   // no work: every block goes straight to the end of the pass
      }
    }
    sflag[4] = n;
  }
  __syncthreads();
  const uint32_t epoch = uint32_t(sflag[1]);
  const int N = sflag[4];

  if (N == 0) {
    // invalid width: nothing is read or written
  } else if (warp >= kWarps) {
    // ================================================================ producer
    const int np = p.mats ? kProducers : 1;
    if (lane == 0 && warp - kWarps < np)
      producer<false, NB>(p, mats, phases, smem_addr(smem), smem_addr(bars), smem_addr(bars + kSlots),
               sflag + 3, warp - kWarps, np, N);

  } else {
    // =============================================================== consumers
    const int g = lane >> 2, t = lane & 3;
    const bool on = g < N;
    const uint32_t ring = smem_addr(smem);
    const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + kSlots);
    // This lane's x columns inside an item slot.  Tensor-copied slices are
    // [unit][row][128 B] with the 16-byte chunks of row r at chunk ^ (r % 8)
    // (128-byte swizzle), so a unit is 1024 bytes and the lane's two chunks
    // 2t, 2t+1 of row g sit at (2t ^ g) and next to it.  Row-copied slices
    // are padded rows of kXRowBytes, and a column g >= N reads a zero row.
    const uint32_t xoff_t0 = uint32_t(kItemXOff + g * 128 + ((2 * t) ^ g) * 16);
    const int xd_t = (g & 1) ? -16 : 16;
    const uint32_t xoff_r = uint32_t(kItemXOff + g * kXRowBytes + t * 32);
    const uint32_t xzero = smem_addr(smem + kZeroRowOff) + t * 32;
    Seq cons;
    cons.init(mats, phases, p);
    bool aborted = false;
    int s = 0;                     // ring slot of the current item
    uint32_t par = 0;              // parity of that slot's current phase
    int cur_ph = -1, cur_mi = -1;
    uint32_t tag = 0;              // tag of this pass and phase
    float acc[NB * kAcc][4];
    // matrix fields cached while the matrix does not change
    int K = 0, KU = 0, MT = 0, fmt = 0, rt = kBlockTiles, kfull = 0, iu = 0;
    int tl = warp, cc = 0;         // this warp's tile and chunk within an item
    uint32_t xoff_t = xoff_t0;     // ... and its x columns (tensor-copied x)
    bool xt = false;               // the matrix's x slice is tensor-copied
    const uint32_t red = smem_addr(smem + kRedOff);   // tile-sum scratch
    while (cons.valid) {
      const int ph = cons.ph;
      // -------------------------------------- ordered: wait for group ph-1
      if (ph != cur_ph) {
        if (p.ordered && ph > 0) {
          if (tid == 0) {
            int ok = 1;
            if (!aborted) {
              const uint32_t *d = p.done + (ph - 1);
              sflag[3] = 1;
              const uint32_t target = uint32_t(phases[ph - 1].rbs);
              if (ld_acquire(d) < target) {
                const uint64_t deadline = globaltimer() + p.timeout_ns;
                uint32_t it = 0;
                // one L2 round trip per poll: the clock and the error word
                // are looked at every 8th poll only
                while (ld_acquire(d) < target) {
                  if ((++it & 7u) == 0) {
                    if (globaltimer() > deadline) {
                      ok = 0;
                      set_error(p.error, kErrDepWait);
                      break;
                    }
                    if (ld_relaxed(reinterpret_cast<const uint32_t *>(p.error)) != 0) {
                      ok = 0;   // another block has failed: results are void
                      break;
                    }
                  }
                  __nanosleep(32);
                }
              }
            }
            sflag[3] = 0;
            sflag[0] = ok ? 0 : 1;
          }
          named_bar(1, kConsumers);
          if (sflag[0]) aborted = true;
          named_bar(1, kConsumers);
        }
        cur_ph = ph;
        tag = epoch * uint32_t(p.nphases) + uint32_t(ph) + 1u;
      }
      if (cons.mi != cur_mi) {
        const MatDev &mm = mats[cons.mi];
        cur_mi = cons.mi;
        K = mm.K;
        KU = mm.KU;
        MT = mm.MT;
        fmt = mm.fmt;
        rt = mm.rt;
        iu = mm.iu;
        kfull = mm.kfull;
        tl = warp / mm.cpi;
        cc = warp - tl * mm.cpi;
        // the warp's chunk starts cc chunks into the item's x slice
        xoff_t = xoff_t0 + uint32_t(cc * mm.cu * 1024 * NB);
        xt = p.mats ? mm.xmap != nullptr : p.x0_tensor != 0;
      }
      if (kFused && fmt == kFmtNorm) {
        // an RMS-norm item: its slot carries no data (take it and give it
        // back), this block's consumers normalise x into y, and the item
        // completes its phase
        if (!aborted) {
          const bool ready = mbar_wait_for(full0 + 8 * s, par, p.timeout_ns);
          if (!__all_sync(0xFFFFFFFFu, ready)) {
            if (lane == 0) set_error(p.error, kErrFullWait);
            aborted = true;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        if (++s == kSlots) {
          s = 0;
          par ^= 1u;
        }
        rms_norm_item(mats[cons.mi], N, reinterpret_cast<float *>(smem + kRedOff), !aborted,
                      cons.rb, 0u);
        if (tid == 0 && !aborted && ph != p.hold_phase) red_add_release(p.done + ph, 1u);
        cons.skip(1, mats, phases, p);
        continue;
      }
      // ------------------------------------------------- one row-block piece
      // the block's contiguous items of one row block: set up once, then a
      // tight loop over its chunks
      const int rb = cons.rb, c0 = cons.c;
      const int len = min(cons.KI - c0, cons.i1 - cons.i);
      const int piece_start = cons.i;
#pragma unroll
      for (int a = 0; a < NB * kAcc; ++a)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[a][e] = 0.f;
      const int mt = rb * rt + tl;
      const bool work = mt < MT;
      int c = c0;
      const int c_end = c0 + len;
      // Fast loop: the common case (tensor-copied x, chunks wholly inside K,
      // the warp's tile inside M) with nothing decided per item but the wait.
      if (!aborted && work && xt) {
        if constexpr (NB > 1) {
          // wider passes: whole chunks only, so this loop does all the work
          const uint32_t code0 = warp * kSlotCodeBytes;
          const uint32_t scl_nv = kItemScaleOff + warp * kNvScaleChunkBytes;
          const uint32_t scl_b = kItemScaleOff + warp * kMxScaleChunkBytes +
                                 (fmt == VG_FMT_MXFP8 ? uint32_t(g * 2 + (t >> 1)) * 8u
                                                      : uint32_t(g) * 16u);
          const int c_full = min(c_end, kfull);
          for (; c < c_full; ++c) {
            const uint32_t item = ring + s * kItemSlotBytes;
            if (!__all_sync(0xFFFFFFFFu, mbar_try_wait(full0 + 8 * s, par)) &&
                !__all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8 * s, par, globaltimer() + p.timeout_ns)))
              break;
            if (fmt == VG_FMT_NVFP4)
              nv_chunk_wide<NB>(item + code0, item + scl_nv, lane, item + xoff_t, xd_t, p.m8, p.m64,
                                acc);
            else if (fmt == VG_FMT_FP8_ROWSCALE)
              f8_chunk_wide<NB, false>(item + code0, 0u, lane, item + xoff_t, xd_t, acc);
            else if (fmt == VG_FMT_MXFP8)
              f8_chunk_wide<NB, true>(item + code0, item + scl_b, lane, item + xoff_t, xd_t, acc);
            else
              i4_chunk_wide<NB>(item + code0, item + scl_b, lane, item + xoff_t, xd_t, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
            if (++s == kSlots) {
              s = 0;
              par ^= 1u;
            }
          }
          if (c < c_full) {
            if (lane == 0) set_error(p.error, kErrFullWait);
            aborted = true;
          }
        } else {
          const uint32_t scl0 = kItemScaleOff + warp * kNvScaleChunkBytes;
          const uint32_t code0 = warp * kSlotCodeBytes;
          const int c_full = min(c_end, kfull);
          if (fmt == VG_FMT_NVFP4) {
            for (; c < c_full; ++c) {
              const uint32_t item = ring + s * kItemSlotBytes;
              if (!__all_sync(0xFFFFFFFFu, mbar_try_wait(full0 + 8 * s, par)) &&
                  !__all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8 * s, par, globaltimer() + p.timeout_ns)))
                break;   // the general loop below records the failure
              // releases the slot itself, before computing its last two units
              nv_chunk_full<true>(item + code0, item + scl0, lane, item + xoff_t, xd_t, p.m8, p.m64,
                                  acc, empty0 + 8 * s);
              if (++s == kSlots) {
                s = 0;
                par ^= 1u;
              }
            }
          } else if (fmt == VG_FMT_MXFP8 || fmt == VG_FMT_INT4G) {
            // these formats take whole chunks and tensor-copied x only, so
            // this loop does all of their work
            const bool mx = fmt == VG_FMT_MXFP8;
            const uint32_t scl_l = kItemScaleOff + warp * kMxScaleChunkBytes +
                                   (mx ? uint32_t(g * 2 + (t >> 1)) * 8u : uint32_t(g) * 16u);
            for (; c < c_full; ++c) {
              const uint32_t item = ring + s * kItemSlotBytes;
              if (!__all_sync(0xFFFFFFFFu, mbar_try_wait(full0 + 8 * s, par)) &&
                  !__all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8 * s, par, globaltimer() + p.timeout_ns)))
                break;
              if (mx) {
                mx_chunk(item + code0, item + scl_l, lane, item + xoff_t, xd_t, acc);
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * s);
              } else {
                // releases the slot itself, before computing its last unit
                i4_chunk(item + code0, item + scl_l, lane, item + xoff_t, xd_t, acc, empty0 + 8 * s);
              }
              if (++s == kSlots) {
                s = 0;
                par ^= 1u;
              }
            }
            if (c < c_full) {          // a wait ran out: nothing else computes them
              if (lane == 0) set_error(p.error, kErrFullWait);
              aborted = true;
            }
          } else {
            for (; c < c_full; ++c) {
              const uint32_t item = ring + s * kItemSlotBytes;
              if (!__all_sync(0xFFFFFFFFu, mbar_try_wait(full0 + 8 * s, par)) &&
                  !__all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8 * s, par, globaltimer() + p.timeout_ns)))
                break;
              f8_chunk<true>(item + code0, lane, item + xoff_t, xd_t, true, true, kF8ChunkUnits, 0,
                             acc);
              __syncwarp();
              if (lane == 0) mbar_arrive(empty0 + 8 * s);
              if (++s == kSlots) {
                s = 0;
                par ^= 1u;
              }
            }
          }
        }
      }
      // General loop: the rest of the piece (K tails, row-copied x, tiles past
      // M, a failed wait).
      for (; c < c_end; ++c) {
        const uint32_t item = ring + s * kItemSlotBytes;
        if (!aborted) {
          // every lane polls; a lane whose wait ran out stops the whole
          // warp, since mma.sync needs all of it
          const bool ready = mbar_wait_for(full0 + 8 * s, par, p.timeout_ns);
          if (!__all_sync(0xFFFFFFFFu, ready)) {
            if (lane == 0) set_error(p.error, kErrFullWait);
            aborted = true;
          }
        }
        if constexpr (NB == 1) {
          if (!aborted && work && fmt <= VG_FMT_FP8_ROWSCALE) {
            const uint32_t xs = xt ? item + xoff_t : (on ? item + xoff_r : xzero);
            const int xd = xt ? xd_t : 16, xu = xt ? 1024 : kUnitK * 2;
            // item c's first column; items past kfull (a K tail) have one chunk
            const int kc = c * iu * kUnitK;
            if (fmt == VG_FMT_NVFP4) {
              const uint32_t scl = item + kItemScaleOff + warp * kNvScaleChunkBytes;
              // warp-uniform test (mma.sync needs the whole warp): the item's
              // whole column range lies inside K
              if (c < kfull) {
                const uint32_t code = item + warp * kSlotCodeBytes;
                if (xt)
                  nv_chunk_full<true>(code, scl, lane, xs, xd, p.m8, p.m64, acc);
                else
                  nv_chunk_full<false>(code, scl, lane, xs, xd, p.m8, p.m64, acc);
              } else {
                const int nu = min(kNvChunkUnits, KU - c * kNvChunkUnits);
                nv_chunk_tail(item + warp * nu * kNvUnitBytes, scl, lane, xs, xu, xd, on, nu,
                              K - kc - 16 * t, p.m8, p.m64, acc);
              }
            } else {
              const bool full = c < kfull;
              const int nu = full ? kF8ChunkUnits : min(kF8ChunkUnits, KU - c * kF8ChunkUnits);
              const uint32_t code = item + warp * nu * kF8UnitBytes;
              if (xt)
                f8_chunk<true>(code, lane, xs, xd, on, full, nu, K - kc - 16 * t, acc);
              else
                f8_chunk<false>(code, lane, xs, xd, on, full, nu, K - kc - 16 * t, acc);
            }
          }
        }
        // release the slot to the producer once every warp has read it
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        if (++s == kSlots) {
          s = 0;
          par ^= 1u;
        }
      }

      // ---------------------------------------------- end of the piece
      if constexpr (NB > 1) {
        if (!finish_piece_wide<NB>(p, mats[cons.mi], cons.items, cons.G, piece_start,
                                   c0 == 0 && len == cons.KI, rb, ph, tag, aborted, tl, cc, red, N,
                                   acc))
          aborted = true;
      } else {
        float accs[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          accs[e] = acc[0][e];
#pragma unroll
          for (int a = 1; a < kAcc; ++a) accs[e] += acc[a][e];
        }
        if (!finish_piece<kFused>(p, mats[cons.mi], cons.items, cons.G, piece_start,
                          c0 == 0 && len == cons.KI, rb, ph, tag, aborted, tl, cc, red, N,
                          accs[0], accs[1], accs[2], accs[3]))
          aborted = true;
      }
      cons.skip(len, mats, phases, p);
    }
  }

  // The last block out resets the per-phase completion counters and
  // advances the pass epoch, so that the next pass's partial sums carry new
  // tags.  Before the tags would overflow 32 bits the epoch restarts at 0
  // and every slot that a call sharing this workspace may have written is
  // cleared (tag 0 never matches): a slot written by an earlier call with a
  // larger grid would otherwise carry a tag that becomes valid again.
  __syncthreads();
  if (tid == 0) sflag[2] = atom_add_relaxed(p.ctas_done, 1u) == uint32_t(p.grid - 1) ? 1 : 0;
  __syncthreads();
  if (sflag[2]) {
    if (tid == 0) {
      fence_acq_rel_gpu();    // every other block has finished with the state
      if (p.done)
        for (int ph = 0; ph < p.nphases; ++ph) p.done[ph] = 0u;
      const bool wrap = (uint64_t(epoch) + 2u) * uint64_t(p.nphases) > 0xFFFFFFFFull;
      *p.epoch = wrap ? 0u : epoch + 1u;
      *p.ctas_done = 0u;
      sflag[0] = wrap ? 1 : 0;
    }
    __syncthreads();
    if (sflag[0]) {
      uint4 *dst = reinterpret_cast<uint4 *>(p.partials);
      const int64_t n = p.clear_words / 2;
      for (int64_t k = tid; k < n; k += kKernelThreads) dst[k] = make_uint4(0, 0, 0, 0);
    }
  }
}

// ================================================================ host side

namespace {

struct DeviceInfo {
  int sms = 0;
  int cc = 0;
  int per_sm = 0;          // resident blocks per SM of every kernel instantiation
  bool attr_set = false;
};
std::mutex g_mu;
DeviceInfo g_dev[64];

// The kernel instantiations: plain N <= 8, fused N <= 8, plain N <= 16,
// plain N <= 32.
const void *const *kernels() {
  static const void *const fns[4] = {
      reinterpret_cast<const void *>(&stream_kernel<false>),
      reinterpret_cast<const void *>(&stream_kernel<true>),
      reinterpret_cast<const void *>(&stream_kernel_wide<2>),
      reinterpret_cast<const void *>(&stream_kernel_wide<4>)};
  return fns;
}
inline int kernel_index(bool fused, int nb) { return nb == 1 ? (fused ? 1 : 0) : nb == 2 ? 2 : 3; }
// Column blocks of 8 for N columns.
inline int col_blocks(int N) { return N <= 8 ? 1 : N <= 16 ? 2 : 4; }

vg_status device_info(int *dev_out, DeviceInfo **info) {
  int dev = 0;
  VG_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return VG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo &d = g_dev[dev];
  if (!d.attr_set) {
    int major = 0, minor = 0;
    VG_CUDA(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev));
    VG_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    VG_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    d.cc = major * 10 + minor;
    if (d.cc != 103) return VG_ERR_UNSUPPORTED;
    for (int k = 0; k < 4; ++k)
      VG_CUDA(cudaFuncSetAttribute(kernels()[k], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kSmemBytes));
    // every instantiation has the same threads and shared memory, and the
    // launch bounds cap their registers alike
    VG_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.per_sm, stream_kernel<true>,
                                                          kKernelThreads, kSmemBytes));
    d.attr_set = true;
  }
  *dev_out = dev;
  *info = &d;
  return VG_OK;
}

// The tensor-map encoder of the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

// x viewed as [K/64 units][N rows][64 columns] (strides 128 bytes and 2K
// bytes), copied in boxes of `units` units x 8 rows with the 128-byte
// swizzle; rows >= N and units past K read as zeros.  False when K is not a
// multiple of 64, when N is below kXTensorMinN, or when the driver does not
// take the map: the caller then copies x row by row.
#ifndef VG_XT_MIN_N
#define VG_XT_MIN_N 1
#endif
constexpr int kXTensorMinN = VG_XT_MIN_N;
// The x tensor map of single GEMVs, kept per host thread for the last
// (x, N, K, units, nb): a decode loop calls with the same buffers every
// step, and encoding a map costs host time on every call otherwise.
struct XmapCache {
  const uint16_t *x = nullptr;
  int N = 0, units = 0, nb = 0;
  int64_t K = 0;
  bool ok = false;
  CUtensorMap map;
};

bool make_xmap(CUtensorMap *map, const uint16_t *x, int N, int64_t K, int units, int nb = 1);

bool cached_xmap(CUtensorMap *map, const uint16_t *x, int N, int64_t K, int units, int nb) {
  thread_local XmapCache c;
  if (!(c.x == x && c.N == N && c.K == K && c.units == units && c.nb == nb)) {
    c.ok = make_xmap(&c.map, x, N, K, units, nb);
    c.x = x;
    c.N = N;
    c.K = K;
    c.units = units;
    c.nb = nb;
  }
  if (c.ok) std::memcpy(map, &c.map, sizeof(CUtensorMap));
  return c.ok;
}

bool make_xmap(CUtensorMap *map, const uint16_t *x, int N, int64_t K, int units, int nb) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_tiled();
  if (!fn || K % kUnitK != 0 || N < kXTensorMinN) return false;
  const cuuint64_t dims[3] = {cuuint64_t(kUnitK), cuuint64_t(N), cuuint64_t(K / kUnitK)};
  const cuuint64_t strides[2] = {cuuint64_t(K) * 2, cuuint64_t(kUnitK) * 2};
  const cuuint32_t box[3] = {cuuint32_t(kUnitK), cuuint32_t(8 * nb), cuuint32_t(units)};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t *>(x), dims, strides, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

MatDev make_mat(int fmt, int64_t M, int64_t K, const void *w, const void *sc, const float *rs,
                float gscale, const uint16_t *x, uint16_t *y) {
  MatDev m;
  std::memset(&m, 0, sizeof m);
  m.w = static_cast<const uint8_t *>(w);
  m.sc = static_cast<const uint8_t *>(sc);
  m.rowscale = rs;
  m.x = x;
  m.y = y;
  m.fmt = fmt;
  m.mult = fmt == VG_FMT_NVFP4 ? kNvEpilogueScale * gscale : 1.0f;
  m.M = int(M);
  m.K = int(K);
  m.MT = int(ceil_div(M, kTileRows));
  m.KU = int(ceil_div(K, kUnitK));
  // 4-bit formats: NVFP4 units and chunks; 8-bit formats: FP8 ones
  const bool nib4 = fmt == VG_FMT_NVFP4 || fmt == VG_FMT_INT4G;
  m.cu = nib4 ? kNvChunkUnits : kF8ChunkUnits;
  m.ub = nib4 ? kNvUnitBytes : kF8UnitBytes;
  m.scb = fmt == VG_FMT_NVFP4 ? kNvScaleChunkBytes
        : fmt == VG_FMT_MXFP8 ? kMxScaleChunkBytes
        : fmt == VG_FMT_INT4G ? kI4ScaleChunkBytes : 0;
  m.KC = int(ceil_div(m.KU, m.cu));
  m.rt = layout_rt(M, K, m.cu);
  m.cpi = kBlockTiles / m.rt;
  m.iu = m.cpi * m.cu;
  m.KI = int(ceil_div(m.KU, m.iu));
  m.kfull = int(K / (int64_t(m.iu) * kUnitK));
  m.RB = int(ceil_div(m.MT, m.rt));
  m.rb_bytes = int64_t(m.rt) * m.KU * m.ub;
  m.op = VG_OP_GEMV;
  m.Mo = m.M;
  return m;
}

// An RMS-norm entry: no weights, no copies; its items are slices of y.
MatDev make_norm_mat(int64_t K, const uint16_t *x, uint16_t *y, const uint16_t *gamma, float eps) {
  MatDev m;
  std::memset(&m, 0, sizeof m);
  m.x = x;
  m.y = y;
  m.gamma = gamma;
  m.eps = eps;
  m.fmt = kFmtNorm;
  m.op = VG_OP_RMSNORM;
  m.M = 1;
  m.Mo = int(K);
  m.K = int(K);
  m.MT = m.KU = m.KC = m.KI = 1;
  // one slice of the output per thread block of a pass (items = slices)
  m.RB = int(i64min(kLayoutSMs, K / 8));
  m.cu = kNvChunkUnits;
  m.ub = kNvUnitBytes;
  m.rt = kBlockTiles;
  m.cpi = 1;
  m.iu = kNvChunkUnits;
  return m;
}

int64_t algorithmic_bytes(const MatDev &m) {
  if (m.fmt == kFmtNorm) return 0;                 // no weights
  const int64_t E = int64_t(m.M) * m.K;
  // a gated pair carries the tensor scales of both halves
  const int64_t gs_bytes = m.op == VG_OP_SWIGLU ? 8 : 4;
  switch (m.fmt) {
    case VG_FMT_NVFP4: return E / 2 + E / 16 + gs_bytes;
    case VG_FMT_MXFP8: return E + E / 32;
    case VG_FMT_INT4G: return E / 2 + 2 * (E / kI4GroupK);
    default: return E + 4 * int64_t(m.M);
  }
}

// Single-GEMV workspace: [header words | partial slots].
// Single-GEMV workspace for nb column blocks of 8: one slot of nb blocks'
// partial sums per thread block.
size_t ws_bytes(int grid, int nb = 1) {
  return kWsHead + size_t(grid) * size_t(nb) * kPartialWords * sizeof(uint64_t);
}

// Whether a matrix can run nb > 1 column blocks: whole items in K (the
// streaming loops do all the work) and an x slice of 8 nb rows per unit
// within the slot's x region.
bool wide_ok(const MatDev &m, int nb) {
  return nb == 1 || (m.kfull == m.KI && m.iu * nb <= kMaxItemUnits);
}

void set_head(Params &p, uint8_t *head) {
  p.error = reinterpret_cast<int *>(head);
  p.ctas_done = reinterpret_cast<uint32_t *>(head + 4);
  p.epoch = reinterpret_cast<uint32_t *>(head + 8);
}

// Every block of a pass must be resident at once (a reducer waits for the
// other contributors), which a cooperative launch guarantees.
vg_status launch(const Params &p, vg_stream_t stream) {
  void *args[] = {const_cast<Params *>(&p)};
  const void *fn = kernels()[kernel_index(p.fused != 0, p.nb)];
  VG_CUDA(cudaLaunchCooperativeKernel(fn, dim3(p.grid),
                                      dim3(kKernelThreads), args, kSmemBytes, as_cuda(stream)));
  return VG_OK;
}

// Blocks per pass: one per SM (fewer when there are fewer items), capped by
// what can be resident at once.
vg_status max_grid(const DeviceInfo &d, int *grid) {
  if (d.per_sm < 1) return VG_ERR_UNSUPPORTED;
  *grid = std::min(d.sms, d.per_sm * d.sms);
  return VG_OK;
}

vg_status gemv_common(const MatDev &m0, int N, void *workspace, size_t workspace_bytes,
                      vg_stream_t stream) {
  int dev;
  DeviceInfo *di;
  if (vg_status s = device_info(&dev, &di)) return s;
  const int64_t T = int64_t(m0.RB) * m0.KI;
  const int nb = col_blocks(N);
  if (!wide_ok(m0, nb)) return VG_ERR_UNSUPPORTED;
  int grid = 0;
  if (vg_status s = max_grid(*di, &grid)) return s;
  grid = int(i64min(grid, T));
  if (!workspace || workspace_bytes < ws_bytes(grid, nb)) return VG_ERR_WORKSPACE;
  if (!aligned16(workspace)) return VG_ERR_ALIGNMENT;
  Params p;
  std::memset(&p, 0, sizeof p);
  p.nphases = 1;
  p.N = N;
  p.nb = nb;
  p.ordered = 0;
  p.hold_phase = -1;
  p.grid = grid;
  p.timeout_ns = 2000000000ull;
  p.m8 = 8;
  p.m64 = 64;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  set_head(p, ws);
  p.partials = reinterpret_cast<uint64_t *>(ws + kWsHead);
  // every call on this device has at most di->sms blocks of at most 4
  // column blocks, so no word past that is ever written
  p.clear_words = i64min(int64_t(di->sms) * 4 * kPartialWords,
                         int64_t((workspace_bytes - kWsHead) / sizeof(uint64_t)));
  p.mat0 = m0;
  p.x0_tensor = cached_xmap(&p.xmap0, m0.x, N, m0.K, m0.iu, nb) ? 1 : 0;
  // items of several chunks, the block-scaled formats and wider passes take
  // x by tensor copy only
  if (!p.x0_tensor && (m0.cpi > 1 || m0.fmt >= VG_FMT_MXFP8 || nb > 1)) return VG_ERR_UNSUPPORTED;
  p.phase0.items = int(T);
  p.phase0.rbs = m0.RB;
  p.phase0.mat_begin = 0;
  p.phase0.mat_end = 1;
  return launch(p, stream);
}

}  // namespace
}  // namespace vg

using namespace vg;

struct vg_verify_plan {
  int dev = 0;
  int N = 0;
  int grid = 0;
  int ordered = 1;
  int nphases = 0;
  int64_t bytes = 0;
  Params params;
  MatDev *d_mats = nullptr;
  PhaseDev *d_phases = nullptr;
  CUtensorMap *d_xmaps = nullptr;  // per matrix (unused entries for row-copied x)
  uint8_t *d_state = nullptr;     // error, counters, partials
  size_t state_bytes = 0;
};

extern "C" vg_status vg_gemv_workspace_size(int64_t M, int64_t K, int format, size_t *bytes) {
  if (vg_status s = check_mk(M, K)) return s;
  if (!bytes || format < VG_FMT_NVFP4 || format > VG_FMT_INT4G) return VG_ERR_INVALID_ARG;
  int dev;
  DeviceInfo *di;
  if (vg_status s = device_info(&dev, &di)) return s;
  const MatDev m = make_mat(format, M, K, nullptr, nullptr, nullptr, 0.f, nullptr, nullptr);
  int grid = 0;
  if (vg_status s = max_grid(*di, &grid)) return s;
  *bytes = ws_bytes(int(i64min(grid, int64_t(m.RB) * m.KI)));
  return VG_OK;
}

extern "C" vg_status vg_gemv_workspace_size_n(int64_t M, int64_t K, int format, int N,
                                              size_t *bytes) {
  if (N < 1 || N > 32) return VG_ERR_INVALID_ARG;
  size_t one = 0;
  if (vg_status s = vg_gemv_workspace_size(M, K, format, &one)) return s;
  *bytes = kWsHead + (one - kWsHead) * size_t(col_blocks(N));
  return VG_OK;
}

static vg_status check_gemv_args(const void *w, const void *x, const void *y, int N, int64_t M,
                                 int64_t K) {
  if (vg_status s = check_mk(M, K)) return s;
  if (N < 1 || N > 32 || !w || !x || !y) return VG_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(x) || !aligned16(y)) return VG_ERR_ALIGNMENT;
  return VG_OK;
}

extern "C" vg_status vg_gemv_nvfp4(const void *w, const void *scales, float gscale,
                                   const uint16_t *x, int N, int64_t M, int64_t K, uint16_t *y,
                                   void *workspace, size_t workspace_bytes, vg_stream_t stream) {
  if (vg_status s = check_gemv_args(w, x, y, N, M, K)) return s;
  if (!scales) return VG_ERR_INVALID_ARG;
  if (!aligned16(scales)) return VG_ERR_ALIGNMENT;
  const MatDev m = make_mat(VG_FMT_NVFP4, M, K, w, scales, nullptr, gscale, x, y);
  return gemv_common(m, N, workspace, workspace_bytes, stream);
}

extern "C" vg_status vg_gemv_fp8_rowscale(const void *w, const float *rowscale, const uint16_t *x,
                                          int N, int64_t M, int64_t K, uint16_t *y,
                                          void *workspace, size_t workspace_bytes,
                                          vg_stream_t stream) {
  if (vg_status s = check_gemv_args(w, x, y, N, M, K)) return s;
  if (!rowscale) return VG_ERR_INVALID_ARG;
  const MatDev m = make_mat(VG_FMT_FP8_ROWSCALE, M, K, w, nullptr, rowscale, 0.f, x, y);
  return gemv_common(m, N, workspace, workspace_bytes, stream);
}

// K of the block-scaled formats: whole chunks only, so that their items are
// whole and run in the streaming loops (which also need the x tensor copy).
static vg_status check_block_format(int fmt, int64_t K) {
  if (fmt == VG_FMT_MXFP8 && K % (kF8ChunkUnits * kUnitK) != 0) return VG_ERR_UNSUPPORTED;
  if (fmt == VG_FMT_INT4G && K % (kNvChunkUnits * kUnitK) != 0) return VG_ERR_UNSUPPORTED;
  return VG_OK;
}

static vg_status gemv_block_scaled(int fmt, const void *w, const void *scales, const uint16_t *x,
                                   int N, int64_t M, int64_t K, uint16_t *y, void *workspace,
                                   size_t workspace_bytes, vg_stream_t stream) {
  if (vg_status s = check_gemv_args(w, x, y, N, M, K)) return s;
  if (vg_status s = check_block_format(fmt, K)) return s;
  if (!scales) return VG_ERR_INVALID_ARG;
  if (!aligned16(scales)) return VG_ERR_ALIGNMENT;
  const MatDev m = make_mat(fmt, M, K, w, scales, nullptr, 1.0f, x, y);
  return gemv_common(m, N, workspace, workspace_bytes, stream);
}

extern "C" vg_status vg_gemv_mxfp8(const void *w, const void *scales, const uint16_t *x, int N,
                                   int64_t M, int64_t K, uint16_t *y, void *workspace,
                                   size_t workspace_bytes, vg_stream_t stream) {
  return gemv_block_scaled(VG_FMT_MXFP8, w, scales, x, N, M, K, y, workspace, workspace_bytes,
                           stream);
}

extern "C" vg_status vg_gemv_int4g(const void *w, const void *scales, const uint16_t *x, int N,
                                   int64_t M, int64_t K, uint16_t *y, void *workspace,
                                   size_t workspace_bytes, vg_stream_t stream) {
  return gemv_block_scaled(VG_FMT_INT4G, w, scales, x, N, M, K, y, workspace, workspace_bytes,
                           stream);
}

extern "C" vg_status vg_gemv_workspace_check(void *workspace, size_t workspace_bytes,
                                             int *device_error, vg_stream_t stream) {
  if (!workspace || !device_error || workspace_bytes < kWsHead) return VG_ERR_INVALID_ARG;
  cudaStream_t st = as_cuda(stream);
  int err = 0;
  VG_CUDA(cudaMemcpyAsync(&err, workspace, sizeof err, cudaMemcpyDeviceToHost, st));
  VG_CUDA(cudaStreamSynchronize(st));
  *device_error = err;
  if (err) {
    VG_CUDA(cudaMemsetAsync(workspace, 0, workspace_bytes, st));
    VG_CUDA(cudaStreamSynchronize(st));
    return VG_ERR_TIMEOUT;
  }
  return VG_OK;
}

// -------------------------------------------------------------- verify plan

extern "C" vg_status vg_verify_plan_create_ex(const vg_matrix_desc *mats, int count, int N,
                                              const vg_plan_options *opt,
                                              vg_verify_plan **plan_out) {
  if (!mats || count < 1 || !plan_out || N < 1 || N > 32) return VG_ERR_INVALID_ARG;
  const int nb = col_blocks(N);
  *plan_out = nullptr;
  vg_plan_options o;
  std::memset(&o, 0, sizeof o);
  o.ordered = 1;
  o.hold_group = -1;
  if (opt) o = *opt;
  int dev;
  DeviceInfo *di;
  if (vg_status s = device_info(&dev, &di)) return s;
  int coop = 0;
  VG_CUDA(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev));
  if (!coop) return VG_ERR_UNSUPPORTED;

  std::vector<MatDev> hm(static_cast<size_t>(count));
  std::vector<PhaseDev> hp;
  int64_t bytes = 0;
  int hold_phase = -1;
  for (int i = 0; i < count; ++i) {
    const vg_matrix_desc &d = mats[i];
    if (i > 0 && d.group < mats[i - 1].group) return VG_ERR_INVALID_ARG;
    // fused operations and dependent x need the group order, and 8 columns
    // at most
    if ((d.op != VG_OP_GEMV || d.x_after_group) && !o.ordered) return VG_ERR_INVALID_ARG;
    if ((d.op != VG_OP_GEMV || d.x_after_group) && nb > 1) return VG_ERR_UNSUPPORTED;
    if (d.x_after_group && (i == 0 || d.group == mats[0].group)) return VG_ERR_INVALID_ARG;
    if (d.op == VG_OP_RMSNORM) {
      if (vg_status s = check_mk(1, d.K)) return s;
      if (!d.x || !d.y || !d.gamma || !(d.eps >= 0.0f) || N < 1 || N > 8)
        return VG_ERR_INVALID_ARG;
      if (!aligned16(d.x) || !aligned16(d.y) || !aligned16(d.gamma)) return VG_ERR_ALIGNMENT;
      hm[i] = make_norm_mat(d.K, d.x, d.y, d.gamma, d.eps);
    } else {
      if (d.op != VG_OP_GEMV && d.op != VG_OP_SWIGLU) return VG_ERR_INVALID_ARG;
      if (vg_status s = check_gemv_args(d.w, d.x, d.y, N, d.M, d.K)) return s;
      if (d.format == VG_FMT_NVFP4) {
        if (!d.scales) return VG_ERR_INVALID_ARG;
        if (!aligned16(d.scales)) return VG_ERR_ALIGNMENT;
      } else if (d.format == VG_FMT_FP8_ROWSCALE) {
        if (!d.rowscale) return VG_ERR_INVALID_ARG;
        if (d.op == VG_OP_SWIGLU && !d.rowscale_up) return VG_ERR_INVALID_ARG;
      } else if (d.format == VG_FMT_MXFP8 || d.format == VG_FMT_INT4G) {
        if (!d.scales || d.op != VG_OP_GEMV) return VG_ERR_INVALID_ARG;
        if (!aligned16(d.scales)) return VG_ERR_ALIGNMENT;
        if (vg_status s = check_block_format(d.format, d.K)) return s;
      } else {
        return VG_ERR_INVALID_ARG;
      }
      hm[i] = make_mat(d.format, d.M, d.K, d.w, d.scales, d.rowscale, d.gscale, d.x, d.y);
      if (d.op == VG_OP_SWIGLU) {
        if (d.M % 16 != 0) return VG_ERR_INVALID_ARG;   // I % 8 == 0
        hm[i].op = VG_OP_SWIGLU;
        hm[i].Mo = int(d.M / 2);
        hm[i].mult2 = kNvEpilogueScale * d.gscale_up;
        hm[i].rowscale2 = d.rowscale_up;
      }
    }
    hm[i].x_after = d.x_after_group ? 1 : 0;
    if (!wide_ok(hm[i], nb)) return VG_ERR_UNSUPPORTED;
    const bool new_phase = hp.empty() || (o.ordered && d.group != mats[i - 1].group);
    if (new_phase) {
      PhaseDev ph;
      ph.items = 0;
      ph.rbs = 0;
      ph.mat_begin = i;
      ph.mat_end = i;
      hp.push_back(ph);
      if (o.ordered && d.group == o.hold_group) hold_phase = int(hp.size()) - 1;
    }
    PhaseDev &ph = hp.back();
    hm[i].item0 = ph.items;
    // a phase's items are counted in 32 bits on the device
    if (int64_t(ph.items) + int64_t(hm[i].RB) * hm[i].KI > int64_t(1) << 30) return VG_ERR_UNSUPPORTED;
    ph.items += hm[i].RB * hm[i].KI;
    ph.rbs += hm[i].RB;
    ph.mat_end = i + 1;
    bytes += algorithmic_bytes(hm[i]);
  }
  // a phase whose y a dependent x of the next phase copies in fences its stores
  for (size_t ph = 0; ph + 1 < hp.size(); ++ph) {
    bool next_dep = false;
    for (int j = hp[ph + 1].mat_begin; j < hp[ph + 1].mat_end; ++j) next_dep |= hm[j].x_after != 0;
    if (next_dep)
      for (int j = hp[ph].mat_begin; j < hp[ph].mat_end; ++j) hm[j].y_async = 1;
  }
  int grid = 0;
  if (vg_status s = max_grid(*di, &grid)) return s;
  if (o.max_ctas > 0) grid = std::min(grid, int(o.max_ctas));

  vg_verify_plan *plan = new vg_verify_plan();
  plan->dev = dev;
  plan->N = N;
  plan->grid = grid;
  plan->ordered = o.ordered ? 1 : 0;
  plan->nphases = int(hp.size());
  plan->bytes = bytes;
  const size_t done_bytes = size_t((hp.size() * 4 + 255) / 256 * 256);
  const size_t part_bytes = size_t(grid) * size_t(nb) * kPartialWords * sizeof(uint64_t);
  plan->state_bytes = kWsHead + done_bytes + part_bytes;
  cudaError_t e = cudaMalloc(&plan->d_mats, sizeof(MatDev) * hm.size());
  if (e == cudaSuccess) e = cudaMalloc(&plan->d_phases, sizeof(PhaseDev) * hp.size());
  if (e == cudaSuccess) e = cudaMalloc(&plan->d_state, plan->state_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&plan->d_xmaps, sizeof(CUtensorMap) * hm.size());
  bool untensored = false;   // an item of several chunks whose x has no tensor map
  if (e == cudaSuccess) {
    std::vector<CUtensorMap> maps(hm.size());
    for (size_t i = 0; i < hm.size(); ++i) {
      if (hm[i].fmt == kFmtNorm) continue;   // no copies
      hm[i].xmap =
          make_xmap(&maps[i], hm[i].x, N, hm[i].K, hm[i].iu, nb) ? plan->d_xmaps + i : nullptr;
      if (!hm[i].xmap && (hm[i].cpi > 1 || hm[i].fmt >= VG_FMT_MXFP8 || nb > 1)) untensored = true;
    }
    e = cudaMemcpy(plan->d_xmaps, maps.data(), sizeof(CUtensorMap) * maps.size(),
                   cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess)
    e = cudaMemcpy(plan->d_mats, hm.data(), sizeof(MatDev) * hm.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(plan->d_phases, hp.data(), sizeof(PhaseDev) * hp.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(plan->d_state, 0, plan->state_bytes);
  if (e == cudaSuccess && untensored) {
    // items of several chunks take x by tensor copy only
    vg_verify_plan_destroy(plan);
    return VG_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) {
    set_cuda_error(e);
    vg_verify_plan_destroy(plan);
    return VG_ERR_CUDA;
  }
  Params &p = plan->params;
  std::memset(&p, 0, sizeof p);
  p.mats = plan->d_mats;
  p.phases = plan->d_phases;
  p.nphases = plan->nphases;
  p.N = N;
  p.nb = nb;
  p.ordered = plan->ordered;
  p.hold_phase = hold_phase;
  p.grid = grid;
  p.timeout_ns = o.wait_timeout_ns > 0 ? uint64_t(o.wait_timeout_ns) : 2000000000ull;
  p.m8 = 8;
  p.m64 = 64;
  set_head(p, plan->d_state);
  p.done = plan->ordered ? reinterpret_cast<uint32_t *>(plan->d_state + kWsHead) : nullptr;
  p.partials = reinterpret_cast<uint64_t *>(plan->d_state + kWsHead + done_bytes);
  p.clear_words = int64_t(grid) * nb * kPartialWords;   // the plan's state is its own
  for (const MatDev &m : hm) p.fused |= m.op != VG_OP_GEMV || m.x_after;
  *plan_out = plan;
  return VG_OK;
}

extern "C" vg_status vg_verify_plan_create(const vg_matrix_desc *mats, int count, int N,
                                           int ordered, vg_verify_plan **plan_out) {
  vg_plan_options o;
  std::memset(&o, 0, sizeof o);
  o.ordered = ordered;
  o.hold_group = -1;
  return vg_verify_plan_create_ex(mats, count, N, &o, plan_out);
}

extern "C" vg_status vg_verify_pass(vg_verify_plan *plan, vg_stream_t stream) {
  if (!plan) return VG_ERR_INVALID_ARG;
  int dev = 0;
  VG_CUDA(cudaGetDevice(&dev));
  if (dev != plan->dev) return VG_ERR_INVALID_ARG;
  return launch(plan->params, stream);
}

extern "C" vg_status vg_verify_plan_set_width(vg_verify_plan *plan, const int32_t *d_width) {
  if (!plan) return VG_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(d_width) & 3u) != 0) return VG_ERR_ALIGNMENT;
  plan->params.width = reinterpret_cast<const int *>(d_width);
  return VG_OK;
}

extern "C" vg_status vg_verify_plan_check(vg_verify_plan *plan, vg_stream_t stream,
                                          int *device_error) {
  if (!plan || !device_error) return VG_ERR_INVALID_ARG;
  cudaStream_t st = as_cuda(stream);
  int err = 0;
  VG_CUDA(cudaMemcpyAsync(&err, plan->d_state, sizeof err, cudaMemcpyDeviceToHost, st));
  VG_CUDA(cudaStreamSynchronize(st));
  *device_error = err;
  if (err) {
    VG_CUDA(cudaMemsetAsync(plan->d_state, 0, plan->state_bytes, st));
    VG_CUDA(cudaStreamSynchronize(st));
    return VG_ERR_TIMEOUT;
  }
  return VG_OK;
}

extern "C" vg_status vg_verify_plan_bytes(const vg_verify_plan *plan, int64_t *bytes) {
  if (!plan || !bytes) return VG_ERR_INVALID_ARG;
  *bytes = plan->bytes;
  return VG_OK;
}

extern "C" vg_status vg_verify_plan_grid(const vg_verify_plan *plan, int *ctas) {
  if (!plan || !ctas) return VG_ERR_INVALID_ARG;
  *ctas = plan->grid;
  return VG_OK;
}

extern "C" vg_status vg_verify_plan_destroy(vg_verify_plan *plan) {
  if (!plan) return VG_OK;
  cudaFree(plan->d_mats);
  cudaFree(plan->d_phases);
  cudaFree(plan->d_xmaps);
  cudaFree(plan->d_state);
  delete plan;
  return VG_OK;
}
