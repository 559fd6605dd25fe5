// vg_gemv.cu -- the weight-streaming GEMV for N = 1..8 BF16 columns over
// NVFP4 or row-scaled FP8 weights, as a single product and as a fused,
// ordered verify pass over a layer stack.
//
// What it computes: y[N,M] = x[N,K] . dequant(W)[M,K]^T with FP32
// accumulation (mtp7-device-confidence engine card, Design table, "GEMVs"
// row; the verify pass of the Decode row runs it for 2-8 columns, a draft
// step for one).  Why it is the hot path: a verify pass reads every weight
// once (card, Measured section: 19.26 GB per pass, its time set by the read
// rate), so the kernel is built to stream bytes at HBM speed.
//
// Design (sm_103a):
//  * Persistent thread blocks, one per SM: 8 consumer warps + 1 producer
//    warp.  The producer streams one pipeline stage per work item with 1-D
//    bulk copies (cp.async.bulk) into a 4-deep shared-memory ring guarded by
//    mbarriers; the weights never pass through registers of the producer.
//  * A work item is one chunk (256 columns NVFP4, 128 FP8) of a row block of
//    16 tiles (256 rows); each consumer warp owns 2 tiles and decodes its
//    codes in registers to BF16 A fragments (bit placement + one BF16x2
//    multiply by the block scale, exact) and runs mma.m16n8k16 with x as the
//    B fragment (x read through L1, shared by all warps), accumulating FP32.
//  * Items are split between thread blocks stream-K style (contiguous item
//    ranges of equal length), so every SM streams the same number of bytes.
//    A row block whose K range is split between blocks is summed from FP32
//    partials by the last block to arrive, in block order (deterministic,
//    no spinning); the counter it used is reset for the next call.
//  * Verify pass: matrices are grouped; in ordered mode the consumers of
//    group g wait (bounded) until group g-1 has completed every row block,
//    while the producer keeps prefetching group g's weights.  All waits are
//    bounded by a timeout on %globaltimer and report an error word instead
//    of hanging.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

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
  int M, K, MT, KU, KC, RB;
  int cu, ub;        // units per chunk, bytes per unit
  int64_t rb_bytes;  // code bytes of a full row block (16 tiles x KU units)
  int64_t item0;     // first item of this matrix within its phase
  int64_t rb_base;   // first arrival counter of this matrix
};

struct PhaseDev {
  int64_t items;
  int64_t rbs;
  int mat_begin, mat_end;
};

struct Params {
  const MatDev *mats;       // nullptr: use mat0 / phase0
  const PhaseDev *phases;
  int nphases;
  int N;
  int ordered;
  int hold_phase;
  int grid;
  uint64_t timeout_ns;
  uint32_t *cnt;
  uint32_t *done;           // per-phase completed row blocks (ordered only)
  uint32_t *ctas_done;
  float *partials;          // [grid][2][16 tiles][32 lanes][4]
  int *error;
  uint32_t m8, m64;         // 8 and 64: shift multipliers kept in registers
  MatDev mat0;
  PhaseDev phase0;
};

constexpr int kPartialFloats = kBlockTiles * 32 * 4;   // one slot
constexpr int kRingBytes = kWarps * kSlots * kSlotBytes;
constexpr int kBarBytes = 2 * kWarps * kSlots * 8;
constexpr int kSmemBytes = kRingBytes + kBarBytes + 64;
constexpr int kConsumers = kWarps * 32;
constexpr int kKernelThreads = kConsumers + 32;        // + one producer warp
constexpr int kErrFullWait = 1, kErrEmptyWait = 2, kErrDepWait = 3;

__host__ __device__ inline int64_t i64min(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ inline int64_t i64max(int64_t a, int64_t b) { return a > b ? a : b; }

__host__ __device__ inline int64_t item_begin(int64_t T, int64_t G, int64_t b) {
  return T * b / G;
}
// Block that owns item i of a phase of T items split over G blocks.
__device__ inline int64_t owner(int64_t T, int64_t G, int64_t i) { return ((i + 1) * G - 1) / T; }

__device__ inline void set_error(int *error, int code) { atomicCAS(error, 0, code); }

// Bounded wait with the clock read only after a first miss.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, uint64_t timeout) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait(bar, parity, globaltimer() + timeout);
}

// The items one thread block processes, in order, across all phases: for
// each phase with items for this block, its contiguous range [i0, i1).  The
// position inside the current matrix (row block rb, chunk c) advances
// incrementally; the only divisions happen when a phase starts.
struct Seq {
  const MatDev *mats;
  const PhaseDev *phases;
  int nphases, ph, mi, mend;
  int rb, c, KC, RB;
  int64_t b, grid, G, i, i0, i1, items;
  bool valid;

  __device__ void init(const MatDev *m, const PhaseDev *p, int np, int64_t blk, int64_t g) {
    mats = m;
    phases = p;
    nphases = np;
    b = blk;
    grid = g;
    ph = -1;
    next_phase();
  }
  __device__ void next_phase() {
    for (++ph; ph < nphases; ++ph) {
      items = phases[ph].items;
      G = i64min(grid, items);
      if (b < G) {
        i0 = item_begin(items, G, b);
        i1 = item_begin(items, G, b + 1);
        i = i0;
        mi = phases[ph].mat_begin;
        mend = phases[ph].mat_end;
        while (mi + 1 < mend && i >= mats[mi].item0 + int64_t(mats[mi].RB) * mats[mi].KC) ++mi;
        KC = mats[mi].KC;
        RB = mats[mi].RB;
        const int64_t rel = i - mats[mi].item0;
        rb = int(rel / KC);
        c = int(rel - int64_t(rb) * KC);
        valid = true;
        return;
      }
    }
    valid = false;
  }
  __device__ __forceinline__ void advance() {
    if (++i == i1) {
      next_phase();
      return;
    }
    if (++c == KC) {
      c = 0;
      if (++rb == RB) {
        rb = 0;
        ++mi;
        KC = mats[mi].KC;
        RB = mats[mi].RB;
      }
    }
  }
};

// One NVFP4 unit of one tile: 4 MMAs (k16 steps) into two accumulators.
__device__ __forceinline__ void nv_unit(const uint4 wv, uint32_t fg, uint32_t fg8, const uint4 xa,
                                        const uint4 xb, uint32_t m8, uint32_t m64,
                                        float (&acc0)[4], float (&acc1)[4]) {
  uint32_t a0, a1, a2, a3;
  nv_decode(wv.x, fg, fg8, m8, m64, a0, a1, a2, a3);
  mma_bf16(acc0, a0, a1, a2, a3, xa.x, xa.y);
  nv_decode(wv.y, fg, fg8, m8, m64, a0, a1, a2, a3);
  mma_bf16(acc1, a0, a1, a2, a3, xa.z, xa.w);
  nv_decode(wv.z, fg, fg8, m8, m64, a0, a1, a2, a3);
  mma_bf16(acc0, a0, a1, a2, a3, xb.x, xb.y);
  nv_decode(wv.w, fg, fg8, m8, m64, a0, a1, a2, a3);
  mma_bf16(acc1, a0, a1, a2, a3, xb.z, xb.w);
}

__device__ __forceinline__ void f8_unit(const uint4 w0, const uint4 w1, const uint4 xa,
                                        const uint4 xb, float (&acc0)[4], float (&acc1)[4]) {
  uint32_t a0, a1, a2, a3;
  f8_decode(w0.x, a0, a1);
  f8_decode(w0.y, a2, a3);
  mma_bf16(acc0, a0, a1, a2, a3, xa.x, xa.y);
  f8_decode(w0.z, a0, a1);
  f8_decode(w0.w, a2, a3);
  mma_bf16(acc1, a0, a1, a2, a3, xa.z, xa.w);
  f8_decode(w1.x, a0, a1);
  f8_decode(w1.y, a2, a3);
  mma_bf16(acc0, a0, a1, a2, a3, xb.x, xb.y);
  f8_decode(w1.z, a0, a1);
  f8_decode(w1.w, a2, a3);
  mma_bf16(acc1, a0, a1, a2, a3, xb.z, xb.w);
}

// x fragment of one unit for lane (g, t): the 16 columns at xp as two
// 16-byte loads, or zeros when `on` is false (column g >= N or K padding).
__device__ __forceinline__ void load_x(const uint16_t *xp, bool on, uint4 &xa, uint4 &xb) {
  if (on) {
    xa = ldg128(xp);
    xb = ldg128(xp + 8);
  } else {
    xa = make_uint4(0, 0, 0, 0);
    xb = xa;
  }
}

// A whole NVFP4 chunk (8 units) of this lane's tile: scale pairs from one
// 16-byte load, codes and x for two units at a time, the next pair loaded
// before the current one is multiplied.
__device__ __forceinline__ void nv_chunk_full(uint32_t slot, int lane, const uint16_t *xp,
                                              bool on, uint32_t m8, uint32_t m64,
                                              float (&acc0)[4], float (&acc1)[4]) {
  const uint4 sc = lds128(slot + kSlotCodeBytes + lane * kNvScaleLaneBytes);
  const uint32_t scw[4] = {sc.x, sc.y, sc.z, sc.w};
  uint4 w0 = lds128(slot + lane * 16), w1 = lds128(slot + kNvUnitBytes + lane * 16);
  uint4 x0a, x0b, x1a, x1b;
  load_x(xp, on, x0a, x0b);
  load_x(xp + kUnitK, on, x1a, x1b);
#pragma unroll
  for (int h = 0; h < kNvChunkUnits / 2; ++h) {
    uint4 nw0, nw1, nx0a, nx0b, nx1a, nx1b;
    if (h + 1 < kNvChunkUnits / 2) {
      nw0 = lds128(slot + (2 * h + 2) * kNvUnitBytes + lane * 16);
      nw1 = lds128(slot + (2 * h + 3) * kNvUnitBytes + lane * 16);
      load_x(xp + (2 * h + 2) * kUnitK, on, nx0a, nx0b);
      load_x(xp + (2 * h + 3) * kUnitK, on, nx1a, nx1b);
    }
    // unit 2h uses scale bytes 0,1 of word h; unit 2h+1 bytes 2,3
    nv_unit(w0, nv_scale_pair(scw[h], 0), nv_scale_pair(scw[h], 1), x0a, x0b, m8, m64, acc0,
            acc1);
    nv_unit(w1, nv_scale_pair(scw[h], 2), nv_scale_pair(scw[h], 3), x1a, x1b, m8, m64, acc0,
            acc1);
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
__device__ __forceinline__ void nv_chunk_tail(uint32_t slot, int lane, const uint16_t *xp,
                                              bool on, int nu, int kleft, uint32_t m8,
                                              uint32_t m64, float (&acc0)[4],
                                              float (&acc1)[4]) {
  const uint4 sc = lds128(slot + kSlotCodeBytes + lane * kNvScaleLaneBytes);
  for (int u = 0; u < nu; ++u) {
    const uint4 wv = lds128(slot + u * kNvUnitBytes + lane * 16);
    uint4 xa, xb;
    load_x(xp + u * kUnitK, on && u * kUnitK < kleft, xa, xb);
    const int q = u >> 1;
    const uint32_t word = q == 0 ? sc.x : q == 1 ? sc.y : q == 2 ? sc.z : sc.w;
    const uint32_t b = uint32_t(u & 1) * 2u;
    nv_unit(wv, nv_scale_pair(word, b), nv_scale_pair(word, b + 1), xa, xb, m8, m64, acc0, acc1);
  }
}

// An FP8 chunk: nu (<= 4) units of 1024 bytes.
__device__ __forceinline__ void f8_chunk(uint32_t slot, int lane, const uint16_t *xp, bool on,
                                         int nu, int kleft, float (&acc0)[4],
                                         float (&acc1)[4]) {
#pragma unroll
  for (int u = 0; u < kF8ChunkUnits; ++u) {
    if (u < nu) {
      const uint4 w0 = lds128(slot + u * kF8UnitBytes + lane * 32);
      const uint4 w1 = lds128(slot + u * kF8UnitBytes + lane * 32 + 16);
      uint4 xa, xb;
      load_x(xp + u * kUnitK, on && u * kUnitK < kleft, xa, xb);
      f8_unit(w0, w1, xa, xb, acc0, acc1);
    }
  }
}

// Producer lane `tile` (0..15): refill consumer warp `tile`'s ring, one item
// at a time, as soon as that warp has released the slot.
__device__ void producer(const Params &p, const MatDev *mats, const PhaseDev *phases, int tile,
                         uint32_t ring, uint32_t full0, uint32_t empty0) {
  const uint64_t policy = policy_evict_first();
  Seq q;
  q.init(mats, phases, p.nphases, blockIdx.x, p.grid);
  int s = 0;
  uint32_t par = 0;
  int64_t issued = 0;
  while (q.valid) {
    if (!mbar_wait_for(empty0 + 8 * s, par ^ 1u, p.timeout_ns)) {
      set_error(p.error, kErrEmptyWait);
      break;
    }
    const MatDev &m = mats[q.mi];
    const uint32_t full = full0 + 8 * s;
    const int tiles = min(kBlockTiles, m.MT - q.rb * kBlockTiles);
    if (tile >= tiles) {
      mbar_arrive_expect_tx(full, 0);
    } else {
      const int nu = min(m.cu, m.KU - q.c * m.cu);
      const uint32_t code_bytes = uint32_t(nu * m.ub);
      const int64_t off = int64_t(q.rb) * m.rb_bytes + int64_t(q.c) * tiles * m.cu * m.ub +
                          int64_t(tile) * nu * m.ub;
      const uint32_t slot = ring + s * kSlotBytes;
      if (m.fmt == VG_FMT_NVFP4) {
        mbar_arrive_expect_tx(full, code_bytes + kNvScaleChunkBytes);
        bulk_g2s(slot, m.w + off, code_bytes, full, policy);
        const int64_t soff =
            (int64_t(q.rb) * kBlockTiles * m.KC + int64_t(q.c) * tiles + tile) * kNvScaleChunkBytes;
        bulk_g2s(slot + kSlotCodeBytes, m.sc + soff, kNvScaleChunkBytes, full, policy);
      } else {
        mbar_arrive_expect_tx(full, code_bytes);
        bulk_g2s(slot, m.w + off, code_bytes, full, policy);
      }
    }
    q.advance();
    ++issued;
    if (++s == kSlots) {
      s = 0;
      par ^= 1u;
    }
  }
  // Never leave while a bulk copy may still be writing shared memory.
  for (int64_t k = i64max(0, issued - kSlots); k < issued; ++k)
    mbar_wait_for(full0 + 8 * int(k % kSlots), uint32_t(k / kSlots) & 1u, p.timeout_ns);
}

__global__ void __launch_bounds__(kKernelThreads, 1) stream_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kRingBytes);
  volatile int *sflag = reinterpret_cast<volatile int *>(smem + kRingBytes + kBarBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const MatDev *mats = p.mats ? p.mats : &p.mat0;
  const PhaseDev *phases = p.mats ? p.phases : &p.phase0;

  if (tid < kWarps * kSlots) {
    mbar_init(smem_addr(bars + tid), 1);                       // full
    mbar_init(smem_addr(bars + kWarps * kSlots + tid), 1);     // empty
  }
  if (tid == 0) {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sflag[0] = 0;
    sflag[1] = 0;
  }
  __syncthreads();

  if (warp == kWarps) {
    // ================================================================ producer
    if (lane < kBlockTiles)
      producer(p, mats, phases, lane, smem_addr(smem + lane * kSlots * kSlotBytes),
               smem_addr(bars + lane * kSlots), smem_addr(bars + kWarps * kSlots + lane * kSlots));
  } else {
    // =============================================================== consumers
    const int g = lane >> 2, t = lane & 3;
    const int N = p.N;
    const bool on = g < N;
    const uint32_t ring = smem_addr(smem + warp * kSlots * kSlotBytes);
    const uint32_t full0 = smem_addr(bars + warp * kSlots);
    const uint32_t empty0 = smem_addr(bars + kWarps * kSlots + warp * kSlots);
    Seq cons;
    cons.init(mats, phases, p.nphases, blockIdx.x, p.grid);
    bool aborted = false;
    int s = 0;                     // ring slot of the current item
    uint32_t par = 0;              // parity of that slot's current phase
    int cur_ph = -1, cur_mi = -1;
    int64_t piece_start = 0;
    int piece_c0 = 0;
    float acc0[4], acc1[4];
    // matrix fields cached while the matrix does not change
    const uint16_t *xbase = nullptr;
    int K = 0, KU = 0, MT = 0, fmt = 0;
    while (cons.valid) {
      const int ph = cons.ph;
      // -------------------------------------- ordered: wait for group ph-1
      if (ph != cur_ph) {
        if (p.ordered && ph > 0) {
          if (tid == 0) {
            int ok = 1;
            if (!aborted) {
              const volatile uint32_t *d = p.done + (ph - 1);
              const uint32_t target = uint32_t(phases[ph - 1].rbs);
              const uint64_t deadline = globaltimer() + p.timeout_ns;
              while (*d < target) {
                if (globaltimer() > deadline) {
                  ok = 0;
                  set_error(p.error, kErrDepWait);
                  break;
                }
                __nanosleep(32);
              }
              __threadfence();
            }
            sflag[0] = ok ? 0 : 1;
          }
          named_bar(1, kConsumers);
          if (sflag[0]) aborted = true;
          named_bar(1, kConsumers);
        }
        cur_ph = ph;
      }
      if (cons.mi != cur_mi) {
        const MatDev &mm = mats[cons.mi];
        cur_mi = cons.mi;
        K = mm.K;
        KU = mm.KU;
        MT = mm.MT;
        fmt = mm.fmt;
        xbase = mm.x + int64_t(g) * K + 16 * t;
      }
      const int rb = cons.rb, c = cons.c;
      if (c == 0 || cons.i == cons.i0) {
        piece_start = cons.i;
        piece_c0 = c;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc0[e] = acc1[e] = 0.f;
      }
      const uint32_t slot = ring + s * kSlotBytes;
      const int mt = rb * kBlockTiles + warp;
      if (!aborted && !mbar_wait_for(full0 + 8 * s, par, p.timeout_ns)) {
        if (lane == 0) set_error(p.error, kErrFullWait);
        aborted = true;
      }
      if (!aborted && mt < MT) {
        if (fmt == VG_FMT_NVFP4) {
          const int kc = c * (kNvChunkUnits * kUnitK);
          // warp-uniform test (mma.sync needs the whole warp): the chunk's
          // whole column range lies inside K
          if (kc + kNvChunkUnits * kUnitK <= K)
            nv_chunk_full(slot, lane, xbase + kc, on, p.m8, p.m64, acc0, acc1);
          else
            nv_chunk_tail(slot, lane, xbase + kc, on, min(kNvChunkUnits, KU - c * kNvChunkUnits),
                          K - kc - 16 * t, p.m8, p.m64, acc0, acc1);
        } else {
          const int kc = c * (kF8ChunkUnits * kUnitK);
          f8_chunk(slot, lane, xbase + kc, on, min(kF8ChunkUnits, KU - c * kF8ChunkUnits),
                   K - kc - 16 * t, acc0, acc1);
        }
      }
      // release the slot to the producer (every lane has read it)
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
      if (++s == kSlots) {
        s = 0;
        par ^= 1u;
      }

      // ---------------------------------------------- end of a row-block piece
      const bool piece_end = c == cons.KC - 1 || cons.i == cons.i1 - 1;
      if (piece_end) {
        const MatDev &m = mats[cons.mi];
        const int64_t T = cons.items, G = cons.G, i0 = cons.i0;
        const bool full_piece = piece_c0 == 0 && c == m.KC - 1;
        float acc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = acc0[e] + acc1[e];
        bool write_out = true;
        if (!full_piece) {
          // partial sums: stash, count arrivals, the last arrival reduces
          const int slotp = int(2 * blockIdx.x + (piece_start == i0 ? 0 : 1));
          float *part = p.partials + int64_t(slotp) * kPartialFloats;
          if (!aborted)
            *reinterpret_cast<float4 *>(part + (warp * 32 + lane) * 4) =
                make_float4(acc[0], acc[1], acc[2], acc[3]);
          named_bar(1, kConsumers);
          const int64_t first = m.item0 + int64_t(rb) * m.KC, last = first + m.KC - 1;
          const int64_t bf = owner(T, G, first), bl = owner(T, G, last);
          if (tid == 0) {
            int is_last = 0;
            if (!aborted) {
              __threadfence();       // publish this block's partials (cumulative)
              uint32_t *cnt = p.cnt + m.rb_base + rb;
              const uint32_t old = atomicAdd(cnt, 1u);
              is_last = old == uint32_t(bl - bf);
              if (is_last) {
                *cnt = 0u;
                __threadfence();     // acquire the other blocks' partials
              }
            }
            sflag[1] = is_last;
          }
          named_bar(1, kConsumers);
          write_out = sflag[1] != 0;
          named_bar(1, kConsumers);
          if (write_out) {
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = 0.f;
            for (int64_t bb = bf; bb <= bl; ++bb) {
              const int64_t ss = 2 * bb + (item_begin(T, G, bb) >= first ? 0 : 1);
              const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                  p.partials + ss * kPartialFloats + (warp * 32 + lane) * 4));
              acc[0] += v.x;
              acc[1] += v.y;
              acc[2] += v.z;
              acc[3] += v.w;
            }
          }
        }
        if (write_out) {
          if (!aborted && mt < m.MT) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int row = mt * kTileRows + g + 8 * h;
              if (row >= m.M) continue;
              const float mult = m.fmt == VG_FMT_NVFP4 ? m.mult : __ldg(m.rowscale + row);
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int nn = 2 * t + e;
                if (nn < N) {
                  const __nv_bfloat16 v = __float2bfloat16_rn(acc[2 * h + e] * mult);
                  m.y[int64_t(nn) * m.M + row] = *reinterpret_cast<const uint16_t *>(&v);
                }
              }
            }
          }
          if (p.done) {
            named_bar(1, kConsumers);
            if (tid == 0 && !aborted && ph != p.hold_phase) {
              __threadfence();       // publish the row block's y (cumulative)
              atomicAdd(p.done + ph, 1u);
            }
          }
        }
      }
      cons.advance();
    }
  }

  // The last block out resets the per-phase completion counters.
  __syncthreads();
  if (p.done && tid == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(p.ctas_done, 1u);
    if (old == uint32_t(p.grid - 1)) {
      for (int ph = 0; ph < p.nphases; ++ph) p.done[ph] = 0u;
      *p.ctas_done = 0u;
      __threadfence();
    }
  }
}

// ================================================================ host side

namespace {

struct DeviceInfo {
  int sms = 0;
  int cc = 0;
  bool attr_set = false;
};
std::mutex g_mu;
DeviceInfo g_dev[64];

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
    VG_CUDA(cudaFuncSetAttribute(stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes));
    d.attr_set = true;
  }
  *dev_out = dev;
  *info = &d;
  return VG_OK;
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
  m.cu = fmt == VG_FMT_NVFP4 ? kNvChunkUnits : kF8ChunkUnits;
  m.ub = fmt == VG_FMT_NVFP4 ? kNvUnitBytes : kF8UnitBytes;
  m.KC = int(ceil_div(m.KU, m.cu));
  m.RB = int(ceil_div(m.MT, kBlockTiles));
  m.rb_bytes = int64_t(kBlockTiles) * m.KU * m.ub;
  return m;
}

int64_t algorithmic_bytes(const MatDev &m) {
  const int64_t E = int64_t(m.M) * m.K;
  return m.fmt == VG_FMT_NVFP4 ? E / 2 + E / 16 + 4 : E + 4 * int64_t(m.M);
}

// Single-GEMV workspace: [error word | counters | partial slots].
constexpr size_t kWsHead = 256;
size_t ws_counters_bytes(int64_t RB) { return size_t((RB * 4 + 255) / 256 * 256); }
size_t ws_bytes(int64_t RB, int grid) {
  return kWsHead + ws_counters_bytes(RB) + size_t(grid) * 2 * kPartialFloats * sizeof(float);
}

vg_status gemv_common(const MatDev &m0, int N, void *workspace, size_t workspace_bytes,
                      vg_stream_t stream) {
  int dev;
  DeviceInfo *di;
  if (vg_status s = device_info(&dev, &di)) return s;
  const int64_t T = int64_t(m0.RB) * m0.KC;
  const int grid = int(i64min(di->sms, T));
  if (!workspace || workspace_bytes < ws_bytes(m0.RB, grid)) return VG_ERR_WORKSPACE;
  if (!aligned16(workspace)) return VG_ERR_ALIGNMENT;
  Params p;
  std::memset(&p, 0, sizeof p);
  p.nphases = 1;
  p.N = N;
  p.ordered = 0;
  p.hold_phase = -1;
  p.grid = grid;
  p.timeout_ns = 2000000000ull;
  p.m8 = 8;
  p.m64 = 64;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  p.error = reinterpret_cast<int *>(ws);
  p.cnt = reinterpret_cast<uint32_t *>(ws + kWsHead);
  p.partials = reinterpret_cast<float *>(ws + kWsHead + ws_counters_bytes(m0.RB));
  p.mat0 = m0;
  p.phase0.items = T;
  p.phase0.rbs = m0.RB;
  p.phase0.mat_begin = 0;
  p.phase0.mat_end = 1;
  stream_kernel<<<grid, kKernelThreads, kSmemBytes, as_cuda(stream)>>>(p);
  VG_LAUNCH_CHECK();
  return VG_OK;
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
  uint8_t *d_state = nullptr;     // error, counters, partials
  size_t state_bytes = 0;
};

extern "C" vg_status vg_gemv_workspace_size(int64_t M, int64_t K, int format, size_t *bytes) {
  if (vg_status s = check_mk(M, K)) return s;
  if (!bytes || (format != VG_FMT_NVFP4 && format != VG_FMT_FP8_ROWSCALE)) return VG_ERR_INVALID_ARG;
  int dev;
  DeviceInfo *di;
  if (vg_status s = device_info(&dev, &di)) return s;
  const MatDev m = make_mat(format, M, K, nullptr, nullptr, nullptr, 0.f, nullptr, nullptr);
  const int grid = int(i64min(di->sms, int64_t(m.RB) * m.KC));
  *bytes = ws_bytes(m.RB, grid);
  return VG_OK;
}

static vg_status check_gemv_args(const void *w, const void *x, const void *y, int N, int64_t M,
                                 int64_t K) {
  if (vg_status s = check_mk(M, K)) return s;
  if (N < 1 || N > 8 || !w || !x || !y) return VG_ERR_INVALID_ARG;
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
  if (!mats || count < 1 || !plan_out || N < 1 || N > 8) return VG_ERR_INVALID_ARG;
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
  int64_t rb_total = 0, bytes = 0;
  int hold_phase = -1;
  for (int i = 0; i < count; ++i) {
    const vg_matrix_desc &d = mats[i];
    if (vg_status s = check_gemv_args(d.w, d.x, d.y, N, d.M, d.K)) return s;
    if (i > 0 && d.group < mats[i - 1].group) return VG_ERR_INVALID_ARG;
    if (d.format == VG_FMT_NVFP4) {
      if (!d.scales) return VG_ERR_INVALID_ARG;
      if (!aligned16(d.scales)) return VG_ERR_ALIGNMENT;
    } else if (d.format == VG_FMT_FP8_ROWSCALE) {
      if (!d.rowscale) return VG_ERR_INVALID_ARG;
    } else {
      return VG_ERR_INVALID_ARG;
    }
    hm[i] = make_mat(d.format, d.M, d.K, d.w, d.scales, d.rowscale, d.gscale, d.x, d.y);
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
    hm[i].rb_base = rb_total;
    ph.items += int64_t(hm[i].RB) * hm[i].KC;
    ph.rbs += hm[i].RB;
    ph.mat_end = i + 1;
    rb_total += hm[i].RB;
    bytes += algorithmic_bytes(hm[i]);
  }
  int grid = di->sms;
  if (o.max_ctas > 0) grid = std::min(grid, int(o.max_ctas));
  int per_sm = 0;
  VG_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stream_kernel, kKernelThreads, kSmemBytes));
  if (per_sm < 1) return VG_ERR_UNSUPPORTED;
  grid = std::min(grid, per_sm * di->sms);

  vg_verify_plan *plan = new vg_verify_plan();
  plan->dev = dev;
  plan->N = N;
  plan->grid = grid;
  plan->ordered = o.ordered ? 1 : 0;
  plan->nphases = int(hp.size());
  plan->bytes = bytes;
  const size_t head = 256;
  const size_t cnt_bytes = size_t((rb_total * 4 + 255) / 256 * 256);
  const size_t done_bytes = size_t((hp.size() * 4 + 4 + 255) / 256 * 256);
  const size_t part_bytes = size_t(grid) * 2 * kPartialFloats * sizeof(float);
  plan->state_bytes = head + cnt_bytes + done_bytes + part_bytes;
  cudaError_t e = cudaMalloc(&plan->d_mats, sizeof(MatDev) * hm.size());
  if (e == cudaSuccess) e = cudaMalloc(&plan->d_phases, sizeof(PhaseDev) * hp.size());
  if (e == cudaSuccess) e = cudaMalloc(&plan->d_state, plan->state_bytes);
  if (e == cudaSuccess)
    e = cudaMemcpy(plan->d_mats, hm.data(), sizeof(MatDev) * hm.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(plan->d_phases, hp.data(), sizeof(PhaseDev) * hp.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(plan->d_state, 0, plan->state_bytes);
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
  p.ordered = plan->ordered;
  p.hold_phase = hold_phase;
  p.grid = grid;
  p.timeout_ns = o.wait_timeout_ns > 0 ? uint64_t(o.wait_timeout_ns) : 2000000000ull;
  p.m8 = 8;
  p.m64 = 64;
  p.error = reinterpret_cast<int *>(plan->d_state);
  p.cnt = reinterpret_cast<uint32_t *>(plan->d_state + head);
  p.done = reinterpret_cast<uint32_t *>(plan->d_state + head + cnt_bytes);
  p.ctas_done = p.done + hp.size();
  p.partials = reinterpret_cast<float *>(plan->d_state + head + cnt_bytes + done_bytes);
  if (!plan->ordered) {
    p.done = nullptr;
    p.ctas_done = nullptr;
  }
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
  void *args[] = {&plan->params};
  VG_CUDA(cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(stream_kernel),
                                      dim3(plan->grid), dim3(kKernelThreads), args, kSmemBytes,
                                      as_cuda(stream)));
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
  cudaFree(plan->d_state);
  delete plan;
  return VG_OK;
}
