/*
 * vgemm.h -- C ABI of the GB300 (sm_103a) NVFP4 / row-scaled FP8 verify-GEMV
 * library (libvgemm.so).
 *
 * The library computes the weight-streaming product of LLM decode and
 * speculative verification,
 *
 *     y[N, M] = x[N, K] . dequant(W)[M, K]^T,     N = 1..8 columns,
 *
 * with W in NVFP4 (E2M1 codes, one E4M3 scale per 16 elements along K, one
 * FP32 tensor scale) or row-scaled FP8-E4M3, x and y in BF16 and FP32
 * accumulation.  This is the "GEMVs" row of the Design table on the
 * mtp7-device-confidence engine card (crit-hub): FP8 and NVFP4 weights fed
 * to BF16 tensor-core fragments for 1-8 columns, where the verify pass of
 * the card's Decode row runs 2-8 columns and a decode step one.  The
 * card's Measured section states what makes it the hot path: a verify pass
 * reads every weight once (19.26 GB), so its time is the weight-read time;
 * the crit README's quality-mode comparison makes the same point for a
 * decode pass.
 *
 * Conventions (all entry points):
 *  - Plain C; nothing throws across the ABI; every call returns a
 *    vg_status.  Argument and alignment errors are detected on the host and
 *    returned before anything is launched.
 *  - Pointers marked "device" are CUDA device (or managed) memory owned by
 *    the caller; "host" pointers are host memory.  Device pointers must be
 *    16-byte aligned.  No entry point allocates device memory per call,
 *    except vg_verify_plan_create, which allocates the plan's own tables
 *    once.
 *  - Work is enqueued on the caller's stream (a cudaStream_t; NULL is the
 *    legacy default stream) and runs asynchronously, except where a
 *    function says it synchronises.
 *  - BF16 values travel as uint16_t bit patterns.
 *  - Limits: 1 <= N <= 32, M >= 1, K >= 16, K % 16 == 0, M * K < 2^40.
 *    Passes wider than 8 columns (batched verification of several requests'
 *    drafts: the NInfer README's one to eight execution lanes, each
 *    verifying its MTP drafts) need whole chunks along K (K % 512 for the
 *    4-bit formats, K % 256 for the 8-bit ones) and x by tensor copy, and
 *    their x slice must fit the kernel's staging: 16 columns for every
 *    layout, 32 for matrices packed in row blocks of 16 tiles (most rows or
 *    K not a multiple of the chunk); otherwise VG_ERR_UNSUPPORTED.  Fused
 *    operations (see vg_matrix_desc) take 8 columns at most.
 *
 * Device weight layout (the "packed" form; canonical forms are below):
 *  NVFP4 codes are stored in 16-row tiles cut into 64-column units of 512
 *  bytes, arranged so that every lane of a warp reads one 16-byte vector
 *  per unit holding 16 consecutive K positions of two rows (one scale block
 *  of each), with the bits of each code placed for a cheap in-register
 *  decode to BF16.  The kernel's unit of work, an item, is 16 tile-chunks
 *  (a chunk is 8 units): one chunk of a row block of 16 tiles, or, for
 *  matrices with few rows (when every item is whole in K), 16 / rt
 *  consecutive chunks of a row block of rt = 8, 4 or 2 tiles.  rt follows
 *  from M, K and the format alone, so the layout is fixed by the matrix
 *  shape.  Units are ordered by row block, then item, then tile, then
 *  chunk, so that every item is one contiguous run of bytes.  Block scales
 *  live in a separate buffer in the same order, 512 bytes per tile per
 *  chunk, re-encoded losslessly so that E4M3 subnormal scales decode like
 *  normal ones.  Row-scaled FP8 codes use 1024-byte units (4 per chunk) in
 *  the same order; their FP32 row scales are a plain [M] array.  Rows past
 *  M and columns past K are zero padding inside the last tile and unit.
 *  The packed buffers are opaque: use the pack / unpack / from_canonical
 *  calls to move between them and the canonical layout.
 *
 * Canonical layout (the plain stored form, as the engine card's Design
 * table "Weights" row calls it):
 *  NVFP4: nib[M][K/2] uint8 (low nibble = even k, high nibble = odd k),
 *         sc[M][K/16] uint8 E4M3 bytes, gscale FP32 multiplier.
 *  FP8:   q[M][K] uint8 E4M3 bytes, rowscale[M] FP32 multipliers.
 */
#ifndef VGEMM_H
#define VGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so that this header does not
 * need the CUDA headers. */
typedef struct CUstream_st *vg_stream_t;

typedef enum vg_status {
    VG_OK = 0,
    VG_ERR_INVALID_ARG = 1,   /* bad size, null pointer, non-finite weight */
    VG_ERR_ALIGNMENT = 2,     /* a device pointer is not 16-byte aligned */
    VG_ERR_UNSUPPORTED = 3,   /* no sm_103a device, or a limit exceeded */
    VG_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    VG_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out */
    VG_ERR_WORKSPACE = 6      /* workspace missing or too small */
} vg_status;

/* Weight formats of vg_matrix_desc.format.
 *   VG_FMT_MXFP8: E4M3 codes, one E8M0 scale 2^(e-127) per 32 elements along
 *     K (e limited to 10..134), K % 256 == 0.
 *   VG_FMT_INT4G: 4-bit codes q with zero point 8 and one BF16 scale s per
 *     128 elements along K of a row, w = (q - 8) * s, K % 512 == 0.
 * These two take x by tensor copy only (see vg_gemv_nvfp4). */
enum { VG_FMT_NVFP4 = 0, VG_FMT_FP8_ROWSCALE = 1, VG_FMT_MXFP8 = 2, VG_FMT_INT4G = 3 };

/* Human-readable name of a status code (static string, never NULL). */
const char *vg_status_string(vg_status s);

/* Library version as 10000*major + 100*minor + patch. */
int vg_version(void);

/* Last CUDA error string seen by the library on this host thread, or "". */
const char *vg_last_cuda_error(void);

/* ------------------------------------------------------------- sizes */

/* Bytes of the packed NVFP4 code buffer (*w_bytes) and block-scale buffer
 * (*scale_bytes) for an M x K matrix.  Either output may be NULL. */
vg_status vg_nvfp4_sizes(int64_t M, int64_t K, size_t *w_bytes, size_t *scale_bytes);

/* Bytes of the packed row-scaled FP8 code buffer for an M x K matrix. */
vg_status vg_fp8_sizes(int64_t M, int64_t K, size_t *w_bytes);

/* ----------------------------------------------------- quantise / pack */

/* NVFP4 round-to-nearest quantisation of an FP32 matrix into the packed
 * layout (load-time re-encoding: the crit landing page's "Models"
 * paragraph names round-to-nearest post-training quantisation to NVFP4;
 * the engine card's Model section re-encodes the head to NVFP4 at load).
 *   W           device FP32 [M][K], row-major, leading dimension K.
 *   w_out       device, vg_nvfp4_sizes(...).w_bytes bytes (written).
 *   scales_out  device, vg_nvfp4_sizes(...).scale_bytes bytes (written;
 *               also used as scratch for the amax reduction).
 *   gscale_out  host; receives the FP32 tensor scale (dequant multiplier).
 * Recipe, in FP32 IEEE arithmetic: gs = amax|W| / 2688; per 16-block
 * s = (blockamax / gs) / 6, scale code = E4M3(s) rounded to nearest even
 * with saturation; d = E4M3value(code) * gs; code of w = E2M1(w / d) to
 * nearest even with saturation (all codes 0 when d == 0).
 * Synchronises the stream once (to read amax).  NaN/Inf in W gives
 * VG_ERR_INVALID_ARG. */
vg_status vg_nvfp4_pack(const float *W, int64_t M, int64_t K,
                        void *w_out, void *scales_out, float *gscale_out,
                        vg_stream_t stream);

/* Row-scaled FP8-E4M3 quantisation (engine card, Model section: the draft
 * layer is stored as FP8 with one scale per row):  rs[m] = rowamax / 448,
 * code = E4M3(w / rs[m]) rounded to nearest even with saturation (all codes
 * 0 when rs[m] == 0).
 *   W            device FP32 [M][K].
 *   w_out        device, vg_fp8_sizes bytes.
 *   rowscale_out device FP32 [M].
 * Synchronises once (to check the row scales).  NaN/Inf in W gives
 * VG_ERR_INVALID_ARG. */
vg_status vg_fp8_pack(const float *W, int64_t M, int64_t K,
                      void *w_out, float *rowscale_out, vg_stream_t stream);

/* Packed NVFP4 -> canonical nib[M][K/2] and sc[M][K/16] (device). */
vg_status vg_nvfp4_unpack(const void *w, const void *scales, int64_t M, int64_t K,
                          uint8_t *nib_out, uint8_t *sc_out, vg_stream_t stream);

/* Packed FP8 -> canonical q[M][K] (device). */
vg_status vg_fp8_unpack(const void *w, int64_t M, int64_t K, uint8_t *q_out,
                        vg_stream_t stream);

/* vg_fp8_pack and vg_fp8_unpack under the names of the row-scaled format: identical
 * arguments, behaviour and errors. */
vg_status vg_fp8_rowscale_pack(const float *W, int64_t M, int64_t K,
                               void *w_out, float *rowscale_out, vg_stream_t stream);
vg_status vg_fp8_rowscale_unpack(const void *w, int64_t M, int64_t K, uint8_t *q_out,
                                 vg_stream_t stream);

/* Canonical NVFP4 (device nib, sc) -> packed layout.  Scale bytes must be
 * non-negative and not NaN (E4M3 bytes 0x00..0x7E); otherwise
 * VG_ERR_INVALID_ARG.  Blocks whose scale is 0 are stored with zero codes
 * (their value is 0 either way).  Synchronises once. */
vg_status vg_nvfp4_from_canonical(const uint8_t *nib, const uint8_t *sc,
                                  int64_t M, int64_t K, void *w_out, void *scales_out,
                                  vg_stream_t stream);

/* Canonical FP8 codes (device q[M][K]) -> packed layout.  NaN codes
 * (0x7F, 0xFF) give VG_ERR_INVALID_ARG.  Synchronises once; w_out's first
 * bytes are used as scratch for the check before being written. */
vg_status vg_fp8_from_canonical(const uint8_t *q, int64_t M, int64_t K, void *w_out,
                                vg_stream_t stream);

/* ------------------------------------------- MXFP8 and groupwise INT4
 * Two more weight formats next to NVFP4 and row-scaled FP8: MXFP8, the OCP
 * Microscaling FP8 format that cuBLASLt takes block-scaled (crit README,
 * Kernels section), and groupwise 4-bit integers, the "groupwise-int"
 * artifacts of the NInfer README (model table) and the 4-bit GPTQ-style
 * groups of Marlin (crit README, Kernels section).
 * Canonical forms:
 *   MXFP8: q[M][K] E4M3 bytes, sc[M][K/32] E8M0 bytes (2^(e-127)).
 *   INT4G: nib[M][K/2] codes 0..15 (low nibble = even k),
 *          sc[M][K/128] BF16 bits; w = (q - 8) * s.
 * Quantisation (FP32 IEEE steps):
 *   MXFP8: per 32-block e = floor(log2(amax)) - 8 + 127 limited to
 *          10..134 (a zero block: 127); q = E4M3(w / 2^(e-127)), nearest
 *          even, saturating.
 *   INT4G: per 128-group s = BF16(amax / 7) (nearest even); q =
 *          clamp(nearest-even integer of w / s, -8, 7) + 8 (8 when s == 0).
 * Sizes of the packed code and scale buffers for any format. */
vg_status vg_weight_sizes(int format, int64_t M, int64_t K, size_t *w_bytes,
                          size_t *scale_bytes);

/* Quantise an FP32 matrix (device [M][K]) into the packed layout.
 * Synchronises once; NaN/Inf gives VG_ERR_INVALID_ARG; K not a multiple of
 * 256 (MXFP8) or 512 (INT4G) gives VG_ERR_UNSUPPORTED. */
vg_status vg_mxfp8_pack(const float *W, int64_t M, int64_t K, void *w_out, void *scales_out,
                        vg_stream_t stream);
vg_status vg_int4g_pack(const float *W, int64_t M, int64_t K, void *w_out, void *scales_out,
                        vg_stream_t stream);

/* Packed -> canonical (device). */
vg_status vg_mxfp8_unpack(const void *w, const void *scales, int64_t M, int64_t K,
                          uint8_t *q_out, uint8_t *sc_out, vg_stream_t stream);
vg_status vg_int4g_unpack(const void *w, const void *scales, int64_t M, int64_t K,
                          uint8_t *nib_out, uint16_t *sc_out, vg_stream_t stream);

/* Canonical -> packed (device).  MXFP8 scale bytes outside 10..134 give
 * VG_ERR_UNSUPPORTED, NaN codes VG_ERR_INVALID_ARG; INT4G scales must be
 * finite (else VG_ERR_INVALID_ARG).  Synchronise once. */
vg_status vg_mxfp8_from_canonical(const uint8_t *q, const uint8_t *sc, int64_t M, int64_t K,
                                  void *w_out, void *scales_out, vg_stream_t stream);
vg_status vg_int4g_from_canonical(const uint8_t *nib, const uint16_t *sc, int64_t M, int64_t K,
                                  void *w_out, void *scales_out, vg_stream_t stream);

/* Gated pair packers for VG_OP_SWIGLU: the gate and up projections of an
 * MLP (each [I][K], I % 8 == 0) packed as one matrix of M = 2*I rows whose
 * every 16-row tile holds 8 gate rows and the same 8 up rows (tile j: gate
 * rows 8j..8j+7, then up rows 8j..8j+7), so that the lane that finishes a
 * gate output also holds the matching up output.  Each half is quantised
 * exactly as vg_nvfp4_pack / vg_fp8_pack would quantise it alone (its own
 * tensor scale or row scales).  Buffers: vg_nvfp4_sizes / vg_fp8_sizes of
 * (2*I, K).  vg_nvfp4_unpack / vg_fp8_unpack of (2*I, K) give the canonical
 * interleaved rows.
 *   Wgate, Wup   device FP32 [I][K].
 *   gscales_out  host float[2]: gate, up tensor scales.
 *   rs_gate_out, rs_up_out  device FP32 [I].
 * Synchronise once; NaN/Inf gives VG_ERR_INVALID_ARG. */
vg_status vg_nvfp4_pack_gated(const float *Wgate, const float *Wup, int64_t I, int64_t K,
                              void *w_out, void *scales_out, float *gscales_out,
                              vg_stream_t stream);
vg_status vg_fp8_pack_gated(const float *Wgate, const float *Wup, int64_t I, int64_t K,
                            void *w_out, float *rs_gate_out, float *rs_up_out,
                            vg_stream_t stream);

/* ------------------------------------------------------------ the GEMV */

/* Workspace bytes that vg_gemv_nvfp4 / vg_gemv_fp8_rowscale need for an
 * M x K matrix on the current device (format: VG_FMT_*): 256 header bytes
 * (a device error word, a count of finished thread blocks, a pass counter)
 * and one 16 KiB slot per thread block for the FP32 partial sums of row
 * blocks whose K range is split between thread blocks.  Each partial sum
 * carries a tag of the pass that wrote it, so stale slots are never mistaken
 * for current ones.  The workspace must be zero-filled once when allocated;
 * afterwards every call leaves it consistent for the next one (error word
 * and block count at zero, pass counter advanced), so it is never cleared
 * again unless vg_gemv_workspace_check reports an error.  Calls that share
 * a workspace must not overlap on the GPU. */
vg_status vg_gemv_workspace_size(int64_t M, int64_t K, int format, size_t *bytes);

/* The same for a GEMV of N columns (N > 8 needs 2x (N <= 16) or 4x the
 * partial-sum space). */
vg_status vg_gemv_workspace_size_n(int64_t M, int64_t K, int format, int N, size_t *bytes);

/* y[n][m] = bf16( sum_k x[n][k] * dequant(W)[m][k] ), NVFP4 weights.
 * One cooperative launch of up to one thread block per SM (all resident at
 * once: the block that sums a split row block waits, bounded, for the
 * others' partial sums).
 *   w, scales   device, packed by vg_nvfp4_pack / vg_nvfp4_from_canonical.
 *   gscale      FP32 tensor scale (from the pack).
 *   x           device BF16 [N][K], row-major, 16-byte aligned.
 *   y           device BF16 [N][M], row-major (written).
 *   workspace   device, >= vg_gemv_workspace_size bytes (see there).
 * Accumulation is FP32; y is rounded to nearest even.  The result for
 * column n does not depend on N or on the other columns, and a repeated
 * call gives the same bits.  With K a multiple of 64, each work item's slice
 * of x is one tensor copy (a tensor map encoded on the host through the
 * driver); otherwise, or if the driver declines the map, x is copied one row
 * at a time (same results, slower).  Items of several chunks (see the weight
 * layout) take x by tensor copy only: if the driver declines their map the
 * call returns VG_ERR_UNSUPPORTED. */
vg_status vg_gemv_nvfp4(const void *w, const void *scales, float gscale,
                        const uint16_t *x, int N, int64_t M, int64_t K, uint16_t *y,
                        void *workspace, size_t workspace_bytes, vg_stream_t stream);

/* Same for row-scaled FP8 weights: dequant(W)[m][k] = E4M3(q[m][k]) * rowscale[m].
 *   rowscale  device FP32 [M]. */
vg_status vg_gemv_fp8_rowscale(const void *w, const float *rowscale,
                               const uint16_t *x, int N, int64_t M, int64_t K, uint16_t *y,
                               void *workspace, size_t workspace_bytes, vg_stream_t stream);

/* The GEMV for MXFP8 and groupwise-INT4 weights (arguments as
 * vg_gemv_nvfp4, minus the tensor scale).  Every block scale is applied
 * exactly: MXFP8 weights are decoded to BF16 with their power-of-two scale,
 * INT4 weights q - 8 go through the MMAs unscaled and each group's FP32 sum
 * is multiplied by its BF16 scale. */
vg_status vg_gemv_mxfp8(const void *w, const void *scales, const uint16_t *x, int N, int64_t M,
                        int64_t K, uint16_t *y, void *workspace, size_t workspace_bytes,
                        vg_stream_t stream);
vg_status vg_gemv_int4g(const void *w, const void *scales, const uint16_t *x, int N, int64_t M,
                        int64_t K, uint16_t *y, void *workspace, size_t workspace_bytes,
                        vg_stream_t stream);

/* Largest workspace, in bytes, that vg_gemv_nvfp4_noalloc can serve. */
#define VG_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

/* vg_gemv_nvfp4 without a caller-supplied workspace, for callers that cannot
 * allocate device memory: code inside a host application that owns all
 * device memory and only lends out input and output buffers, code that must
 * not call cudaMalloc because it may synchronise the whole device, or code
 * held to a fixed memory budget.  The pages have no counterpart to this
 * entry point; it exists for such callers only.
 *   Arguments and results are those of vg_gemv_nvfp4, minus the workspace.
 *   The workspace is one fixed device array of VG_NOALLOC_SCRATCH_BYTES
 *   (4 MiB) inside the library, created on each device when the library's
 *   module is first used there and held until the process exits.  A call
 *   that needs more (vg_gemv_workspace_size_n; any N <= 8 fits on devices of
 *   up to 255 SMs) gives VG_ERR_UNSUPPORTED.
 *   Nothing is allocated: the call looks up the array's device address
 *   (cudaGetSymbolAddress, on every call, so a device reset is harmless),
 *   clears the array's error word (4 bytes, cudaMemsetAsync on `stream`),
 *   then runs the GEMV on it; the rest of the array stays consistent from
 *   call to call.  The first call on a device loads the library's module
 *   there: make it before any stream capture.  Errors are those of
 *   vg_gemv_nvfp4 detected on the host; a bounded device-side wait that runs
 *   out is not reported by the return value (the launch has already
 *   returned) but left in the array's error word, which
 *   vg_gemv_nvfp4_noalloc_check reads.  All calls share the one array, so
 *   calls that overlap on the GPU (other streams, other host threads) race
 *   and give wrong results: serialise them. */
vg_status vg_gemv_nvfp4_noalloc(const void *w, const void *scales, float gscale,
                                const uint16_t *x, int N, int64_t M, int64_t K, uint16_t *y,
                                vg_stream_t stream);

/* Error report of vg_gemv_nvfp4_noalloc, also allocation-free: synchronises
 * `stream`, reads the fixed array's error word left by the most recent call
 * into *device_error (0, or the code of the first bounded wait that ran out)
 * and, if it is set, zero-fills the whole array and returns VG_ERR_TIMEOUT
 * (the y of that call is void).  The pages have no counterpart to it. */
vg_status vg_gemv_nvfp4_noalloc_check(int *device_error, vg_stream_t stream);

/* Reads and clears the device error word of a GEMV workspace (synchronous).
 * *device_error receives 0, or a nonzero code if a bounded wait inside a
 * kernel ran out (then the workspace is also re-zeroed). */
vg_status vg_gemv_workspace_check(void *workspace, size_t workspace_bytes,
                                  int *device_error, vg_stream_t stream);

/* ------------------------------------------------------ HBM read probe */

/* Read-only bandwidth probe (the "physics-based" ceiling that crit's Eval
 * measures, crit README, Eval section; the engine card's Measured section
 * sets the verify pass against the card's read rate).  Reads `bytes` of the
 * device buffer `buf` once and folds them into `sink` (device, >= one word
 * per thread block: the SM count for mode 1, SMs x resident blocks for
 * mode 0).  mode 0: 16-byte vector loads; modes 1 and 2: per-warp rings
 * of `slots` bulk copies of `chunk` bytes (chunk a multiple of 256,
 * chunk * slots <= 12288); mode 1 interleaves chunks over the whole device,
 * mode 2 gives each block one contiguous range (the GEMV's order), mode 3
 * is mode 2 plus a chunk/8-byte side copy per slot from a second region
 * (codes plus block scales; then (chunk + chunk/8) * slots <= 12288).
 * Time it with events on `stream`. */
vg_status vg_hbm_read_probe(const void *buf, size_t bytes, int mode, int chunk, int slots,
                            uint32_t *sink, int sink_words, vg_stream_t stream);

/* -------------------------------------------------- fused verify pass */

/* Operations of a verify pass entry (vg_matrix_desc.op). */
enum {
    VG_OP_GEMV = 0,      /* y = x . dequant(W)^T */
    VG_OP_SWIGLU = 1,    /* gated MLP pair: y = SiLU(x . Wgate^T) * (x . Wup^T) */
    VG_OP_RMSNORM = 2    /* y = x * gamma / sqrt(mean(x^2) + eps), no weights */
};

/* One entry of a verify pass (a layer stack).  Entries must be listed with
 * non-decreasing group; group g+1 depends on group g.  Zero-initialise, then
 * set: the fields after y default to a plain GEMV whose x does not depend
 * on the pass.
 *
 * VG_OP_GEMV: y[N][M] = x[N][K] . dequant(W)[M][K]^T.
 * VG_OP_SWIGLU, the gated activation fused into the epilogue of the MLP's
 *   gate and up projections (engine card, Model section: the MLPs): W is a
 *   gated pair packed by vg_nvfp4_pack_gated / vg_fp8_pack_gated, M = 2*I
 *   (I gate rows and I up rows, I % 8 == 0), and
 *     y[n][i] = bf16( SiLU(g) * u ),  g = x[n] . Wgate[i],  u = x[n] . Wup[i],
 *   with g and u kept in FP32 (never rounded to BF16); y is [N][I].  NVFP4:
 *   gscale is the gate half's tensor scale, gscale_up the up half's; FP8:
 *   rowscale / rowscale_up are the halves' FP32 row scales [I].
 * VG_OP_RMSNORM, the row reduction before a layer's projections (engine
 *   card, Checks section: row reductions are checked next to the GEMVs):
 *     y[n][k] = bf16( x[n][k] * gamma[k] / sqrt(sum_k x[n][k]^2 / K + eps) ),
 *   sums and scaling in FP32; x and y [N][K], gamma BF16 [K]; format, M, w,
 *   scales and rowscale are ignored.  Every thread block of the pass sums
 *   whole rows and writes one slice of y (N must be at most 8).
 * x_after_group = 1 says that x is written earlier in the same pass (by the
 *   previous group, e.g. the down projection's x = the gated pair's y, or
 *   q/k/v's x = an RMS norm's y): its copy into the kernel is then issued
 *   only after the previous group has completed.  0 (default): x is ready
 *   before the pass starts and is copied ahead of the group order. */
typedef struct vg_matrix_desc {
    int32_t format;          /* VG_FMT_* */
    int32_t group;           /* dependency group */
    int64_t M, K;
    const void *w;           /* device, packed codes */
    const void *scales;      /* device, packed block scales (NVFP4, MXFP8, INT4G), else NULL */
    const float *rowscale;   /* device FP32 [M] (FP8; SWIGLU: gate rows [I]), else NULL */
    float gscale;            /* tensor scale (NVFP4; SWIGLU: of the gate rows) */
    const uint16_t *x;       /* device BF16 [N][K] */
    uint16_t *y;             /* device BF16 [N][M] ([N][M/2] SWIGLU, [N][K] RMSNORM) */
    int32_t op;              /* VG_OP_* (0: GEMV) */
    int32_t x_after_group;   /* 1: x is written by the previous group of this pass */
    float gscale_up;         /* SWIGLU, NVFP4: tensor scale of the up rows */
    float eps;               /* RMSNORM */
    const float *rowscale_up;/* SWIGLU, FP8: device FP32 row scales of the up rows [I] */
    const uint16_t *gamma;   /* RMSNORM: device BF16 weights [K] */
} vg_matrix_desc;

typedef struct vg_verify_plan vg_verify_plan;

/* Options of vg_verify_plan_create_ex (zero-initialise, then set). */
typedef struct vg_plan_options {
    int32_t ordered;          /* 1: group g's products wait for group g-1 (default);
                                 0: no waits (an upper bound) */
    int32_t max_ctas;         /* 0: one thread block per SM */
    int64_t wait_timeout_ns;  /* bound of every device-side wait; 0: 2 s */
    int32_t hold_group;       /* fault-injection: if >= 0, the completion of this
                                 group is never signalled, so the next group's
                                 wait runs out (VG_ERR_TIMEOUT); -1: off */
    int32_t reserved;
} vg_plan_options;

/* Plan a fused verify pass over `count` matrices for N columns: one
 * persistent, cooperative launch streams every weight once, groups in
 * order (engine card, Decode row: one verify step checks all drafted
 * tokens at once, 2-8 columns; Measured section: 19.26 GB read per pass).  Allocates the
 * plan's descriptor table, counters and partial-sum space once.
 * Descriptors (pointers included) are copied; buffer contents may change
 * between passes.  Each item's slice of x is copied into shared memory by
 * copies that run ahead of the group order, so an x may alias a y of the
 * same plan only when its descriptor sets x_after_group (its copies then
 * wait until the previous group has completed, and that group's y is the
 * x); any other x must not alias any y of the plan. */
vg_status vg_verify_plan_create(const vg_matrix_desc *mats, int count, int N,
                                int ordered, vg_verify_plan **plan_out);
vg_status vg_verify_plan_create_ex(const vg_matrix_desc *mats, int count, int N,
                                   const vg_plan_options *opt, vg_verify_plan **plan_out);

/* Enqueue one verify pass on `stream`.  Passes of one plan must not overlap
 * on the GPU. */
vg_status vg_verify_pass(vg_verify_plan *plan, vg_stream_t stream);

/* Width dispatch on the device (engine card, Design table, Decode row: the
 * verify pass runs for however many drafts the round made, 2-8 columns, with
 * no host wait mid-round).  After this call every pass of `plan` reads its
 * width from the device word *d_width when the pass starts, instead of
 * using the N the plan was created with: the pass computes and writes y
 * columns 0..width-1 only (the other columns of each y are left untouched,
 * and rows >= width of each x are never used), so one plan, or one CUDA
 * graph holding its pass, serves every width 1..N and a kernel earlier on
 * the stream can choose it.  A width outside 1..N makes the pass do nothing
 * and set the device error word to 5 (read by vg_verify_plan_check).
 *   d_width  device int32 (4-byte aligned), or NULL to return to the fixed N.
 * The pointer is captured by the launch (and by graph capture), the value
 * is read by each pass. */
vg_status vg_verify_plan_set_width(vg_verify_plan *plan, const int32_t *d_width);

/* Synchronises the stream, reads the plan's device error word and, if it is
 * set, clears it and resets the plan's counters.  *device_error: 0 or a
 * nonzero code (a bounded wait ran out).  Returns VG_ERR_TIMEOUT if set. */
vg_status vg_verify_plan_check(vg_verify_plan *plan, vg_stream_t stream, int *device_error);

/* Weight+scale bytes one pass streams (the algorithmic byte count). */
vg_status vg_verify_plan_bytes(const vg_verify_plan *plan, int64_t *bytes);

/* Number of thread blocks the pass launches. */
vg_status vg_verify_plan_grid(const vg_verify_plan *plan, int *ctas);

vg_status vg_verify_plan_destroy(vg_verify_plan *plan);

#ifdef __cplusplus
}
#endif
#endif /* VGEMM_H */
