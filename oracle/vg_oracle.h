/*
 * vg_oracle.h -- plain, slow, obviously correct CPU reference for the
 * NVFP4 / row-scaled FP8 decode-and-verify GEMV.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py may load this library.  It shares no code,
 * header, table or constant with the CUDA path in verify_gemm_gb300/csrc.
 *
 * Everything here works on the CANONICAL layout:
 *   nib[m][k/2]  : E2M1 codes, low nibble = even k, high nibble = odd k
 *   sc[m][k/16]  : one E4M3 byte per 16-element block along K
 *   gs           : FP32 tensor scale (dequantisation multiplier)
 *   q[m][k]      : FP8-E4M3 codes (row-scaled FP8), rs[m] FP32 row scale
 *   x[n][k]      : BF16 bit patterns, y[n][m] results
 *
 * The product being checked is y[N,M] = x[N,K] . dequant(W)[M,K]^T, the
 * weight-streaming product that the mtp7-device-confidence engine card
 * (crit-hub), Design table, "GEMVs" row, runs for 1-8 columns, and that
 * the same card's Measured section (19.26 GB read per verify pass) and
 * Checks section (the FP8 and NVFP4 GEMVs for 1-8 columns compared with an
 * FP64 reference) describe.  Accumulation is FP64; products of decoded weights and BF16
 * activations are exact in FP64.
 */
#ifndef VG_ORACLE_H
#define VG_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Value of a 4-bit E2M1 code: sign = bit 3, magnitude from the 8-entry
 * table {0, 0.5, 1, 1.5, 2, 3, 4, 6}. */
double vgo_e2m1_value(int code);

/* Value of an OCP FP8 E4M3 ("FN") byte: bias 7, subnormals f*2^-9,
 * 0x7F/0xFF are NaN, no infinities, max 448. */
double vgo_e4m3_value(int byte);

/* Value of a BF16 bit pattern. */
double vgo_bf16_value(uint16_t bits);

/* Round-to-nearest-even, saturating E4M3 encoder of an FP32 value
 * (sign kept; |v| >= 448 gives +-448; NaN gives 0x7F|sign). */
int vgo_e4m3_encode(float v);

/* Round-to-nearest-even, saturating E2M1 encoder of an FP32 value
 * (sign bit copied from v, so -0.1 gives 0x8). */
int vgo_e2m1_encode(float v);

/* NVFP4 round-to-nearest quantisation (load-time re-encoding, crit landing
 * page, "Models" paragraph: post-training quantisation to NVFP4 by
 * round-to-nearest).  K % 16 == 0.  Returns 0, or -1 if W holds a NaN/Inf. */
int vgo_nvfp4_quantise(const float *W, int64_t M, int64_t K,
                       uint8_t *nib, uint8_t *sc, float *gs_out);

/* Largest |W[i]| over n elements (FP32, exact). */
float vgo_amax(const float *W, int64_t n);

/* The per-block part of vgo_nvfp4_quantise for a given tensor scale gs,
 * so that a subset of rows can be quantised with the whole matrix's gs. */
void vgo_nvfp4_quantise_gs(const float *W, int64_t M, int64_t K, float gs,
                           uint8_t *nib, uint8_t *sc);

/* Row-scaled FP8-E4M3 quantisation (engine card, Model section: a layer
 * stored as FP8 with one scale per row).  Returns 0, or -1 if W holds a
 * NaN/Inf. */
int vgo_fp8_quantise(const float *W, int64_t M, int64_t K,
                     uint8_t *q, float *rs_out);

/* Dequantised weights in FP64 (exact). */
void vgo_nvfp4_dequant(const uint8_t *nib, const uint8_t *sc, float gs,
                       int64_t M, int64_t K, double *What);
void vgo_fp8_dequant(const uint8_t *q, const float *rs,
                     int64_t M, int64_t K, double *What);

/* y[n][r] = sum_k What[rows[r]][k] * x[n][k] and a[n][r] = sum_k |What x|
 * in FP64 for the listed rows (rows == NULL: all M rows, r = m).  Output
 * arrays are [N][nrows].  threads <= 1 runs on the calling thread. */
void vgo_gemv_nvfp4(const uint8_t *nib, const uint8_t *sc, float gs,
                    const uint16_t *x, int N, int64_t M, int64_t K,
                    const int64_t *rows, int64_t nrows,
                    double *y, double *a, int threads);
void vgo_gemv_fp8(const uint8_t *q, const float *rs,
                  const uint16_t *x, int N, int64_t M, int64_t K,
                  const int64_t *rows, int64_t nrows,
                  double *y, double *a, int threads);

/* ------------------------------------------------------ other formats
 * Two more weight formats the pages name next to NVFP4 and FP8: MXFP8
 * (crit README, Kernels section: cuBLASLt's block-scaled MXFP8) and
 * groupwise integer weights (NInfer README, model table: "groupwise-int"
 * artifacts; crit README, Kernels section: Marlin's 4-bit weights in
 * GPTQ-style groups against 16-bit activations).  The pages define neither;
 * the readings are the plain public ones:
 *   MXFP8 (OCP Microscaling): E4M3 elements, one E8M0 scale 2^(e-127) per
 *     32 consecutive K elements; quantisation takes the shared exponent
 *     floor(log2(block amax)) - 8 (8 = the largest E4M3 exponent), scale
 *     byte e = that + 127 limited to 10..134 (scales 2^-117..2^7, the range
 *     in which every scaled element is a normal BF16 value), a zero block
 *     gets e = 127; codes are E4M3(w / 2^(e-127)) rounded to nearest even
 *     with saturation.
 *   groupwise-int ("int4-g128"): 4-bit codes q in 0..15 with the zero point
 *     8, one BF16 scale s per 128 consecutive K elements of a row,
 *     w = (q - 8) * s; quantisation s = bf16(amax / 7) (FP32 division, one
 *     rounding to BF16), q = clamp(rne(w / s), -8, 7) + 8 (all 8 when
 *     s == 0). */

/* Value of an E8M0 scale byte: 2^(e-127); 0xFF is NaN. */
double vgo_e8m0_value(int byte);

/* MXFP8 quantisation, K % 32 == 0: q[M][K] E4M3 bytes, sc[M][K/32] E8M0
 * bytes.  Returns 0, or -1 if W holds a NaN/Inf. */
int vgo_mxfp8_quantise(const float *W, int64_t M, int64_t K, uint8_t *q, uint8_t *sc);

/* Groupwise INT4 quantisation, K % 128 == 0: nib[M][K/2] (low nibble =
 * even k), sc[M][K/128] BF16 bits.  Returns 0, or -1 on NaN/Inf. */
int vgo_int4g_quantise(const float *W, int64_t M, int64_t K, uint8_t *nib, uint16_t *sc);

void vgo_mxfp8_dequant(const uint8_t *q, const uint8_t *sc, int64_t M, int64_t K, double *What);
void vgo_int4g_dequant(const uint8_t *nib, const uint16_t *sc, int64_t M, int64_t K,
                       double *What);

/* The GEMV of vgo_gemv_nvfp4 for these formats (same outputs). */
void vgo_gemv_mxfp8(const uint8_t *q, const uint8_t *sc, const uint16_t *x, int N, int64_t M,
                    int64_t K, const int64_t *rows, int64_t nrows, double *y, double *a,
                    int threads);
void vgo_gemv_int4g(const uint8_t *nib, const uint16_t *sc, const uint16_t *x, int N, int64_t M,
                    int64_t K, const int64_t *rows, int64_t nrows, double *y, double *a,
                    int threads);

/* ------------------------------------------------- fused neighbours
 * Operations that sit next to the GEMV in a layer and that the verify pass
 * can run in the same launch (engine card, Checks section: the operator
 * checks cover row reductions next to the GEMVs; the card's Model section
 * names the MLPs, whose gate and up projections feed a gated activation).
 * The pages give no formulas; these are the plain definitions of the
 * SiLU-gated MLP activation and of RMS normalisation used by the model
 * family the card runs. */

/* BF16 bit pattern nearest to v: round to nearest, ties to the even
 * significand, with BF16's subnormals (spacing 2^-133); one rounding from
 * the FP64 value.  |v| past the largest finite BF16 gives +-inf. */
uint16_t vgo_bf16_round(double v);

/* SiLU(g) = g * sigmoid(g) = g / (1 + exp(-g)), FP64. */
double vgo_silu(double g);

/* Gated activation of n gate/up pairs: h[i] = SiLU(g[i]) * u[i] (FP64),
 * and the acceptance bound of a BF16 h computed from a gate and an up
 * product that each carry the GEMV tolerance: with eg = 4e-3*ag + 1e-6 and
 * eu = 4e-3*au + 1e-6 (ag, au = sum|w x| of the two products),
 *   bound = 1.1*eg*(|u| + eu) + |SiLU(g)|*eu + 2^-8*|h| + 1e-6,
 * where 1.1 bounds |SiLU'| everywhere and 2^-8*|h| covers the BF16
 * rounding of h. */
void vgo_swiglu(const double *g, const double *u, const double *ag, const double *au,
                int64_t n, double *h, double *bound);

/* RMS normalisation of N rows of K BF16 values with BF16 weights gamma[K]:
 *   out[n][k] = bf16( x[n][k] * gamma[k] / sqrt(sum_k x[n][k]^2 / K + eps) )
 * evaluated in FP64 with one rounding to BF16 at the end. */
void vgo_rmsnorm(const uint16_t *x, const uint16_t *gamma, int N, int64_t K, double eps,
                 uint16_t *out);

/* Count elements with |y - yref| > rel*a + abs; *worst gets the largest
 * |y - yref| / (rel*a + abs).  y is BF16 bits. */
int64_t vgo_check(const uint16_t *y, const double *yref, const double *a,
                  int64_t n, double rel, double abs_tol, double *worst);

#ifdef __cplusplus
}
#endif
#endif
