/*
 * vmx_oracle.h -- the plain CPU definition of float_moment, float_psnr and
 * integer_psnr.
 *
 * TEST INFRASTRUCTURE ONLY. This is the oracle the CUDA library is checked
 * against. Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load it; the library never calls it and shares no code with it.
 *
 * Samples are read as unsigned codewords: uint8 when bpc == 8, else uint16
 * (host byte order). Frame f of a batch starts at base + f * height * stride.
 */
#ifndef VMX_ORACLE_H
#define VMX_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* float_moment of one frame pair: out[0..3] = ref first moment, dis first
 * moment, ref second moment, dis second moment. If s2_rows is not NULL it
 * receives [2][height] exact per-row sums of the float squares in units of
 * 1/scaler^2 (ref rows, then dis rows). */
void vmx_oracle_moment(const void *ref, const void *dis, int width, int height,
                       int64_t stride_bytes, int bpc, double out[4],
                       uint64_t *s2_rows);

/* The four accumulators of vmx_oracle_moment() before the division by the
 * pixel count: the CPU's running doubles (true scale) after the last pixel. */
void vmx_oracle_moment_acc(const void *ref, const void *dis, int width, int height,
                           int64_t stride_bytes, int bpc, double acc[4]);

/* The psnr noise accumulator before the division by the pixel count (the
 * CPU's row-order double, true scale); rows as vmx_oracle_psnr(). */
double vmx_oracle_psnr_noise(const void *ref, const void *dis, int width, int height,
                             int64_t stride_bytes, int bpc, uint64_t *rows);

/* float_psnr of one frame pair: rows[height] receives each row's sum of the
 * float squared differences in units of 1/scaler^2; *mse the frame noise
 * divided by the pixel count. rows may be NULL. */
void vmx_oracle_psnr(const void *ref, const void *dis, int width, int height,
                     int64_t stride_bytes, int bpc, uint64_t *rows, double *mse);

/* integer_psnr of one plane pair: rows[height] (may be NULL) receives each
 * row's exact sum of squared codeword differences, *sse the plane's, and
 * *mse that sum divided by the pixel count (codeword units). */
void vmx_oracle_integer_psnr(const void *ref, const void *dis, int width, int height,
                             int64_t stride_bytes, int bpc, uint64_t *rows, uint64_t *sse,
                             double *mse);
void vmx_oracle_integer_psnr_batch(const void *ref, const void *dis, int width, int height,
                                   int64_t stride_bytes, int bpc, int first, int count,
                                   uint64_t *rows /* [count][height] or NULL */,
                                   uint64_t *sse /* [count] */, double *mse /* [count] */);

/* PSNR from the mean squared error on the 8-bit scale:
 * 10 * log10(peak^2 / max(mse, 1e-10)), peak = (2^bpc - 1) / 2^(bpc - 8),
 * capped at psnr_max when psnr_max > 0. */
double vmx_oracle_psnr_db(double mse, int bpc, double psnr_max);

/* Batch helpers: frames [first, first + count) of a batch. */
void vmx_oracle_moment_batch(const void *ref, const void *dis, int width, int height,
                             int64_t stride_bytes, int bpc, int first, int count,
                             double *out /* [count][4] */);
void vmx_oracle_psnr_batch(const void *ref, const void *dis, int width, int height,
                           int64_t stride_bytes, int bpc, int first, int count,
                           uint64_t *rows /* [count][height] or NULL */,
                           double *mse /* [count] */);

/* Which planted mistake this build carries (0 = none). */
int vmx_oracle_mutation(void);

#ifdef __cplusplus
}
#endif
#endif
