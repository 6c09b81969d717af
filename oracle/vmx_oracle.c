/*
 * vmx_oracle.c -- the plain CPU definition of float_moment, float_psnr and
 * integer_psnr.
 *
 * TEST INFRASTRUCTURE ONLY: the oracle the CUDA library is checked against.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use
 * it. It shares no code with the library.
 *
 * What it computes is the CPU extractors as the pages describe them, written
 * out loop by loop, with no blocking, no reordering and no integer tricks:
 *
 *   - picture_copy() puts every codeword on the 8-bit scale as the binary32
 *     value p / scaler, scaler = 2^(bpc - 8) (Research-2081 "Finding": the
 *     CPU's power-of-two normalisation; ADR-1499 "Decision" point 4).
 *   - float_moment, moment.c::compute_2nd_moment(): one binary32 square per
 *     pixel, added into a double in raster order, divided by the pixel count
 *     (ADR-1497 "Context"). The first moment is the same loop over the
 *     binary32 values themselves.
 *   - float_psnr, float_psnr.c::extract(): the binary32 square of each
 *     sample difference, a row's squares added into a double (noise_line()),
 *     the rows added into one double in row order, then divided by the pixel
 *     count (ADR-1499 "Context" and "Decision").
 *   - integer_psnr, one plane pair at a time (psnr_y, psnr_cb, psnr_cr): the
 *     exact integer sum of squared codeword differences and that sum over
 *     the pixel count (the Metal kernel batch page names the feature and its
 *     integer partials; the formula is the plain reading).
 *
 * Build: -O2 -fno-fast-math -ffp-contract=off -fno-tree-vectorize, so that
 * every float product is rounded to binary32 on its own (no fused multiply-
 * add) and every double add happens in the loop's order, one pixel at a time
 * (the scalar order; ADR-1497 "Consequences" notes that lane-order SIMD adds
 * are not the scalar sum past 2^53 units).
 *
 * ORACLE_MUTATION=k builds a copy with one planted mistake, used only to
 * show that the tests pinning this file catch each of them.
 */
#include "vmx_oracle.h"

#include <math.h>
#include <stddef.h>
#include <string.h>

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

int vmx_oracle_mutation(void) { return ORACLE_MUTATION; }

/* One codeword, read as unsigned; uint16 samples may sit at any address. */
static unsigned sample_at(const unsigned char *row, int j, int bpc)
{
    if (bpc == 8)
        return row[j];
    uint16_t v;
    memcpy(&v, row + 2 * (size_t)j, sizeof v);
    return v;
}

static const unsigned char *row_ptr(const void *plane, int64_t stride, int i)
{
    return (const unsigned char *)plane + (int64_t)i * stride;
}

/* The scaler of the CPU's normalisation, 2^(bpc - 8), as a binary32. */
static float scaler_of(int bpc)
{
#if ORACLE_MUTATION == 8
    return (float)(1 << (bpc - 7));
#else
    return (float)(1 << (bpc - 8));
#endif
}

static int last_column(int width)
{
#if ORACLE_MUTATION == 5
    return width - 1;
#else
    return width;
#endif
}

static double pixel_count(int width, int height)
{
#if ORACLE_MUTATION == 7
    return (double)width * (double)height - 1.0;
#else
    return (double)width * (double)height;
#endif
}

/* First moment: the mean of the normalised samples (ADR-1212 normalisation
 * as recalled in Research-2081 "Selected restoration"), raster order. */
static double first_moment_acc(const void *plane, int w, int h, int64_t stride, int bpc)
{
    const float scaler = scaler_of(bpc);
#if ORACLE_MUTATION == 9
    float acc = 0.0f;
#else
    double acc = 0.0;
#endif
    for (int i = 0; i < h; ++i) {
        const unsigned char *row = row_ptr(plane, stride, i);
        for (int j = 0; j < last_column(w); ++j) {
            float f = (float)sample_at(row, j, bpc) / scaler;
            acc += (double)f;
        }
    }
    return (double)acc;
}

/* Second moment, moment.c::compute_2nd_moment() as ADR-1497 "Context"
 * states it: one binary32 square per pixel added into a double in raster
 * order, then divided by the pixel count. */
static double second_moment_acc(const void *plane, int w, int h, int64_t stride, int bpc)
{
    const float scaler = scaler_of(bpc);
#if ORACLE_MUTATION == 2
    float acc = 0.0f;
#else
    double acc = 0.0;
#endif
#if ORACLE_MUTATION == 6
    for (int j = 0; j < last_column(w); ++j) {
        for (int i = 0; i < h; ++i) {
            const unsigned char *row = row_ptr(plane, stride, i);
#else
    for (int i = 0; i < h; ++i) {
        const unsigned char *row = row_ptr(plane, stride, i);
        for (int j = 0; j < last_column(w); ++j) {
#endif
            float f = (float)sample_at(row, j, bpc) / scaler;
#if ORACLE_MUTATION == 1
            double sq = (double)f * (double)f;
            acc += sq;
#else
            float sq = f * f;
            acc += (double)sq;
#endif
        }
    }
    return (double)acc;
}

/* Each row's sum of binary32 squares in units of 1/scaler^2. A row has at
 * most 2^15 terms below 2^32 units, so its double sum is exact in any order
 * (ADR-1499 "Decision" point 1) and scaling by scaler^2 is exact. */
static void second_moment_rows(const void *plane, int w, int h, int64_t stride, int bpc,
                               uint64_t *rows)
{
    const float scaler = scaler_of(bpc);
    const int k2 = 2 * (bpc - 8);
    for (int i = 0; i < h; ++i) {
        const unsigned char *row = row_ptr(plane, stride, i);
        double acc = 0.0;
        for (int j = 0; j < last_column(w); ++j) {
            float f = (float)sample_at(row, j, bpc) / scaler;
#if ORACLE_MUTATION == 1
            acc += (double)f * (double)f;
#else
            float sq = f * f;
            acc += (double)sq;
#endif
        }
        rows[i] = (uint64_t)ldexp(acc, k2);
    }
}

void vmx_oracle_moment_acc(const void *ref, const void *dis, int width, int height,
                           int64_t stride_bytes, int bpc, double acc[4])
{
#if ORACLE_MUTATION == 11
    const void *a = dis, *b = ref;
#else
    const void *a = ref, *b = dis;
#endif
    acc[0] = first_moment_acc(a, width, height, stride_bytes, bpc);
    acc[1] = first_moment_acc(b, width, height, stride_bytes, bpc);
    acc[2] = second_moment_acc(a, width, height, stride_bytes, bpc);
    acc[3] = second_moment_acc(b, width, height, stride_bytes, bpc);
}

void vmx_oracle_moment(const void *ref, const void *dis, int width, int height,
                       int64_t stride_bytes, int bpc, double out[4], uint64_t *s2_rows)
{
    double acc[4];
    vmx_oracle_moment_acc(ref, dis, width, height, stride_bytes, bpc, acc);
    for (int i = 0; i < 4; ++i)
        out[i] = acc[i] / pixel_count(width, height);
    if (s2_rows) {
#if ORACLE_MUTATION == 11
        const void *a = dis, *b = ref;
#else
        const void *a = ref, *b = dis;
#endif
        second_moment_rows(a, width, height, stride_bytes, bpc, s2_rows);
        second_moment_rows(b, width, height, stride_bytes, bpc, s2_rows + height);
    }
}

/* Not the CPU's result: the second moment as a SIMD path that adds in lanes
 * forms it (the page on the exact second-moment sum, "Neutral / follow-ups":
 * the NEON and SVE2 paths of the CPU extractor add in lanes, so past 2^53
 * units they are not the scalar sum). Reading taken: `lanes` double
 * accumulators, the pixel at raster position n going to lane n mod lanes,
 * the lanes added left to right at the end. lanes == 1 is the scalar loop.
 * Kept to measure that divergence; nothing in the library targets it. */
double vmx_oracle_second_moment_lanes(const void *plane, int width, int height,
                                      int64_t stride_bytes, int bpc, int lanes)
{
    double acc[16] = {0.0};
    if (lanes < 1) lanes = 1;
    if (lanes > 16) lanes = 16;
    const float scaler = scaler_of(bpc);
    long long n = 0;
    for (int i = 0; i < height; ++i) {
        const unsigned char *row = row_ptr(plane, stride_bytes, i);
        for (int j = 0; j < width; ++j) {
            float f = (float)sample_at(row, j, bpc) / scaler;
            float sq = f * f;
            acc[n % lanes] += (double)sq;
            ++n;
        }
    }
    double total = acc[0];
    for (int l = 1; l < lanes; ++l) total += acc[l];
    return total / pixel_count(width, height);
}

/* float_psnr.c::extract() as ADR-1499 "Context" states it: the binary32
 * square of each sample difference, a row's squares into a double
 * (noise_line()), the rows into one double in row order, then the CPU's
 * divisions (by scaler^2 through the normalisation, and by the pixel
 * count). */
double vmx_oracle_psnr_noise(const void *ref, const void *dis, int width, int height,
                             int64_t stride_bytes, int bpc, uint64_t *rows)
{
    const float scaler = scaler_of(bpc);
    const int k2 = 2 * (bpc - 8);
#if ORACLE_MUTATION == 4
    uint64_t exact_total = 0;
#endif
    double noise = 0.0;
#if ORACLE_MUTATION == 10
    double row_acc = 0.0;
#endif
    for (int i = 0; i < height; ++i) {
        const unsigned char *rr = row_ptr(ref, stride_bytes, i);
        const unsigned char *dr = row_ptr(dis, stride_bytes, i);
#if ORACLE_MUTATION != 10
        double row_acc = 0.0;
#endif
        for (int j = 0; j < last_column(width); ++j) {
            float fr = (float)sample_at(rr, j, bpc) / scaler;
            float fd = (float)sample_at(dr, j, bpc) / scaler;
            float e = fr - fd;
            float e2 = e * e;
#if ORACLE_MUTATION == 3
            noise += (double)e2;
#endif
            row_acc += (double)e2;
        }
        if (rows)
            rows[i] = (uint64_t)ldexp(row_acc, k2);
#if ORACLE_MUTATION == 4
        exact_total += (uint64_t)ldexp(row_acc, k2);
#elif ORACLE_MUTATION != 3
        noise += row_acc;
#endif
    }
#if ORACLE_MUTATION == 4
    noise = ldexp((double)exact_total, -k2);
#endif
    return noise;
}

void vmx_oracle_psnr(const void *ref, const void *dis, int width, int height,
                     int64_t stride_bytes, int bpc, uint64_t *rows, double *mse)
{
    const double noise = vmx_oracle_psnr_noise(ref, dis, width, height, stride_bytes, bpc, rows);
#if ORACLE_MUTATION == 13
    *mse = (double)((float)noise / (float)pixel_count(width, height));
#else
    *mse = noise / pixel_count(width, height);
#endif
}

/* integer_psnr of one plane pair (psnr_y, psnr_cb, psnr_cr each take one;
 * the page on the Metal kernel batch T8-1c..k, "Feature scope" and "Integer
 * kernels": integer partials, reduced in double on the host). The pages give
 * no formula; the reading taken is the plain one: the sum of squared
 * codeword differences, an exact integer per row and per plane (no
 * normalisation, no rounding), and the MSE that sum divided by the pixel
 * count in double. */
void vmx_oracle_integer_psnr(const void *ref, const void *dis, int width, int height,
                             int64_t stride_bytes, int bpc, uint64_t *rows, uint64_t *sse,
                             double *mse)
{
    uint64_t total = 0;
    for (int i = 0; i < height; ++i) {
        const unsigned char *rr = row_ptr(ref, stride_bytes, i);
        const unsigned char *dr = row_ptr(dis, stride_bytes, i);
        uint64_t row = 0;
        for (int j = 0; j < last_column(width); ++j) {
            const int64_t d = (int64_t)sample_at(rr, j, bpc) - (int64_t)sample_at(dr, j, bpc);
#if ORACLE_MUTATION == 14
            row += (uint64_t)(d < 0 ? -d : d);
#else
            row += (uint64_t)(d * d);
#endif
        }
        if (rows)
            rows[i] = row;
        total += row;
    }
    *sse = total;
#if ORACLE_MUTATION == 15
    *mse = (double)total / (double)width;
#else
    *mse = (double)total / pixel_count(width, height);
#endif
}

void vmx_oracle_integer_psnr_batch(const void *ref, const void *dis, int width, int height,
                                   int64_t stride_bytes, int bpc, int first, int count,
                                   uint64_t *rows, uint64_t *sse, double *mse)
{
    const int64_t pitch = (int64_t)height * stride_bytes;
    for (int f = 0; f < count; ++f) {
        const int64_t off = (int64_t)(first + f) * pitch;
        vmx_oracle_integer_psnr((const unsigned char *)ref + off, (const unsigned char *)dis + off,
                                width, height, stride_bytes, bpc,
                                rows ? rows + (size_t)f * height : NULL, sse + f, mse + f);
    }
}

/* PSNR from the MSE. The pages leave the formula open; this is the reading
 * taken: the peak is the largest codeword on the 8-bit scale, the MSE is
 * floored at 1e-10, and the result is capped only when psnr_max > 0. */
double vmx_oracle_psnr_db(double mse, int bpc, double psnr_max)
{
    const double peak = (double)((1 << bpc) - 1) / (double)(1 << (bpc - 8));
    const double floor_mse = mse > 1e-10 ? mse : 1e-10;
    double db = 10.0 * log10(peak * peak / floor_mse);
    if (psnr_max > 0.0 && db > psnr_max)
        db = psnr_max;
    return db;
}

void vmx_oracle_moment_batch(const void *ref, const void *dis, int width, int height,
                             int64_t stride_bytes, int bpc, int first, int count,
                             double *out)
{
    const int64_t pitch = (int64_t)height * stride_bytes;
    for (int f = 0; f < count; ++f) {
        const int64_t off = (int64_t)(first + f) * pitch;
        vmx_oracle_moment((const unsigned char *)ref + off, (const unsigned char *)dis + off,
                          width, height, stride_bytes, bpc, out + 4 * (size_t)f, NULL);
    }
}

void vmx_oracle_psnr_batch(const void *ref, const void *dis, int width, int height,
                           int64_t stride_bytes, int bpc, int first, int count,
                           uint64_t *rows, double *mse)
{
    const int64_t pitch = (int64_t)height * stride_bytes;
    for (int f = 0; f < count; ++f) {
        const int64_t off = (int64_t)(first + f) * pitch;
        vmx_oracle_psnr((const unsigned char *)ref + off, (const unsigned char *)dis + off,
                        width, height, stride_bytes, bpc,
                        rows ? rows + (size_t)f * height : NULL, mse + f);
    }
}
