// vmx_intpsnr.cu -- integer_psnr: per plane, the exact sum of squared
// codeword differences (psnr_y, psnr_cb and psnr_cr each take one plane;
// the page on the Metal kernel batch T8-1c..k, "Feature scope" and "Integer
// kernels": integer partials, reduced on the host in double). Every sum is
// an integer, so the order of the additions cannot change it: rows are
// reduced by warps in any order and added into the plane's sum with 64-bit
// integer atomics.
//
// One warp per row (grid-stride over the batch's rows). A 32-bit word holds
// two 16-bit samples (four 8-bit ones). The absolute differences come from
// a SIMD absolute difference; a 16-bit difference a = 256 h + l squares as
// 256 a h + a l, the two-way 16x8-bit dot products of the word of
// differences with its own bytes rearranged as [l0, l1, h0, h1] (the same
// byte split as the float_psnr row sums); 8-bit differences square by a
// four-way dot product with themselves.

#include <stdint.h>

#include <cuda_runtime.h>

#include "vmx.h"
#include "vmx_internal.h"
#include "vmx_intpsnr.h"

namespace vmx {
namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr int kPsnrThreads = 256;

// Failed index checks of a checked build (bit 1), per device; read and
// cleared by integer_psnr_check_flags().
__device__ uint32_t g_check_flags;

// With VMX_CHECK: whether i < n; if not, the failure is recorded and the
// caller skips the access. Without: always true.
__device__ __forceinline__ bool in_extent(size_t i, size_t n)
{
#if VMX_CHECK
    if (i < n) return true;
    atomicOr(&g_check_flags, 2u);
    return false;
#else
    (void)i;
    (void)n;
    return true;
#endif
}

__device__ __forceinline__ uint4 ld_stream_v4(const void *ptr)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr));
    return v;
}

// 16-byte vector v of a row of `width` samples of `bytes` bytes, zero past
// the row's end; VEC: the row starts on a 16-byte boundary.
template <int BYTES, bool VEC>
__device__ __forceinline__ uint4 row_vec(const unsigned char *row, int v, int width)
{
    constexpr int kPer = 16 / BYTES;
    const int j0 = v * kPer;
    if (VEC && j0 + kPer <= width) return ld_stream_v4(row + 16 * (size_t)v);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        if (j0 + i < width) {
            if (BYTES == 2) {
                const uint32_t s = __ldg(reinterpret_cast<const unsigned short *>(row) + j0 + i);
                w[i >> 1] |= s << (16 * (i & 1));
            } else {
                const uint32_t s = __ldg(row + j0 + i);
                w[i >> 2] |= s << (8 * (i & 3));
            }
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Warp total of values below 2^51 (a lane's share of a row is below 2^42).
__device__ __forceinline__ uint64_t warp_total(uint64_t v)
{
    const uint32_t lo = __reduce_add_sync(kAll, (uint32_t)v & 0xFFFFFFu);
    const uint32_t hi = __reduce_add_sync(kAll, (uint32_t)(v >> 24));
    return ((uint64_t)hi << 24) + lo;
}

// This lane's share of a row's sum of squared differences.
template <int BYTES, bool VEC>
__device__ uint64_t lane_sse(const unsigned char *rr, const unsigned char *dr, int width, int lane)
{
    constexpr int kPer = 16 / BYTES;
    const int nv = (width + kPer - 1) / kPer;
    uint64_t acc = 0;
    if (BYTES == 2) {
        // 32-bit dot-product sums of at most 256 samples a lane stay below
        // 2^32 (256 times 65535 times 255) before they move to acc.
        uint32_t lo = 0, hi = 0, pend = 0;
        for (int v = lane; v < nv; v += 32) {
            const uint4 R = row_vec<BYTES, VEC>(rr, v, width), D = row_vec<BYTES, VEC>(dr, v, width);
            const uint32_t r4[4] = {R.x, R.y, R.z, R.w}, d4[4] = {D.x, D.y, D.z, D.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t a = __vabsdiffu2(r4[w], d4[w]);
                const uint32_t x = __byte_perm(a, 0, 0x3120);
                lo = __dp2a_lo(a, x, lo);
                hi = __dp2a_hi(a, x, hi);
            }
            pend += 8;
            if (pend == 256) {
                acc += ((uint64_t)hi << 8) + lo;
                lo = hi = pend = 0;
            }
        }
        acc += ((uint64_t)hi << 8) + lo;
    } else {
        // A lane holds at most 1024 8-bit samples of a row: below 2^26.
        uint32_t s = 0;
        for (int v = lane; v < nv; v += 32) {
            const uint4 R = row_vec<BYTES, VEC>(rr, v, width), D = row_vec<BYTES, VEC>(dr, v, width);
            const uint32_t r4[4] = {R.x, R.y, R.z, R.w}, d4[4] = {D.x, D.y, D.z, D.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t a = __vabsdiffu4(r4[w], d4[w]);
                s = __dp4a(a, a, s);
            }
        }
        acc = s;
    }
    return acc;
}

template <int BYTES, bool VEC>
__global__ void __launch_bounds__(kPsnrThreads) sse_kernel(const unsigned char *ref,
                                                           const unsigned char *dis, int width,
                                                           int height, int64_t stride, int frames,
                                                           unsigned long long *sse,
                                                           uint64_t *rows, uint32_t shrink)
{
    const int lane = (int)(threadIdx.x & 31);
    const int64_t nrows = (int64_t)frames * height;
    const int64_t warps = (int64_t)gridDim.x * (kPsnrThreads / 32);
    for (int64_t w = (int64_t)blockIdx.x * (kPsnrThreads / 32) + (threadIdx.x >> 5); w < nrows;
         w += warps) {
        const int f = (int)(w / height);
        if (!in_extent((size_t)w, (size_t)nrows)) continue;  // the row lies inside the planes
        const int64_t off = w * stride;  // row w of the batch: frame f, row w - f * height
        const uint64_t row = warp_total(lane_sse<BYTES, VEC>(ref + off, dis + off, width, lane));
        if (lane == 0) {
            // (a test of a checked build takes the rows' extent as one less)
            if (rows && in_extent((size_t)w, (size_t)nrows - shrink)) rows[w] = row;
            if (in_extent((size_t)f, (size_t)frames)) atomicAdd(sse + f, (unsigned long long)row);
        }
    }
}

__global__ void mse_kernel(const unsigned long long *sse, double *mse, int frames, double n)
{
    const int f = (int)(blockIdx.x * blockDim.x + threadIdx.x);
    if (f < frames) mse[f] = (double)sse[f] / n;
}

template <int BYTES>
cudaError_t launch_sse(const IntPsnrArgs &a, bool vec, int grid, cudaStream_t s)
{
    if (vec)
        sse_kernel<BYTES, true><<<grid, kPsnrThreads, 0, s>>>(
            a.ref, a.dis, a.width, a.height, a.stride, a.frames,
            reinterpret_cast<unsigned long long *>(a.sse), a.rows, a.check_shrink);
    else
        sse_kernel<BYTES, false><<<grid, kPsnrThreads, 0, s>>>(
            a.ref, a.dis, a.width, a.height, a.stride, a.frames,
            reinterpret_cast<unsigned long long *>(a.sse), a.rows, a.check_shrink);
    return cudaGetLastError();
}

}  // namespace

cudaError_t integer_psnr_check_flags(uint32_t *flags, cudaStream_t stream)
{
    *flags = 0;
    if (!VMX_CHECK) return cudaSuccess;
    cudaError_t err = cudaMemcpyFromSymbolAsync(flags, g_check_flags, sizeof(uint32_t), 0,
                                                cudaMemcpyDeviceToHost, stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
    const uint32_t zero = 0;
    if (err == cudaSuccess) err = cudaMemcpyToSymbol(g_check_flags, &zero, sizeof zero);
    return err;
}

cudaError_t launch_integer_psnr(const IntPsnrArgs &a, cudaStream_t stream)
{
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    const int64_t nrows = (int64_t)a.frames * a.height;
    const int64_t want = (nrows + kPsnrThreads / 32 - 1) / (kPsnrThreads / 32);
    const int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    const bool vec = (uintptr_t)a.ref % 16 == 0 && (uintptr_t)a.dis % 16 == 0 && a.stride % 16 == 0;
    err = cudaMemsetAsync(a.sse, 0, (size_t)a.frames * sizeof(uint64_t), stream);
    if (err != cudaSuccess) return err;
    err = a.bytes == 2 ? launch_sse<2>(a, vec, grid, stream) : launch_sse<1>(a, vec, grid, stream);
    if (err != cudaSuccess) return err;
    mse_kernel<<<(a.frames + 127) / 128, 128, 0, stream>>>(
        reinterpret_cast<const unsigned long long *>(a.sse), a.mse, a.frames,
        (double)a.width * (double)a.height);
    return cudaGetLastError();
}

}  // namespace vmx
