/*
 * vmx.h -- C ABI of libvmx: bit-exact float_moment and float_psnr of 8- to
 * 16-bit luma frame pairs on a CUDA GPU (sm_103a).
 *
 * What is computed (the CPU extractors the results must equal bit for bit):
 *
 *   Samples p are unsigned codewords; scaler = 2^(bpc - 8); the CPU puts every
 *   sample on the 8-bit scale as the binary32 value p / scaler.
 *
 *   float_moment (ADR-1497 "Context"; Research-2081 "Selected restoration"):
 *     first moment  = mean of p / scaler, raster order, double accumulator;
 *     second moment = one binary32 square per pixel, fl32((p/scaler)^2), added
 *                     into a double in raster order, divided by the pixel
 *                     count. Past 2^53 units the CPU's running double rounds
 *                     on every add; the library reproduces that rounding
 *                     value for value (ADR-1497 "Decision").
 *   float_psnr (ADR-1499 "Context" and "Decision"):
 *     each row's sum of binary32 squared sample differences (exact, below
 *     2^47 units), the rows added into one double in row order, divided by
 *     the pixel count: the MSE on the 8-bit scale.
 *
 *   "Units" are 1/scaler^2: every float square is an integer below 2^32 in
 *   them, and the library forms every sum as an integer in these units.
 *
 * Layout of the inputs: frame f of a batch starts at base + f * height *
 * stride_bytes; row i of a frame at + i * stride_bytes. bpc == 8 means uint8
 * samples, 9..16 means uint16 samples in host (little-endian) byte order.
 * Samples above 2^bpc - 1 are used as they are (the CPU does not clamp).
 *
 * Limits: 1 <= width <= 32768 (a row has at most 2^15 terms, ADR-1499
 * "Decision" point 1), height >= 1, width * height <= 2^25, nframes >= 1,
 * stride_bytes >= width * bytes per sample.
 *
 * Streams: every call enqueues its work on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and returns without waiting, except where a
 * function says it synchronises. Calls that share one workspace must not run
 * concurrently.
 *
 * Errors: every int-returning function returns VMX_OK (0) or a negative code.
 * On an argument error nothing is launched and no output is written.
 */
#ifndef VMX_H
#define VMX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VMX_OK 0
#define VMX_EINVAL (-1)    /* bad argument: pointer, size, bpc, stride, workspace size */
#define VMX_ENOMEM (-2)    /* the library could not allocate device memory */
#define VMX_ECUDA (-3)     /* a CUDA call failed; vmx_strerror() names it */
#define VMX_ETIMEOUT (-4)  /* a bounded device wait gave up; outputs are not valid */
#define VMX_ESCRATCH (-5)  /* the shape needs more than VMX_NOALLOC_SCRATCH_BYTES */
#define VMX_ECHECK (-6)    /* a checked build only: an index check failed (the access was skipped) */

#define VMX_FEATURE_MOMENT 1 /* float_moment: 4 doubles per frame */
#define VMX_FEATURE_PSNR 2   /* float_psnr: row sums and the MSE per frame */

/* Bytes of device workspace a call needs for this shape and these features
 * (VMX_FEATURE_* bits). Returns 0 for arguments the calls would reject. */
size_t vmx_workspace_bytes(int width, int height, int bpc, int nframes, int features);

/*
 * float_moment of nframes frame pairs (ADR-1497; Research-2081).
 *   ref, dis      device pointers to the first frame of each batch.
 *   moments       device, [nframes][4] doubles: ref first moment, dis first
 *                 moment, ref second moment, dis second moment.
 *   s2_rows       device or NULL, [nframes][2][height] uint64: each row's
 *                 exact sum of the binary32 squares in units (ref rows, then
 *                 dis rows).
 *   s2_sums       device or NULL, [nframes][2] uint64: the CPU's rounded
 *                 second-moment accumulators after the last pixel, in units
 *                 (the doubles the CPU divides by the pixel count, exactly).
 *   workspace     device memory of at least vmx_workspace_bytes(...,
 *                 VMX_FEATURE_MOMENT) bytes, caller-owned and 256-byte
 *                 aligned; or NULL, in which case the call allocates it on
 *                 `stream`, waits for the result, frees it and returns the
 *                 device status itself (the call is then synchronous).
 * Asynchronous on `stream` when a workspace is given. A bounded device wait
 * that gave up is reported by vmx_workspace_status() on that workspace.
 */
int vmx_moment_frames(const void *ref, const void *dis, int width, int height,
                      int64_t stride_bytes, int bpc, int nframes, double *moments,
                      uint64_t *s2_rows, uint64_t *s2_sums, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * integer_psnr of nframes plane pairs (the page on the Metal kernel batch
 * T8-1c..k, "Feature scope": psnr_y, psnr_cb and psnr_cr, one call per plane;
 * "Integer kernels": integer partials). The pages give no formula; the
 * reading taken: the exact sum of squared codeword differences (no
 * normalisation, no rounding) and the MSE in codeword units.
 *   ref, dis    device planes as vmx_moment_frames() (a chroma plane passes its
 *               own width, height and stride).
 *   sse         device, [nframes] uint64: each plane's sum (cleared and
 *               written by the call).
 *   mse         device, [nframes] doubles: sse / (width * height).
 *   rows        device or NULL, [nframes][height] uint64: each row's sum.
 * PSNR in dB on the host: vmx_integer_psnr_db(). No workspace; asynchronous
 * on `stream`. Errors: VMX_EINVAL (as vmx_moment_frames(); sse and mse
 * required; nothing launched), VMX_ECUDA. Each row's sum goes into its
 * plane's sum by a 64-bit integer atomic add (exact in any order).
 */
int vmx_integer_psnr_frames(const void *ref, const void *dis, int width, int height,
                            int64_t stride_bytes, int bpc, int nframes, uint64_t *sse,
                            double *mse, uint64_t *rows, void *stream);

/*
 * float_psnr of nframes frame pairs (ADR-1499).
 *   rows        device, [nframes][height] uint64: each row's exact sum of the
 *               binary32 squared differences in units of 1/scaler^2.
 *   mse         device, [nframes] doubles: the CPU's row-order noise / pixels.
 *   noise_sums  device or NULL, [nframes] uint64: the CPU's row-order noise
 *               accumulator in units.
 * The PSNR itself is a host function of the MSE: vmx_psnr_db().
 * Workspace, stream and errors as vmx_moment_frames().
 */
int vmx_float_psnr_frames(const void *ref, const void *dis, int width, int height,
                          int64_t stride_bytes, int bpc, int nframes, uint64_t *rows,
                          double *mse, uint64_t *noise_sums, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * Both features in one read of both planes. Same arguments as the two calls
 * above; the workspace is vmx_workspace_bytes(..., VMX_FEATURE_MOMENT |
 * VMX_FEATURE_PSNR). Outputs as above; s2_rows, s2_sums and noise_sums may
 * be NULL.
 */
int vmx_moment_psnr_frames(const void *ref, const void *dis, int width, int height,
                           int64_t stride_bytes, int bpc, int nframes, double *moments,
                           uint64_t *s2_rows, uint64_t *s2_sums, uint64_t *psnr_rows,
                           double *mse, uint64_t *noise_sums, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * Pipelined batches. vmx_frames_ex() is vmx_moment_psnr_frames() with the
 * features as bits (as in vmx_frames_host()) and `flags`:
 *   VMX_FLAG_CLEARED  skip the call's clear of the workspace's control words:
 *                     vmx_workspace_clear() did it on this stream since the
 *                     workspace was last used.
 *   VMX_FLAG_OVERLAP  launch the kernel so that it may start while the
 *                     previous kernel on `stream` is still running
 *                     (programmatic dependent launch: its blocks take the SM
 *                     slots that kernel's blocks leave; with small batches
 *                     several calls run at a time). The caller guarantees
 *                     that this call reads and writes nothing that an earlier
 *                     kernel on `stream` still running may write (another
 *                     workspace, other outputs) and that the workspace was
 *                     cleared beforehand (VMX_FLAG_CLEARED): a clear enqueued
 *                     between the two kernels would separate them. The kernel
 *                     does not finish before the previous one, so later work
 *                     on the stream follows both.
 * Both flags need a workspace. Errors as the other calls; unknown flags are
 * VMX_EINVAL. The pages have no counterpart: this is how a stream of batches
 * of one shape keeps the GPU busy between batches.
 */
#define VMX_FLAG_CLEARED 1u
#define VMX_FLAG_OVERLAP 2u
int vmx_workspace_clear(void *workspace, size_t workspace_bytes, int width, int height, int bpc,
                        int nframes, int features, void *stream);
/*
 * vmx_workspace_clear() of `count` workspaces laid out back to back in one
 * allocation, workspace i at workspace + i * workspace_bytes, by one strided
 * set on `stream` (one node when captured in a graph, where one clear per
 * workspace would be `count`): the batches of one replay cleared at once.
 * workspace_bytes a multiple of 256, at least vmx_workspace_bytes() for the
 * shape; workspace 256-byte aligned. Errors: VMX_EINVAL (NULL, count 0,
 * a shape the library rejects, sizes or alignment; nothing enqueued),
 * VMX_ECUDA.
 */
int vmx_workspace_clear_n(void *workspace, size_t workspace_bytes, size_t count, int width, int height,
                          int bpc, int nframes, int features, void *stream);
int vmx_frames_ex(const void *ref, const void *dis, int width, int height, int64_t stride_bytes,
                  int bpc, int nframes, int features, double *moments, uint64_t *s2_rows,
                  uint64_t *s2_sums, uint64_t *psnr_rows, double *mse, uint64_t *noise_sums,
                  void *workspace, size_t workspace_bytes, unsigned flags, void *stream);

/*
 * Status of the last call that used `workspace`: VMX_OK, VMX_ETIMEOUT if a
 * bounded device wait gave up, or (a checked build only) VMX_ECHECK if an
 * index check failed. Synchronises `stream`.
 */
int vmx_workspace_status(const void *workspace, void *stream);

/*
 * How the last call on `workspace` formed its second-moment sums, summed over
 * its frames and planes (host array of 4): rows added exactly, rows added by
 * their run, rows walked term by term, and 2048-term chunks the term walk
 * scanned (including the psnr row walk). Synchronises `stream`.
 */
int vmx_workspace_stats(const void *workspace, void *stream, uint64_t *out4);

/*
 * PSNR in dB from the MSE on the 8-bit scale, on the host:
 * 10 * log10(peak^2 / max(mse, 1e-10)) with peak = (2^bpc - 1) / 2^(bpc - 8),
 * capped at psnr_max when psnr_max > 0. The pages give no formula; this is
 * the reading the library takes. Host arrays of n doubles.
 */
int vmx_psnr_db(const double *mse, int n, int bpc, double psnr_max, double *psnr);

/*
 * PSNR in dB of integer_psnr MSE values (the page on the Metal kernel batch
 * T8-1c..k, "Feature scope": psnr_y, psnr_cb, psnr_cr; no formula given):
 * the MSE in codeword units over 4^(bpc - 8) (exact: a power of two), which
 * is the MSE on the 8-bit scale, then vmx_psnr_db() of it. Host arrays of n
 * doubles; psnr_max as vmx_psnr_db(). Errors: VMX_EINVAL (a NULL array,
 * n < 0, bpc outside 8..16; nothing written).
 */
int vmx_integer_psnr_db(const double *mse, int n, int bpc, double psnr_max, double *psnr);

/*
 * Host-memory entry point: frames in host memory, results in host memory,
 * same layout and outputs as the device calls, `chunk_frames` frames per
 * launch on `stream`. Page-locked (mapped) inputs are read in place by the
 * kernel over the host link, with no staging copy; other host memory is
 * copied chunk by chunk into the workspace on a stream the call creates
 * while the previous chunk computes. Each chunk's results are copied back
 * on `stream`. Returns after everything has finished. features: VMX_FEATURE_* bits; outputs of a
 * feature not asked for may be NULL, as may s2_rows and psnr (psnr needs
 * VMX_FEATURE_PSNR; it is vmx_psnr_db() of mse with psnr_max).
 *   workspace  device memory of vmx_host_workspace_bytes(...) bytes, 256-byte
 *              aligned, or NULL (then allocated and freed by the call).
 */
size_t vmx_host_workspace_bytes(int width, int height, int64_t stride_bytes, int bpc,
                                int chunk_frames, int features);
int vmx_frames_host(const void *ref, const void *dis, int width, int height,
                    int64_t stride_bytes, int bpc, int nframes, int features,
                    double *moments, uint64_t *s2_rows, uint64_t *psnr_rows, double *mse,
                    double *psnr, double psnr_max, int chunk_frames, void *workspace,
                    size_t workspace_bytes, void *stream);

/* Bytes of host<->device traffic one vmx_frames_host() call moves for these
 * arguments (inputs in, outputs out), for reporting. */
void vmx_frames_host_traffic(int width, int height, int64_t stride_bytes, int bpc,
                             int nframes, int features, int want_s2_rows,
                             uint64_t *h2d_bytes, uint64_t *d2h_bytes);

/*
 * Both features (or either) with no allocation at all. The pages have no
 * counterpart to this call: it exists for callers that cannot allocate
 * device memory while they run, e.g. a stage whose process has handed the
 * whole device to another framework's memory pool, or a real-time pipeline
 * that must not call cudaMalloc/cudaFree (which can synchronise the device).
 *
 * Its scratch is one fixed array of VMX_NOALLOC_SCRATCH_BYTES in the
 * library's static device memory, one per device (present whether or not
 * this call is used). Shapes whose vmx_workspace_bytes(width, height, bpc,
 * nframes, features) exceeds that are rejected with VMX_ESCRATCH before
 * anything is enqueued; split the batch into fewer frames.
 *
 * Set-up: the first call on each device (that device current) looks up the
 * array's address with cudaGetSymbolAddress, which may load the library's
 * device code; make that first call before any stream capture begins. Later
 * calls on the device only enqueue work.
 *
 * Each call clears the control words the kernel needs at zero (a memset on
 * `stream`), then launches the same frame kernel as vmx_moment_psnr_frames.
 * Overlapping calls on one device share the one scratch array and RACE:
 * issue them on one stream, or order them with events, from one thread at
 * a time.
 *   features    VMX_FEATURE_* bits; outputs of a feature not asked for may
 *               be NULL, and s2_rows, s2_sums, noise_sums may be NULL.
 *   outputs     device pointers, layout as vmx_moment_psnr_frames().
 *   status      device or NULL, one uint32: set on `stream` after the
 *               kernel to 0, or to bit 0 when a bounded device wait gave up
 *               and (a checked build only) bit 1 when an index check failed
 *               (the outputs are then not valid).
 * Asynchronous on `stream`. Returns VMX_OK, VMX_EINVAL (arguments, as the
 * other calls), VMX_ESCRATCH, or VMX_ECUDA. Every argument is checked, and
 * VMX_EINVAL or VMX_ESCRATCH returned, before any CUDA call.
 */
#define VMX_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int vmx_frames_noalloc(const void *ref, const void *dis, int width, int height,
                       int64_t stride_bytes, int bpc, int nframes, int features,
                       double *moments, uint64_t *s2_rows, uint64_t *s2_sums,
                       uint64_t *psnr_rows, double *mse, uint64_t *noise_sums,
                       uint32_t *status, void *stream);

/*
 * Checked builds (compiled with VMX_CHECK=1, a debug and test variant of the
 * library): every index the kernels compute into one of their arrays is
 * compared with the array's extent before the access; an index out of range
 * skips the access and is reported, never trapped. No counterpart in the
 * pages. vmx_checked_build() returns 1 in such a build, 0 otherwise. The
 * frame kernel reports a failed check in its call's status (VMX_ECHECK from
 * vmx_workspace_status() or a call with a NULL workspace); integer_psnr has
 * no status word, so vmx_check_status() returns VMX_ECHECK if a check failed
 * in any integer_psnr launch on the current device since the last call (and
 * clears it), else VMX_OK; it synchronises `stream`. In other builds it
 * returns VMX_OK at once.
 */
int vmx_checked_build(void);
int vmx_check_status(void *stream);

/*
 * Timing builds (compiled with VMX_PHASE_TIMES=1, a profiling variant of the
 * library; no counterpart in the pages): the frame kernel adds each phase's
 * SM clock cycles, summed over its warps, and stamps a few events with the
 * GPU's global nanosecond timer, into 16 counters on the current device that
 * accumulate over launches:
 *   [0] first warp's start (ns)      [1] last warp's end (ns)
 *   [2] streaming items (cycles)     [3] look-back, waits included (cycles)
 *   [4] plans and row runs (cycles)  [5] completion of items (cycles)
 *   [6] last warp out of items (ns)  [7] first warp out of items (ns)
 *   [8] walks, waits included (cycles) [9] last walk's end (ns)
 *   [10] walks taken                 [11] items streamed
 *   [12] longest walk (cycles)       [13] first walk's start (ns)
 *   [14] row runs formed             [15] the SM clock rate (kHz)
 * vmx_phase_times copies them into `out` (16 values, when not NULL), then
 * clears them when `reset` is non-zero (the minima to all ones). It
 * synchronises the device's default stream; call it with no launch of the
 * library in flight. Errors: VMX_EINVAL in other builds or with neither an
 * `out` nor `reset`, VMX_ECUDA.
 */
int vmx_phase_times(uint64_t *out, int reset);

/* Name of a status code (and the last CUDA error for VMX_ECUDA). */
const char *vmx_strerror(int status);

/* Launches of the library's own kernels since load (a counter). */
uint64_t vmx_kernel_launches(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int vmx_version(void);

#ifdef __cplusplus
}
#endif
#endif /* VMX_H */
