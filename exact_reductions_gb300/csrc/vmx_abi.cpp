// vmx_abi.cpp -- the C ABI of libvmx: argument checks, the workspace layout,
// the launch of the frame kernel, and the host-memory pipeline.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "vmx.h"
#include "vmx_internal.h"
#include "vmx_intpsnr.h"

namespace vmx {

namespace {

std::atomic<uint64_t> g_launches{0};
thread_local char g_last_cuda[160] = "";

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int cuda_fail(cudaError_t e)
{
    std::snprintf(g_last_cuda, sizeof g_last_cuda, "%s: %s", cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return e == cudaErrorMemoryAllocation ? VMX_ENOMEM : VMX_ECUDA;
}

// Host-side fault injection for tests: VMX_TEST_FAIL_AT=alloc|launch|status
// makes that stage fail without touching the GPU.
bool fail_at(const char *stage)
{
    const char *v = std::getenv("VMX_TEST_FAIL_AT");
    return v && std::strcmp(v, stage) == 0;
}

// Tests of the bounded device waits: VMX_TEST_SPIN_LIMIT=n polls instead of
// kSpinLimit, and VMX_TEST_WAIT_STALL=1 makes the walks wait for a block count
// that is never reached, so that every such wait gives up and sets the
// status word (the kernel still returns; nothing faults).
uint32_t spin_limit_setting()
{
    const char *v = std::getenv("VMX_TEST_SPIN_LIMIT");
    if (!v) return kSpinLimit;
    const long n = std::strtol(v, nullptr, 10);
    return n > 0 && n < (long)kSpinLimit ? (uint32_t)n : kSpinLimit;
}

bool wait_stall_setting()
{
    const char *v = std::getenv("VMX_TEST_WAIT_STALL");
    return v && std::strcmp(v, "1") == 0;
}

// Tests of a checked build: VMX_TEST_CHECK_SHRINK=1 makes the kernel take the
// per-plane row arrays as one element shorter than they are, so that an
// index check fails (and skips its access; nothing goes out of bounds).
uint32_t check_shrink_setting()
{
    const char *v = std::getenv("VMX_TEST_CHECK_SHRINK");
    return v && std::strcmp(v, "1") == 0 ? 1u : 0u;
}

// A device status word: bit 1 an index check failed (checked builds), bit 0
// a bounded wait gave up.
int status_of_word(uint32_t w)
{
    if (w & 2u) return VMX_ECHECK;
    return w != 0u ? VMX_ETIMEOUT : VMX_OK;
}

// Tests of forward progress: VMX_TEST_GRID_MULT=n (2..16) launches n times
// as many CTAs as the GPU holds at once, so that most of the grid starts only
// as earlier CTAs exit.
int grid_mult_setting()
{
    const char *v = std::getenv("VMX_TEST_GRID_MULT");
    if (!v) return 1;
    const long n = std::strtol(v, nullptr, 10);
    return n >= 2 && n <= 16 ? (int)n : 1;
}

int bytes_per_sample(int bpc) { return bpc == 8 ? 1 : 2; }

}  // namespace

// Items a call has at least, rows allowing (shorter items for small calls).
#ifndef VMX_FEW_ITEMS
#define VMX_FEW_ITEMS 512
#endif
constexpr int kFewItems = VMX_FEW_ITEMS;

bool make_layout(int width, int height, int bpc, int frames, int features, Layout *L)
{
    if (width < 1 || width > 32768 || height < 1 || frames < 1 || bpc < 8 || bpc > 16)
        return false;
    if ((int64_t)width * height > (int64_t)1 << 25) return false;
    if (features < 1 || features > 3) return false;
    const int64_t n = (int64_t)width * height;
    const bool m = features & VMX_FEATURE_MOMENT;
    // Terms are below 2^32 units: a frame of n pixels stays at or below 2^53
    // units when n <= 2^21 and below 2^55 when n <= 2^23.
    L->ordered = m && bpc > 8 && n > ((int64_t)1 << 21);
    L->full = L->ordered && n > ((int64_t)1 << 23);
    const int target = L->full ? kItemPixelsFull : kItemPixels;
    int rpi = std::min(kMaxRowsPerItem, std::max(1, (target + width - 1) / width));
    // A call of very few items (a small frame or two) would leave most of
    // the GPU idle and each warp walking its item's rows one after another:
    // shorter items then, down to one row, until the call has kFewItems.
    if (!L->full) rpi = (int)std::max<int64_t>(1, std::min<int64_t>(rpi, (int64_t)frames * height / kFewItems));
    const int ipf = (height + rpi - 1) / rpi;
    const int bpf = (ipf + kBlockItems - 1) / kBlockItems;
    if ((int64_t)frames * ipf >= (int64_t)INT_MAX / 2) return false;
    const size_t F = (size_t)frames, I = (size_t)ipf, B = (size_t)bpf, H = (size_t)height;
    L->width = width;
    L->height = height;
    L->frames = frames;
    L->bpc = bpc;
    L->features = features;
    L->rows_per_item = rpi;
    L->items_per_frame = ipf;
    L->blocks_per_frame = bpf;
    size_t off = 0;
    L->off_ctrl = off;
    off = align256(off + (kCtrlWords + F * B + (L->full ? F * I : 0)) * sizeof(uint32_t));
    L->ctrl_bytes = off;
    L->off_blocks = off;
    off = align256(off + F * B * sizeof(Agg));
    L->off_items = off;
    off = align256(off + F * I * sizeof(Agg));
    L->off_item_inc = off;
    if (L->full) off = align256(off + F * I * 2 * sizeof(uint64_t));
    L->off_s2_rows = off;
    if (m) off = align256(off + F * 2 * H * sizeof(uint64_t));
    L->off_odd_rows = off;
    if (L->ordered) off = align256(off + F * 2 * H * sizeof(uint32_t));
    L->off_rec = off;
    if (L->full) off = align256(off + F * 2 * H * sizeof(RowRec));
    L->total = off;
    return true;
}

namespace {

struct Outputs {
    double *moments;
    uint64_t *s2_rows, *s2_sums, *psnr_rows;
    double *mse;
    uint64_t *noise_sums;
};

// The checks of a frame call's planes, shape and outputs (no CUDA call):
// VMX_OK with the workspace layout in *L, else VMX_EINVAL.
int check_frames_args(const void *ref, const void *dis, int width, int height, int64_t stride,
                      int bpc, int nframes, int features, const Outputs &o, Layout *L)
{
    if (!ref || !dis || !make_layout(width, height, bpc, nframes, features, L)) return VMX_EINVAL;
    if (stride < (int64_t)width * bytes_per_sample(bpc)) return VMX_EINVAL;
    if ((features & VMX_FEATURE_MOMENT) && !o.moments) return VMX_EINVAL;
    if ((features & VMX_FEATURE_PSNR) && (!o.psnr_rows || !o.mse)) return VMX_EINVAL;
    if (bpc > 8 && ((uintptr_t)ref % 2 || (uintptr_t)dis % 2 || stride % 2)) return VMX_EINVAL;
    return VMX_OK;
}

// status: where a bounded wait that gave up is recorded; NULL for the
// workspace's own status word (cleared with the other control words).
int run_frames(const void *ref, const void *dis, int width, int height, int64_t stride,
               int bpc, int nframes, int features, const Outputs &o, void *workspace,
               size_t workspace_bytes, cudaStream_t stream, uint32_t *status_word = nullptr,
               unsigned flags = 0)
{
    if (flags & ~(unsigned)(VMX_FLAG_CLEARED | VMX_FLAG_OVERLAP)) return VMX_EINVAL;
    if (flags && !workspace) return VMX_EINVAL;
    Layout L;
    const int bad = check_frames_args(ref, dis, width, height, stride, bpc, nframes, features, o, &L);
    if (bad != VMX_OK) return bad;
    const bool own = workspace == nullptr;
    if (!own && (workspace_bytes < L.total || (uintptr_t)workspace % 256)) return VMX_EINVAL;
    if (own && fail_at("alloc")) return VMX_ENOMEM;
    if (fail_at("launch")) {
        std::snprintf(g_last_cuda, sizeof g_last_cuda, "injected launch failure");
        return VMX_ECUDA;
    }
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    cudaError_t err;
    if (own) {
        void *p = nullptr;
        err = cudaMallocAsync(&p, L.total, stream);
        if (err != cudaSuccess) return cuda_fail(err);
        ws = static_cast<unsigned char *>(p);
    }
    Params p;
    p.ref = static_cast<const unsigned char *>(ref);
    p.dis = static_cast<const unsigned char *>(dis);
    p.stride = stride;
    p.pitch = stride * height;
    p.width = width;
    p.height = height;
    p.frames = nframes;
    p.k = bpc - 8;
    p.rows_per_item = L.rows_per_item;
    p.items_per_frame = L.items_per_frame;
    p.blocks_per_frame = L.blocks_per_frame;
    p.ctrl = reinterpret_cast<uint32_t *>(ws + L.off_ctrl);
    p.block_fin = p.ctrl + kCtrlWords;
    p.flags = p.block_fin + (size_t)nframes * L.blocks_per_frame;
    p.status = status_word ? status_word : p.ctrl + kCtrlStatus;
    p.items = reinterpret_cast<Agg *>(ws + L.off_items);
    p.blocks = reinterpret_cast<Agg *>(ws + L.off_blocks);
    p.item_inc = reinterpret_cast<uint64_t *>(ws + L.off_item_inc);
    p.odd_rows = reinterpret_cast<uint32_t *>(ws + L.off_odd_rows);
    p.s2_rows = o.s2_rows ? o.s2_rows : reinterpret_cast<uint64_t *>(ws + L.off_s2_rows);
    p.psnr_rows = o.psnr_rows;
    p.rec = reinterpret_cast<RowRec *>(ws + L.off_rec);
    p.moments = o.moments;
    p.mse = o.mse;
    p.s2_sums = o.s2_sums;
    p.noise_sums = o.noise_sums;
    p.spin_limit = spin_limit_setting();
    p.test_stall = wait_stall_setting() ? 1u : 0u;
    p.test_grid_mult = grid_mult_setting();
    p.check_shrink = check_shrink_setting();
    p.overlap = (flags & VMX_FLAG_OVERLAP) ? 1u : 0u;
    const bool vec = (uintptr_t)ref % 16 == 0 && (uintptr_t)dis % 16 == 0 && stride % 16 == 0;
    err = (flags & VMX_FLAG_CLEARED) ? cudaSuccess
                                     : cudaMemsetAsync(ws + L.off_ctrl, 0, L.ctrl_bytes, stream);
    if (err == cudaSuccess) {
        err = launch_frames(p, L, features, vec, stream);
        if (err == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    if (!own) return err == cudaSuccess ? VMX_OK : cuda_fail(err);
    int status = VMX_OK;
    uint32_t dev_status = 0;
    if (err == cudaSuccess)
        err = cudaMemcpyAsync(&dev_status, p.ctrl + kCtrlStatus, sizeof dev_status,
                              cudaMemcpyDeviceToHost, stream);
    const cudaError_t ferr = cudaFreeAsync(ws, stream);
    if (err == cudaSuccess) err = ferr;
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) status = cuda_fail(err);
    else status = status_of_word(dev_status);
    return status;
}

}  // namespace
}  // namespace vmx

using namespace vmx;

extern "C" {

int vmx_version(void) { return 10200; }

int vmx_checked_build(void) { return VMX_CHECK ? 1 : 0; }

int vmx_phase_times(uint64_t *out, int reset)
{
    if (!VMX_PHASE_TIMES || (!out && !reset)) return VMX_EINVAL;
    const cudaError_t err = phase_times(out, reset != 0);
    return err == cudaSuccess ? VMX_OK : cuda_fail(err);
}

int vmx_check_status(void *stream)
{
    if (!VMX_CHECK) return VMX_OK;
    uint32_t v = 0;
    const cudaError_t err = integer_psnr_check_flags(&v, static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err);
    return v ? VMX_ECHECK : VMX_OK;
}

uint64_t vmx_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char *vmx_strerror(int status)
{
    switch (status) {
    case VMX_OK: return "ok";
    case VMX_EINVAL: return "invalid argument";
    case VMX_ENOMEM: return "out of device memory";
    case VMX_ECUDA: return g_last_cuda[0] ? g_last_cuda : "CUDA error";
    case VMX_ETIMEOUT: return "a bounded device wait gave up";
    case VMX_ESCRATCH: return "shape needs more scratch than the no-alloc call holds";
    case VMX_ECHECK: return "an index check failed (checked build)";
    default: return "unknown status";
    }
}

size_t vmx_workspace_bytes(int width, int height, int bpc, int nframes, int features)
{
    Layout L;
    if (!make_layout(width, height, bpc, nframes, features, &L)) return 0;
    return L.total;
}

int vmx_moment_frames(const void *ref, const void *dis, int width, int height,
                      int64_t stride_bytes, int bpc, int nframes, double *moments,
                      uint64_t *s2_rows, uint64_t *s2_sums, void *workspace,
                      size_t workspace_bytes, void *stream)
{
    const Outputs o{moments, s2_rows, s2_sums, nullptr, nullptr, nullptr};
    return run_frames(ref, dis, width, height, stride_bytes, bpc, nframes, VMX_FEATURE_MOMENT, o,
                      workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int vmx_float_psnr_frames(const void *ref, const void *dis, int width, int height,
                          int64_t stride_bytes, int bpc, int nframes, uint64_t *rows,
                          double *mse, uint64_t *noise_sums, void *workspace,
                          size_t workspace_bytes, void *stream)
{
    const Outputs o{nullptr, nullptr, nullptr, rows, mse, noise_sums};
    return run_frames(ref, dis, width, height, stride_bytes, bpc, nframes, VMX_FEATURE_PSNR, o,
                      workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int vmx_integer_psnr_frames(const void *ref, const void *dis, int width, int height,
                            int64_t stride_bytes, int bpc, int nframes, uint64_t *sse,
                            double *mse, uint64_t *rows, void *stream)
{
    if (!ref || !dis || !sse || !mse) return VMX_EINVAL;
    if (width < 1 || width > 32768 || height < 1 || nframes < 1 || bpc < 8 || bpc > 16)
        return VMX_EINVAL;
    if ((int64_t)width * height > (int64_t)1 << 25) return VMX_EINVAL;
    if (stride_bytes < (int64_t)width * bytes_per_sample(bpc)) return VMX_EINVAL;
    if (bpc > 8 && ((uintptr_t)ref % 2 || (uintptr_t)dis % 2 || stride_bytes % 2)) return VMX_EINVAL;
    if (fail_at("launch")) {
        std::snprintf(g_last_cuda, sizeof g_last_cuda, "injected launch failure");
        return VMX_ECUDA;
    }
    IntPsnrArgs a;
    a.ref = static_cast<const unsigned char *>(ref);
    a.dis = static_cast<const unsigned char *>(dis);
    a.width = width;
    a.height = height;
    a.frames = nframes;
    a.stride = stride_bytes;
    a.bytes = bytes_per_sample(bpc);
    a.sse = sse;
    a.mse = mse;
    a.rows = rows;
    a.check_shrink = check_shrink_setting();
    const cudaError_t err = launch_integer_psnr(a, static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err);
    g_launches.fetch_add(2, std::memory_order_relaxed);
    return VMX_OK;
}

int vmx_moment_psnr_frames(const void *ref, const void *dis, int width, int height,
                           int64_t stride_bytes, int bpc, int nframes, double *moments,
                           uint64_t *s2_rows, uint64_t *s2_sums, uint64_t *psnr_rows,
                           double *mse, uint64_t *noise_sums, void *workspace,
                           size_t workspace_bytes, void *stream)
{
    const Outputs o{moments, s2_rows, s2_sums, psnr_rows, mse, noise_sums};
    return run_frames(ref, dis, width, height, stride_bytes, bpc, nframes,
                      VMX_FEATURE_MOMENT | VMX_FEATURE_PSNR, o, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream));
}

int vmx_workspace_clear(void *workspace, size_t workspace_bytes, int width, int height, int bpc,
                        int nframes, int features, void *stream)
{
    Layout L;
    if (!workspace || !make_layout(width, height, bpc, nframes, features, &L)) return VMX_EINVAL;
    if (workspace_bytes < L.total || (uintptr_t)workspace % 256) return VMX_EINVAL;
    const cudaError_t err =
        cudaMemsetAsync(static_cast<unsigned char *>(workspace) + L.off_ctrl, 0, L.ctrl_bytes,
                        static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? VMX_OK : cuda_fail(err);
}

int vmx_workspace_clear_n(void *workspace, size_t workspace_bytes, size_t count, int width, int height,
                          int bpc, int nframes, int features, void *stream)
{
    Layout L;
    if (!workspace || count == 0 || !make_layout(width, height, bpc, nframes, features, &L)) return VMX_EINVAL;
    if (workspace_bytes < L.total || workspace_bytes % 256 || (uintptr_t)workspace % 256) return VMX_EINVAL;
    // One strided set covers every workspace's control words: one graph node.
    const cudaError_t err =
        cudaMemset2DAsync(static_cast<unsigned char *>(workspace) + L.off_ctrl, workspace_bytes, 0,
                          L.ctrl_bytes, count, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? VMX_OK : cuda_fail(err);
}

int vmx_frames_ex(const void *ref, const void *dis, int width, int height, int64_t stride_bytes,
                  int bpc, int nframes, int features, double *moments, uint64_t *s2_rows,
                  uint64_t *s2_sums, uint64_t *psnr_rows, double *mse, uint64_t *noise_sums,
                  void *workspace, size_t workspace_bytes, unsigned flags, void *stream)
{
    const Outputs o{moments, s2_rows, s2_sums, psnr_rows, mse, noise_sums};
    return run_frames(ref, dis, width, height, stride_bytes, bpc, nframes, features, o, workspace,
                      workspace_bytes, static_cast<cudaStream_t>(stream), nullptr, flags);
}

int vmx_workspace_status(const void *workspace, void *stream)
{
    if (!workspace) return VMX_EINVAL;
    if (fail_at("status")) return VMX_ETIMEOUT;
    uint32_t v = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint32_t *ctrl = reinterpret_cast<const uint32_t *>(workspace);
    cudaError_t err = cudaMemcpyAsync(&v, ctrl + kCtrlStatus, sizeof v, cudaMemcpyDeviceToHost, s);
    if (err == cudaSuccess) err = cudaStreamSynchronize(s);
    if (err != cudaSuccess) return cuda_fail(err);
    return status_of_word(v);
}

int vmx_workspace_stats(const void *workspace, void *stream, uint64_t *out4)
{
    if (!workspace || !out4) return VMX_EINVAL;
    uint32_t v[4] = {0, 0, 0, 0};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint32_t *ctrl = reinterpret_cast<const uint32_t *>(workspace);
    cudaError_t err =
        cudaMemcpyAsync(v, ctrl + kCtrlRowsExact, sizeof v, cudaMemcpyDeviceToHost, s);
    if (err == cudaSuccess) err = cudaStreamSynchronize(s);
    if (err != cudaSuccess) return cuda_fail(err);
    for (int i = 0; i < 4; ++i) out4[i] = v[i];
    return VMX_OK;
}

int vmx_psnr_db(const double *mse, int n, int bpc, double psnr_max, double *psnr)
{
    if (!mse || !psnr || n < 0 || bpc < 8 || bpc > 16) return VMX_EINVAL;
    const double peak = (double)((1 << bpc) - 1) / (double)(1 << (bpc - 8));
    for (int i = 0; i < n; ++i) {
        const double m = mse[i] > 1e-10 ? mse[i] : 1e-10;
        double db = 10.0 * std::log10(peak * peak / m);
        if (psnr_max > 0.0 && db > psnr_max) db = psnr_max;
        psnr[i] = db;
    }
    return VMX_OK;
}

int vmx_integer_psnr_db(const double *mse, int n, int bpc, double psnr_max, double *psnr)
{
    if (!mse || !psnr || n < 0 || bpc < 8 || bpc > 16) return VMX_EINVAL;
    // MSE in codeword units over 4^(bpc - 8) (a power of two: exact) is the
    // MSE on the 8-bit scale that vmx_psnr_db takes.
    const double scale = 1.0 / (double)(1ull << (2 * (bpc - 8)));
    for (int i = 0; i < n; ++i) {
        const double m = mse[i] * scale;
        const int rc = vmx_psnr_db(&m, 1, bpc, psnr_max, psnr + i);
        if (rc != VMX_OK) return rc;
    }
    return VMX_OK;
}

// ---------------------------------------------------- host-memory pipeline

namespace {

struct HostPlan {
    size_t in_bytes;      // one plane of one chunk
    size_t out_bytes;     // one chunk's outputs
    size_t ws_bytes;      // the frame kernel's workspace for one chunk
    size_t off_in[2][2];  // [slot][plane]
    size_t off_out[2];
    size_t off_ws;
    size_t off_status;    // u32 status over all chunks
    size_t total;
    // Offsets inside one chunk's outputs.
    size_t o_moments, o_s2_rows, o_psnr_rows, o_mse;
};

bool host_plan(int width, int height, int64_t stride, int bpc, int chunk, int features,
               HostPlan *hp)
{
    Layout L;
    if (chunk < 1 || !make_layout(width, height, bpc, chunk, features, &L)) return false;
    if (stride < (int64_t)width * bytes_per_sample(bpc)) return false;
    const size_t c = (size_t)chunk, H = (size_t)height;
    hp->in_bytes = c * H * (size_t)stride;
    size_t o = 0;
    hp->o_moments = o;
    o = align256(o + c * 4 * sizeof(double));
    hp->o_s2_rows = o;
    o = align256(o + c * 2 * H * sizeof(uint64_t));
    hp->o_psnr_rows = o;
    o = align256(o + c * H * sizeof(uint64_t));
    hp->o_mse = o;
    o = align256(o + c * sizeof(double));
    hp->out_bytes = o;
    hp->ws_bytes = L.total;
    size_t off = 0;
    for (int s = 0; s < 2; ++s)
        for (int pl = 0; pl < 2; ++pl) {
            hp->off_in[s][pl] = off;
            off = align256(off + hp->in_bytes);
        }
    for (int s = 0; s < 2; ++s) {
        hp->off_out[s] = off;
        off = align256(off + hp->out_bytes);
    }
    hp->off_ws = off;
    off = align256(off + hp->ws_bytes);
    hp->off_status = off;
    off = align256(off + sizeof(uint32_t));
    hp->total = off;
    return true;
}

// The device's address for `bytes` of host memory at ptr when the device can
// read all of it in place (page-locked, mapped memory), else false.
bool device_view(const void *ptr, size_t bytes, const unsigned char **dev)
{
    cudaPointerAttributes a, b;
    const unsigned char *p = static_cast<const unsigned char *>(ptr);
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess ||
        cudaPointerGetAttributes(&b, p + (bytes - 1)) != cudaSuccess) {
        cudaGetLastError();  // not an error for the call: use staged copies
        return false;
    }
    if (a.type != cudaMemoryTypeHost || b.type != cudaMemoryTypeHost || !a.devicePointer ||
        !b.devicePointer)
        return false;
    const unsigned char *d = static_cast<const unsigned char *>(a.devicePointer);
    if (static_cast<const unsigned char *>(b.devicePointer) != d + (bytes - 1)) return false;
    *dev = d;
    return true;
}

}  // namespace

size_t vmx_host_workspace_bytes(int width, int height, int64_t stride_bytes, int bpc,
                                int chunk_frames, int features)
{
    HostPlan hp;
    if (!host_plan(width, height, stride_bytes, bpc, chunk_frames, features, &hp)) return 0;
    return hp.total;
}

void vmx_frames_host_traffic(int width, int height, int64_t stride_bytes, int bpc,
                             int nframes, int features, int want_s2_rows,
                             uint64_t *h2d_bytes, uint64_t *d2h_bytes)
{
    const uint64_t F = (uint64_t)std::max(nframes, 0), H = (uint64_t)std::max(height, 0);
    (void)width;
    (void)bpc;
    if (h2d_bytes) *h2d_bytes = 2 * F * H * (uint64_t)std::max<int64_t>(stride_bytes, 0);
    uint64_t out = 0;
    if (features & VMX_FEATURE_MOMENT) {
        out += F * 4 * sizeof(double);
        if (want_s2_rows) out += F * 2 * H * sizeof(uint64_t);
    }
    if (features & VMX_FEATURE_PSNR) out += F * H * sizeof(uint64_t) + F * sizeof(double);
    if (d2h_bytes) *d2h_bytes = out;
}

int vmx_frames_host(const void *ref, const void *dis, int width, int height,
                    int64_t stride_bytes, int bpc, int nframes, int features,
                    double *moments, uint64_t *s2_rows, uint64_t *psnr_rows, double *mse,
                    double *psnr, double psnr_max, int chunk_frames, void *workspace,
                    size_t workspace_bytes, void *stream)
{
    if (!ref || !dis || nframes < 1 || features < 1 || features > 3) return VMX_EINVAL;
    const bool m = features & VMX_FEATURE_MOMENT, ps = features & VMX_FEATURE_PSNR;
    if ((m && !moments) || (ps && (!psnr_rows || !mse)) || (psnr && !ps)) return VMX_EINVAL;
    const int chunk = std::min(std::max(chunk_frames, 1), nframes);
    HostPlan hp;
    if (!host_plan(width, height, stride_bytes, bpc, chunk, features, &hp)) return VMX_EINVAL;
    const bool own = workspace == nullptr;
    if (!own && (workspace_bytes < hp.total || (uintptr_t)workspace % 256)) return VMX_EINVAL;
    if (fail_at("alloc")) return VMX_ENOMEM;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaStream_t copy = nullptr;
    cudaEvent_t copied[2] = {nullptr, nullptr}, computed[2] = {nullptr, nullptr};
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    int status = VMX_OK;
    cudaError_t err = cudaSuccess;
    if (own) {
        void *p = nullptr;
        err = cudaMalloc(&p, hp.total);
        if (err != cudaSuccess) return cuda_fail(err);
        ws = static_cast<unsigned char *>(p);
    }
    const size_t H = (size_t)height;
    const size_t frame_bytes = H * (size_t)stride_bytes;
    // Page-locked inputs are read in place by the kernel (over the host link,
    // no staging copy); others are copied chunk by chunk into the workspace.
    const unsigned char *zr = nullptr, *zd = nullptr;
    const bool in_place = device_view(ref, (size_t)nframes * frame_bytes, &zr) &&
                          device_view(dis, (size_t)nframes * frame_bytes, &zd);
    if (!in_place) {
        err = cudaStreamCreateWithFlags(&copy, cudaStreamNonBlocking);
        for (int s = 0; s < 2 && err == cudaSuccess; ++s) {
            err = cudaEventCreateWithFlags(&copied[s], cudaEventDisableTiming);
            if (err == cudaSuccess)
                err = cudaEventCreateWithFlags(&computed[s], cudaEventDisableTiming);
        }
    }
    uint32_t *dstatus = reinterpret_cast<uint32_t *>(ws + hp.off_status);
    if (err == cudaSuccess) err = cudaMemsetAsync(dstatus, 0, sizeof(uint32_t), cs);
    for (int c0 = 0, it = 0; c0 < nframes && err == cudaSuccess && status == VMX_OK;
         c0 += chunk, ++it) {
        const int n = std::min(chunk, nframes - c0);
        const int slot = in_place ? 0 : it & 1;
        const unsigned char *in_r = in_place ? zr + c0 * frame_bytes : ws + hp.off_in[slot][0];
        const unsigned char *in_d = in_place ? zd + c0 * frame_bytes : ws + hp.off_in[slot][1];
        unsigned char *out = ws + hp.off_out[slot];
        if (!in_place) {
            // Inputs of this chunk: wait until the slot's previous chunk computed.
            unsigned char *sr = ws + hp.off_in[slot][0], *sd = ws + hp.off_in[slot][1];
            if (it >= 2) err = cudaStreamWaitEvent(copy, computed[slot], 0);
            if (err == cudaSuccess)
                err = cudaMemcpyAsync(sr, static_cast<const unsigned char *>(ref) + c0 * frame_bytes,
                                      n * frame_bytes, cudaMemcpyHostToDevice, copy);
            if (err == cudaSuccess)
                err = cudaMemcpyAsync(sd, static_cast<const unsigned char *>(dis) + c0 * frame_bytes,
                                      n * frame_bytes, cudaMemcpyHostToDevice, copy);
            if (err == cudaSuccess) err = cudaEventRecord(copied[slot], copy);
            if (err == cudaSuccess) err = cudaStreamWaitEvent(cs, copied[slot], 0);
        }
        if (err != cudaSuccess) break;
        Outputs o;
        o.moments = m ? reinterpret_cast<double *>(out + hp.o_moments) : nullptr;
        o.s2_rows = m ? reinterpret_cast<uint64_t *>(out + hp.o_s2_rows) : nullptr;
        o.s2_sums = nullptr;
        o.psnr_rows = ps ? reinterpret_cast<uint64_t *>(out + hp.o_psnr_rows) : nullptr;
        o.mse = ps ? reinterpret_cast<double *>(out + hp.o_mse) : nullptr;
        o.noise_sums = nullptr;
        status = run_frames(in_r, in_d, width, height, stride_bytes, bpc, n, features, o,
                            ws + hp.off_ws, hp.ws_bytes, cs, dstatus);
        if (status != VMX_OK) break;
        if (m) {
            err = cudaMemcpyAsync(moments + (size_t)c0 * 4, o.moments, n * 4 * sizeof(double),
                                  cudaMemcpyDeviceToHost, cs);
            if (err == cudaSuccess && s2_rows)
                err = cudaMemcpyAsync(s2_rows + (size_t)c0 * 2 * H, o.s2_rows,
                                      n * 2 * H * sizeof(uint64_t), cudaMemcpyDeviceToHost, cs);
        }
        if (ps && err == cudaSuccess) {
            err = cudaMemcpyAsync(psnr_rows + (size_t)c0 * H, o.psnr_rows, n * H * sizeof(uint64_t),
                                  cudaMemcpyDeviceToHost, cs);
            if (err == cudaSuccess)
                err = cudaMemcpyAsync(mse + c0, o.mse, n * sizeof(double), cudaMemcpyDeviceToHost, cs);
        }
        if (err == cudaSuccess && !in_place) err = cudaEventRecord(computed[slot], cs);
    }
    // A bounded wait that gave up in any chunk fails the call.
    uint32_t st = 0;
    if (err == cudaSuccess && status == VMX_OK)
        err = cudaMemcpyAsync(&st, dstatus, sizeof st, cudaMemcpyDeviceToHost, cs);
    if (err == cudaSuccess) err = cudaStreamSynchronize(cs);
    if (err == cudaSuccess && status == VMX_OK && st) status = status_of_word(st);
    if (copy) cudaStreamSynchronize(copy);
    for (int s = 0; s < 2; ++s) {
        if (copied[s]) cudaEventDestroy(copied[s]);
        if (computed[s]) cudaEventDestroy(computed[s]);
    }
    if (copy) cudaStreamDestroy(copy);
    if (own) cudaFree(ws);
    if (status == VMX_OK && err != cudaSuccess) status = cuda_fail(err);
    if (status == VMX_OK && psnr) status = vmx_psnr_db(mse, nframes, bpc, psnr_max, psnr);
    return status;
}

// The no-alloc call's scratch address per device, looked up on the first
// call made with that device current.
namespace {
constexpr int kMaxDevices = 64;
std::atomic<void *> g_noalloc_ptr[kMaxDevices];
std::mutex g_noalloc_mu;
}  // namespace

int vmx_frames_noalloc(const void *ref, const void *dis, int width, int height,
                       int64_t stride_bytes, int bpc, int nframes, int features,
                       double *moments, uint64_t *s2_rows, uint64_t *s2_sums,
                       uint64_t *psnr_rows, double *mse, uint64_t *noise_sums,
                       uint32_t *status, void *stream)
{
    // Every argument check first: nothing touches the device for a rejected
    // call (the planes, the shape, the outputs, then the scratch limit).
    Layout L;
    const Outputs o{moments, s2_rows, s2_sums, psnr_rows, mse, noise_sums};
    const int bad = check_frames_args(ref, dis, width, height, stride_bytes, bpc, nframes, features,
                                      o, &L);
    if (bad != VMX_OK) return bad;
    if (L.total > VMX_NOALLOC_SCRATCH_BYTES) return VMX_ESCRATCH;
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return cuda_fail(err);
    if (dev < 0 || dev >= kMaxDevices) return VMX_EINVAL;
    void *ws = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (!ws) {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        ws = g_noalloc_ptr[dev].load(std::memory_order_relaxed);
        if (!ws) {
            err = noalloc_scratch_address(&ws);
            if (err != cudaSuccess) return cuda_fail(err);
            if (!ws) return cuda_fail(cudaErrorInvalidSymbol);
            g_noalloc_ptr[dev].store(ws, std::memory_order_release);
        }
    }
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // run_frames clears the control words (tickets, counters, the status
    // word) on `cs` before its launch; the rest of the scratch is written
    // before it is read.
    const int rc = run_frames(ref, dis, width, height, stride_bytes, bpc, nframes, features, o,
                              ws, VMX_NOALLOC_SCRATCH_BYTES, cs);
    if (rc != VMX_OK || !status) return rc;
    const uint32_t *dev_status =
        reinterpret_cast<const uint32_t *>(static_cast<unsigned char *>(ws) + L.off_ctrl) +
        kCtrlStatus;
    err = cudaMemcpyAsync(status, dev_status, sizeof(uint32_t), cudaMemcpyDeviceToDevice, cs);
    return err == cudaSuccess ? VMX_OK : cuda_fail(err);
}

}  // extern "C"

