// vmx_internal.h -- workspace layout and kernel parameters shared by the
// C-ABI (vmx_abi.cpp) and the kernels (vmx_kernels.cu).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime.h>

#include "ordsum.cuh"

namespace vmx {

constexpr int kThreads = 256;              // threads per CTA
constexpr int kWarps = kThreads / 32;      // one row at a time per warp
constexpr int kMaxRowsPerTile = 64;        // rows a CTA takes per ticket, at most
constexpr int kUnroll = 4;                 // 256-pixel segments in flight per warp
constexpr uint32_t kSpinLimit = 1u << 22;  // bounded look-back wait (polls)

// Control words at the start of the workspace (cleared before each call).
enum Ctrl : int {
    kCtrlTicket = 0,     // next tile ticket
    kCtrlStatus = 1,     // 0, or 1 when a bounded wait gave up
    kCtrlRowsExact = 2,  // walk statistics: rows added exactly
    kCtrlRowsRun = 3,    //   rows added by their run
    kCtrlRowsTerms = 4,  //   rows walked term by term
    kCtrlTermChunks = 5, //   2048-term chunks the term walk scanned
    kCtrlWords = 8,
};

// Where everything lives in the workspace. All offsets are 256-byte aligned.
struct Layout {
    int width, height, frames, bpc, features;
    int rows_per_tile, tiles_per_frame;
    bool ordered;        // second moments may pass 2^53 units: look-back + runs
    size_t off_ctrl;     // u32 [kCtrlWords] + done[F] + flag[F * T]
    size_t ctrl_bytes;   // bytes cleared per call
    size_t off_tile_agg; // u64 [F * T][2] exact second-moment sums per tile
    size_t off_tile_inc; // u64 [F * T][2] inclusive exact prefix per tile
    size_t off_tile_s1;  // u64 [F * T][2] first-moment sums per tile
    size_t off_s2_rows;  // u64 [F][2][H] (when the caller passes none)
    size_t off_psnr_rows;// u64 [F][H]    (when the caller passes none)
    size_t off_rec;      // RowRec [F][2][H]
    size_t total;
};

// Returns false for shapes the library rejects.
bool make_layout(int width, int height, int bpc, int frames, int features, Layout *out);

struct Params {
    const unsigned char *ref, *dis;
    int64_t stride;   // bytes between rows
    int64_t pitch;    // bytes between frames
    int width, height, frames;
    int k;            // bpc - 8
    int rows_per_tile, tiles_per_frame;
    uint32_t *ctrl, *done, *flags;
    uint32_t *status;  // set to 1 when a bounded wait gives up
    uint64_t *tile_agg, *tile_inc, *tile_s1;
    uint64_t *s2_rows, *psnr_rows;
    RowRec *rec;
    double *moments, *mse;
    uint64_t *s2_sums, *noise_sums;
    uint32_t spin_limit;
};

// Enqueue the frame kernel. `features` VMX_FEATURE_* bits; `vec` true when
// every row starts on a 16-byte boundary.
cudaError_t launch_frames(const Params &p, const Layout &L, int features, bool vec,
                          cudaStream_t stream);

}  // namespace vmx
