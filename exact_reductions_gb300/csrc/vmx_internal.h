// vmx_internal.h -- workspace layout and kernel parameters shared by the
// C-ABI (vmx_abi.cpp) and the kernels (vmx_kernels.cu).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime.h>

#include "ordsum.cuh"

namespace vmx {

#ifndef VMX_THREADS
#define VMX_THREADS 32
#endif
// Threads per CTA: one warp (the warps share nothing but a CTA's slot), so
// that the register cap alone sets the warps per SM (28 at kMaxRegs; four-
// warp CTAs at 80 registers held 24), and a warp that runs out of items
// frees its slot for the next call's kernel at once.
constexpr int kThreads = VMX_THREADS;
constexpr int kWarps = kThreads / 32;
#ifndef VMX_MAX_REGS
#define VMX_MAX_REGS 72
#endif
#ifndef VMX_MAX_REGS_FULL
#define VMX_MAX_REGS_FULL 80
#endif
#ifndef VMX_UNROLL
#define VMX_UNROLL 3
#endif
// Registers per thread of the frame kernel, at most (registers go out 256 a
// warp): 72 keeps 28 one-warp CTAs on an SM; 80, 25, for the instances with
// the look-back, whose phase B spills more under 72. A cap, rather than
// launch bounds asking for a CTA count, measured faster at the same count.
constexpr int kMaxRegs = VMX_MAX_REGS;
constexpr int kMaxRegsFull = VMX_MAX_REGS_FULL;
constexpr int kMaxRowsPerItem = 32;        // rows per item, at most
#ifndef VMX_MAX_CHUNK
#define VMX_MAX_CHUNK 4
#endif
constexpr int kMaxChunk = VMX_MAX_CHUNK;   // items a warp takes per ticket, at most
#ifndef VMX_ITEM_PIXELS
#define VMX_ITEM_PIXELS 12288
#endif
constexpr int kItemPixels = VMX_ITEM_PIXELS; // target pixels per warp item
#ifndef VMX_ITEM_PIXELS_FULL
#define VMX_ITEM_PIXELS_FULL 32768
#endif
// Target pixels per item where the look-back runs (frames that can pass
// 2^55): its wait and the item's ticket are paid per item, so items are
// larger there.
constexpr int kItemPixelsFull = VMX_ITEM_PIXELS_FULL;
constexpr int kUnroll = VMX_UNROLL;        // 16-byte vectors in flight per lane per plane
#ifndef VMX_FLUSH_SAMPLES
#define VMX_FLUSH_SAMPLES 256
#endif
constexpr int kFlushSamples = VMX_FLUSH_SAMPLES; // 16-bit samples per lane and plane between flushes
#ifndef VMX_STAGES
#define VMX_STAGES 0
#endif
// Row chunks each warp keeps in shared memory, filled by bulk asynchronous
// copies; 0 (the default): 16-byte loads straight into registers, which
// measure faster on the 16-bit rows (with 3 stages and 16 warps per SM the
// 16-bit 3840x2160 batch takes about 9% longer).
constexpr int kStages = VMX_STAGES;
constexpr uint32_t kPipeSpinLimit = 1u << 20;  // polls of one chunk's barrier, at most
#ifndef VMX_LOW_DEPTH
#define VMX_LOW_DEPTH 1  // depths up to 12 bits: exact-square passes where samples allow
#endif
#ifndef VMX_FIRST_UNROLL
#define VMX_FIRST_UNROLL 16
#endif
constexpr int kFirstUnroll = VMX_FIRST_UNROLL;  // loads in flight per lane in the walks' sequential sums
// Timing builds (VMX_PHASE_TIMES=1, a profiling variant of the library):
// the frame kernel sums each phase's clock cycles over its warps and stamps
// a few events with the global timer, into counters vmx_phase_times() reads.
#ifndef VMX_PHASE_TIMES
#define VMX_PHASE_TIMES 0
#endif
enum PhaseCounter : int {
    kPtStart = 0,       // first warp's start (global timer, ns)
    kPtEnd = 1,         // last warp's end (ns)
    kPtStream = 2,      // phase A: items streamed (cycles, summed over warps)
    kPtLookback = 3,    // phase B: look-back, waits included (cycles)
    kPtRuns = 4,        // phase B: plans and row runs (cycles)
    kPtComplete = 5,    // phase C: completion (cycles)
    kPtOutLast = 6,     // last warp out of items (ns)
    kPtOutFirst = 7,    // first warp out of items (ns)
    kPtWalks = 8,       // phase D: walks, waits included (cycles)
    kPtWalksEnd = 9,    // last walk's end (ns)
    kPtWalkTasks = 10,  // walks taken
    kPtItems = 11,      // items streamed
    kPtWalkMax = 12,    // longest walk (cycles)
    kPtWalksStart = 13, // first walk's start (ns)
    kPtRunRows = 14,    // row runs formed in phase B
    kPtClockKHz = 15,   // the device's SM clock rate (kHz; filled by the reader)
    kPtCount = 16
};

#ifndef VMX_CHECK
// 1: a checked build (a test variant). Every index the kernels compute into
// one of their arrays is compared with the array's extent first; one out of
// range sets bit 1 of the call's status word (VMX_ECHECK on the host) and the
// access is skipped. Nothing traps. 0: the checks compile to nothing.
#define VMX_CHECK 0
#endif
#ifndef VMX_WHOLE_LOADS
#define VMX_WHOLE_LOADS 1  // passes wholly inside a row load without per-vector checks
#endif
constexpr uint32_t kSpinLimit = 1u << 22;  // bounded look-back wait (polls)

// Control words at the start of the workspace (cleared before each call).
enum Ctrl : int {
    kCtrlTicket = 0,     // next item ticket
    kCtrlStatus = 1,     // 0, or 1 when a bounded wait gave up
    kCtrlRowsExact = 2,  // walk statistics: rows added exactly
    kCtrlRowsRun = 3,    //   rows added by a closed form or a run
    kCtrlRowsTerms = 4,  //   rows walked term by term
    kCtrlPasses = 5,     //   search passes and chunks the walks scanned
    kCtrlWalkTicket = 6, // next frame to walk
    kCtrlWords = 8,
};

// Per-item and per-block sums the walk reads (64 bytes): the exact
// second-moment sums (ref, dis), the first-moment sums, the psnr sum and the
// odd-term counts (ref in the low half of odd, dis in the high half). A
// block's record is written by the block's last item to finish, from its
// items' records. Whether a record is out is kept apart, in words cleared by
// every call (a block's count of finished items; an item's flag where the
// look-back runs).
struct alignas(16) Agg {
    uint64_t s2[2];
    uint64_t s1[2];
    uint64_t psnr;
    uint64_t odd;
    uint64_t pad[2];
};
constexpr int kBlockItems = 32;  // items folded into one block aggregate

// Where everything lives in the workspace. All offsets are 256-byte aligned.
struct Layout {
    int width, height, frames, bpc, features;
    int rows_per_item, items_per_frame, blocks_per_frame;
    bool ordered;        // second moments may pass 2^53 units: odd counts per row
    bool full;           // ... and 2^55: look-back and row runs from binade 55 up
    size_t off_ctrl;     // u32 [kCtrlWords] + finished items per block [F * B] + item flags [F * I] (full)
    size_t ctrl_bytes;   // bytes cleared per call: the control words, counts and flags
    size_t off_blocks;   // Agg [F * B], written by each block's last item
    size_t off_items;    // Agg [F * I]
    size_t off_item_inc; // u64 [F * I][2] inclusive exact prefix per item (look-back)
    size_t off_s2_rows;  // u64 [F][2][H] (when the caller passes none)
    size_t off_odd_rows; // u32 [F][2][H] odd terms per row
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
    int rows_per_item, items_per_frame, blocks_per_frame;
    uint32_t *ctrl;
    uint32_t *flags;      // per item, frames that can pass 2^55 only: 0, 1 (its record is
                          // out), 2 (and its inclusive prefix)
    uint32_t *block_fin;  // items of each block that have finished (32-bit counts)
    uint32_t *status;  // set to 1 when a bounded wait gives up
    Agg *items, *blocks;
    uint64_t *item_inc;
    uint64_t *s2_rows, *psnr_rows;
    uint32_t *odd_rows;
    RowRec *rec;
    double *moments, *mse;
    uint64_t *s2_sums, *noise_sums;
    uint32_t spin_limit;
    uint32_t overlap; // launched to overlap the previous kernel on the stream
    uint32_t test_stall;  // tests only: the walks wait for a count never reached
    int test_grid_mult;   // tests only (host side): launch this many times the resident CTAs
    uint32_t check_shrink;  // tests of a checked build: the row-sum arrays' extent is taken as one less
};

// Enqueue the frame kernel. `features` VMX_FEATURE_* bits; `vec` true when
// every row starts on a 16-byte boundary.
cudaError_t launch_frames(const Params &p, const Layout &L, int features, bool vec,
                          cudaStream_t stream);

// A timing build's counters (kPtCount) of the current device into `out`
// (when not null), then, when `reset`, cleared for the next launches.
cudaError_t phase_times(uint64_t *out, bool reset);

// Device address of the current device's static scratch array of
// VMX_NOALLOC_SCRATCH_BYTES bytes (cudaGetSymbolAddress; no allocation).
cudaError_t noalloc_scratch_address(void **ptr);

}  // namespace vmx
