// vmx_kernels.cu -- the frame kernel: float_moment and float_psnr of a batch
// of frame pairs, every sum an exact integer in units of 1/scaler^2, and the
// CPU's rounded double sums reproduced value for value.
//
// One persistent kernel per call; every warp works on its own. A warp takes
// items (a few whole rows of one frame, both planes) from a ticket counter,
// frame by frame, the batch's last frames row by row across frames, with no
// CTA barrier anywhere:
//
//   A. It streams the item's rows once with coalesced 16-byte loads and forms
//      each row's exact sums: first moments (sum of p), second-moment terms
//      (binary32 squares, ADR-1497 "Context"), psnr terms (binary32 squares of
//      the differences, ADR-1499 "Context") and, when the second moments can
//      pass 2^53 units, the number of odd terms per row. No float partials,
//      no atomics on data.
//   B. Only for frames above 2^23 pixels, whose sums can pass 2^55 units: the
//      item's exact sums are published, and once the warp has streamed its
//      next item the exact sum before the item is read by a decoupled
//      look-back over the frame's earlier items (bounded wait). Rows planned
//      in a binade from 55 up get their run (ADR-1497 "Decision", third
//      point): the rows are asked into L2 and read again, each lane running
//      one binary32 trajectory through a contiguous stretch of the row, the
//      lanes' runs composed in order.
//   C. The item counts itself in its block (32 items) by a 32-bit release
//      add (acquire-release with B); the block's last item to finish adds the
//      block's item records into the block's record and marks it done. Warps that
//      find no item left take frames to walk: the crossing of 2^53 is found
//      as soon as the blocks before it are complete, that row is walked term
//      by term, and once the frame is complete each plane's later rows are
//      added in closed form (binades 53 and 54, from the rows' exact sums and
//      odd counts), by their runs (from 55 up), or term by term where a row
//      crosses a binade; psnr adds the exact row sums in row order (ADR-1499
//      "Decision"). It writes the doubles the CPU divides out.
#include <climits>

#include "vmx.h"
#include "vmx_internal.h"

namespace vmx {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kA = 0x4B000000u;                   // bits of 2^23 (g = kA + p)

// ---------------------------------------------------------------- loads ---

__device__ __forceinline__ uint4 ld_nc_v4(const void *ptr)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr));
    return v;
}

__device__ __forceinline__ uint32_t ld_u16(const unsigned char *ptr)
{
    return __ldg(reinterpret_cast<const unsigned short *>(ptr));
}

__device__ __forceinline__ uint32_t ld_u8(const unsigned char *ptr) { return __ldg(ptr); }

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *ptr)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(uint32_t *ptr, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

// Adds v at GPU scope with acquire-release order; returns the old value.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t *ptr, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
    return old;
}

// Adds v at GPU scope with release order; returns the old value.
__device__ __forceinline__ uint32_t atom_add_release(uint32_t *ptr, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
    return old;
}

// Orders the thread's earlier reads (a release RMW it observed) before its
// later memory accesses, at GPU scope.
__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }



// --------------------------------------------------------- checked builds ---
// With VMX_CHECK, chk() compares an index with its array's extent and, when it
// is out of range, sets bit 1 of the call's status word and returns false so
// that the access is skipped (a load gives 0). Without, it is always true.
#if VMX_CHECK
__device__ __forceinline__ bool chk(uint32_t *status, size_t i, size_t n)
{
    if (i < n) return true;
    atomicOr(status, 2u);
    return false;
}
#else
__device__ __forceinline__ bool chk(uint32_t *, size_t, size_t) { return true; }
#endif

// Timing-build counters (PhaseCounter): lane 0 of a warp adds or stamps.
__device__ unsigned long long g_phase[kPtCount];
#if VMX_PHASE_TIMES
__device__ __forceinline__ unsigned long long pt_now()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ long long pt_clock() { return clock64(); }
__device__ __forceinline__ void pt_add(int k, unsigned long long v)
{
    if ((threadIdx.x & 31u) == 0u) atomicAdd(&g_phase[k], v);
}
__device__ __forceinline__ void pt_cycles(int k, long long since) { pt_add(k, (unsigned long long)(clock64() - since)); }
__device__ __forceinline__ void pt_max(int k, unsigned long long v)
{
    if ((threadIdx.x & 31u) == 0u) atomicMax(&g_phase[k], v);
}
__device__ __forceinline__ void pt_min(int k, unsigned long long v)
{
    if ((threadIdx.x & 31u) == 0u) atomicMin(&g_phase[k], v);
}
#else
__device__ __forceinline__ unsigned long long pt_now() { return 0ull; }
__device__ __forceinline__ long long pt_clock() { return 0ll; }
__device__ __forceinline__ void pt_add(int, unsigned long long) {}
__device__ __forceinline__ void pt_cycles(int, long long) {}
__device__ __forceinline__ void pt_max(int, unsigned long long) {}
__device__ __forceinline__ void pt_min(int, unsigned long long) {}
#endif

// Extents (elements) of the kernel's arrays; a test of a checked build takes
// the per-plane row arrays' as one less, so that a check fires.
__device__ __forceinline__ size_t ext_plane_rows(const Params &p)
{
    return (size_t)p.frames * 2 * p.height - p.check_shrink;
}
__device__ __forceinline__ size_t ext_frame_rows(const Params &p) { return (size_t)p.frames * p.height; }
__device__ __forceinline__ size_t ext_items(const Params &p) { return (size_t)p.frames * p.items_per_frame; }
__device__ __forceinline__ size_t ext_blocks(const Params &p) { return (size_t)p.frames * p.blocks_per_frame; }

// Sample type traits: a 16-byte vector holds 8 uint16 or 16 uint8 samples.
template <typename TS>
struct Samples;

template <>
struct Samples<uint16_t> {
    static constexpr int kPerVec = 8;
    static constexpr int kShift = 3;
    __device__ static uint32_t one(const unsigned char *row, int j) { return ld_u16(row + 2 * j); }
    __device__ static uint64_t term(uint32_t s) { return term_of_sample(s); }
};

template <>
struct Samples<uint8_t> {
    static constexpr int kPerVec = 16;
    static constexpr int kShift = 4;
    __device__ static uint32_t one(const unsigned char *row, int j) { return ld_u8(row + j); }
    __device__ static uint64_t term(uint32_t s) { return (uint64_t)(s * s); }
};

// Vector v of a row of `width` samples: 16 bytes, zero past the row's end.
template <typename TS, bool VEC>
__device__ __forceinline__ uint4 load_vec(const unsigned char *row, int v, int width)
{
    using S = Samples<TS>;
    const int j0 = v << S::kShift;
    if (VEC && j0 + S::kPerVec <= width) return ld_nc_v4(row + 16 * (size_t)v);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < S::kPerVec; ++i) {
        if (j0 + i < width) {
            const uint32_t s = S::one(row, j0 + i);
            if (sizeof(TS) == 2) w[i >> 1] |= s << (16 * (i & 1));
            else w[i >> 2] |= s << (8 * (i & 3));
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ int lane_id_early() { return (int)(threadIdx.x & 31); }

// ------------------------------------ bulk copies into shared memory ---
//
// A warp streams the whole 16-byte vectors of its item's rows through
// kStages chunk buffers of its own in shared memory. A chunk is one pass of
// the row loop: kUnroll x 32 vectors of each plane, copied by two bulk
// asynchronous copies that lane 0 starts on the buffer's mbarrier; the warp
// waits for the barrier's phase and reads the chunk with shared loads. A
// buffer is refilled only after every lane has read it (a warp barrier, then
// a proxy fence orders those reads before the copy's writes).

constexpr int kChunkVecs = 32 * kUnroll;          // vectors per plane in a chunk
constexpr uint32_t kNStages = kStages > 0 ? (uint32_t)kStages : 1u;  // buffers (at least one, for the modulo)
constexpr uint32_t kChunkBytes = 16u * kChunkVecs;
constexpr uint32_t kStageBytes = 2u * kChunkBytes;  // both planes
constexpr size_t kPipeSmem = kStages > 0 ? (size_t)kWarps * kStages * (kStageBytes + 8u) : 0;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0u;
}

// Bytes (a multiple of 16) from a 16-byte aligned global address to shared
// memory, completing on `bar`.
__device__ __forceinline__ void bulk_to_smem(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Asks `bytes` (a multiple of 16) from a 16-byte aligned global address into
// L2, without waiting.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// A warp's chunk stream: chunks consumed (k) and started (n) over the warp's
// life, which give each chunk its buffer (index mod kStages) and barrier
// phase (index / kStages mod 2), and the next chunk of the current item to
// start (row, chunk in the row).
struct Pipe {
    uint32_t buf, bar;  // shared addresses of the warp's buffers and barriers
    uint32_t k, n;
    int prow, pc;
    bool broken;  // a wait gave up: later waits are skipped
};

// The rows [prow, r1) of one frame: chunks per row and plane bases.
struct PipeSrc {
    const unsigned char *fr, *fd;
    int64_t stride;
    int r1, cpr;
};

// Starts chunks until kStages are in flight or unread, or the item has no
// more. Called by the whole warp (lane 0 issues) after a warp barrier.
__device__ __forceinline__ void pipe_fill(Pipe &pp, const PipeSrc &src)
{
    while (src.cpr > 0 && pp.prow < src.r1 && pp.n < pp.k + (uint32_t)kStages) {
        if (lane_id_early() == 0) {
            const uint32_t st = pp.n % kNStages;
            const uint32_t dst = pp.buf + st * kStageBytes, bar = pp.bar + 8u * st;
            const int64_t off = (int64_t)pp.prow * src.stride + (int64_t)pp.pc * kChunkBytes;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_expect_tx(bar, kStageBytes);
            bulk_to_smem(dst, src.fr + off, kChunkBytes, bar);
            bulk_to_smem(dst + kChunkBytes, src.fd + off, kChunkBytes, bar);
        }
        ++pp.n;
        if (++pp.pc == src.cpr) {
            pp.pc = 0;
            ++pp.prow;
        }
    }
}

// Waits (bounded) until chunk i is in shared memory.
__device__ __forceinline__ void pipe_wait(Pipe &pp, uint32_t i, uint32_t *status)
{
    if (pp.broken) return;
    const uint32_t bar = pp.bar + 8u * (i % kNStages), par = (i / kNStages) & 1u;
    uint32_t spins = 0;
    while (!mbar_try_wait(bar, par)) {
        if (++spins > kPipeSpinLimit) {
            if (lane_id_early() == 0) atomicOr(status, 1u);
            pp.broken = true;
            break;
        }
    }
    pp.broken = __any_sync(0xffffffffu, pp.broken);
}

// ------------------------------------------------------- warp primitives ---

__device__ __forceinline__ int lane_id() { return (int)(threadIdx.x & 31); }

// Warp total modulo 2^32 (one warp-wide reduction instruction).
__device__ __forceinline__ uint32_t warp_sum32(uint32_t v) { return __reduce_add_sync(kFull, v); }

// Warp total of values below 2^51 each (row and item sums): the low 24 bits
// and the rest reduced apart as 32-bit sums, neither of which can wrap
// (32 times 2^24, 32 times 2^27).
__device__ __forceinline__ uint64_t warp_sum_lt51(uint64_t v)
{
    const uint32_t lo = warp_sum32((uint32_t)v & 0xFFFFFFu);
    const uint32_t hi = warp_sum32((uint32_t)(v >> 24));
    return ((uint64_t)hi << 24) + lo;
}

__device__ __forceinline__ uint64_t warp_sum(uint64_t v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    return v;
}

// A pair of running sums: the exact sum of terms and how many were odd.
struct SC {
    uint64_t s, c;
};

__device__ __forceinline__ SC sc_add(SC a, SC b) { return SC{a.s + b.s, a.c + b.c}; }

__device__ __forceinline__ SC shfl_sc(SC x, int src)
{
    return SC{__shfl_sync(kFull, x.s, src), __shfl_sync(kFull, x.c, src)};
}

// Exclusive prefix of the lanes' pairs, in lane order; *total the warp total.
__device__ __forceinline__ SC warp_excl_sc(SC x, SC *total)
{
    const int lane = lane_id();
    SC v = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const SC o{__shfl_up_sync(kFull, v.s, off), __shfl_up_sync(kFull, v.c, off)};
        if (lane >= off) v = sc_add(v, o);
    }
    *total = shfl_sc(v, 31);
    return SC{v.s - x.s, v.c - x.c};
}

__device__ __forceinline__ Run shfl_run(const Run &r, int src)
{
    return Run{{__shfl_sync(kFull, r.inc[0], src), __shfl_sync(kFull, r.inc[1], src)}};
}

// Exclusive composition of the lanes' runs in lane order (earlier first).
__device__ __forceinline__ Run warp_excl_run(const Run &x, int sh, Run *total)
{
    const int lane = lane_id();
    Run v = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const Run o{{__shfl_up_sync(kFull, v.inc[0], off), __shfl_up_sync(kFull, v.inc[1], off)}};
        if (lane >= off) v = compose(o, v, sh);
    }
    *total = shfl_run(v, 31);
    Run ex{{__shfl_up_sync(kFull, v.inc[0], 1), __shfl_up_sync(kFull, v.inc[1], 1)}};
    if (lane == 0) ex = run_identity();
    return ex;
}

// --------------------------------------------------- phase A: row sums ---

// A row's sums as the warp keeps them in shared memory for its item.
struct alignas(8) RowSlot {
    uint64_t x, y, z, w;  // ref and dis second-moment sums, psnr sum, odd counts (ref | dis << 32)
    uint64_t s1;          // the row's first-moment sums (ref | dis << 32)
};

// A lane's row sums that only the flushes touch, in shared memory (one slot
// per lane of each warp) so that they hold no registers across the passes.
struct LaneRowAcc {
    uint64_t t2r[32], t2d[32], tp[32];
};

struct RowSums {
    uint64_t t2r, t2d, tp, s1r, s1d;
    uint32_t oddr, oddd;
};

// Per-lane accumulators of a 16-bit row. A 32-bit word holds two samples.
//
// Sums of squares: with p = 256 h + l (bytes h, l), p^2 = 256 p h + p l, and
// the two-way 16x8-bit dot products (dp2a) of a word with its own bytes
// rearranged as [l0, l1, h0, h1] give p0 l0 + p1 l1 and p0 h0 + p1 h1 in
// 32-bit accumulators; with the other plane's bytes they give the cross sums
// p q of float_psnr's sum d^2 = sum p^2 + sum q^2 - 2 sum p q.
// The binary32 square is p^2 minus its rounding error e = fma(f, f, -fl(f f)),
// with f = p exact in binary32 (g = 2^23 + p as bits, less 2^23); the errors
// are integers of at most 2^7 and add exactly in binary32.
// Odd terms: a binary32 square of a codeword is odd exactly when the codeword
// is odd and below 4096, i.e. its bits 0 and 12-15 read 1 and 0; the even
// terms are counted (a halfword minimum marks them, 0 or 1 in each
// halfword, and the marks are added as packed halfword counts) and the row's
// end takes them from its number of samples.
// First moments: two packed adds a word (the word itself and its high
// sample). The dot products run on the FMA-heavy pipe, as do the packed
// binary32 operations; the adds run on the integer ALU, which has room.
// Each flush folds its rounding errors into the row's term sums (kept in
// shared memory) at once.
struct Acc16 {
    uint32_t lr, hr, ld, hd, lx, hx;  // dot-product sums since the last flush
    uint32_t nzr, nzd;                // the row's even terms so far (two halfword counts each)
    float2 er, ed, ep;                // rounding errors since the last flush
    uint32_t s1r, s1d;                // row sums of the words (first moments, packed)
    uint32_t s1rh, s1dh;              // row sums of the words' high samples
    uint64_t tp;                      // psnr alone: the row's sum of the terms
};

__device__ __forceinline__ float2 neg2(float2 v) { return make_float2(-v.x, -v.y); }

// Each unsigned halfword of x, or 1 if that is smaller.
__device__ __forceinline__ uint32_t halfword_min1(uint32_t x) { return __vminu2(x, 0x00010001u); }

// First moments of a word of two 16-bit samples into the lane's row sums by
// two adds: the word itself (p0 + 2^16 p1, modulo 2^32) and its high sample.
__device__ __forceinline__ void acc16_s1(uint32_t &s, uint32_t &sh, uint32_t w)
{
    s += w;
    sh += w >> 16;
}

// The lane's first-moment sum of a row from its two sums (the low samples'
// sum, s - 2^16 sh modulo 2^32, is below 2^32).
__device__ __forceinline__ uint32_t s1_total(uint32_t s, uint32_t sh) { return (s - (sh << 16)) + sh; }

// The lane's count of even terms of a row from its halfword counts (marks of
// 0 or 1 added as two halfwords, each at most 512 a row).
__device__ __forceinline__ uint32_t even_total(uint32_t n) { return (n & 0xffffu) + (n >> 16); }

template <bool M, bool P, bool ODD>
__device__ __forceinline__ void acc16_word(Acc16 &a, uint32_t r, uint32_t d)
{
    const uint32_t gr0 = __byte_perm(r, kA, 0x7610), gr1 = __byte_perm(r, kA, 0x7632);
    const uint32_t gd0 = __byte_perm(d, kA, 0x7610), gd1 = __byte_perm(d, kA, 0x7632);
    const float2 m23 = make_float2(-8388608.0f, -8388608.0f);
    const float2 fr = __fadd2_rn(make_float2(__uint_as_float(gr0), __uint_as_float(gr1)), m23);
    const float2 fd = __fadd2_rn(make_float2(__uint_as_float(gd0), __uint_as_float(gd1)), m23);
    if (M) {
        const uint32_t xr = __byte_perm(r, 0, 0x3120), xd = __byte_perm(d, 0, 0x3120);
        a.lr = __dp2a_lo(r, xr, a.lr);
        a.hr = __dp2a_hi(r, xr, a.hr);
        a.ld = __dp2a_lo(d, xd, a.ld);
        a.hd = __dp2a_hi(d, xd, a.hd);
        if (P) {
            a.lx = __dp2a_lo(r, xd, a.lx);
            a.hx = __dp2a_hi(r, xd, a.hx);
        }
        acc16_s1(a.s1r, a.s1rh, r);
        acc16_s1(a.s1d, a.s1dh, d);
        a.er = __fadd2_rn(a.er, __ffma2_rn(fr, fr, neg2(__fmul2_rn(fr, fr))));
        a.ed = __fadd2_rn(a.ed, __ffma2_rn(fd, fd, neg2(__fmul2_rn(fd, fd))));
        if (ODD) {
            // Per 16-bit sample: zero exactly when it is odd and below 4096;
            // the unsigned halfword minimum with 1 marks the others.
            const uint32_t tr = (r & 0xF001F001u) ^ 0x00010001u, td = (d & 0xF001F001u) ^ 0x00010001u;
            a.nzr += halfword_min1(tr);
            a.nzd += halfword_min1(td);
        }
    }
    if (P) {
        const float2 x = __fadd2_rn(fr, neg2(fd));  // exact
        a.ep = __fadd2_rn(a.ep, __ffma2_rn(x, x, neg2(__fmul2_rn(x, x))));
        if (!M) {  // psnr alone: d^2 from the signed difference, straight into the row sum
            const int32_t i0 = (int32_t)(gr0 - gd0), i1 = (int32_t)(gr1 - gd1);
            a.tp += (uint64_t)((int64_t)i0 * i0);
            a.tp += (uint64_t)((int64_t)i1 * i1);
        }
    }
}

// The same sums for a word pair whose four samples are all below 4096 (the
// pass checked it): their binary32 squares, and those of their differences,
// are exact, so there are no rounding errors to take off, and a term is odd
// exactly when its sample is.
template <bool M, bool P, bool ODD>
__device__ __forceinline__ void acc16_word_low(Acc16 &a, uint32_t r, uint32_t d)
{
    if (M) {
        const uint32_t xr = __byte_perm(r, 0, 0x3120), xd = __byte_perm(d, 0, 0x3120);
        a.lr = __dp2a_lo(r, xr, a.lr);
        a.hr = __dp2a_hi(r, xr, a.hr);
        a.ld = __dp2a_lo(d, xd, a.ld);
        a.hd = __dp2a_hi(d, xd, a.hd);
        if (P) {
            a.lx = __dp2a_lo(r, xd, a.lx);
            a.hx = __dp2a_hi(r, xd, a.hx);
        }
        acc16_s1(a.s1r, a.s1rh, r);
        acc16_s1(a.s1d, a.s1dh, d);
        if (ODD) {
            a.nzr += ~r & 0x00010001u;
            a.nzd += ~d & 0x00010001u;
        }
    } else if (P) {
        const int32_t i0 = (int32_t)(r & 0xffffu) - (int32_t)(d & 0xffffu);
        const int32_t i1 = (int32_t)(r >> 16) - (int32_t)(d >> 16);
        a.tp += (uint64_t)(i0 * i0) + (uint64_t)(i1 * i1);
    }
}

// Folds the sums since the last flush into the row sums. At most
// kFlushSamples (256) samples per lane and plane since the last flush keep
// every dot-product sum below 2^32 (256 times 65535 times 255), every error
// sum below 2^15 (exact in binary32) and every even-term count at most 256.
template <bool M, bool P, bool ODD>
__device__ __forceinline__ void acc16_flush(Acc16 &a, LaneRowAcc &sa, int lane)
{
    const int64_t ep = P ? small_f_to_i(__fadd_rn(a.ep.x, a.ep.y)) : 0;
    if (M) {
        const uint64_t pr = ((uint64_t)a.hr << 8) + a.lr;  // sums of p^2, q^2
        const uint64_t pd = ((uint64_t)a.hd << 8) + a.ld;
        sa.t2r[lane] += pr - (uint64_t)(int64_t)small_f_to_i(__fadd_rn(a.er.x, a.er.y));
        sa.t2d[lane] += pd - (uint64_t)(int64_t)small_f_to_i(__fadd_rn(a.ed.x, a.ed.y));
        if (P) {
            const uint64_t px = ((uint64_t)a.hx << 8) + a.lx;  // sum of p q
            sa.tp[lane] += pr + pd - 2ull * px - (uint64_t)ep;
            a.lx = a.hx = 0;
        }
        a.lr = a.hr = a.ld = a.hd = 0;
        a.er = a.ed = make_float2(0.0f, 0.0f);
    } else if (P) {
        a.tp -= (uint64_t)ep;
    }
    if (P) a.ep = make_float2(0.0f, 0.0f);
}

// With STG the row's whole chunks come through the warp's chunk stream (the
// row is the stream's next `cpr` chunks), the rest of the row straight from
// global memory.
// With LOW (depths up to 12 bits) a pass whose samples are all below 4096
// takes the exact-square body; any other pass (a container value past the
// depth) the full one.
template <bool M, bool P, bool ODD, bool VEC, bool STG, bool LOW>
__device__ RowSums row_sums16(const unsigned char *rr, const unsigned char *dr, int width, Pipe &pp,
                              const PipeSrc &src, uint32_t *status)
{
    static_assert(kUnroll * 8 <= kFlushSamples, "an iteration holds at most kFlushSamples per lane");
    static_assert(kFlushSamples <= 256, "dot-product sums must stay below 2^32");
    const int lane = lane_id();
    Acc16 a = {};
    __shared__ LaneRowAcc lane_acc[kWarps];
    LaneRowAcc &sa = lane_acc[threadIdx.x >> 5];
    if (M) sa.t2r[lane] = sa.t2d[lane] = sa.tp[lane] = 0;
    const int nvt = (width + 7) >> 3;
    // Vectors wholly inside the row (all of them but a ragged last one).
    const int nfull = width >> 3;
    uint32_t pend = 0;  // samples per lane per plane since the last flush
    int base = 0;
    if (STG) {
        const uint32_t lane_off = 16u * (uint32_t)lane;
        for (int c = 0; c < src.cpr; ++c, base += kChunkVecs) {
            if (pend + 8 * kUnroll > kFlushSamples) {
                acc16_flush<M, P, ODD>(a, sa, lane);
                pend = 0;
            }
            __syncwarp();  // every lane is done with the previous chunk's buffer
            pipe_fill(pp, src);
            pipe_wait(pp, pp.k, status);
            const uint32_t at = pp.buf + (pp.k % kNStages) * kStageBytes + lane_off;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const uint4 R = lds128(at + 512u * u);
                const uint4 D = lds128(at + kChunkBytes + 512u * u);
                acc16_word<M, P, ODD>(a, R.x, D.x);
                acc16_word<M, P, ODD>(a, R.y, D.y);
                acc16_word<M, P, ODD>(a, R.z, D.z);
                acc16_word<M, P, ODD>(a, R.w, D.w);
            }
            ++pp.k;
            pend += 8 * kUnroll;
        }
    }
    for (; base < nvt; base += 32 * kUnroll) {
        // Vectors per lane this time (the same for the whole warp): kUnroll
        // but at the row's end, where vectors past it are skipped.
        const int nu = min(kUnroll, (nvt - base + 31) >> 5);
        if (pend + 8 * nu > kFlushSamples) {
            acc16_flush<M, P, ODD>(a, sa, lane);
            pend = 0;
        }
        uint4 R[kUnroll], D[kUnroll];
#if VMX_WHOLE_LOADS
        // Every vector of this iteration inside the row (the warp agrees):
        // plain 16-byte loads without per-vector checks.
        if (VEC && base + 32 * kUnroll <= nfull) {
            const uint4 *vr = reinterpret_cast<const uint4 *>(rr) + base + lane;
            const uint4 *vd = reinterpret_cast<const uint4 *>(dr) + base + lane;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (VMX_CHECK && !chk(status, base + 32 * u + lane, nfull)) {
                    R[u] = D[u] = make_uint4(0u, 0u, 0u, 0u);
                    continue;
                }
                R[u] = ld_nc_v4(vr + 32 * u);
                D[u] = ld_nc_v4(vd + 32 * u);
            }
        } else
#endif
        {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (u < nu) {
                    const int v = base + u * 32 + lane;
                    R[u] = load_vec<uint16_t, VEC>(rr, v, width);
                    D[u] = load_vec<uint16_t, VEC>(dr, v, width);
                }
            }
        }
        bool low = false;
        if (LOW) {
            uint32_t o = 0;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (u < nu) o |= R[u].x | R[u].y | R[u].z | R[u].w | D[u].x | D[u].y | D[u].z | D[u].w;
            low = !__any_sync(kFull, (o & 0xF000F000u) != 0u);
        }
        if (LOW && low) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (u < nu) {
                    acc16_word_low<M, P, ODD>(a, R[u].x, D[u].x);
                    acc16_word_low<M, P, ODD>(a, R[u].y, D[u].y);
                    acc16_word_low<M, P, ODD>(a, R[u].z, D[u].z);
                    acc16_word_low<M, P, ODD>(a, R[u].w, D[u].w);
                }
            }
        } else {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (u < nu) {
                    acc16_word<M, P, ODD>(a, R[u].x, D[u].x);
                    acc16_word<M, P, ODD>(a, R[u].y, D[u].y);
                    acc16_word<M, P, ODD>(a, R[u].z, D[u].z);
                    acc16_word<M, P, ODD>(a, R[u].w, D[u].w);
                }
            }
        }
        pend += 8 * nu;
    }
    acc16_flush<M, P, ODD>(a, sa, lane);
    RowSums out = {0, 0, 0, 0, 0, 0, 0};
    if (M) {
        out.t2r = sa.t2r[lane];
        out.t2d = sa.t2d[lane];
        // Row totals of the first moments (a lane's share is below 2^26,
        // the row's below 2^31).
        out.s1r = warp_sum32(s1_total(a.s1r, a.s1rh));
        out.s1d = warp_sum32(s1_total(a.s1d, a.s1dh));
    }
    const uint32_t even = ODD ? even_total(a.nzr) | (even_total(a.nzd) << 16) : 0u;
    if (P) out.tp = M ? sa.tp[lane] : a.tp;
    // Row totals (a lane's sums of a row stay below 2^42: at most 1024 terms
    // below 2^32).
    out.t2r = warp_sum_lt51(out.t2r);
    out.t2d = warp_sum_lt51(out.t2d);
    out.tp = warp_sum_lt51(out.tp);
    if (ODD) {  // both counts fit 16 bits (a row has at most 2^15 samples)
        const uint32_t nl = 8u * (uint32_t)((nvt + 31) >> 5);  // samples per lane and plane
        const uint32_t packed = warp_sum32((nl | (nl << 16)) - even);
        out.oddr = packed & 0xffffu;
        out.oddd = packed >> 16;
    }
    return out;
}

// 8-bit rows: every square is below 2^16, exact; byte dot products.
template <bool M, bool P, bool VEC>
__device__ RowSums row_sums8(const unsigned char *rr, const unsigned char *dr, int width)
{
    const int lane = lane_id();
    uint32_t s1r = 0, s1d = 0, s2r = 0, s2d = 0, srd = 0;
    const int nvt = (width + 15) >> 4;
    for (int base = 0; base < nvt; base += 32 * kUnroll) {
        uint4 R[kUnroll], D[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = base + u * 32 + lane;
            R[u] = load_vec<uint8_t, VEC>(rr, v, width);
            D[u] = load_vec<uint8_t, VEC>(dr, v, width);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint32_t r4[4] = {R[u].x, R[u].y, R[u].z, R[u].w};
            const uint32_t d4[4] = {D[u].x, D[u].y, D[u].z, D[u].w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                s2r = __dp4a(r4[w], r4[w], s2r);
                s2d = __dp4a(d4[w], d4[w], s2d);
                if (M) {
                    s1r = __dp4a(r4[w], 0x01010101u, s1r);
                    s1d = __dp4a(d4[w], 0x01010101u, s1d);
                }
                if (P) srd = __dp4a(r4[w], d4[w], srd);
            }
        }
    }
    RowSums out;
    // A row's sums of 8-bit products stay below 2^31 (2^15 samples below 2^16).
    out.t2r = warp_sum32(s2r);
    out.t2d = warp_sum32(s2d);
    out.tp = P ? out.t2r + out.t2d - 2ull * warp_sum32(srd) : 0ull;
    out.s1r = M ? warp_sum32(s1r) : 0;  // row totals (below 2^23)
    out.s1d = M ? warp_sum32(s1d) : 0;
    out.oddr = out.oddd = 0;
    return out;
}

// ------------------------------------------------ phase B: row runs ---

// 16-byte vector v of a 16-bit row through L1 (zero past the row's end):
// the run pass reads each lane's vectors three apart, so neighbouring loads
// share cache lines.
template <bool VEC>
__device__ __forceinline__ uint4 load_vec16_l1(const unsigned char *row, int v, int width)
{
    const int j0 = v << 3;
    if (VEC && j0 + 8 <= width) return __ldg(reinterpret_cast<const uint4 *>(row) + v);
    return load_vec<uint16_t, VEC>(row, v, width);
}

// The binary32 squares of a word's two 16-bit samples as the exact
// integers they are (term_from_float in ordsum.cuh, two samples at a time):
// p^2 less the product's rounding error, which a fused multiply-add gives.
__device__ __forceinline__ void terms_of_word(uint32_t w, uint32_t *t0, uint32_t *t1)
{
    const uint32_t p0 = w & 0xffffu, p1 = w >> 16;
    const float2 m23 = make_float2(-8388608.0f, -8388608.0f);
    const float2 f = __fadd2_rn(make_float2(__uint_as_float(p0 | kA), __uint_as_float(p1 | kA)), m23);
    const float2 e = __ffma2_rn(f, f, neg2(__fmul2_rn(f, f)));  // integers in [-128, 128]
    const float2 ei = __fadd2_rn(e, make_float2(12582912.0f, 12582912.0f));
    *t0 = p0 * p0 - (__float_as_uint(ei.x) - 0x4B400000u);
    *t1 = p1 * p1 - (__float_as_uint(ei.y) - 0x4B400000u);
}

// A lane's binary32 trajectories under last place u = 2^sh (the method of
// lane_run_fp in ordsum.cuh), both start parities advanced by one packed add
// per term: after n terms, the compact run of those n terms. Exact while
// n * 2u < 2^22 (the trajectory offsets stay exact small integers). Only a
// term's residue v = t mod 2u matters for its rounding, and the run's parity
// needs the terms' sum only modulo 2u, which the residues' sum gives: each
// residue is kept as the bits of the binary32 2^23 + v (one three-input
// logic op), whose integer sum carries v's sum in its low 24 bits.
struct Traj {
    float2 F;
    uint32_t gsum;  // sum of the residues' binary32 bits: low 24 bits the residues' sum
};

// The trajectories' start: 1.5 * 2^23 * u (even) and one place higher (odd).
__device__ __forceinline__ float2 traj_start(int sh)
{
    const float uf = __uint_as_float((uint32_t)(127 + sh) << 23);  // 2^sh
    const float f0e = __fmul_rn(12582912.0f, uf);
    return make_float2(f0e, __fadd_rn(f0e, uf));
}

template <int N>
__device__ __forceinline__ void traj_extend(Traj &T, const uint32_t (&t)[N], uint32_t vmask)
{
    static_assert(N % 2 == 0, "terms come in pairs");
    const float2 m23 = make_float2(-8388608.0f, -8388608.0f);
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        const uint32_t g0 = (t[i] & vmask) | kA, g1 = (t[i + 1] & vmask) | kA;
        T.gsum += g0 + g1;
        const float2 vf = __fadd2_rn(make_float2(__uint_as_float(g0), __uint_as_float(g1)), m23);
        T.F = __fadd2_rn(T.F, make_float2(vf.x, vf.x));
        T.F = __fadd2_rn(T.F, make_float2(vf.y, vf.y));
    }
}

// The compact run: tlo the terms' sum modulo 2u (all that composing and the
// parities read of it), d each parity's increment less the terms' sum.
__device__ __forceinline__ LaneRun traj_run(const Traj &T, float2 f0)
{
    const float2 dF = __fadd2_rn(T.F, make_float2(-f0.x, -f0.y));
    const int32_t vsum = (int32_t)(T.gsum & 0xFFFFFFu);  // below 2^22
    LaneRun r;
    r.tlo = (uint32_t)vsum;
    r.d[0] = (int32_t)(__float_as_uint(__fadd_rn(dF.x, 12582912.0f)) - 0x4B400000u) - vsum;
    r.d[1] = (int32_t)(__float_as_uint(__fadd_rn(dF.y, 12582912.0f)) - 0x4B400000u) - vsum;
    return r;
}

// The compact run of the N terms t (N = 24 is exact up to sh = 16).
template <int N>
__device__ __forceinline__ LaneRun lane_run_fp2(const uint32_t (&t)[N], int sh)
{
    const float2 f0 = traj_start(sh);
    Traj T{f0, 0u};
    traj_extend(T, t, (2u << sh) - 1u);
    return traj_run(T, f0);
}

// Lanes' runs composed in lane order by a shuffle tree (lane i takes lane
// i + off): every lane gets the run of all 32.
__device__ __forceinline__ LaneRun warp_run_of_lanes(LaneRun l, int sh)
{
    const int lane = lane_id();
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        LaneRun o;
        o.tlo = __shfl_down_sync(kFull, l.tlo, off);
        o.d[0] = __shfl_down_sync(kFull, l.d[0], off);
        o.d[1] = __shfl_down_sync(kFull, l.d[1], off);
        if ((lane & (2 * off - 1)) == 0) l = lane_compose(l, o, sh);
    }
    LaneRun w;
    w.tlo = __shfl_sync(kFull, l.tlo, 0);
    w.d[0] = __shfl_sync(kFull, l.d[0], 0);
    w.d[1] = __shfl_sync(kFull, l.d[1], 0);
    return w;
}

// The run of a 16-bit row under binade e (so sh = e - 52 <= 10). In rounds
// of at most 32 x 128 vectors, each lane takes a contiguous stretch of the
// round (at most 1024 terms: 1024 * 2^11 < 2^22 keeps its trajectory exact
// for every binade up to 62) and runs one trajectory through it; the lanes'
// runs are composed in lane order, the rounds in row order. A lane reads its
// stretch three vectors at a time, the next three already on their way.
// Samples past the lane's stretch are zero terms, which leave a run as it is.
template <bool VEC>
__device__ __forceinline__ Run row_run16(const unsigned char *row, int width, int e, uint64_t exact)
{
    constexpr int kRunVecs = 3;     // vectors per lane and step
    constexpr int kLaneVecs = 128;  // vectors per lane and round, at most
    const int lane = lane_id();
    const int sh = e - 52;
    const uint32_t vmask = (2u << sh) - 1u;
    const float2 f0 = traj_start(sh);
    const int nvt = (width + 7) >> 3;
    LaneRun acc = lane_identity();
    for (int base = 0; base < nvt; base += 32 * kLaneVecs) {
        const int left = min(nvt - base, 32 * kLaneVecs);
        const int per = (left + 31) >> 5;  // the round's vectors per lane
        const int v0 = base + lane * per, v1 = min(base + left, v0 + per);
        const auto load = [row, width, v1](int v) {
            return v < v1 ? load_vec16_l1<VEC>(row, v, width) : make_uint4(0u, 0u, 0u, 0u);
        };
        Traj T{f0, 0u};
        uint4 nx[kRunVecs];
#pragma unroll
        for (int u = 0; u < kRunVecs; ++u) nx[u] = load(v0 + u);
        for (int k = 0; k < per; k += kRunVecs) {
            uint4 cv[kRunVecs];
#pragma unroll
            for (int u = 0; u < kRunVecs; ++u) cv[u] = nx[u];
            if (k + kRunVecs < per) {
#pragma unroll
                for (int u = 0; u < kRunVecs; ++u) nx[u] = load(v0 + k + kRunVecs + u);
            }
            uint32_t t[8 * kRunVecs];
#pragma unroll
            for (int u = 0; u < kRunVecs; ++u) {
                const uint32_t w4[4] = {cv[u].x, cv[u].y, cv[u].z, cv[u].w};
#pragma unroll
                for (int w = 0; w < 4; ++w) terms_of_word(w4[w], &t[8 * u + 2 * w], &t[8 * u + 2 * w + 1]);
            }
            traj_extend(T, t, vmask);
        }
        acc = lane_compose(acc, warp_run_of_lanes(traj_run(T, f0), sh), sh);
    }
    return lane_to_run(acc, exact);
}

// ------------------------------------------------------ phase C: walk ---

__device__ __forceinline__ void count(uint32_t *ctrl, int which, uint32_t n)
{
    if (lane_id() == 0 && n) atomicAdd(ctrl + which, n);
}

// Two-level search. Among the elements [lo, hi) (pairs from fetch(i)), finds
// the first index m whose inclusive prefix (summed from lo) makes bad() true;
// bad must be monotone along the prefix. *before gets the prefix before m
// (the whole sum when no element is bad; then hi is returned). Each pass
// gives every lane a contiguous range, scans the lanes' sums and narrows to
// the range where bad() turns true, until a range of at most 4 per lane.
template <class Fetch, class Bad>
__device__ int warp_first(Fetch fetch, int lo, int hi, Bad bad, SC *before, uint32_t *ctrl)
{
    const int lane = lane_id();
    SC base{0, 0};
    for (;;) {
        count(ctrl, kCtrlPasses, 1);
        const int len = hi - lo;
        if (len <= 0) {
            *before = base;
            return hi;
        }
        const int c = (len + 31) / 32;
        const int a = lo + lane * c;
        const int b = min(hi, a + c);
        if (c <= 4) {
            SC v[4];
            SC loc{0, 0};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[i] = (a + i < b) ? fetch(a + i) : SC{0, 0};
                loc = sc_add(loc, v[i]);
            }
            SC tot;
            SC cur = sc_add(base, warp_excl_sc(loc, &tot));
            int cand = INT_MAX;
            SC cb{0, 0};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (cand != INT_MAX || a + i >= b) continue;
                const SC nx = sc_add(cur, v[i]);
                if (bad(nx)) {
                    cand = a + i;
                    cb = cur;
                }
                cur = nx;
            }
            const unsigned m = __ballot_sync(kFull, cand != INT_MAX);
            if (!m) {
                *before = sc_add(base, tot);
                return hi;
            }
            const int src = __ffs(m) - 1;
            *before = shfl_sc(cb, src);
            return __shfl_sync(kFull, cand, src);
        }
        SC loc{0, 0};
#pragma unroll kFirstUnroll
        for (int i = a; i < b; ++i) loc = sc_add(loc, fetch(i));
        SC tot;
        const SC ex = warp_excl_sc(loc, &tot);
        const bool hit = a < b && bad(sc_add(base, sc_add(ex, loc)));
        const unsigned m = __ballot_sync(kFull, hit);
        if (!m) {
            *before = sc_add(base, tot);
            return hi;
        }
        const int src = __ffs(m) - 1;
        base = sc_add(base, shfl_sc(ex, src));
        const int nlo = lo + src * c;
        hi = min(hi, nlo + c);
        lo = nlo;
    }
}

// Runs in order from S (S >= 2^53, binade b fixed): returns the first index m
// in [lo, hi) whose element has no valid run or would take S to 2^(b+1) or
// more, and leaves in S the value before m (after all, when m == hi).
// run_at(i, sh, &ok) gives element i's run under last place 2^sh.
template <class RunAt>
__device__ int warp_run_walk(RunAt run_at, int lo, int hi, uint64_t &S, uint32_t *ctrl)
{
    const int lane = lane_id();
    const int b = binade_of(S), sh = b - 52;
    const uint64_t top = 2ull << b;
    for (int c0 = lo; c0 < hi; c0 += 128) {
        count(ctrl, kCtrlPasses, 1);
        const int q0 = c0 + lane * 4;
        Run r[4];
        bool ok[4];
        Run lr = run_identity();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ok[i] = true;
            r[i] = run_identity();
            if (q0 + i < hi) r[i] = run_at(q0 + i, sh, &ok[i]);
            if (!ok[i]) r[i] = run_identity();
            lr = compose(lr, r[i], sh);
        }
        Run tot;
        uint64_t cur = apply(warp_excl_run(lr, sh, &tot), S, sh);
        int cand = INT_MAX;
        uint64_t cb = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (cand != INT_MAX || q0 + i >= hi) continue;
            const uint64_t nx = apply(r[i], cur, sh);
            if (!ok[i] || nx >= top) {
                cand = q0 + i;
                cb = cur;
            } else {
                cur = nx;
            }
        }
        const unsigned m = __ballot_sync(kFull, cand != INT_MAX);
        if (!m) {
            S = apply(tot, S, sh);
            continue;
        }
        const int src = __ffs(m) - 1;
        S = __shfl_sync(kFull, cb, src);
        return __shfl_sync(kFull, cand, src);
    }
    return hi;
}

// Adds the terms of one row (the binary32 squares of its samples) to S by
// the CPU's rule: exact adds while the sum stays at or below 2^53, the closed
// forms in binades 53 and 54, runs from 55 up, and the full rounding of each
// term that crosses into the next binade.
template <typename TS>
__device__ uint64_t resolve_row(const unsigned char *row, int width, uint64_t S, uint32_t *ctrl,
                               int pos = 0)
{
    auto term = [row](int j) -> uint64_t { return Samples<TS>::term(Samples<TS>::one(row, j)); };
    while (pos < width) {
        int m;
        if (S < kTwo53) {
            SC before;
            m = warp_first([&](int j) { return SC{term(j), 0}; }, pos, width,
                           [S](SC x) { return S + x.s > kTwo53; }, &before, ctrl);
            S += before.s;
        } else if (binade_of(S) <= 54) {
            const int b = binade_of(S);
            const uint64_t top = 2ull << b;
            SC before;
            m = warp_first(
                [&](int j) {
                    const uint64_t t = term(j);
                    return SC{t, t & 1ull};
                },
                pos, width, [S, b, top](SC x) { return closed_form_after(S, x.s, x.c, b) >= top; },
                &before, ctrl);
            S = closed_form_after(S, before.s, before.c, b);
        } else {
            m = warp_run_walk(
                [&](int j, int sh, bool *ok) {
                    *ok = true;
                    return run_of_term(term(j), sh);
                },
                pos, width, S, ctrl);
        }
        if (m < width) S = rnd53(S + term(m));
        pos = m + 1;
    }
    return S;
}

// The CPU's second-moment sum of plane X of frame f from row r on, S the sum
// before row r: rows added exactly, in closed form (binades 53 and 54, from
// the row's exact sum and odd count), by their run (from 55 up), else term
// by term from the samples. The general path; walk_plane_fast() takes the
// common case in a few passes and falls back here.
__device__ uint64_t resolve_row_fast(const unsigned char *row, int width, uint64_t S, uint32_t *ctrl);

template <typename TS, bool VEC, bool FULL>
__device__ uint64_t walk_plane_from(const Params &p, int f, int X, int r, uint64_t S)
{
    const int H = p.height;
    const size_t off = ((size_t)f * 2 + X) * H, nrows = ext_plane_rows(p);
    const uint64_t *R = p.s2_rows + off;
    const uint32_t *O = p.odd_rows + off;
    const RowRec *rec = p.rec + off;
    const unsigned char *plane = (X == 0 ? p.ref : p.dis) + (int64_t)f * p.pitch;
    const auto ldR = [&p, R, off, nrows](int i) { return chk(p.status, off + i, nrows) ? __ldcg(R + i) : 0ull; };
    const auto ldO = [&p, O, off, nrows](int i) {
        return chk(p.status, off + i, nrows) ? (uint64_t)__ldcg(O + i) : 0ull;
    };
    while (r < H) {
        int m;
        if (S < kTwo53) {
            SC before;
            m = warp_first([&ldR](int i) { return SC{ldR(i), 0}; }, r, H,
                           [S](SC x) { return S + x.s > kTwo53; }, &before, p.ctrl);
            S += before.s;
            count(p.ctrl, kCtrlRowsExact, (uint32_t)(m - r));
        } else if (binade_of(S) <= 54) {
            const int b = binade_of(S);
            const uint64_t top = 2ull << b;
            SC before;
            m = warp_first([&ldR, &ldO](int i) { return SC{ldR(i), ldO(i)}; }, r, H,
                           [S, b, top](SC x) { return closed_form_after(S, x.s, x.c, b) >= top; },
                           &before, p.ctrl);
            S = closed_form_after(S, before.s, before.c, b);
            count(p.ctrl, kCtrlRowsRun, (uint32_t)(m - r));
        } else if (FULL) {
            const int b = binade_of(S);
            m = warp_run_walk(
                [&p, &ldR, rec, off, nrows, b](int i, int sh, bool *ok) {
                    const uint64_t rs = ldR(i);
                    if (rs == 0) {
                        *ok = true;
                        return run_identity();
                    }
                    const uint4 w = chk(p.status, off + i, nrows)
                                        ? __ldcg(reinterpret_cast<const uint4 *>(rec + i))
                                        : make_uint4(0u, 0u, 0u, 0u);
                    const uint64_t inc0 = ((uint64_t)w.y << 32) | w.x;
                    const int e = (int)(w.w & 0xffu), kind = (int)((w.w >> 8) & 0xffu);
                    *ok = kind == kRowRun && e == b;
                    return Run{{inc0, inc0 + (uint64_t)(int64_t)(int32_t)w.z}};
                },
                r, H, S, p.ctrl);
            count(p.ctrl, kCtrlRowsRun, (uint32_t)(m - r));
        } else {
            m = r;  // no runs kept (a frame this small cannot reach 2^55)
        }
        r = m;
        if (r < H) {
            const unsigned char *rp = plane + (int64_t)r * p.stride;
            if (VEC && sizeof(TS) == 2) S = resolve_row_fast(rp, p.width, S, p.ctrl);
            else S = resolve_row<TS>(rp, p.width, S, p.ctrl);
            count(p.ctrl, kCtrlRowsTerms, 1);
            ++r;
        }
    }
    return S;
}

// The CPU's psnr noise of frame f in units: the exact row sums added in
// row order.
__device__ uint64_t walk_rows(const Params &p, int f)
{
    const int H = p.height;
    const size_t off = (size_t)f * H, n = ext_frame_rows(p);
    const uint64_t *rows = p.psnr_rows + off;
    uint32_t *ctrl = p.ctrl;
    const auto ld = [&p, rows, off, n](int i) { return chk(p.status, off + i, n) ? __ldcg(rows + i) : 0ull; };
    uint64_t S = 0;
    int r = 0;
    while (r < H) {
        int m;
        if (S < kTwo53) {
            SC before;
            m = warp_first([&ld](int i) { return SC{ld(i), 0}; }, r, H,
                           [S](SC x) { return S + x.s > kTwo53; }, &before, ctrl);
            S += before.s;
        } else {
            m = warp_run_walk(
                [&ld](int i, int sh, bool *ok) {
                    *ok = true;
                    return run_of_term(ld(i), sh);
                },
                r, H, S, ctrl);
        }
        if (m < H) S = rnd53(S + ld(m));
        r = m + 1;
    }
    return S;
}

__device__ __forceinline__ double scaled_mean(uint64_t units, int shift, double n)
{
    // units * 2^-shift is exact (a power-of-two scaling of an exact double);
    // the division is the CPU's, correctly rounded.
    const double scale = 1.0 / (double)(1ull << shift);
    return __ddiv_rn(__dmul_rn((double)units, scale), n);
}

__device__ __forceinline__ void store_agg(Agg *a, const Agg &g)
{
    uint4 *v = reinterpret_cast<uint4 *>(a);
    __stcg(v, make_uint4((uint32_t)g.s2[0], (uint32_t)(g.s2[0] >> 32), (uint32_t)g.s2[1],
                         (uint32_t)(g.s2[1] >> 32)));
    __stcg(v + 1, make_uint4((uint32_t)g.s1[0], (uint32_t)(g.s1[0] >> 32), (uint32_t)g.s1[1],
                             (uint32_t)(g.s1[1] >> 32)));
    __stcg(v + 2, make_uint4((uint32_t)g.psnr, (uint32_t)(g.psnr >> 32), (uint32_t)g.odd,
                             (uint32_t)(g.odd >> 32)));
}

__device__ __forceinline__ Agg agg_zero() { return Agg{{0, 0}, {0, 0}, 0, 0, {0, 0}}; }

// Items block b of a frame holds.
__device__ __forceinline__ uint32_t block_items(const Params &p, int b)
{
    return (uint32_t)min(kBlockItems, p.items_per_frame - b * kBlockItems);
}

// Whether block b of frame f has its record out: its last item to finish
// wrote the record, then set the block's count one past its items (release).
__device__ __forceinline__ bool block_done(const Params &p, int f, int b)
{
    const size_t i = (size_t)f * p.blocks_per_frame + b;
    return chk(p.status, i, ext_blocks(p)) && ld_acquire(p.block_fin + i) == block_items(p, b) + 1u;
}

// Whether item i of frame f has its record out (its flag is 1, or 2 once the
// look-back has published its inclusive prefix).
__device__ __forceinline__ bool item_done(const Params &p, int f, int i)
{
    const size_t k = (size_t)f * p.items_per_frame + i;
    return chk(p.status, k, ext_items(p)) && ld_acquire(p.flags + k) != 0u;
}

// Called by the whole warp of block b's last item to finish, after lane 0
// has acquired the block's count (every item released its record before it
// counted itself): each lane reads one item's record, the warp adds them,
// and lane 0 writes the block's record and then, with release order, sets
// the block's count one past its items. Item sums stay below 2^48 (at most
// 2^16 pixels of terms below 2^32).
__device__ __noinline__ void fold_block(const Params &p, int f, int b)
{
    const int lane = lane_id(), I = p.items_per_frame;
    const int i = b * kBlockItems + lane;
    Agg g = agg_zero();
    if (lane < (int)block_items(p, b) && chk(p.status, (size_t)f * I + i, ext_items(p))) {
        const Agg *it = p.items + (size_t)f * I + i;
        g.s2[0] = __ldcg(&it->s2[0]);
        g.s2[1] = __ldcg(&it->s2[1]);
        g.s1[0] = __ldcg(&it->s1[0]);
        g.s1[1] = __ldcg(&it->s1[1]);
        g.psnr = __ldcg(&it->psnr);
        g.odd = __ldcg(&it->odd);
    }
    Agg t = agg_zero();
    t.s2[0] = warp_sum_lt51(g.s2[0]);
    t.s2[1] = warp_sum_lt51(g.s2[1]);
    t.s1[0] = warp_sum_lt51(g.s1[0]);
    t.s1[1] = warp_sum_lt51(g.s1[1]);
    t.psnr = warp_sum_lt51(g.psnr);
    t.odd = warp_sum_lt51(g.odd);  // two counts below 2^17, summed in their halves
    const size_t k = (size_t)f * p.blocks_per_frame + b;
    if (lane == 0 && chk(p.status, k, ext_blocks(p))) {
        store_agg(p.blocks + k, t);
        st_release(p.block_fin + k, block_items(p, b) + 1u);
    }
}

// Waits (bounded) until every block of frame f is out, then returns the
// frame's sums that part `part` needs: plane X's second- and first-moment
// sums and odd terms (X = part < 2), or the psnr sum.
__device__ Agg frame_totals(const Params &p, int f, int part)
{
    const int lane = lane_id(), NB = p.blocks_per_frame;
    const Agg *bl = p.blocks + (size_t)f * NB;
    uint32_t spins = 0;
    for (;;) {
        bool ok = true;
        for (int b = lane; b < NB; b += 32) ok = ok && block_done(p, f, b);
        if (__all_sync(kFull, ok)) break;
        if (++spins > p.spin_limit) {
            if (lane == 0) atomicOr(p.status, 1u);
            break;
        }
        __nanosleep(128);
    }
    Agg t = agg_zero();
    if (part < 2) {
        const int X = part;
        uint64_t s2 = 0, s1 = 0, odd = 0;
        for (int b = lane; b < NB; b += 32) {
            if (!chk(p.status, (size_t)f * NB + b, ext_blocks(p))) continue;
            s2 += __ldcg(&bl[b].s2[X]);
            s1 += __ldcg(&bl[b].s1[X]);
            odd += __ldcg(&bl[b].odd);
        }
        t.s2[X] = warp_sum(s2);
        t.s1[X] = warp_sum(s1);
        t.odd = warp_sum(odd);
    } else {
        uint64_t ps = 0;
        for (int b = lane; b < NB; b += 32)
            if (chk(p.status, (size_t)f * NB + b, ext_blocks(p))) ps += __ldcg(&bl[b].psnr);
        t.psnr = warp_sum(ps);
    }
    return t;
}

// A window of up to 32 consecutive aggregates, lane i holding element i and
// whether it is complete: the first lane not complete (32 if none), the sum
// of the complete prefix, and the first lane of that prefix whose inclusive
// prefix from `run` passes 2^53 (-1 if none) with the prefix before it.
struct WindowScan {
    int first_open, hit;
    SC before, tot;
};

__device__ WindowScan scan_window(bool done, SC v, SC run)
{
    WindowScan w;
    const int lane = lane_id();
    const unsigned open = __ballot_sync(kFull, !done);
    w.first_open = open ? __ffs(open) - 1 : 32;
    if (lane >= w.first_open) v = SC{0, 0};
    const SC ex = warp_excl_sc(v, &w.tot);
    const unsigned hit = __ballot_sync(kFull, lane < w.first_open && run.s + ex.s + v.s > kTwo53);
    w.hit = hit ? __ffs(hit) - 1 : -1;
    w.before = sc_add(run, shfl_sc(ex, w.hit >= 0 ? w.hit : 0));
    return w;
}

// The first item of frame f whose inclusive exact prefix of plane X passes
// 2^53, found as soon as the items up to it are complete (later items may
// still be running); I when the whole frame stays at or below 2^53. Complete
// blocks are summed from their block sums (the prefix is kept; each poll
// looks at the 32 blocks from the first incomplete one), the first
// incomplete block item by item: an item is complete once its flag is set. A wait on one block is bounded. *before gets the prefix
// (sum, odd terms) before the item returned.
template <bool FLAGS>
__device__ int crossing_item(const Params &p, int f, int X, SC *before)
{
    const int lane = lane_id(), NB = p.blocks_per_frame, I = p.items_per_frame;
    const Agg *bl = p.blocks + (size_t)f * NB;
    const Agg *it = p.items + (size_t)f * I;
    const int shift = X ? 32 : 0;
    const auto sums = [X, shift](const Agg *a) {
        return SC{__ldcg(&a->s2[X]), (__ldcg(&a->odd) >> shift) & 0xffffffffull};
    };
    const size_t nb = ext_blocks(p), ni = ext_items(p);
    SC run{0, 0};  // exact prefix of blocks [0, base), all complete
    int base = 0;
    uint32_t spins = 0;
    while (base < NB) {
        count(p.ctrl, kCtrlPasses, 1);
        const int b = base + lane;
        bool done = true;
        SC v{0, 0};
        if (b < NB) {
            done = block_done(p, f, b);
            if (done && chk(p.status, (size_t)f * NB + b, nb)) v = sums(bl + b);
        }
        const WindowScan w = scan_window(done, v, run);
        if (w.hit >= 0) {  // a complete block: every item in it is out
            const int i = (base + w.hit) * kBlockItems + lane;
            const WindowScan wi = scan_window(
                true, i < I && chk(p.status, (size_t)f * I + i, ni) ? sums(it + i) : SC{0, 0}, w.before);
            *before = wi.before;
            return (base + w.hit) * kBlockItems + wi.hit;
        }
        run = sc_add(run, w.tot);
        base += w.first_open;
        if (w.first_open > 0) continue;
        if (!FLAGS) {  // items keep no flags of their own: wait for the block
            if (++spins > p.spin_limit) {
                if (lane == 0) atomicOr(p.status, 1u);
                *before = run;
                return I;
            }
            __nanosleep(64);
            continue;
        }
        // Block `base` is incomplete: poll its items alone until the
        // crossing shows among its complete ones or all of them are out.
        const int i = base * kBlockItems + lane;
        for (;;) {
            bool di = true;
            SC vi{0, 0};
            if (i < I) {
                di = item_done(p, f, i);
                if (di && chk(p.status, (size_t)f * I + i, ni)) vi = sums(it + i);
            }
            const WindowScan wi = scan_window(di, vi, run);
            if (wi.hit >= 0) {
                *before = wi.before;
                return base * kBlockItems + wi.hit;
            }
            if (wi.first_open == 32) {  // the whole block is out
                run = sc_add(run, wi.tot);
                ++base;
                break;
            }
            if (++spins > p.spin_limit) {  // an item never completed
                if (lane == 0) atomicOr(p.status, 1u);
                *before = run;
                return I;
            }
            __nanosleep(64);
        }
    }
    *before = run;
    return I;
}

// S after a run of terms with exact sum and odd count x, in the regime S is
// in: exact adds at or below 2^53, else the closed form of binade b (53, 54).
__device__ __forceinline__ uint64_t regime_after(uint64_t S, SC x, bool exact, int b)
{
    return exact ? S + x.s : closed_form_after(S, x.s, x.c, b);
}

__device__ __forceinline__ bool regime_left(uint64_t v, bool exact, int b)
{
    return exact ? v > kTwo53 : v >= (2ull << b);
}

// Zeroes the samples of V (64 consecutive samples from j0) before pos; a zero
// sample adds nothing.
__device__ __forceinline__ void mask_before(uint4 (&V)[8], int j0, int pos)
{
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        uint32_t w[4] = {V[v].x, V[v].y, V[v].z, V[v].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = j0 + v * 8 + 2 * q;
            w[q] &= (j >= pos ? 0x0000ffffu : 0u) | (j + 1 >= pos ? 0xffff0000u : 0u);
        }
        V[v] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// The exact sum and the odd-term count of the binary32 squares of 64
// samples, by the row pass's arithmetic: byte-split dot products for the
// squares, rounding errors in binary32, odd terms four at a time.
__device__ __forceinline__ void sums64(const uint4 (&V)[8], uint64_t *sum, uint32_t *odd)
{
    uint32_t lo_sum = 0, hi_sum = 0, ob = 0;
    float2 e = make_float2(0.0f, 0.0f);
    const float2 m23 = make_float2(-8388608.0f, -8388608.0f);
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        const uint32_t w[4] = {V[v].x, V[v].y, V[v].z, V[v].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t x = __byte_perm(w[q], 0, 0x3120);
            lo_sum = __dp2a_lo(w[q], x, lo_sum);
            hi_sum = __dp2a_hi(w[q], x, hi_sum);
            const uint32_t g0 = __byte_perm(w[q], kA, 0x7610), g1 = __byte_perm(w[q], kA, 0x7632);
            const float2 f = __fadd2_rn(make_float2(__uint_as_float(g0), __uint_as_float(g1)), m23);
            e = __fadd2_rn(e, __ffma2_rn(f, f, neg2(__fmul2_rn(f, f))));
        }
#pragma unroll
        for (int q = 0; q < 4; q += 2) {
            const uint32_t lo = __byte_perm(w[q], w[q + 1], 0x6420);
            const uint32_t hi = __byte_perm(w[q], w[q + 1], 0x7531);
            const uint32_t big = ((hi & 0x7F7F7F7Fu) + 0x70707070u) | hi;  // bit 7: byte >= 16
            ob += lo & ~(big >> 7) & 0x01010101u;
        }
    }
    *sum = ((uint64_t)hi_sum << 8) + lo_sum - (uint64_t)(int64_t)small_f_to_i(__fadd_rn(e.x, e.y));
    *odd = (ob & 0xffu) + ((ob >> 8) & 0xffu) + ((ob >> 16) & 0xffu) + (ob >> 24);
}

// Exclusive composition, in lane order, of the lanes' compact runs and of
// their exact sums; *tot and *tot_s get the warp's.
__device__ __forceinline__ void warp_excl_lane_run(const LaneRun &x, uint64_t xs, int sh, LaneRun *ex,
                                                   uint64_t *ex_s, LaneRun *tot, uint64_t *tot_s)
{
    const int lane = lane_id();
    LaneRun v = x;
    uint64_t vs = xs;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        LaneRun o;
        o.tlo = __shfl_up_sync(kFull, v.tlo, off);
        o.d[0] = __shfl_up_sync(kFull, v.d[0], off);
        o.d[1] = __shfl_up_sync(kFull, v.d[1], off);
        const uint64_t os = __shfl_up_sync(kFull, vs, off);
        if (lane >= off) {
            v = lane_compose(o, v, sh);
            vs += os;
        }
    }
    tot->tlo = __shfl_sync(kFull, v.tlo, 31);
    tot->d[0] = __shfl_sync(kFull, v.d[0], 31);
    tot->d[1] = __shfl_sync(kFull, v.d[1], 31);
    *tot_s = __shfl_sync(kFull, vs, 31);
    LaneRun e;
    e.tlo = __shfl_up_sync(kFull, v.tlo, 1);
    e.d[0] = __shfl_up_sync(kFull, v.d[0], 1);
    e.d[1] = __shfl_up_sync(kFull, v.d[1], 1);
    uint64_t es = __shfl_up_sync(kFull, vs, 1);
    if (lane == 0) {
        e = lane_identity();
        es = 0;
    }
    *ex = e;
    *ex_s = es;
}

// The terms of a 16-bit row starting on a 16-byte boundary, added to S from
// term `pos` on, for S from 2^55 up (binade b, last place u = 2^(b-52)), in
// rounds of 2048 terms: each lane forms the compact run of its 64
// consecutive terms (eight 8-term runs from eight 16-byte loads, composed in
// order), the warp composes the lanes' runs in order, and a round whose run
// keeps S below 2^(b+1) is added at once (ADR-1497 "Decision": a run's
// increments composed in order; every intermediate sum lies below the final
// one). Otherwise the first lane whose run takes S there puts its 64 samples
// in shared memory, the warp composes their one-term runs two per lane, the
// term that leaves the binade is rounded in full, and the round is taken up
// again from the next term in the new binade.
__device__ __noinline__ uint64_t resolve_row_runs(const unsigned char *row, int width, uint64_t S, int pos,
                                                  uint32_t *ctrl)
{
    __shared__ uint32_t swords[kWarps][32];
    const int lane = lane_id(), wid = (int)(threadIdx.x >> 5);
    int base = pos & ~2047;
    while (base < width) {
        const int b = binade_of(S), sh = b - 52;
        const uint64_t top = 2ull << b;
        count(ctrl, kCtrlPasses, 1);
        const int j0 = base + lane * 64;
        uint4 V[8];
#pragma unroll
        for (int v = 0; v < 8; ++v) V[v] = load_vec<uint16_t, true>(row, (j0 >> 3) + v, width);
        if (j0 < pos) mask_before(V, j0, pos);  // terms before pos are already in S
        LaneRun lr = lane_identity();
        uint64_t ls = 0;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            uint32_t t[8];
            const uint32_t w4[4] = {V[v].x, V[v].y, V[v].z, V[v].w};
#pragma unroll
            for (int w = 0; w < 4; ++w) terms_of_word(w4[w], &t[2 * w], &t[2 * w + 1]);
#pragma unroll
            for (int i = 0; i < 8; ++i) ls += t[i];
            lr = lane_compose(lr, lane_run_fp2(t, sh), sh);
        }
        LaneRun ex, tot;
        uint64_t ex_s, tot_s;
        warp_excl_lane_run(lr, ls, sh, &ex, &ex_s, &tot, &tot_s);
        const uint64_t whole = apply(lane_to_run(tot, tot_s), S, sh);
        if (whole < top) {
            S = whole;
            base += 32 * 64;
            pos = base;
            continue;
        }
        const uint64_t sb = apply(lane_to_run(ex, ex_s), S, sh);
        const uint64_t sa = apply(lane_to_run(lr, ls), sb, sh);
        const int src = __ffs(__ballot_sync(kFull, sa >= top)) - 1;
        const uint64_t s_src = __shfl_sync(kFull, sb, src);
        if (lane == src) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                swords[wid][4 * v] = V[v].x;
                swords[wid][4 * v + 1] = V[v].y;
                swords[wid][4 * v + 2] = V[v].z;
                swords[wid][4 * v + 3] = V[v].w;
            }
        }
        __syncwarp();
        const uint32_t w = swords[wid][lane];
        __syncwarp();
        const uint64_t t0 = term_of_sample(w & 0xffffu), t1 = term_of_sample(w >> 16);
        const Run r0 = run_of_term(t0, sh), r1 = run_of_term(t1, sh);
        Run tot2;
        const Run ex2 = warp_excl_run(compose(r0, r1, sh), sh, &tot2);
        const uint64_t c0 = apply(ex2, s_src, sh);
        const uint64_t c1 = apply(r0, c0, sh);
        const bool bad0 = c1 >= top;
        const bool bad1 = !bad0 && apply(r1, c1, sh) >= top;
        const int src2 = __ffs(__ballot_sync(kFull, bad0 || bad1)) - 1;
        const bool second = __shfl_sync(kFull, (int)bad1, src2);
        const uint64_t before = __shfl_sync(kFull, bad0 ? c0 : c1, src2);
        const uint64_t tm = __shfl_sync(kFull, bad0 ? t0 : t1, src2);
        S = rnd53(before + tm);  // the term that leaves the binade, rounded in full
        pos = base + src * 64 + 2 * src2 + (second ? 1 : 0) + 1;
    }
    return S;
}

// The terms of a 16-bit row starting on a 16-byte boundary, added to S from
// term `pos` on, in rounds of 2048 terms (64 consecutive terms per lane, from
// eight 16-byte loads). A round that keeps S at or below 2^53, or in its
// binade by the closed form, is added at once. Otherwise the first lane
// where that fails puts its 64 samples in shared memory, the warp scans them
// two per lane, the first term that leaves the regime is rounded in full,
// and the rest of the round is added from the round's sums. From binade 55
// up the general term walk takes over.
__device__ uint64_t resolve_row_fast(const unsigned char *row, int width, uint64_t S,
                                     uint32_t *ctrl)
{
    __shared__ uint32_t words[kWarps][32];
    const int lane = lane_id(), wid = (int)(threadIdx.x >> 5);
    int base = 0, pos = 0;
    while (base < width) {
        if (S >= kTwo53 && binade_of(S) >= 55) return resolve_row_runs(row, width, S, pos, ctrl);
        count(ctrl, kCtrlPasses, 1);
        const int j0 = base + lane * 64;
        uint4 V[8];
#pragma unroll
        for (int v = 0; v < 8; ++v) V[v] = load_vec<uint16_t, true>(row, (j0 >> 3) + v, width);
        if (j0 < pos) mask_before(V, j0, pos);  // terms before pos are already in S
        uint64_t ls;
        uint32_t lc32;
        sums64(V, &ls, &lc32);
        const uint64_t lc = lc32;
        SC tot;
        const SC ex = warp_excl_sc(SC{ls, lc}, &tot);
        const bool exact = S < kTwo53;
        const int b = exact ? 53 : binade_of(S);
        if (!regime_left(regime_after(S, tot, exact, b), exact, b)) {
            S = regime_after(S, tot, exact, b);
            base += 32 * 64;
            pos = base;
            continue;
        }
        const int src = __ffs(__ballot_sync(
                            kFull, regime_left(regime_after(S, sc_add(ex, SC{ls, lc}), exact, b), exact, b))) -
                        1;
        if (lane == src) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                words[wid][4 * v] = V[v].x;
                words[wid][4 * v + 1] = V[v].y;
                words[wid][4 * v + 2] = V[v].z;
                words[wid][4 * v + 3] = V[v].w;
            }
        }
        __syncwarp();
        const uint32_t w = words[wid][lane];
        __syncwarp();
        const int jb = base + src * 64 + 2 * lane;
        uint64_t t0 = term_of_sample(w & 0xffffu), t1 = term_of_sample(w >> 16);
        if (jb < pos || jb >= width) t0 = 0;
        if (jb + 1 < pos || jb + 1 >= width) t1 = 0;
        SC tot2;
        const SC ex2 = warp_excl_sc(SC{t0 + t1, (t0 & 1) + (t1 & 1)}, &tot2);
        const SC srcpre = shfl_sc(ex, src);
        const uint64_t c0 = regime_after(S, sc_add(srcpre, ex2), exact, b);
        const uint64_t c1 = regime_after(c0, SC{t0, t0 & 1}, exact, b);
        const bool bad0 = regime_left(c1, exact, b);
        const bool bad1 = !bad0 && regime_left(regime_after(c1, SC{t1, t1 & 1}, exact, b), exact, b);
        const int src2 = __ffs(__ballot_sync(kFull, bad0 || bad1)) - 1;
        const bool second = __shfl_sync(kFull, (int)bad1, src2);
        const uint64_t sb = __shfl_sync(kFull, bad0 ? c0 : c1, src2);
        const uint64_t tm = __shfl_sync(kFull, bad0 ? t0 : t1, src2);
        const uint64_t tfirst = __shfl_sync(kFull, t0, src2);
        const int m = base + src * 64 + 2 * src2 + (second ? 1 : 0);
        S = rnd53(sb + tm);
        // The round's terms after m, from its sums.
        SC through = sc_add(srcpre, shfl_sc(ex2, src2));
        if (second) through = sc_add(through, SC{tfirst, tfirst & 1});
        through = sc_add(through, SC{tm, tm & 1});
        const SC rest{tot.s - through.s, tot.c - through.c};
        const bool exact2 = S < kTwo53;
        const int b2 = exact2 ? 53 : binade_of(S);
        if (b2 <= 54 && !regime_left(regime_after(S, rest, exact2, b2), exact2, b2)) {
            S = regime_after(S, rest, exact2, b2);
            base += 32 * 64;
            pos = base;
            continue;
        }
        pos = m + 1;  // the round crosses again: walk it from the next term
    }
    return S;
}

// The second-moment sum of plane X. The first block whose exact prefix
// passes 2^53 is found as soon as the blocks before it are complete, then
// its item and row (one pass each); that row is walked term by term while
// the frame's later rows may still be running. Once the frame is complete,
// all later rows are added by one closed form if the sum then stays in its
// binade (always so below 2^55); anything else continues on the general
// path. *t gets the frame's sums.
template <typename TS, bool VEC, bool FULL>
__device__ uint64_t walk_plane_fast(const Params &p, int f, int X, Agg *t)
{
    const int I = p.items_per_frame, H = p.height;
    const size_t off = ((size_t)f * 2 + X) * H, nrows = ext_plane_rows(p);
    const uint64_t *R = p.s2_rows + off;
    const uint32_t *O = p.odd_rows + off;
    const auto ldRO = [&p, R, O, off, nrows](int i) {
        return chk(p.status, off + i, nrows) ? SC{__ldcg(R + i), (uint64_t)__ldcg(O + i)} : SC{0, 0};
    };
    SC pre_items;
    const int it = crossing_item<FULL>(p, f, X, &pre_items);
    if (it >= I) {
        *t = frame_totals(p, f, X);
        count(p.ctrl, kCtrlRowsExact, (uint32_t)H);
        return t->s2[X];
    }
    SC b2{0, 0};
    const int r0 = it * p.rows_per_item;
    const int row = p.rows_per_item == 1  // the item is the row
                        ? r0
                        : warp_first(ldRO, r0, min(H, r0 + p.rows_per_item),
                                     [pre_items](SC x) { return pre_items.s + x.s > kTwo53; }, &b2,
                                     p.ctrl);
    const SC pre = sc_add(pre_items, b2);
    count(p.ctrl, kCtrlRowsExact, (uint32_t)row);
    const unsigned char *plane = (X == 0 ? p.ref : p.dis) + (int64_t)f * p.pitch;
    const unsigned char *rp = plane + (int64_t)row * p.stride;
    uint64_t S = pre.s;
    if (VEC && sizeof(TS) == 2) S = resolve_row_fast(rp, p.width, S, p.ctrl);
    else S = resolve_row<TS>(rp, p.width, S, p.ctrl);
    count(p.ctrl, kCtrlRowsTerms, 1);
    const SC rsc = ldRO(row);
    const uint64_t rs = rsc.s, rc = rsc.c;
    *t = frame_totals(p, f, X);
    const uint64_t tot = t->s2[X], tot_odd = X ? (t->odd >> 32) : (t->odd & 0xffffffffull);
    const uint64_t rest_s = tot - pre.s - rs, rest_c = tot_odd - pre.c - rc;
    if (S >= kTwo53 && binade_of(S) <= 54) {
        const int b = binade_of(S);
        const uint64_t Sn = closed_form_after(S, rest_s, rest_c, b);
        if (Sn < (2ull << b)) {
            count(p.ctrl, kCtrlRowsRun, (uint32_t)(H - row - 1));
            return Sn;
        }
    }
    return walk_plane_from<TS, VEC, FULL>(p, f, X, row + 1, S);
}

// One part of a frame's results: part 0 and 1 the moments of ref and dis
// (when moments are asked for), the last part the psnr noise.
template <typename TS, bool M, bool P, bool ODD, bool FULL, bool VEC>
__device__ __noinline__ void walk_part(const Params &p, int f, int part)
{
    const double N = (double)p.width * (double)p.height;
    const bool lead = lane_id() == 0;
    if (M && part < 2) {
        const int X = part;
        Agg t;
        uint64_t s2;
        if (ODD) {
            s2 = walk_plane_fast<TS, VEC, FULL>(p, f, X, &t);
        } else {  // such frames stay at or below 2^53 units
            t = frame_totals(p, f, X);
            s2 = t.s2[X];
            count(p.ctrl, kCtrlRowsExact, (uint32_t)p.height);
        }
        if (lead && chk(p.status, (size_t)f * 4 + 2 + X, (size_t)p.frames * 4)) {
            p.moments[(size_t)f * 4 + X] = scaled_mean(t.s1[X], p.k, N);
            p.moments[(size_t)f * 4 + 2 + X] = scaled_mean(s2, 2 * p.k, N);
            if (p.s2_sums) p.s2_sums[(size_t)f * 2 + X] = s2;
        }
    } else if (P) {
        const Agg t = frame_totals(p, f, 2);
        const uint64_t d = t.psnr <= kTwo53 ? t.psnr
                                            : walk_rows(p, f);
        if (lead && chk(p.status, (size_t)f, (size_t)p.frames)) {
            p.mse[f] = scaled_mean(d, 2 * p.k, N);
            if (p.noise_sums) p.noise_sums[f] = d;
        }
    }
}

// ---------------------------------------------------------- the kernel ---

// The exact second-moment sums of the frame's items before item j, by a
// decoupled look-back over flags (1: the item's own sums are out, 2: the
// inclusive sums are out), 32 predecessors at a time: the flag-1 sums up to
// the nearest inclusive prefix are added at once; a nearer item with nothing
// out yet is waited for. Called by the whole warp; lane 0's aggr, aggd are
// the item's own sums. A wait longer than p.spin_limit polls sets the status
// word and gives up.
__device__ __noinline__ void lookback(const Params &p, int f, int j, uint64_t aggr, uint64_t aggd,
                                      uint64_t *pre_r, uint64_t *pre_d)
{
    const int lane = lane_id();
    const size_t base = (size_t)f * p.items_per_frame;
    const size_t idx = base + j;
    uint64_t pr = 0, pd = 0;
    if (j > 0) {
        int q = j - 1;
        uint32_t spins = 0;
        for (;;) {
            const int i = q - lane;  // lane 0 the nearest predecessor
            const uint32_t fl =
                i < 0 ? 2u : (chk(p.status, base + i, ext_items(p)) ? ld_acquire(p.flags + base + i) : 2u);
            const unsigned zero = __ballot_sync(kFull, fl == 0u);
            const unsigned incl = __ballot_sync(kFull, fl == 2u);
            const int fz = zero ? __ffs(zero) - 1 : 32;
            const int fi = incl ? __ffs(incl) - 1 : 32;
            if (fz < fi) {
                if (++spins > p.spin_limit) {
                    if (lane == 0) atomicOr(p.status, 1u);
                    break;
                }
                __nanosleep(64);
                continue;
            }
            uint64_t vr = 0, vd = 0;
            if (i >= 0 && !chk(p.status, base + i, ext_items(p))) {
            } else if (i >= 0 && lane < fi) {
                vr = __ldcg(&p.items[base + i].s2[0]);
                vd = __ldcg(&p.items[base + i].s2[1]);
            } else if (i >= 0 && lane == fi) {
                vr = __ldcg(p.item_inc + (base + i) * 2);
                vd = __ldcg(p.item_inc + (base + i) * 2 + 1);
            }
            pr += warp_sum(vr);
            pd += warp_sum(vd);
            if (fi < 32) break;  // an inclusive prefix (item 0 always publishes one)
            q -= 32;
        }
    }
    if (lane == 0 && chk(p.status, idx, ext_items(p))) {
        __stcg(p.item_inc + idx * 2, pr + aggr);
        __stcg(p.item_inc + idx * 2 + 1, pd + aggd);
        st_release(p.flags + idx, 2u);
    }
    *pre_r = pr;
    *pre_d = pd;
}

// Phase B of item j of frame f (rows [r0, r1), lane i holding row r0 + i's
// exact sums my_r, my_d; aggr, aggd the item's): the exact sums before the
// item by the look-back, each row's plan from its exact prefix, and the run
// of every row planned from binade 55 up (its record, else a record of no
// run). A function of its own, so that its state holds no registers in the
// row loop.
template <bool VEC>
__device__ __noinline__ void plan_and_runs(const Params &p, int f, int j, int r0, int r1, uint64_t my_r,
                                           uint64_t my_d, uint64_t aggr, uint64_t aggd)
{
    const int lane = lane_id(), H = p.height;
    uint64_t pr = 0, pd = 0;
    const long long t0 = pt_clock();
    lookback(p, f, j, aggr, aggd, &pr, &pd);
    const long long t1 = pt_clock();
    pt_add(kPtLookback, (unsigned long long)(t1 - t0));
    // Lane i plans row r0 + i of both planes from the row's exact prefix.
    SC tot;
    const uint64_t exr = warp_excl_sc(SC{my_r, 0}, &tot).s;
    const uint64_t exd = warp_excl_sc(SC{my_d, 0}, &tot).s;
    const bool mine = lane < r1 - r0;
    const int er = mine ? plan_binade(pr + exr, my_r) : 0;
    const int ed = mine ? plan_binade(pd + exd, my_d) : 0;
    // The rows to run are read a second time, one after another: all of
    // them are asked into L2 at once, so that only the first waits on DRAM.
    const uint32_t bytes = ((uint32_t)p.width * 2u) & ~15u;
    if (VEC && bytes > 0u && mine && chk(p.status, (size_t)f * H + r0 + lane, ext_frame_rows(p))) {
        const int64_t off = (int64_t)f * p.pitch + (int64_t)(r0 + lane) * p.stride;
        if (er >= 55) prefetch_l2(p.ref + off, bytes);
        if (ed >= 55) prefetch_l2(p.dis + off, bytes);
    }
    for (int X = 0; X < 2; ++X) {
        const unsigned char *plane = (X ? p.dis : p.ref) + (int64_t)f * p.pitch;
        for (int r = r0; r < r1; ++r) {
            const int li = r - r0;
            const int e = __shfl_sync(kFull, X ? ed : er, li);
            RowRec rec = {0ull, 0, 0, kRowNone, 0};
            if (e >= 55) {
                const uint64_t rs = __shfl_sync(kFull, X ? my_d : my_r, li);
                const Run run = row_run16<VEC>(plane + (int64_t)r * p.stride, p.width, e, rs);
                pt_add(kPtRunRows, 1ull);
                rec.inc0 = run.inc[0];
                rec.dinc = (int32_t)(run.inc[1] - run.inc[0]);
                rec.e = (uint8_t)e;
                rec.kind = kRowRun;
            }
            const size_t k = ((size_t)f * 2 + X) * H + r;
            if (lane == 0 && chk(p.status, k, ext_plane_rows(p))) p.rec[k] = rec;
        }
    }
    pt_cycles(kPtRuns, t1);
}

// C. completion of item j of frame f: the item counts itself in its block
// (32-bit), one release per item (its records, then its count); the block's
// last item to finish acquires them all (with one fence unless the count
// was taken acquire-release) and writes the block's record. (A test of the
// bounded waits asks for one item more than a block holds: no block
// completes.) Called by the whole warp.
template <bool FULL>
__device__ __forceinline__ void complete_item(const Params &p, int f, int j)
{
    const long long t0 = pt_clock();
    const int b = j / kBlockItems, NB = p.blocks_per_frame;
    uint32_t last = 0;
    if (lane_id() == 0) {
        uint32_t *cnt = p.block_fin + (size_t)f * NB + b;
        const uint32_t old = !chk(p.status, (size_t)f * NB + b, ext_blocks(p)) ? 0u
                             : FULL ? atom_add_acq_rel(cnt, 1u)
                                    : atom_add_release(cnt, 1u);
        last = old + 1u == block_items(p, b) + p.test_stall ? 1u : 0u;
        if (last && !FULL) fence_acq_rel();
    }
    if (__shfl_sync(kFull, last, 0)) {
        __syncwarp();  // lane 0's acquire before the other lanes' reads
        fold_block(p, f, b);
    }
    pt_cycles(kPtComplete, t0);
}

// A streamed item whose plan is still to come: its frame and index, its
// exact sums, and each row's (lane i's row r0 + i).
struct ParkSlot {
    uint64_t rows[2][kMaxRowsPerItem];
    uint64_t agg[2];
    int f, j;
};

// Phases B and C of the item in a warp's slot. Called by the whole warp.
template <bool VEC, bool FULL>
__device__ __noinline__ void resume_parked(const Params &p, const ParkSlot &q)
{
    const int lane = lane_id();
    const int f = q.f, j = q.j;
    const int r0 = j * p.rows_per_item, r1 = min(p.height, r0 + p.rows_per_item);
    uint64_t my_r = 0, my_d = 0;
    if (lane < r1 - r0) {
        my_r = q.rows[0][lane];
        my_d = q.rows[1][lane];
    }
    plan_and_runs<VEC>(p, f, j, r0, r1, my_r, my_d, q.agg[0], q.agg[1]);
    complete_item<FULL>(p, f, j);
}

// The order items are handed out in: frame by frame, except that the last
// kTailFrames frames (all of them in a batch of at most that many) go row by
// row across those frames. A frame's crossing row (about three quarters down
// a frame of uniform noise) is then out well before the batch's last rows,
// so its walk runs while they stream instead of after them.
#ifndef VMX_TAIL_FRAMES
#define VMX_TAIL_FRAMES 16
#endif
constexpr int kTailFrames = VMX_TAIL_FRAMES;
__device__ __forceinline__ void item_of_ticket(int tk, int F, int I, int *f, int *j)
{
    const int K = min(F, kTailFrames);
    const int head = (F - K) * I;
    if (tk < head) {
        *f = tk / I;
        *j = tk - *f * I;
    } else {
        const int t = tk - head;
        *j = t / K;
        *f = F - K + (t - *j * K);
    }
}

template <typename TS, bool M, bool P, bool ODD, bool FULL, bool VEC, bool LOW>
__global__ void __maxnreg__(FULL ? kMaxRegsFull : kMaxRegs) frames_kernel(Params p)
{
    const int lane = lane_id();
    const int I = p.items_per_frame;
    const int nitems = p.frames * I;
    const int H = p.height;
    // Items are handed out by a ticket counter only, in chunks of
    // consecutive items, one atomic per chunk, the chunk size shrinking from
    // kMaxChunk to 1 as the items run out; so an item belongs to a warp that
    // is running, whatever part of the grid is resident. With look-back a
    // chunk is one item: an item's look-back waits for the item before it,
    // and in a longer chunk that item would wait for its owner's earlier
    // items, so the chunks would run one after another. Waits stay
    // deadlock-free: streaming an item never waits, and a look-back (taken
    // up for a parked item once the warp has streamed its next one) waits
    // only for earlier items to have streamed, each of which a running warp
    // holds or has finished.
    // The parameters as the functions the kernel calls without inlining see
    // them: a copy in shared memory, so that no thread keeps a copy of its
    // own in local memory for them to point at (the kernel reads its own).
    // Measured per instance: the 16-bit aligned full-depth instance without
    // the look-back runs about 1% faster with the per-thread copy (16 x
    // 3840x2160: 98.6 against 99.7 us a call in a stream), every other one
    // 1-5% faster with the shared copy.
    constexpr bool kOwnCopy = sizeof(TS) == 2 && VEC && !FULL && !LOW;
    __shared__ Params shared_params;
    if (!kOwnCopy) {
        if (threadIdx.x == 0) shared_params = p;
        __syncthreads();
    }
    const Params &sp = kOwnCopy ? p : shared_params;
    __shared__ RowSlot item_rows[kWarps][kMaxRowsPerItem];  // sums of an item's rows
    __shared__ ParkSlot park[FULL && M ? kWarps : 1];         // an item waiting for its plan
    bool parked = false;
    const int wid = (int)(threadIdx.x >> 5);
    // 16-bit rows on 16-byte boundaries stream through shared memory.
    constexpr bool STG = kStages > 0 && VEC && sizeof(TS) == 2;
    extern __shared__ __align__(128) unsigned char pipe_smem[];
    Pipe pp{0u, 0u, 0u, 0u, 0, 0, false};
    const int cpr = STG ? (p.width >> 3) / kChunkVecs : 0;  // whole chunks per row
    if (STG) {
        pp.buf = smem_u32(pipe_smem) + (uint32_t)wid * kStages * kStageBytes;
        pp.bar = smem_u32(pipe_smem) + (uint32_t)kWarps * kStages * kStageBytes + 8u * kStages * (uint32_t)wid;
        if (lane == 0) {
            for (int st = 0; st < kStages; ++st) mbar_init(pp.bar + 8u * st);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncwarp();
    }
    // A kernel launched to overlap this one (the next call on the stream,
    // which touches nothing this one writes) may be scheduled at once: its
    // blocks take the SM slots this grid's blocks leave.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t nwarps = gridDim.x * (uint32_t)kWarps;
    uint32_t cur = 0u, end = 0u, seen = 0u;
    pt_min(kPtStart, pt_now());
    for (;;) {
        if (cur >= end) {
            const uint32_t left = (uint32_t)nitems > seen ? (uint32_t)nitems - seen : 0u;
            const uint32_t k = FULL ? 1u : max(1u, min((uint32_t)kMaxChunk, left / (4u * nwarps)));
            uint32_t c = 0;
            if (lane == 0) c = atomicAdd(p.ctrl + kCtrlTicket, k);
            c = __shfl_sync(kFull, c, 0);
            seen = c + k;
            cur = c;
            end = c + k;
        }
        const int tk = (int)cur++;
        if (tk >= nitems) break;
        int f, j;
        item_of_ticket(tk, p.frames, I, &f, &j);
        const long long ta = pt_clock();
        const int r0 = j * p.rows_per_item, r1 = min(H, r0 + p.rows_per_item);
        const unsigned char *fr = p.ref + (int64_t)f * p.pitch;
        const unsigned char *fd = p.dis + (int64_t)f * p.pitch;
        const PipeSrc src{fr, fd, p.stride, r1, cpr};
        if (STG) {  // start the item's first chunks
            pp.prow = r0;
            pp.pc = 0;
            __syncwarp();
            pipe_fill(pp, src);
        }

        // A. exact row sums. Lane 0 records each row and keeps its sums in
        // the warp's shared slots, so that no item totals stay live in
        // registers across rows; lane i reads row i's back afterwards.
        for (int r = r0; r < r1; ++r) {
            // (a checked build: the row and the frame lie inside the planes)
            if (!chk(p.status, (size_t)f * H + r, ext_frame_rows(p))) continue;
            const unsigned char *rr = fr + (int64_t)r * p.stride;
            const unsigned char *dr = fd + (int64_t)r * p.stride;
            const RowSums rs = sizeof(TS) == 2
                                   ? row_sums16<M, P, ODD, VEC, STG, LOW>(rr, dr, p.width, pp, src, p.status)
                                   : row_sums8<M, P, VEC>(rr, dr, p.width);
            if (lane == 0) {
                const size_t k0 = ((size_t)f * 2) * H + r, k1 = ((size_t)f * 2 + 1) * H + r;
                const size_t np = ext_plane_rows(p);
                if (M && chk(p.status, k0, np)) p.s2_rows[k0] = rs.t2r;
                if (M && chk(p.status, k1, np)) p.s2_rows[k1] = rs.t2d;
                if (ODD && chk(p.status, k0, np)) p.odd_rows[k0] = rs.oddr;
                if (ODD && chk(p.status, k1, np)) p.odd_rows[k1] = rs.oddd;
                if (P) p.psnr_rows[(size_t)f * H + r] = rs.tp;  // (f, r) checked above
            }
            if (lane == 0 && chk(p.status, r - r0, kMaxRowsPerItem))
                item_rows[wid][r - r0] = RowSlot{rs.t2r, rs.t2d, rs.tp, (uint64_t)rs.oddr | ((uint64_t)rs.oddd << 32),
                                                 rs.s1r | (rs.s1d << 32)};
        }
        __syncwarp();
        uint64_t my_r = 0, my_d = 0, my_p = 0, my_o = 0;  // this lane's row of the item
        uint32_t s1r = 0, s1d = 0;
        if (lane < r1 - r0 && chk(p.status, lane, kMaxRowsPerItem)) {
            const RowSlot v = item_rows[wid][lane];
            my_r = v.x;
            my_d = v.y;
            my_p = v.z;
            my_o = v.w;
            s1r = (uint32_t)v.s1;
            s1d = (uint32_t)(v.s1 >> 32);
        }
        __syncwarp();
        // Lane 0 alone stores and adds the item's sums: a one-row item has
        // them in lane 0 already. A row's first-moment sum is below 2^31.
        Agg g = agg_zero();
        const bool one = r1 - r0 == 1;
        if (M) {
            g.s2[0] = one ? my_r : warp_sum_lt51(my_r);  // a row's sum is below 2^47
            g.s2[1] = one ? my_d : warp_sum_lt51(my_d);
            g.s1[0] = warp_sum_lt51(s1r);
            g.s1[1] = warp_sum_lt51(s1d);
        }
        if (ODD && !one) {  // each count fits 32 bits
            g.odd = (uint64_t)warp_sum32((uint32_t)my_o) | ((uint64_t)warp_sum32((uint32_t)(my_o >> 32)) << 32);
        } else if (ODD) {
            g.odd = my_o;
        }
        if (P) g.psnr = one ? my_p : warp_sum_lt51(my_p);
        if (lane == 0 && chk(p.status, (size_t)f * I + j, ext_items(p))) {
            Agg *ia = p.items + (size_t)f * I + j;
            store_agg(ia, g);
            // The look-back reads each item's flag: its sums are out.
            if (FULL) st_release(p.flags + (size_t)f * I + j, 1u);
        }

        pt_cycles(kPtStream, ta);
        pt_add(kPtItems, 1ull);
        // B. frames that can pass 2^55: runs of the rows planned from 55 up.
        // An item's plan waits for every item of the frame before it, so it
        // is taken up only after the warp has streamed its next item (the
        // item parked meanwhile in the warp's shared slot): by then those
        // items are out, and the warp seldom waits.
        if (FULL && M) {
            if (parked) resume_parked<VEC, FULL>(sp, park[wid]);
            __syncwarp();
            if (lane < r1 - r0) {
                park[wid].rows[0][lane] = my_r;
                park[wid].rows[1][lane] = my_d;
            }
            if (lane == 0) {
                park[wid].agg[0] = g.s2[0];
                park[wid].agg[1] = g.s2[1];
                park[wid].f = f;
                park[wid].j = j;
            }
            __syncwarp();
            parked = true;
            continue;
        }

        // C. completion.
        complete_item<FULL>(sp, f, j);
    }
    if (FULL && M && parked) resume_parked<VEC, FULL>(sp, park[wid]);
    pt_max(kPtOutLast, pt_now());
    pt_min(kPtOutFirst, pt_now());

    // Every chunk a warp started it has read, unless a wait gave up: then
    // wait (bounded) for the copies still landing in its buffers.
    if (STG && pp.broken) {
        pp.broken = false;
        for (uint32_t i = pp.n > (uint32_t)kStages ? pp.n - kStages : 0u; i < pp.n; ++i) pipe_wait(pp, i, p.status);
    }

    // D. Walks. A warp out of items takes a part of a frame to walk (the ref
    // moments, the dis moments, the psnr noise). A warp gets here only once
    // every item has been handed out, so each item a walk waits for is held
    // by a running warp, which finishes it without waiting on the walks; the
    // waits are bounded all the same.
    constexpr int kParts = (M ? 2 : 0) + (P ? 1 : 0);
    for (;;) {
        int wt = 0;
        if (lane == 0) wt = (int)atomicAdd(p.ctrl + kCtrlWalkTicket, 1u);
        wt = __shfl_sync(kFull, wt, 0);
        if (wt >= p.frames * kParts) break;
        const int wf = wt / kParts, part = wt - wf * kParts;
        const long long tw = pt_clock();
        pt_min(kPtWalksStart, pt_now());
        walk_part<TS, M, P, ODD, FULL, VEC>(sp, wf, M ? part : 2);
        pt_cycles(kPtWalks, tw);
        pt_max(kPtWalkMax, (unsigned long long)(pt_clock() - tw));
        pt_add(kPtWalkTasks, 1ull);
        pt_max(kPtWalksEnd, pt_now());
    }
    // Launched to overlap the previous kernel: the grid finishes after it, so
    // that the stream's later work still follows both. One block waiting is
    // enough for that; the others leave at once, and their slots go to the
    // next calls (with small batches several calls run at a time).
    if (p.overlap && blockIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    pt_max(kPtEnd, pt_now());
}

template <typename TS, bool M, bool P, bool ODD, bool FULL, bool VEC, bool LOW>
cudaError_t launch_one(const Params &p, const Layout &L, cudaStream_t stream)
{
    static int blocks_per_sm[64] = {0};  // per device ordinal, filled once
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    // Chunk buffers of the 16-bit kernels that stream through shared memory.
    const size_t smem = kStages > 0 && VEC && sizeof(TS) == 2 ? kPipeSmem : 0;
    if (blocks_per_sm[dev] == 0) {
        if (smem > 0) {
            err = cudaFuncSetAttribute(frames_kernel<TS, M, P, ODD, FULL, VEC, LOW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (err != cudaSuccess) return err;
        }
        int n = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, frames_kernel<TS, M, P, ODD, FULL, VEC, LOW>, kThreads, smem);
        if (err != cudaSuccess) return err;
        blocks_per_sm[dev] = n > 0 ? n : 1;
    }
    int sms = 0;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    const long long warps = (long long)L.frames * L.items_per_frame;
    const long long blocks = (warps + kWarps - 1) / kWarps;
    int grid = (int)std::min<long long>(blocks, (long long)sms * blocks_per_sm[dev]);
    if (p.test_grid_mult > 1) grid = sms * blocks_per_sm[dev] * p.test_grid_mult;
    if (!p.overlap) {
        frames_kernel<TS, M, P, ODD, FULL, VEC, LOW><<<grid, kThreads, smem, stream>>>(p);
        return cudaGetLastError();
    }
    // Programmatic dependent launch: may start once every block of the
    // previous kernel on the stream has run out of items or exited.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, frames_kernel<TS, M, P, ODD, FULL, VEC, LOW>, p);
}

template <typename TS, bool M, bool P, bool ODD, bool FULL, bool LOW = false>
cudaError_t launch_vec(const Params &p, const Layout &L, bool vec, cudaStream_t s)
{
    return vec ? launch_one<TS, M, P, ODD, FULL, true, LOW>(p, L, s)
               : launch_one<TS, M, P, ODD, FULL, false, LOW>(p, L, s);
}

template <bool M, bool P>
cudaError_t launch_u16(const Params &p, const Layout &L, bool vec, cudaStream_t s)
{
    // Depths up to 12 bits check each pass for samples below 4096.
    const bool low = VMX_LOW_DEPTH && L.bpc <= 12;
    if (L.full) return launch_vec<uint16_t, M, P, true, true>(p, L, vec, s);
    if (L.ordered)
        return low ? launch_vec<uint16_t, M, P, true, false, true>(p, L, vec, s)
                   : launch_vec<uint16_t, M, P, true, false>(p, L, vec, s);
    return low ? launch_vec<uint16_t, M, P, false, false, true>(p, L, vec, s)
               : launch_vec<uint16_t, M, P, false, false>(p, L, vec, s);
}

}  // namespace

cudaError_t launch_frames(const Params &p, const Layout &L, int features, bool vec,
                          cudaStream_t stream)
{
    const bool m = features & VMX_FEATURE_MOMENT, ps = features & VMX_FEATURE_PSNR;
    if (L.bpc == 8) {
        if (m && ps) return launch_vec<uint8_t, true, true, false, false>(p, L, vec, stream);
        if (m) return launch_vec<uint8_t, true, false, false, false>(p, L, vec, stream);
        return launch_vec<uint8_t, false, true, false, false>(p, L, vec, stream);
    }
    if (m && ps) return launch_u16<true, true>(p, L, vec, stream);
    if (m) return launch_u16<true, false>(p, L, vec, stream);
    return VMX_LOW_DEPTH && L.bpc <= 12 ? launch_vec<uint16_t, false, true, false, false, true>(p, L, vec, stream)
                       : launch_vec<uint16_t, false, true, false, false>(p, L, vec, stream);
}

// Scratch of vmx_frames_noalloc: a fixed array in the module's static device
// memory, one per device, 256-byte aligned like a caller's workspace.
static __device__ __align__(256) unsigned char g_noalloc_scratch[VMX_NOALLOC_SCRATCH_BYTES];

cudaError_t phase_times(uint64_t *out, bool reset)
{
    if (out) {
        cudaError_t err = cudaMemcpyFromSymbol(out, g_phase, sizeof(g_phase));
        if (err != cudaSuccess) return err;
        int dev = 0, khz = 0;
        err = cudaGetDevice(&dev);
        if (err == cudaSuccess) err = cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev);
        if (err != cudaSuccess) return err;
        out[kPtClockKHz] = (uint64_t)khz;
    }
    if (!reset) return cudaSuccess;
    unsigned long long z[kPtCount] = {0};
    z[kPtStart] = z[kPtOutFirst] = z[kPtWalksStart] = ~0ull;
    return cudaMemcpyToSymbol(g_phase, z, sizeof(z));
}

cudaError_t noalloc_scratch_address(void **ptr)
{
    return cudaGetSymbolAddress(ptr, g_noalloc_scratch);
}

}  // namespace vmx
