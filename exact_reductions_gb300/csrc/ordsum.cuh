// ordsum.cuh -- integer arithmetic of the CPU's rounded double sums.
//
// Host and device. In units of 1/scaler^2 every value the CPU's double
// accumulator takes is an integer, and one step of its loop is the exact
// integer sum rounded to 53 significant bits, ties to even (ADR-1497
// "Decision", first point). From 2^53 up, while the running sum S stays in one
// binade [2^e, 2^(e+1)), S is a multiple of the binade's last place
// u = 2^(e-52), and adding a term t moves S to the multiple of u nearest to
// S + t, a tie going to the even multiple (second point). A run of terms
// therefore acts on S through one bit, the parity of S / u: it is a pair of
// increments, one for an even and one for an odd start, and runs compose
// associatively but not commutatively.
//
// Everything here is u64/u32 integer arithmetic, except lane_run_fp(), which
// rounds with binary32 adds whose last place is u (see there).
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define VMX_HD __host__ __device__ __forceinline__
#else
#define VMX_HD inline
#endif

#if defined(VMX_MODEL_MUTATIONS)
// Planted mistakes, compiled only into the CPU model used by the tests.
extern "C" int vmx_model_mutation;
#define VMX_MUT(k) (vmx_model_mutation == (k))
#else
#define VMX_MUT(k) false
#endif

namespace vmx {

constexpr uint64_t kTwo53 = 1ull << 53;

VMX_HD int bit_length(uint64_t x)
{
#if defined(__CUDA_ARCH__)
    return 64 - __clzll((long long)x);
#else
    return x ? 64 - __builtin_clzll(x) : 0;
#endif
}

// floor(log2 S) for S >= 2^53: the binade the CPU's sum is in.
VMX_HD int binade_of(uint64_t s) { return bit_length(s) - 1; }

// The multiple of 2^sh nearest to x, a tie going to the even multiple.
// sh >= 1. The result may be the next power of two.
VMX_HD uint64_t round_to_ulp(uint64_t x, int sh)
{
    const uint64_t mask = (1ull << sh) - 1;
    uint64_t lsb = (x >> sh) & 1ull;
    if (VMX_MUT(1)) lsb ^= 1ull;  // ties to odd
    return (x + (mask >> 1) + lsb) & ~mask;
}

// One step of the CPU's loop in units: x rounded to 53 significant bits,
// ties to even.
VMX_HD uint64_t rnd53(uint64_t x)
{
    if (VMX_MUT(6)) return x;  // no rounding at all
    if (x <= kTwo53) return x;
    return round_to_ulp(x, bit_length(x) - 53);
}

// A run: the increment it adds to S for an even (inc[0]) and an odd (inc[1])
// start S / u, in units, under one binade's last place u = 2^sh.
struct Run {
    uint64_t inc[2];
};

VMX_HD Run run_identity() { return Run{{0ull, 0ull}}; }

// The run of one term t under last place 2^sh.
VMX_HD Run run_of_term(uint64_t t, int sh)
{
    const uint64_t u = 1ull << sh;
    Run r;
    r.inc[0] = round_to_ulp(t, sh);
    r.inc[1] = round_to_ulp(u + t, sh) - u;
    return r;
}

// Parity of S / u after a run added `inc` to a start of parity p.
VMX_HD unsigned parity_after(unsigned p, uint64_t inc, int sh)
{
    return p ^ (unsigned)((inc >> sh) & 1ull);
}

// a then b.
VMX_HD Run compose(const Run &a, const Run &b, int sh)
{
    if (VMX_MUT(3)) {  // composed in reverse
        Run c;
        for (int p = 0; p < 2; ++p)
            c.inc[p] = b.inc[p] + a.inc[parity_after((unsigned)p, b.inc[p], sh)];
        return c;
    }
    Run c;
    c.inc[0] = a.inc[0] + b.inc[parity_after(0u, a.inc[0], sh)];
    c.inc[1] = a.inc[1] + b.inc[parity_after(1u, a.inc[1], sh)];
    return c;
}

// S after a run, for S a multiple of u = 2^sh in the run's binade.
VMX_HD uint64_t apply(const Run &r, uint64_t s, int sh)
{
    if (VMX_MUT(2)) return s + r.inc[0];  // parity ignored
    return s + r.inc[(s >> sh) & 1ull];
}

VMX_HD float as_float(uint32_t u)
{
#if defined(__CUDA_ARCH__)
    return __uint_as_float(u);
#else
    float f;
    __builtin_memcpy(&f, &u, sizeof f);
    return f;
#endif
}

VMX_HD uint32_t as_uint(float f)
{
#if defined(__CUDA_ARCH__)
    return __float_as_uint(f);
#else
    uint32_t u;
    __builtin_memcpy(&u, &f, sizeof u);
    return u;
#endif
}

// Binary32 add, multiply and fused multiply-add, each rounded once to
// nearest even, never contracted or reassociated.
VMX_HD float f32_add(float a, float b)
{
#if defined(__CUDA_ARCH__)
    return __fadd_rn(a, b);
#else
    volatile float r = a + b;
    return r;
#endif
}

VMX_HD float f32_mul(float a, float b)
{
#if defined(__CUDA_ARCH__)
    return __fmul_rn(a, b);
#else
    volatile float r = a * b;
    return r;
#endif
}

VMX_HD float f32_fma(float a, float b, float c)
{
#if defined(__CUDA_ARCH__)
    return __fmaf_rn(a, b, c);
#else
    return __builtin_fmaf(a, b, c);
#endif
}

// Small integers to and from binary32 without a conversion instruction:
// 2^23 + v has v in its low mantissa bits for 0 <= v < 2^23, and
// 1.5 * 2^23 + i has i + 2^22 there for |i| < 2^22.
constexpr uint32_t kMagicU = 0x4B000000u;  // 2^23
constexpr uint32_t kMagicI = 0x4B400000u;  // 1.5 * 2^23
VMX_HD float small_u_to_f(uint32_t v) { return f32_add(as_float(v | kMagicU), -8388608.0f); }
VMX_HD int32_t small_f_to_i(float x)
{
    return (int32_t)(as_uint(f32_add(x, 12582912.0f)) - kMagicI);
}
// Inverse of small_u_to_f for an integral 0 <= x < 2^23.
VMX_HD uint32_t small_f_to_u(float x) { return as_uint(f32_add(x, 8388608.0f)) - kMagicU; }

// The binary32 square of a codeword p < 2^16 given f = (float)p, as the
// exact integer it is (p^2 rounded to 24 significant bits): p^2 minus the
// product's rounding error, which the fused multiply-add gives exactly.
VMX_HD uint32_t term_from_float(uint32_t p, float f)
{
    const float tf = f32_mul(f, f);
    const float ef = f32_fma(f, f, -tf);  // p^2 - tf, an integer in [-128, 128]
    return p * p - (uint32_t)small_f_to_i(ef);
}

// The CPU's term in units for a codeword p < 2^16.
VMX_HD uint32_t term_of_sample(uint32_t p) { return term_from_float(p, small_u_to_f(p)); }

// The binary32 square of a difference of codewords, |d| < 2^16.
VMX_HD uint32_t term_of_diff(uint32_t a, uint32_t b)
{
    return term_of_sample(a > b ? a - b : b - a);
}

// A lane's run of consecutive terms, in compact form: a number congruent to
// the terms' sum modulo 2u (all that composing and the parities read; the
// CPU model keeps the sum modulo 2^32, the device the residues' sum) and, for
// each start parity, the run's increment minus the exact sum of its terms (a
// small signed number).
struct LaneRun {
    uint32_t tlo;
    int32_t d[2];
};

VMX_HD LaneRun lane_identity() { return LaneRun{0u, {0, 0}}; }

VMX_HD unsigned lane_parity_after(unsigned p, const LaneRun &r, int sh)
{
    return p ^ (((r.tlo + (uint32_t)r.d[p]) >> sh) & 1u);
}

// a then b, compact form.
VMX_HD LaneRun lane_compose(const LaneRun &a, const LaneRun &b, int sh)
{
    LaneRun c;
    if (VMX_MUT(3)) {  // composed in reverse
        c.tlo = a.tlo + b.tlo;
        c.d[0] = b.d[0] + a.d[lane_parity_after(0u, b, sh)];
        c.d[1] = b.d[1] + a.d[lane_parity_after(1u, b, sh)];
        return c;
    }
    c.tlo = a.tlo + b.tlo;
    c.d[0] = a.d[0] + b.d[lane_parity_after(0u, a, sh)];
    c.d[1] = a.d[1] + b.d[lane_parity_after(1u, a, sh)];
    return c;
}

// The full run of a compact run whose terms add to `exact` units.
VMX_HD Run lane_to_run(const LaneRun &r, uint64_t exact)
{
    Run out;
    out.inc[0] = exact + (uint64_t)(int64_t)r.d[0];
    out.inc[1] = exact + (uint64_t)(int64_t)r.d[1];
    return out;
}

// The compact run of n terms under last place u = 2^sh, sh >= 1, while
// n * 2u < 2^22 (the device runs each lane's stretch of a row, up to 1024
// terms, the same way).
//
// Only t mod 2u matters for how a term rounds: writing t = 2u*m + v with
// 0 <= v < 2u, the increment is 2u*m plus the rounded increment of v from the
// same parity (a shift by 2u keeps the parity). The rounded increments of the
// small v are formed by binary32 adds: a float F in [2^23 u, 2^24 u) has last
// place exactly u, and F + v rounds to the nearest multiple of u, a tie to the
// even F / u, which is the CPU's rule with F / u standing for S / u. The even
// trajectory starts at 1.5 * 2^23 * u (F / u even), the odd one a place
// higher; n adds of v < 2u never leave the binade while n * 2u < 2^22.
VMX_HD LaneRun lane_run_fp(const uint32_t *t, int n, int sh)
{
    const float uf = as_float((uint32_t)(127 + sh) << 23);  // 2^sh
    const float f0e = f32_mul(12582912.0f, uf);              // 1.5 * 2^23 * u
    const float f0o = f32_add(f0e, uf);
    float fe = f0e, fo = f0o;
    uint32_t tlo = 0, vsum = 0;
    const uint32_t vmask = (2u << sh) - 1u;
    for (int i = 0; i < n; ++i) {
        const uint32_t v = t[i] & vmask;
        tlo += t[i];
        vsum += v;
        const float vf = small_u_to_f(v);
        fe = f32_add(fe, vf);
        fo = f32_add(fo, vf);
    }
    LaneRun r;
    r.tlo = tlo;
    r.d[0] = small_f_to_i(f32_add(fe, -f0e)) - (int32_t)vsum;
    r.d[1] = small_f_to_i(f32_add(fo, -f0o)) - (int32_t)vsum;
    if (VMX_MUT(2)) r.d[1] = r.d[0];  // parity ignored
    return r;
}

// Closed forms for the binades 53 and 54. Every term of this method is the
// binary32 square of a codeword (or of a difference of codewords) below 2^16,
// and every such square t satisfies t mod 8 in {0, 1, 4}, with t odd exactly
// when the codeword is odd and below 4096 (checked over all 65 536 codewords).
// So under last place 2 (binade 53) a term is either a multiple of 4 (added
// exactly, parity kept) or a tie that lands S on a multiple of 4: from an
// even start every tie rounds down by 1; from an odd start the first tie
// rounds up by 1 and the rest down. Under last place 4 (binade 54) the
// residues 0 and 4 add exactly and residue 1 rounds down, for either parity.
// With `sum` the exact sum of a run of such terms and `odd` how many of them
// are odd, the run adds:
//   binade 53: sum - odd, plus 2 when the start is odd and odd > 0;
//   binade 54: sum - odd.
VMX_HD uint64_t closed_form_after(uint64_t s, uint64_t sum, uint64_t odd, int binade)
{
    if (VMX_MUT(2)) return s + sum - odd;  // parity ignored
    uint64_t r = s + sum - odd;
    if (binade == 53 && odd > 0 && ((s >> 1) & 1ull)) r += 2;
    return r;
}

// Kinds of per-row record the streaming pass leaves for the walk.
enum RowKind : uint8_t {
    kRowNone = 0,  // no run: the walk adds the row exactly or from its terms
    kRowRun = 1,   // a run of the whole row under binade `e`
};

struct RowRec {
    uint64_t inc0;  // increment for an even start
    int32_t dinc;   // inc1 - inc0
    uint8_t e;      // binade the run was formed under
    uint8_t kind;   // RowKind
    uint16_t pad;
};

// The binade a row is planned in from the exact sum before it, P: the row
// gets a run when P >= 2^53 and P plus the row's exact sum stays below the
// next power of two; otherwise 0 (no run). Any plan is correct: the walk
// checks each run against the CPU's actual sum and falls back to the terms.
VMX_HD int plan_binade(uint64_t prefix, uint64_t row_sum)
{
    if (prefix < kTwo53) return 0;
    const int e = binade_of(prefix);
    if (e >= 63) return 0;
    if (prefix + row_sum >= (1ull << (e + 1))) return 0;
    return e;
}

}  // namespace vmx
