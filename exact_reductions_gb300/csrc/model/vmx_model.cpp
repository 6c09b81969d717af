// vmx_model.cpp -- the library's ordered-sum steps run one after another on
// the CPU, for tests only.
//
// The CUDA kernels form the CPU's second-moment sum of a 16-bit plane in
// steps: exact row sums, a per-row plan from their exact prefix, per-row runs
// built from lane runs (lane_run_fp; 8 terms here, 24 on the device, the
// same algebra) composed in order, and a walk
// that adds each row exactly, by its run, or term by term. This file runs the
// same arithmetic (ordsum.cuh) sequentially so the tests can hold it against
// the CPU oracle without a GPU, with real plans, deliberately wrong plans and
// planted mistakes (VMX_MODEL_MUTATIONS). It is not part of libvmx.
#include <stdint.h>
#include <string.h>

#include <vector>

#include "../ordsum.cuh"

extern "C" {
int vmx_model_mutation = 0;
void vmx_model_set_mutation(int k) { vmx_model_mutation = k; }
}

namespace {

using namespace vmx;

// Terms of the plane in raster order: the binary32 square of each sample.
struct Plane {
    const uint16_t *p;
    int w, h;
    int64_t stride;  // in samples
    uint32_t term(int i, int j) const { return term_of_sample(p[(int64_t)i * stride + j]); }
};

uint64_t lcg(uint64_t &s)
{
    s = s * 6364136223846793005ull + 1442695040888963407ull;
    return s >> 33;
}

// A row's run under last place 2^sh: 256-term segments of 32 lanes of 8
// terms, lanes and segments composed in raster order.
Run row_run(const Plane &pl, int i, int sh, uint64_t exact)
{
    LaneRun row = lane_identity();
    for (int seg = 0; seg < pl.w; seg += 256) {
        LaneRun s = lane_identity();
        for (int lane = 0; lane < 32; ++lane) {
            uint32_t t[8];
            int n = 0;
            for (int k = 0; k < 8; ++k) {
                const int j = seg + lane * 8 + k;
                t[k] = j < pl.w ? pl.term(i, j) : 0u;
                n = 8;
            }
            s = lane_compose(s, lane_run_fp(t, n, sh), sh);
        }
        row = lane_compose(row, s, sh);
    }
    return lane_to_run(row, exact);
}

// Adds terms one by one from any S with the cheapest valid form of the step:
// an exact add while the sum stays at or below 2^53, the binade's run of the
// term while it stays below the next power of two, else the full rounding.
uint64_t apply_terms(uint64_t s, const uint32_t *t, int n, uint64_t *count)
{
    for (int k = 0; k < n; ++k) {
        const uint64_t x = s + t[k];
        if (VMX_MUT(5) || x <= kTwo53) {
            s = x;  // (mutation 5: the fallback adds exactly)
        } else if (s >= kTwo53 && x < (2ull << binade_of(s))) {
            const int sh = binade_of(s) - 52;
            s = apply(run_of_term(t[k], sh), s, sh);
        } else if (VMX_MUT(7) && s >= kTwo53) {
            s = round_to_ulp(x, binade_of(s) - 52);  // crossing rounded at the old place
        } else {
            s = rnd53(x);
        }
    }
    if (count) *count += (uint64_t)n;
    return s;
}

// The same walk step by step with the closed forms of binades 53 and 54
// (closed_form_after) and single-term runs from 55 up.
uint64_t apply_terms_cf(uint64_t s, const uint32_t *t, int n, uint64_t *count)
{
    for (int k = 0; k < n; ++k) {
        const uint64_t x = s + t[k];
        if (VMX_MUT(5) || x <= kTwo53) {
            s = x;
            continue;
        }
        if (s >= kTwo53) {
            const int b = binade_of(s);
            const uint64_t top = 2ull << b;
            uint64_t next;
            if (b <= 54) next = closed_form_after(s, t[k], t[k] & 1u, b);
            else next = apply(run_of_term(t[k], b - 52), s, b - 52);
            if (next < top) {
                s = next;
                continue;
            }
        }
        s = (VMX_MUT(7) && s >= kTwo53) ? round_to_ulp(x, binade_of(s) - 52) : rnd53(x);
    }
    if (count) *count += (uint64_t)n;
    return s;
}

}  // namespace

extern "C" {

// The CPU's second-moment sum through the closed-form route: per row the
// exact sum and the count of odd terms; rows in binades 53 and 54 are added
// in closed form, rows planned in binades from 55 up by their run, all other
// rows term by term. stats as vmx_model_plane_s2.
uint64_t vmx_model_plane_s2_cf(const uint16_t *plane, int w, int h, int64_t stride_samples,
                               uint64_t *stats)
{
    Plane pl{plane, w, h, stride_samples};
    std::vector<uint64_t> rows(h), odd(h);
    std::vector<RowRec> rec(h);
    uint64_t prefix = 0;
    for (int i = 0; i < h; ++i) {
        uint64_t s = 0, c = 0;
        for (int j = 0; j < w; ++j) {
            const uint32_t t = pl.term(i, j);
            s += t;
            c += t & 1u;
        }
        rows[i] = s;
        odd[i] = c;
        memset(&rec[i], 0, sizeof rec[i]);
        const int e = plan_binade(prefix, s);
        if (e >= 55) {
            const Run r = row_run(pl, i, VMX_MUT(4) ? e - 51 : e - 52, s);
            rec[i].inc0 = r.inc[0];
            rec[i].dinc = (int32_t)(r.inc[1] - r.inc[0]);
            rec[i].e = (uint8_t)e;
            rec[i].kind = kRowRun;
        }
        prefix += s;
    }
    uint64_t st[4] = {0, 0, 0, 0};
    uint64_t s = 0;
    std::vector<uint32_t> t(w);
    for (int i = 0; i < h; ++i) {
        const uint64_t r = rows[i];
        if (s + r <= kTwo53 || r == 0) {
            s += r;
            ++st[0];
            continue;
        }
        if (s >= kTwo53) {
            const int b = binade_of(s);
            uint64_t next = 0;
            bool have = false;
            if (b <= 54) {
                next = closed_form_after(s, r, odd[i], b);
                have = true;
            } else if (rec[i].kind == kRowRun && rec[i].e == b) {
                Run run;
                run.inc[0] = rec[i].inc0;
                run.inc[1] = rec[i].inc0 + (uint64_t)(int64_t)rec[i].dinc;
                next = apply(run, s, b - 52);
                have = true;
            }
            if (have && next < (2ull << b)) {
                s = next;
                ++st[1];
                continue;
            }
        }
        for (int j = 0; j < w; ++j) t[j] = pl.term(i, j);
        s = apply_terms_cf(s, t.data(), w, &st[3]);
        ++st[2];
    }
    if (stats) memcpy(stats, st, sizeof st);
    return s;
}

// The CPU's second-moment sum (units) of one 16-bit plane through the
// library's steps. plan: 0 = plan from the exact prefix, 1 = a random binade
// (or none) per row, 2 = no runs at all. stats (may be NULL): [0] rows added
// exactly, [1] rows added by their run, [2] rows walked term by term,
// [3] terms walked.
uint64_t vmx_model_plane_s2(const uint16_t *plane, int w, int h, int64_t stride_samples,
                            int plan, uint64_t seed, uint64_t *stats)
{
    Plane pl{plane, w, h, stride_samples};
    std::vector<uint64_t> rows(h);
    for (int i = 0; i < h; ++i) {
        uint64_t s = 0;
        for (int j = 0; j < w; ++j) s += pl.term(i, j);
        rows[i] = s;
    }
    // Plans and runs.
    std::vector<RowRec> rec(h);
    uint64_t prefix = 0, rng = seed ? seed : 1;
    for (int i = 0; i < h; ++i) {
        int e = 0;
        if (plan == 0) e = plan_binade(prefix, rows[i]);
        else if (plan == 1) {
            const uint64_t r = lcg(rng) % 7;
            e = r == 0 ? 0 : (int)(52 + r);  // none, or 53..58
        }
        memset(&rec[i], 0, sizeof rec[i]);
        if (e) {
            const int sh = VMX_MUT(4) ? e - 51 : e - 52;  // (mutation 4: wrong units)
            const Run r = row_run(pl, i, sh, rows[i]);
            rec[i].inc0 = r.inc[0];
            rec[i].dinc = (int32_t)(r.inc[1] - r.inc[0]);
            rec[i].e = (uint8_t)e;
            rec[i].kind = kRowRun;
        }
        prefix += rows[i];
    }
    // The walk.
    uint64_t st[4] = {0, 0, 0, 0};
    uint64_t s = 0;
    std::vector<uint32_t> t(w);
    for (int i = 0; i < h; ++i) {
        const uint64_t r = rows[i];
        if (s + r <= kTwo53 || r == 0) {
            s += r;
            ++st[0];
            continue;
        }
        if (s >= kTwo53 && rec[i].kind == kRowRun && rec[i].e == binade_of(s)) {
            const int sh = rec[i].e - 52;
            Run run;
            run.inc[0] = rec[i].inc0;
            run.inc[1] = rec[i].inc0 + (uint64_t)(int64_t)rec[i].dinc;
            const uint64_t next = apply(run, s, sh);
            if (next < (2ull << rec[i].e)) {
                s = next;
                ++st[1];
                continue;
            }
        }
        for (int j = 0; j < w; ++j) t[j] = pl.term(i, j);
        s = apply_terms(s, t.data(), w, &st[3]);
        ++st[2];
    }
    if (stats) memcpy(stats, st, sizeof st);
    return s;
}

// S after adding n terms in order from `start` (any term size below 2^58),
// by the same cheapest-valid-step rule the walk's fallback uses.
uint64_t vmx_model_ordered_terms(const uint64_t *terms, int n, uint64_t start)
{
    uint64_t s = start;
    for (int k = 0; k < n; ++k) {
        const uint64_t x = s + terms[k];
        if (VMX_MUT(5) || x <= kTwo53) {
            s = x;
        } else if (s >= kTwo53 && x < (2ull << binade_of(s))) {
            const int sh = binade_of(s) - 52;
            s = apply(run_of_term(terms[k], sh), s, sh);
        } else if (VMX_MUT(7) && s >= kTwo53) {
            s = round_to_ulp(x, binade_of(s) - 52);
        } else {
            s = rnd53(x);
        }
    }
    return s;
}

// Compose the single-term runs of n terms in order under last place 2^sh,
// both as full runs and as compact lane runs (8 at a time), and return the
// full run (out[0..1]) and the compact one converted back (out[2..3]).
void vmx_model_run_of_terms(const uint32_t *t, int n, int sh, uint64_t *out)
{
    Run r = run_identity();
    LaneRun l = lane_identity();
    uint64_t exact = 0;
    for (int k = 0; k < n; ++k) {
        r = compose(r, run_of_term(t[k], sh), sh);
        exact += t[k];
    }
    for (int k = 0; k < n; k += 8) {
        const int m = n - k < 8 ? n - k : 8;
        l = lane_compose(l, lane_run_fp(t + k, m, sh), sh);
    }
    const Run lr = lane_to_run(l, exact);
    out[0] = r.inc[0];
    out[1] = r.inc[1];
    out[2] = lr.inc[0];
    out[3] = lr.inc[1];
}

// One compact lane run over all n terms at once (the device forms its lane
// runs of 24 consecutive terms this way), converted to the full run.
void vmx_model_lane_run(const uint32_t *t, int n, int sh, uint64_t *out)
{
    uint64_t exact = 0;
    for (int k = 0; k < n; ++k) exact += t[k];
    const Run r = lane_to_run(lane_run_fp(t, n, sh), exact);
    out[0] = r.inc[0];
    out[1] = r.inc[1];
}

uint64_t vmx_model_rnd53(uint64_t x) { return rnd53(x); }
uint32_t vmx_model_term(uint32_t p) { return term_of_sample(p); }

}  // extern "C"
