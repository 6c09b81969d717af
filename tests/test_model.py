"""The library's ordered-sum steps, run sequentially on the CPU (no GPU).

``libvmx_model.so`` compiles the same header the CUDA kernels use
(``ordsum.cuh``) into a sequential model of the streaming pass and the walk:
exact row sums, a per-row plan, row runs built from 8-term lane runs, and a
walk that adds rows exactly, by their run, or term by term. It must give the
oracle's double on every frame, with real plans and with wrong plans
(ADR-1497 "Decision": any plan, even a wrong one, stays correct), and each
planted mistake of ADR-1497's guard list must break it.
"""

import ctypes

import numpy as np
import pytest

import oracle
from exact import ordered_sum, rnd53, scaled_mean
from exact_reductions_gb300 import build, synth

_model = None


def model():
    global _model
    if _model is None:
        lib = ctypes.CDLL(build.build_model())
        u64, i32, i64, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        lib.vmx_model_plane_s2.argtypes = [vp, i32, i32, i64, i32, u64, vp]
        lib.vmx_model_plane_s2.restype = u64
        lib.vmx_model_plane_s2_cf.argtypes = [vp, i32, i32, i64, vp]
        lib.vmx_model_plane_s2_cf.restype = u64
        lib.vmx_model_ordered_terms.argtypes = [vp, i32, u64]
        lib.vmx_model_ordered_terms.restype = u64
        lib.vmx_model_run_of_terms.argtypes = [vp, i32, i32, vp]
        lib.vmx_model_run_of_terms.restype = None
        lib.vmx_model_lane_run.argtypes = [vp, i32, i32, vp]
        lib.vmx_model_lane_run.restype = None
        lib.vmx_model_set_mutation.argtypes = [i32]
        lib.vmx_model_rnd53.argtypes = [u64]
        lib.vmx_model_rnd53.restype = u64
        lib.vmx_model_term.argtypes = [ctypes.c_uint32]
        lib.vmx_model_term.restype = ctypes.c_uint32
        _model = lib
    return _model


def plane_s2(plane, plan=0, seed=1):
    """plan 0/1/2: real, random or no plans with general runs; 3: the
    closed-form route (binades 53/54 in closed form, runs from 55 up)."""
    plane = np.ascontiguousarray(plane, dtype=np.uint16)
    h, w = plane.shape
    stats = np.zeros(4, dtype=np.uint64)
    if plan == 3:
        s = model().vmx_model_plane_s2_cf(plane.ctypes.data, w, h, w, stats.ctypes.data)
    else:
        s = model().vmx_model_plane_s2(plane.ctypes.data, w, h, w, plan, seed, stats.ctypes.data)
    return int(s), stats


def _frames():
    out = [("T1", *synth.WORKLOADS["T1"].frame(0)),
           ("C4", *synth.WORKLOADS["C4"].frame(0)),
           ("T2", *synth.WORKLOADS["T2"].frame(0)),
           ("T4a", *synth.WORKLOADS["T4"].frame(0)),
           ("T4b", *synth.WORKLOADS["T4"].frame(1)),
           ("C5b0", *synth.WORKLOADS["C5b"].frame(0)),
           ("C5b2", *synth.WORKLOADS["C5b"].frame(2)),
           ("T3", *synth.WORKLOADS["T3"].frame(0)),
           ("C5c", *synth.WORKLOADS["C5c"].frame(0))]
    return out


_FRAMES = None
_SUMS = {}


def frames():
    global _FRAMES
    if _FRAMES is None:
        _FRAMES = _frames()
    return _FRAMES


def oracle_sums(name, ref, dis):
    if name not in _SUMS:
        _SUMS[name] = oracle.moment_sums(ref, dis, 16)
    return _SUMS[name]


def check_frames(plans=(0, 1, 2), names=None):
    """The model's CPU sum of each plane equals the oracle's accumulator,
    exactly, in units."""
    for name, ref, dis in frames():
        if names and name not in names:
            continue
        want = oracle_sums(name, ref, dis)
        for plan in plans:
            for idx, plane in ((2, ref), (3, dis)):
                s, _ = plane_s2(plane, plan=plan, seed=idx + 7)
                assert s == want[idx], f"{name} plane {idx - 2} plan {plan}: {s} != {want[idx]}"


def test_run_semantics_against_rounded_adds():
    """A run's two increments are what the CPU's rounded adds do from an even
    and an odd start inside one binade (ADR-1497 "Decision", second point)."""
    rng = np.random.default_rng(3)
    m = model()
    for trial in range(400):
        sh = int(rng.integers(1, 6))
        e = 52 + sh
        n = int(rng.integers(1, 40))
        kind = trial % 3
        if kind == 0:
            t = rng.integers(0, 2**32, size=n, dtype=np.uint64)
        elif kind == 1:
            t = rng.integers(0, 4096, size=n, dtype=np.uint64) ** 2
        else:
            t = rng.integers(0, 4 << sh, size=n, dtype=np.uint64)
        t32 = t.astype(np.uint32)
        out = np.zeros(4, dtype=np.uint64)
        m.vmx_model_run_of_terms(t32.ctypes.data, n, sh, out.ctypes.data)
        u = 1 << sh
        for p in (0, 1):
            s0 = (1 << e) + (2 * int(rng.integers(0, 2**40)) + p) * u
            s = s0
            for v in t32.tolist():
                s = rnd53(s + v)
            assert s < (2 << e)
            assert int(out[p]) == s - s0, (trial, p)
            assert int(out[2 + p]) == s - s0, (trial, p, "compact")


def test_long_lane_runs_against_rounded_adds():
    """A lane's compact run of 24 consecutive terms (the device's length)
    formed in one pass, for last places 2^3..2^10 (binades 55..62, every
    binade a 16-bit frame can reach): its increments are the CPU's rounded
    adds from an even and an odd start (ADR-1497 "Decision")."""
    rng = np.random.default_rng(8)
    m = model()
    for trial in range(600):
        sh = 3 + trial % 8
        e = 52 + sh
        n = 24 if trial % 4 else int(rng.integers(1, 48))
        kind = trial % 3
        if kind == 0:
            t = rng.integers(0, 2**32, size=n, dtype=np.uint64)
        elif kind == 1:
            t = rng.integers(0, 65536, size=n, dtype=np.uint64)
            t = np.array([m.vmx_model_term(int(p)) for p in t.tolist()], dtype=np.uint64)
        else:
            t = rng.integers(0, 4 << sh, size=n, dtype=np.uint64)
        t32 = t.astype(np.uint32)
        out = np.zeros(2, dtype=np.uint64)
        m.vmx_model_lane_run(t32.ctypes.data, n, sh, out.ctypes.data)
        u = 1 << sh
        for p in (0, 1):
            s0 = (1 << e) + (2 * int(rng.integers(0, 2**40)) + p) * u
            s = s0
            for v in t32.tolist():
                s = rnd53(s + v)
            assert s < (2 << e)
            assert int(out[p]) == s - s0, (trial, n, sh, p)


def test_rnd53_and_terms():
    m = model()
    rng = np.random.default_rng(5)
    for x in rng.integers(0, 2**58, size=20000, dtype=np.uint64).tolist():
        assert m.vmx_model_rnd53(x) == rnd53(x)
    for p in range(0, 65536, 7):
        assert m.vmx_model_term(p) == int(np.float32(p) * np.float32(p))


def test_model_real_plans_match_oracle():
    check_frames(plans=(0,))


def test_model_closed_forms_match_oracle():
    """Binades 53 and 54 in closed form from (row sum, odd count)."""
    check_frames(plans=(3,))


def test_closed_form_residues_of_all_codewords():
    """The fact the closed forms rest on: every binary32 square of a codeword
    is 0, 1 or 4 mod 8, and odd exactly for odd codewords below 4096."""
    from exact import rnd24
    p = np.arange(65536, dtype=np.uint64)
    t = rnd24(p * p)
    assert set((t % 8).tolist()) == {0, 1, 4}
    assert np.array_equal((t & 1) == 1, ((p & 1) == 1) & (p < 4096))


def test_model_wrong_and_no_plans_match_oracle():
    check_frames(plans=(1, 2), names=("T1", "C4", "T4a", "C5b2", "T3"))


def test_model_real_plan_uses_runs():
    """With the real plan almost every row past 2^53 is added by its run."""
    ref, _ = synth.WORKLOADS["C4"].frame(0)
    _, st = plane_s2(ref, plan=0)
    exact, by_run, walked = int(st[0]), int(st[1]), int(st[2])
    assert exact + by_run + walked == ref.shape[0]
    assert by_run > 300 and walked <= 3


def test_model_ordered_terms_psnr_rows():
    ref, dis = synth.WORKLOADS["C5a"].frame(0)
    rows, mse = oracle.psnr(ref, dis, 16)
    d = model().vmx_model_ordered_terms(rows.ctypes.data, rows.size, 0)
    assert d == ordered_sum(rows)
    assert scaled_mean(d, 16, ref.size) == mse


GUARDS = {1: "a tie to the odd value", 2: "the parity ignored",
          3: "the tree composed in reverse", 4: "a run's units under the wrong binade",
          5: "the term-by-term fallback as exact adds", 6: "no rounding at all",
          7: "a binade crossing rounded at the old last place"}


@pytest.mark.parametrize("k", sorted(GUARDS), ids=lambda k: f"break{k}")
def test_planted_break_fails(k):
    """ADR-1497 "Consequences" (guards): each hand-made break of the
    ordered-sum arithmetic makes the model disagree with the oracle."""
    m = model()
    m.vmx_model_set_mutation(k)
    try:
        with pytest.raises(AssertionError):
            check_frames(plans=(0, 2, 3), names=("C4", "T4a", "T4b", "C5b2", "T3", "C5c"))
    finally:
        m.vmx_model_set_mutation(0)
