"""Edge cases on the GPU: ragged widths, padded strides, misaligned planes,
one-pixel rows and columns, the widest rows, the largest frames, repeated
calls, and the host-memory entry point. Each compared with the oracle."""

import numpy as np
import pytest
import torch

from exact_reductions_gb300 import api, synth
from gpu_helpers import oracle_frames, run_and_check, same_doubles, to_device, u64

pytestmark = pytest.mark.gpu


def _pair(seed, F, H, S, bpc, mode="uniform", W=None):
    rng = np.random.default_rng(seed)
    refs, diss = [], []
    for _ in range(F):
        r, d = synth.random_plane_pair(rng, W or S, H, bpc, stride_samples=S, mode=mode)
        refs.append(r)
        diss.append(d)
    return np.stack(refs), np.stack(diss)


@pytest.mark.parametrize("bpc", [8, 10, 12, 16])
@pytest.mark.parametrize("W,H", [(1, 1), (1, 37), (37, 1), (7, 5), (255, 3), (257, 9),
                                 (1000, 17), (2049, 11)])
def test_ragged_shapes(W, H, bpc):
    for mode in ("uniform", "extreme"):
        ref, dis = _pair(W * 131 + H + bpc, 2, H, W, bpc, mode)
        run_and_check(ref, dis, bpc)


@pytest.mark.parametrize("bpc", [8, 16])
def test_padded_stride_with_garbage(bpc):
    """Samples past the width are garbage and must not count."""
    W, S, H = 1000, 1024 + 8, 40
    ref, dis = _pair(5, 3, H, S, bpc, W=W)
    run_and_check(ref, dis, bpc, width=W)


@pytest.mark.parametrize("bpc", [8, 16])
def test_misaligned_planes(bpc):
    """Planes 2 or 1 samples past a 16-byte boundary use scalar loads."""
    ref, dis = _pair(6, 2, 64, 640, bpc)
    run_and_check(ref, dis, bpc, misalign=1)


def test_misaligned_past_2_53():
    """The scalar-load path through runs and the walk (16-bit, 2560x1440)."""
    wl = synth.WORKLOADS["T1"]
    ref, dis = wl.batch()
    run_and_check(ref, dis, 16, misalign=1)


@pytest.mark.parametrize("bpc", [9, 11, 13, 14, 15])
def test_other_depths(bpc):
    """Scalers 2^1, 2^3, 2^5, 2^6, 2^7: ragged and packed rows, and a frame
    above 2^21 pixels (the odd-counting instance)."""
    ref, dis = _pair(100 + bpc, 2, 37, 1001, bpc, mode="extreme")
    run_and_check(ref, dis, bpc)
    rng = np.random.default_rng(200 + bpc)
    top = 1 << bpc
    ref = rng.integers(top // 2, top, size=(1, 1100, 2048), dtype=np.uint16)
    dis = rng.integers(0, top, size=(1, 1100, 2048), dtype=np.uint16)
    run_and_check(ref, dis, bpc)


def test_misaligned_past_2_55():
    """The scalar-load path through the look-back, the row runs from binade
    55 up and the general walk (16-bit 4096x2560 near full scale)."""
    wl = synth.WORKLOADS["T2"]
    ref, dis = wl.batch()
    run_and_check(ref, dis, 16, misalign=1)


@pytest.mark.parametrize("bpc", [10, 12])
def test_low_depths_with_container_values_past_the_depth(bpc):
    """Depths up to 12 bits take an exact-square pass while every sample in
    it is below 4096. Container values past the depth (up to 65535) must send
    their passes through the full body: here mixed within rows and across
    rows, and, at 3.7 M pixels, a frame whose rows past 2^53 units (their odd
    terms counted on the exact-square passes) follow overrange rows."""
    rng = np.random.default_rng(40 + bpc)
    top = 1 << bpc
    ref = rng.integers(0, top, size=(2, 64, 3000)).astype(np.uint16)
    dis = rng.integers(0, top, size=(2, 64, 3000)).astype(np.uint16)
    ref[:, ::3, :700] = rng.integers(4096, 65536, size=ref[:, ::3, :700].shape)
    dis[:, 1::3, 1500:1510] = 65535
    for features in (3, 1, 2):
        run_and_check(ref, dis, bpc, features=features)
    H, W = 1440, 2560
    ref = rng.integers(0, top, size=(1, H, W)).astype(np.uint16)
    dis = rng.integers(0, top, size=(1, H, W)).astype(np.uint16)
    ref[:, :1008] = rng.integers(60000, 65536, size=(1, 1008, W))
    _, stats = run_and_check(ref, dis, bpc)
    assert int(stats[1]) > 0  # rows past 2^53 added by a closed form


def test_past_2_55_ragged_last_items():
    """Look-back items of several rows on frames whose height is not a
    multiple of them (4000 wide: 9-row items, 2400 rows leave a 6-row last
    item) past 2^55 units, so that the runs, the look-back and the walk meet
    a short last item of every frame."""
    rng = np.random.default_rng(31)
    ref = rng.integers(60000, 65536, size=(2, 2400, 4000), dtype=np.uint16)
    dis = rng.integers(60000, 65536, size=(2, 2400, 4000), dtype=np.uint16)
    _, stats = run_and_check(ref, dis, 16)
    assert int(stats[1]) > 0  # rows added by a closed form or a run


def test_ragged_width_past_2_53():
    """A width that is not a multiple of 8 (a partial last vector) on a frame
    past 2^53 units: the crossing row walk reads the row's tail by samples."""
    rng = np.random.default_rng(12)
    ref = rng.integers(40000, 65536, size=(2, 1440, 2563), dtype=np.uint16)
    dis = rng.integers(40000, 65536, size=(2, 1440, 2563), dtype=np.uint16)
    run_and_check(ref, dis, 16)


def test_widest_rows_largest_frame():
    """32768-sample rows (2^15 terms, ADR-1499 "Decision" point 1) and a
    2^25-pixel frame past 2^53 units."""
    rng = np.random.default_rng(9)
    ref = rng.integers(30000, 65536, size=(1, 1024, 32768), dtype=np.uint16)
    dis = rng.integers(0, 65536, size=(1, 1024, 32768), dtype=np.uint16)
    run_and_check(ref, dis, 16)


def test_single_column_tall_frame():
    """Width 1: every row is one term; frames of 2^21 + 1 pixels count odd
    terms, in items of 32 one-sample rows."""
    rng = np.random.default_rng(10)
    H = (1 << 21) + 1
    ref = rng.integers(60000, 65536, size=(1, H, 1), dtype=np.uint16)
    dis = rng.integers(0, 65536, size=(1, H, 1), dtype=np.uint16)
    run_and_check(ref, dis, 16)


def test_repeated_calls_identical_and_workspace_reused():
    wl = synth.WORKLOADS["T4"]
    ref, dis = wl.batch()
    r, d = to_device(ref), to_device(dis)
    first = api.frames(r, d, 16, sums=True)
    for _ in range(3):
        again = api.frames(r, d, 16, sums=True, ws=first["_workspace"])
        torch.cuda.synchronize()
        assert torch.equal(again["moments"].view(torch.int64), first["moments"].view(torch.int64))
        assert torch.equal(again["psnr_rows"].view(torch.int64),
                           first["psnr_rows"].view(torch.int64))
        assert torch.equal(again["s2_sums"].view(torch.int64), first["s2_sums"].view(torch.int64))


def test_host_entry_matches_device_entry():
    """vmx_frames_host (host buffers, copies inside the call, chunks of 2)
    gives the device call's outputs, and the PSNR of the oracle's MSE."""
    import oracle
    wl = synth.WORKLOADS["C5a"]
    ref, dis = wl.batch(5)
    host = api.frames_host(ref, dis, 16, features=3, chunk_frames=2, s2_rows=True)
    dev = api.frames(to_device(ref), to_device(dis), 16, s2_rows=True)
    torch.cuda.synchronize()
    assert same_doubles(host["moments"], dev["moments"].cpu().numpy())
    assert np.array_equal(host["psnr_rows"], u64(dev["psnr_rows"]))
    assert np.array_equal(host["s2_rows"], u64(dev["s2_rows"]))
    assert same_doubles(host["mse"], dev["mse"].cpu().numpy())
    want_mse = [w["mse"] for w in oracle_frames(ref, dis, 16, range(5))]
    assert same_doubles(host["mse"], want_mse)
    assert same_doubles(host["psnr"], [oracle.psnr_db(m, 16, 0.0) for m in want_mse])


@pytest.mark.parametrize("chunk", [2, 5])
def test_host_entry_reads_pinned_frames_in_place(chunk):
    """Page-locked host frames are read in place by the kernel (no staging
    copy); the outputs equal the device call's and the pageable call's."""
    wl = synth.WORKLOADS["C5a"]
    ref, dis = wl.batch(5)
    pin_r = torch.from_numpy(ref).pin_memory()
    pin_d = torch.from_numpy(dis).pin_memory()
    assert pin_r.is_pinned() and pin_d.is_pinned()
    pinned = api.frames_host(pin_r.numpy(), pin_d.numpy(), 16, features=3, chunk_frames=chunk,
                             s2_rows=True)
    pageable = api.frames_host(ref, dis, 16, features=3, chunk_frames=chunk, s2_rows=True)
    dev = api.frames(to_device(ref), to_device(dis), 16, s2_rows=True)
    torch.cuda.synchronize()
    for k in ("moments", "mse", "psnr"):
        assert same_doubles(pinned[k], pageable[k]), k
    for k in ("psnr_rows", "s2_rows"):
        assert np.array_equal(pinned[k], pageable[k]), k
    assert same_doubles(pinned["moments"], dev["moments"].cpu().numpy())
    assert np.array_equal(pinned["s2_rows"], u64(dev["s2_rows"]))


def test_graph_replays_match_calls():
    """A captured call replayed on new inputs copied into the same tensors
    gives the plain call's outputs (and the oracle's) every time."""
    wl = synth.WORKLOADS["T1"]
    ref, dis = wl.batch(1)
    rng = np.random.default_rng(11)
    R, D = to_device(ref), to_device(dis)
    fg = api.FrameGraph(R, D, 16, s2_rows=True, sums=True)
    for step in range(3):
        if step:
            ref = rng.integers(40000, 65536, size=ref.shape, dtype=np.uint16)
            R.copy_(torch.from_numpy(ref))
        out = fg.replay()
        plain = api.frames(R, D, 16, s2_rows=True, sums=True)
        torch.cuda.synchronize()
        assert fg.status() == 0
        for k in ("moments", "mse"):
            assert same_doubles(out[k].cpu().numpy(), plain[k].cpu().numpy()), (step, k)
        for k in ("psnr_rows", "s2_rows", "s2_sums", "noise_sums"):
            assert np.array_equal(u64(out[k]), u64(plain[k])), (step, k)
        want = oracle_frames(ref, dis, 16, [0])[0]
        assert same_doubles(out["moments"].cpu().numpy()[0], want["moments"])
        assert np.array_equal(u64(out["s2_sums"])[0], want["s2_sums"])


def test_overlapped_batches_match_calls():
    """Four batches per replay, each kernel launched to overlap the one
    before: every batch's outputs equal a plain call's on its inputs."""
    wl = synth.WORKLOADS["C4"]
    ref, dis = wl.batch(4)
    Rs = [to_device(ref[i:i + 1]) for i in range(4)]
    Ds = [to_device(dis[i:i + 1]) for i in range(4)]
    fg = api.FrameGraph(Rs[0], Ds[0], 16, s2_rows=True, sums=True, depth=4, refs=Rs, diss=Ds)
    for _ in range(2):
        fg.replay()
        torch.cuda.synchronize()
        assert fg.status() == 0
        for i in range(4):
            plain = api.frames(Rs[i], Ds[i], 16, s2_rows=True, sums=True)
            torch.cuda.synchronize()
            got = fg.outs[i]
            for k in ("moments", "mse"):
                assert same_doubles(got[k].cpu().numpy(), plain[k].cpu().numpy()), (i, k)
            for k in ("psnr_rows", "s2_rows", "s2_sums", "noise_sums"):
                assert np.array_equal(u64(got[k]), u64(plain[k])), (i, k)


def test_overlapped_look_back_batches_match_the_oracle():
    """Four one-frame 7680x4320 batches (sums past 2^55: look-back, row runs,
    walks) per replay, each kernel launched to overlap the one before, so
    that several run at once: every batch's outputs equal the oracle's."""
    wl = synth.WORKLOADS["C5c"]
    ref, dis = wl.batch(4)
    Rs = [to_device(ref[i:i + 1]) for i in range(4)]
    Ds = [to_device(dis[i:i + 1]) for i in range(4)]
    fg = api.FrameGraph(Rs[0], Ds[0], 16, s2_rows=True, sums=True, depth=4, refs=Rs, diss=Ds)
    want = oracle_frames(ref, dis, 16, range(4))
    for _ in range(2):
        fg.replay()
        torch.cuda.synchronize()
        assert fg.status() == 0
        for i in range(4):
            got, w = fg.outs[i], want[i]
            assert same_doubles(got["moments"].cpu().numpy()[0], w["moments"]), i
            assert same_doubles(got["mse"].cpu().numpy()[0], w["mse"]), i
            assert np.array_equal(u64(got["s2_rows"])[0], w["s2_rows"]), i
            assert np.array_equal(u64(got["s2_sums"])[0], w["s2_sums"]), i
            assert np.array_equal(u64(got["psnr_rows"])[0], w["psnr_rows"]), i
            assert int(u64(got["noise_sums"])[0]) == w["noise_sum"], i


def test_bounded_wait_gives_up_and_context_stays_usable(monkeypatch):
    """A walk that waits for a block count nothing reaches gives up after the
    poll limit, the call reports VMX_ETIMEOUT, and the next call is exact."""
    from exact_reductions_gb300 import _lib
    wl = synth.WORKLOADS["T1"]
    ref, dis = wl.batch(1)
    R, D = to_device(ref), to_device(dis)
    monkeypatch.setenv("VMX_TEST_SPIN_LIMIT", "2000")
    monkeypatch.setenv("VMX_TEST_WAIT_STALL", "1")
    out = api.frames(R, D, 16)
    torch.cuda.synchronize()
    assert api.workspace_status(out["_workspace"]) == _lib.VMX_ETIMEOUT
    # With no workspace the call waits for the result and returns the status.
    with pytest.raises(_lib.VmxError) as err:
        lib = _lib.load()
        o = torch.empty((1, 4), dtype=torch.float64, device="cuda:0")
        _lib.check(lib.vmx_moment_frames(R.data_ptr(), D.data_ptr(), wl.width, wl.height,
                                         wl.width * 2, 16, 1, o.data_ptr(), None, None, None, 0,
                                         torch.cuda.current_stream().cuda_stream), "stalled")
    assert err.value.status == _lib.VMX_ETIMEOUT
    monkeypatch.delenv("VMX_TEST_WAIT_STALL")
    monkeypatch.delenv("VMX_TEST_SPIN_LIMIT")
    run_and_check(ref, dis, 16)


def test_launch_counter_counts_calls():
    wl = synth.WORKLOADS["C1"]
    ref, dis = wl.batch()
    before = api.kernel_launches()
    run_and_check(ref, dis, 8)
    assert api.kernel_launches() == before + 1


@pytest.mark.parametrize("key,frames", [("C4", 16), ("T2", 1), ("T4", 2)])
def test_grid_larger_than_the_gpu_holds(monkeypatch, key, frames):
    """Forward progress does not rest on the whole grid being resident at
    once: with four times as many CTAs as the GPU holds (most of them start
    only as earlier ones exit, and find no items left), the call comes back
    with status 0 and every output equal to the oracle's. Items go out by
    ticket only, so each item a walk waits for is held by a running warp."""
    monkeypatch.setenv("VMX_TEST_GRID_MULT", "4")
    wl = synth.WORKLOADS[key]
    ref, dis = wl.batch(frames)
    run_and_check(ref, dis, wl.bpc, frames=sorted({0, frames - 1}))
