"""The timing build (VMX_PHASE_TIMES=1, where the bench's --phase-times split
comes from): outputs still equal to the oracle's, and counters that account
for the call: every item streamed once, look-back and runs only where a
frame can pass 2^55, one walk per frame and part, stamps in order."""

import numpy as np
import pytest
import torch

from exact_reductions_gb300 import _lib, build, synth
from gpu_helpers import run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def timed():
    return _lib.bind(build.build_variant("phase_times", ["VMX_PHASE_TIMES=1"]))


def _read_and_reset(lib):
    c = np.zeros(16, dtype=np.uint64)
    assert lib.vmx_phase_times(c.ctypes.data, 1) == _lib.VMX_OK
    return [int(x) for x in c]


# (workload, frames, whether its frames can pass 2^55: look-back items of
# ceil(32768 / width) rows, else ceil(12288 / width) rows, the defaults)
@pytest.mark.parametrize("key,frames,full", [("T2", 1, True), ("C4", 2, False)])
def test_phase_times_account_for_the_call(monkeypatch, timed, key, frames, full):
    monkeypatch.setattr(_lib, "_lib", timed)
    wl = synth.WORKLOADS[key]
    ref, dis = wl.batch(frames)
    torch.cuda.synchronize()
    _read_and_reset(timed)
    run_and_check(ref, dis, wl.bpc)  # one call, every output against the oracle
    c = _read_and_reset(timed)
    rows = -(-(32768 if full else 12288) // wl.width)
    assert c[11] == frames * -(-wl.height // rows)  # items streamed
    assert c[10] == 3 * frames                      # walks: ref, dis moments and psnr
    assert c[2] > 0 and c[5] > 0 and c[8] > 0
    if full:
        assert c[3] > 0 and c[14] > 0  # look-back, and rows past 2^55 run
    else:
        assert c[3] == 0 and c[4] == 0 and c[14] == 0
    assert c[0] <= c[7] <= c[6] <= c[1]
    assert c[13] <= c[9] <= c[1]
    assert c[12] <= c[8]
    assert c[15] > 0
    assert _read_and_reset(timed)[11] == 0  # cleared
