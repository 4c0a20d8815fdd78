"""A bounded wait of the TMA prefill kernel that runs out is reported as SSM_ERR_TIMEOUT, and the device
stays usable: the next call on the same stream is correct.

The wait limit is set to 0 ns through the C ABI (ssm_set_wait_limit_ns), so that a warp gives up at the
first staged tile it finds not yet arrived; nothing faults, traps or waits without end. The warps that give
up still wait (with the fixed 2 s bound) for the copies they have in flight before they exit. To make sure
some tile is not there yet when its warp first looks, the inputs (270 MB) are larger than L2 and L2 is
flushed right before the call: every warp's first tiles then come from DRAM, behind the requests of all
the other warps.
"""
import numpy as np
import pytest

import ssm_inputs
from gpu_util import dev_inputs
from tolerance import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("disc", ["euler", "zoh"])
def test_wait_that_runs_out_reports_timeout_then_recovers(orc, disc):
    import torch
    import selective_state_space_124_b300 as lib
    from selective_state_space_124_b300 import _ffi
    batch, L, D, N = 1, 65536, 512, 16  # N = 16, 16-byte aligned rows: the TMA-staged kernel
    inp = ssm_inputs.make_inputs(batch, L, D, N, seed=61)
    d = dev_inputs(inp, "f32")
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 18, device="cuda")  # 512 MiB, four times the L2
    lib.check_device()  # nothing pending from earlier tests
    prev = lib.set_wait_limit_ns(0)
    try:
        assert prev == 2_000_000_000
        flush.zero_()
        y, fs = lib.ssm_scan_fwd(d["x"], d["delta"], d["A_log"], d["B"], d["C"], disc=disc)  # enqueues fine
        with pytest.raises(_ffi.SsmError) as err:
            lib.check_device(stream)
        assert err.value.status == _ffi.SSM_ERR_TIMEOUT
        lib.check_device(stream)  # the status word was read and cleared
    finally:
        assert lib.set_wait_limit_ns(prev) == 0
    # the same stream, the default limit: a normal, correct result
    y, fs = lib.ssm_scan_fwd(d["x"], d["delta"], d["A_log"], d["B"], d["C"], disc=disc)
    lib.check_device(stream)
    chans = [0, 63, 64, 200, 511]  # the oracle on a few whole channels (L = 65536 steps each)
    yr, sr = orc.scan_fwd(inp["x"], inp["delta"], inp["A_log"], inp["B"], inp["C"], disc=disc, channels=chans)
    assert rel_err(y[0, :, chans].T.cpu().numpy(), yr) <= TOL["f32"]
    assert rel_err(fs[0, chans].cpu().numpy(), sr) <= TOL["f32"]

