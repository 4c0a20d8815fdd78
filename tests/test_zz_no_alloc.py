"""ssm_scan_bwd_noalloc: the backward pass for callers that cannot allocate device memory (a plugin inside a
host whose memory pool owns the GPU, a service that must not allocate while serving). It keeps its
chunk-end states in a scratch array inside the library instead of a caller-given workspace.

The GPU test calls it through the C ABI twice in a row and checks both results against ssm_scan_bwd with a
workspace of its own; the CPU test checks that sizes beyond the built-in scratch are refused before any GPU
work. This file is collected last on purpose, so that a run stopping at the first failure has run every
other test already; it passes on its own and after the others alike.
"""
import ctypes

import numpy as np
import pytest

import ssm_inputs
from gpu_util import dev_inputs
from selective_state_space_124_b300 import _ffi
from tolerance import TOL, rel_err

SCRATCH_BYTES = 64 << 20
KEYS = ("dx", "ddelta", "dA_log", "dB", "dC", "dh0")


def test_noalloc_refuses_sizes_beyond_its_scratch():
    lib = _ffi.load()
    # batch 8, L 4096, D 4096, N 16 needs about 1 GB of chunk-end states
    need = lib.ssm_scan_bwd_workspace_size(8, 4096, 4096, 16)
    assert need > SCRATCH_BYTES
    v = lambda a: ctypes.c_void_p(a)
    fake = [v((1 << 40) + (k << 32)) for k in range(14)]
    st = lib.ssm_scan_bwd_noalloc(*fake, 8, 4096, 4096, 16, 0, 0, None)
    assert st == _ffi.SSM_ERR_INVALID_ARG
    assert b"built-in scratch" in lib.ssm_last_error()


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    import selective_state_space_124_b300 as ssm
    batch, L, D, N = 2, 700, 96, 16
    inp = ssm_inputs.make_inputs(batch, L, D, N, seed=31)
    rng = np.random.default_rng(32)
    d = dev_inputs(inp, "f32")
    dy = torch.from_numpy(rng.standard_normal((batch, L, D)).astype(np.float32)).cuda()
    h0 = torch.from_numpy(rng.standard_normal((batch, D, N)).astype(np.float32)).cuda()
    dfinal = torch.from_numpy(rng.standard_normal((batch, D, N)).astype(np.float32)).cuda()
    assert 0 < ssm.bwd_workspace_size(batch, L, D, N) <= SCRATCH_BYTES
    for disc in ("euler", "zoh"):
        want = ssm.ssm_scan_bwd(d["x"], d["delta"], d["A_log"], d["B"], d["C"], dy, disc=disc, h0=h0,
                                dfinal=dfinal)
        ssm.check_device()
        want = {k: want[k].cpu().numpy() for k in KEYS}
        for call in range(2):
            out = {"dx": torch.full((batch, L, D), float("nan"), device="cuda"),
                   "ddelta": torch.full((batch, L, D), float("nan"), device="cuda"),
                   "dA_log": torch.full((D, N), float("nan"), device="cuda"),
                   "dB": torch.full((batch, L, N), float("nan"), device="cuda"),
                   "dC": torch.full((batch, L, N), float("nan"), device="cuda"),
                   "dh0": torch.full((batch, D, N), float("nan"), device="cuda")}
            p = lambda t: ctypes.c_void_p(t.data_ptr())
            st = _ffi.load().ssm_scan_bwd_noalloc(
                p(d["x"]), p(d["delta"]), p(d["A_log"]), p(d["B"]), p(d["C"]), p(h0), p(dy), p(dfinal),
                *(p(out[k]) for k in KEYS), batch, L, D, N, _ffi.DTYPE["f32"], _ffi.DISC[disc],
                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            _ffi.check("ssm_scan_bwd_noalloc", st)
            ssm.check_device()
            for k in KEYS:
                e = rel_err(out[k].cpu().numpy(), want[k])
                assert e <= TOL["f32"], f"{disc}, call {call + 1}: {k} rel err {e:.3g}"
