"""Parity of the host-streaming prefill (ssm_scan_fwd_host through the C ABI: host arrays, segments uploaded,
scanned and downloaded in turn) with the fp64 oracle: several segment lengths (one segment, a ragged last
segment, single-step segments), batch > 1 (strided host rows), N < 16 and unaligned D (the general kernel per
segment), bf16, ZOH with an initial state, pageable host memory, and a caller stream other than the default."""
import numpy as np
import pytest

import ssm_inputs
from gpu_util import host_values
from tolerance import TOL, rel_err

pytestmark = pytest.mark.gpu


def _host(a, dtype, pin=True):
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(ssm_inputs.bf16_round(a).view(np.int16).copy()).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    return t.pin_memory() if pin else t


CASES = [
    # batch, L, D, N, disc, dtype, seg_L, with h0
    (1, 1000, 128, 16, "euler", "f32", 256, False),   # 4 segments, the last ragged
    (1, 1000, 128, 16, "zoh", "f32", 4096, True),     # one segment
    (3, 777, 70, 8, "zoh", "f32", 100, True),         # strided rows, general kernel, ragged
    (2, 600, 256, 16, "euler", "bf16", 128, False),   # bf16, 5 segments
    (1, 50, 64, 16, "euler", "f32", 1, True),         # single-step segments
]


@pytest.mark.parametrize("case", CASES, ids=[f"b{c[0]}_L{c[1]}_D{c[2]}_N{c[3]}_{c[4]}_{c[5]}_seg{c[6]}"
                                             + ("_h0" if c[7] else "") for c in CASES])
def test_host_prefill_parity(orc, case):
    import selective_state_space_124_b300 as lib
    batch, L, D, N, disc, dtype, seg, with_h0 = case
    inp = ssm_inputs.make_inputs(batch, L, D, N, seed=7 * L + D, dtype=dtype)
    h0 = np.random.default_rng(L).standard_normal((batch, D, N)).astype(np.float32) if with_h0 else None
    hx = {k: _host(inp[k], dtype) for k in ("x", "delta", "B", "C")}
    y, fs = lib.ssm_scan_fwd_host(hx["x"], hx["delta"], _host(inp["A_log"], "f32"), hx["B"], hx["C"], disc=disc,
                                  h0=None if h0 is None else _host(h0, "f32"), seg_L=seg)
    lib.check_device()
    assert y.device.type == "cpu" and fs.device.type == "cpu"
    vals = host_values(inp, dtype)
    yr, sr = orc.scan_fwd(vals["x"], vals["delta"], inp["A_log"], vals["B"], vals["C"], disc=disc, h0=h0)
    assert rel_err(y.float().numpy(), yr) <= TOL[dtype]
    assert rel_err(fs.numpy(), sr) <= TOL[dtype]


def test_host_prefill_pageable_memory_and_side_stream(orc):
    """Pageable host arrays (no overlap, same results) on a caller stream that is not the default one; the
    binding routes CPU tensors given to ssm_scan_fwd through the same entry point."""
    import torch
    import selective_state_space_124_b300 as lib
    batch, L, D, N = 2, 900, 96, 16
    inp = ssm_inputs.make_inputs(batch, L, D, N, seed=77)
    hx = {k: _host(inp[k], "f32", pin=False) for k in ("x", "delta", "B", "C", "A_log")}
    side = torch.cuda.Stream()
    y, fs = lib.ssm_scan_fwd_host(hx["x"], hx["delta"], hx["A_log"], hx["B"], hx["C"], disc="zoh", seg_L=200,
                                  stream=side)
    y2, fs2 = lib.ssm_scan_fwd(hx["x"], hx["delta"], hx["A_log"], hx["B"], hx["C"], disc="zoh")
    lib.check_device()
    yr, sr = orc.scan_fwd(inp["x"], inp["delta"], inp["A_log"], inp["B"], inp["C"], disc="zoh")
    for got_y, got_s in ((y, fs), (y2, fs2)):
        assert rel_err(got_y.numpy(), yr) <= TOL["f32"]
        assert rel_err(got_s.numpy(), sr) <= TOL["f32"]


def test_host_prefill_reuses_one_workspace():
    """Back-to-back calls on one caller-owned workspace: each call is ordered after the previous one's
    copy-out, so the second call's uploads cannot overwrite data the first still reads."""
    import torch
    import selective_state_space_124_b300 as lib
    batch, L, D, N = 1, 3000, 128, 16
    a = ssm_inputs.make_inputs(batch, L, D, N, seed=1)
    b = ssm_inputs.make_inputs(batch, L, D, N, seed=2)
    ws = torch.empty(lib.host_workspace_size(batch, D, N, "f32", 500), dtype=torch.uint8, device="cuda")
    outs = []
    for inp in (a, b, a):
        hx = {k: _host(inp[k], "f32") for k in ("x", "delta", "B", "C", "A_log")}
        outs.append(lib.ssm_scan_fwd_host(hx["x"], hx["delta"], hx["A_log"], hx["B"], hx["C"], seg_L=500,
                                          workspace=ws))
    lib.check_device()
    assert torch.equal(outs[0][0], outs[2][0]) and torch.equal(outs[0][1], outs[2][1])
    assert not torch.equal(outs[0][0], outs[1][0])
