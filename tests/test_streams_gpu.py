"""Calls on two streams at once: the library keeps no state between calls except the device status words
(set only when a bounded wait runs out), so a prefill, a decode step, a backward pass (each with its own
workspace) and an SSD layer enqueued on two streams without ordering between them give each stream the
oracle's result for its own inputs."""
import numpy as np
import pytest

import ssm_inputs
from tolerance import TOL, rel_err

pytestmark = pytest.mark.gpu


def test_two_streams_concurrently(orc):
    import torch
    import selective_state_space_124_b300 as lib

    b, L, D, N, disc = 2, 1200, 256, 16, "euler"
    cuda = torch.device("cuda")

    def f32(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(cuda)

    def bf16(bits, shape):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).reshape(shape).to(cuda)

    cases = []
    for seed in (3, 4):
        rng = np.random.default_rng(seed + 50)
        c = dict(scan=ssm_inputs.make_inputs(b, L, D, N, seed=seed), tok=ssm_inputs.token_inputs(b, D, N, seed=seed),
                 dy=rng.standard_normal((b, L, D)).astype(np.float32),
                 ssd=ssm_inputs.make_ssd_inputs(1, 500, 2, 64, 128, seed=seed))
        c["dev"] = {k: f32(c["scan"][k]) for k in ("x", "delta", "A_log", "B", "C")}
        c["tokd"] = {k: f32(c["tok"][k]) for k in ("x", "delta", "B", "C")}
        c["dyd"] = f32(c["dy"])
        q = c["ssd"]
        c["ssdd"] = (bf16(q["x_bits"], (1, 500, 2, 64)), f32(q["delta"]), f32(q["A_log"]),
                     bf16(q["B_bits"], (1, 500, 128)), bf16(q["C_bits"], (1, 500, 128)))
        cases.append(c)
    torch.cuda.synchronize()

    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for c, s in zip(cases, streams):  # enqueue everything; the streams are not ordered against each other
        with torch.cuda.stream(s):
            d = c["dev"]
            c["y"], c["fs"] = lib.ssm_scan_fwd(d["x"], d["delta"], d["A_log"], d["B"], d["C"], disc)
            c["state"] = c["fs"].clone()
            t = c["tokd"]
            c["y_t"] = lib.ssm_scan_step(c["state"], t["x"], t["delta"], d["A_log"], t["B"], t["C"], disc)
            c["grads"] = lib.ssm_scan_bwd(d["x"], d["delta"], d["A_log"], d["B"], d["C"], c["dyd"], disc)
            c["ys"], c["fss"] = lib.ssm_ssd_fwd(*c["ssdd"], disc)
    torch.cuda.synchronize()
    lib.check_device()

    for c in cases:
        s = c["scan"]
        yr, fr = orc.scan_fwd(s["x"], s["delta"], s["A_log"], s["B"], s["C"], disc=disc)
        assert rel_err(c["y"].cpu().numpy(), yr) <= TOL["f32"]
        assert rel_err(c["fs"].cpu().numpy(), fr) <= TOL["f32"]
        t = c["tok"]
        sr, ytr = orc.scan_step(c["fs"].cpu().numpy().astype(np.float64), t["x"], t["delta"], s["A_log"], t["B"],
                                t["C"], disc=disc)
        assert rel_err(c["y_t"].cpu().numpy(), ytr) <= TOL["f32"]
        assert rel_err(c["state"].cpu().numpy(), sr) <= TOL["f32"]
        gr = orc.scan_bwd(s["x"], s["delta"], s["A_log"], s["B"], s["C"], c["dy"], disc=disc)
        for k in ("dx", "ddelta", "dA_log", "dB", "dC", "dh0"):
            assert rel_err(c["grads"][k].cpu().numpy(), gr[k]) <= TOL["f32"], k
        q = c["ssd"]
        ysr, fsr = orc.ssd_fwd(q["x"], q["delta"], q["A_log"], q["B"], q["C"], disc=disc)
        assert rel_err(c["ys"].float().cpu().numpy(), ysr) <= TOL["bf16"]
        assert rel_err(c["fss"].cpu().numpy(), fsr) <= TOL["bf16"]
