"""Parity of the CUDA decode step (ssm_scan_step, through the C ABI) with the fp64 oracle."""
import numpy as np
import pytest

import ssm_inputs
from tolerance import TOL, rel_err

pytestmark = pytest.mark.gpu


def _dev(a, dtype):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(ssm_inputs.bf16_round(a).view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def _vals(a, dtype):
    return ssm_inputs.bf16_to_f32(ssm_inputs.bf16_round(a)).reshape(a.shape) if dtype == "bf16" else a


@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 70, 5), (4, 257, 16), (2, 1000, 8), (5, 64, 3)])
@pytest.mark.parametrize("disc", ["euler", "zoh"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_step_shapes(orc, shape, disc, dtype):
    import torch
    import selective_state_space_124_b300 as lib
    batch, D, N = shape
    rng = np.random.default_rng(batch * 1000 + D)
    st = rng.standard_normal((batch, D, N)).astype(np.float32)
    x = rng.standard_normal((batch, D)).astype(np.float32)
    dt = np.log1p(np.exp(rng.normal(-2, 1, (batch, D)))).astype(np.float32)
    B = rng.standard_normal((batch, N)).astype(np.float32)
    C = rng.standard_normal((batch, N)).astype(np.float32)
    A_log = ssm_inputs.a_log_s4d(D, N)
    state = torch.from_numpy(st).cuda()
    y = lib.ssm_scan_step(state, _dev(x, dtype), _dev(dt, dtype), torch.from_numpy(A_log).cuda(),
                          _dev(B, dtype), _dev(C, dtype), disc=disc)
    lib.check_device()
    sr, yr = orc.scan_step(st.astype(np.float64), _vals(x, dtype), _vals(dt, dtype), A_log, _vals(B, dtype),
                           _vals(C, dtype), disc=disc)
    assert rel_err(y.float().cpu().numpy(), yr) <= TOL[dtype]
    assert rel_err(state.cpu().numpy(), sr) <= TOL[dtype]


@pytest.mark.parametrize("disc", ["euler", "zoh"])
def test_step_matches_fwd(orc, disc):
    """A prefill followed by decode steps equals one prefill over the whole sequence."""
    import torch
    import selective_state_space_124_b300 as lib
    from gpu_util import dev_inputs
    batch, L, D, N, k = 2, 64, 96, 16, 40
    inp = ssm_inputs.make_inputs(batch, L, D, N, seed=12)
    d = dev_inputs(inp, "f32")
    y, fs = lib.ssm_scan_fwd(d["x"], d["delta"], d["A_log"], d["B"], d["C"], disc=disc)
    sl = lambda t, a, b_: t[:, a:b_].contiguous()
    _, state = lib.ssm_scan_fwd(sl(d["x"], 0, k), sl(d["delta"], 0, k), d["A_log"], sl(d["B"], 0, k),
                                sl(d["C"], 0, k), disc=disc)
    for t in range(k, L):
        yt = lib.ssm_scan_step(state, d["x"][:, t].contiguous(), d["delta"][:, t].contiguous(), d["A_log"],
                               d["B"][:, t].contiguous(), d["C"][:, t].contiguous(), disc=disc)
        assert rel_err(yt.cpu().numpy(), y[:, t].cpu().numpy()) <= 1e-5
    assert rel_err(state.cpu().numpy(), fs.cpu().numpy()) <= 1e-5


@pytest.mark.slow
def test_workload_decode_1000_steps(orc):
    """batch 128, D 5120, N 16, fp32 state in HBM, 1000 consecutive steps. The oracle carries the whole
    state in fp64 alongside. Every step's y and state are checked on 1,027 sampled channels (the first and
    last channels, the last batch row, and a random spread); steps 1, 100, 200, ..., 1000 are checked on
    every one of the 655,360 channels, y and state."""
    import torch
    import selective_state_space_124_b300 as lib
    cfg = ssm_inputs.WORKLOADS["decode"]
    ds = ssm_inputs.DecodeStream(**cfg)
    batch, D, N = cfg["batch"], cfg["D"], cfg["N"]
    rng = np.random.default_rng(77)
    chans = np.unique(np.concatenate([rng.choice(batch * D, 1024, replace=False), [0, D - 1, batch * D - 1]]))
    b_idx, d_idx = np.divmod(chans, D)
    chans_dev = torch.from_numpy(chans).cuda()
    state = torch.from_numpy(ds.state0).cuda()
    A_log = torch.from_numpy(ds.A_log).cuda()
    ref = ds.state0.astype(np.float64)  # [batch, D, N], the oracle's own state
    full_checks = 0
    for step in range(cfg["steps"]):
        s = ds.next_step()
        y = lib.ssm_scan_step(state, _dev(s["x"], "f32"), _dev(s["delta"], "f32"), A_log, _dev(s["B"], "f32"),
                              _dev(s["C"], "f32"), disc=cfg["disc"])
        ref, yr = orc.scan_step(ref, s["x"], s["delta"], ds.A_log, s["B"], s["C"], disc=cfg["disc"])
        if step == 0 or (step + 1) % 100 == 0:
            yg = y.cpu().numpy()
            sg = state.cpu().numpy()
            ey, es = rel_err(yg, yr), rel_err(sg, ref)
            full_checks += 1
        else:
            yg = y.cpu().numpy()[b_idx, d_idx]
            sg = state.view(batch * D, N)[chans_dev].cpu().numpy()
            ey, es = rel_err(yg, yr[b_idx, d_idx]), rel_err(sg, ref.reshape(batch * D, N)[chans])
        assert ey <= TOL["f32"], f"step {step}: y rel err {ey:.3g}"
        assert es <= TOL["f32"], f"step {step}: state rel err {es:.3g}"
    assert full_checks == 11
    lib.check_device()


@pytest.mark.parametrize("disc", ["euler", "zoh"])
def test_step_misaligned_A_log_and_many_quads(orc, disc):
    """The four-lanes-per-channel kernel over more (channel, quad) items than one grid pass holds, and the
    one-thread-per-channel kernel when A_log is not 16-byte aligned; both against the oracle."""
    import torch
    import selective_state_space_124_b300 as lib
    batch, D, N = 40, 3000, 16   # 480k quads: several trips of the persistent grid, ragged last trip
    rng = np.random.default_rng(51)
    st = rng.standard_normal((batch, D, N)).astype(np.float32)
    x = rng.standard_normal((batch, D)).astype(np.float32)
    dt = np.log1p(np.exp(rng.normal(-2, 1, (batch, D)))).astype(np.float32)
    B = rng.standard_normal((batch, N)).astype(np.float32)
    C = rng.standard_normal((batch, N)).astype(np.float32)
    A_log = ssm_inputs.a_log_s4d(D, N)
    sr, yr = orc.scan_step(st.astype(np.float64), x, dt, A_log, B, C, disc=disc)
    flat = torch.zeros(D * N + 1, device="cuda")
    flat[1:] = torch.from_numpy(A_log).cuda().reshape(-1)
    for A_dev in (torch.from_numpy(A_log).cuda(), flat[1:].view(D, N)):
        state = torch.from_numpy(st).cuda()
        y = lib.ssm_scan_step(state, _dev(x, "f32"), _dev(dt, "f32"), A_dev, _dev(B, "f32"), _dev(C, "f32"), disc=disc)
        lib.check_device()
        assert rel_err(y.cpu().numpy(), yr) <= TOL["f32"]
        assert rel_err(state.cpu().numpy(), sr) <= TOL["f32"]
