"""Parity of the backward pass (ssm_scan_bwd through the C ABI) with the fp64 oracle's adjoint recurrence:
every gradient, both discretisations, fp32 and bf16 inputs, with and without an initial state and a
gradient on the final state; shapes that cut rows into several pieces (so both carries -- the state from
the left and the adjoint from the right -- are rebuilt), ragged channel counts, N < 16, sequences shorter
than one recomputed chunk, and the full Mamba-130M-shaped layer on sampled channels."""
import numpy as np
import pytest

import ssm_inputs
from gpu_util import dev_inputs, host_values
from tolerance import TOL, rel_err

pytestmark = pytest.mark.gpu

KEYS = ("dx", "ddelta", "dA_log", "dB", "dC", "dh0")


def _dev(a, dtype):
    import torch
    if a is None:
        return None
    if dtype == "bf16":
        return torch.from_numpy(ssm_inputs.bf16_round(a).view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def _f32(a):
    import torch
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def _dy(rng, shape, dtype):
    dy = rng.standard_normal(shape).astype(np.float32)
    if dtype == "bf16":
        dy = ssm_inputs.bf16_to_f32(ssm_inputs.bf16_round(dy)).reshape(shape)
    return dy


def _run(orc, batch, L, D, N, disc, dtype, with_state, seed, mu=-2.0, a_log=None):
    import selective_state_space_124_b300 as lib
    inp = ssm_inputs.make_inputs(batch, L, D, N, seed=seed, dtype=dtype, mu=mu, a_log=a_log)
    rng = np.random.default_rng(seed + 1)
    dy = _dy(rng, (batch, L, D), dtype)
    h0 = rng.standard_normal((batch, D, N)).astype(np.float32) if with_state else None
    dfinal = rng.standard_normal((batch, D, N)).astype(np.float32) if with_state else None
    d = dev_inputs(inp, dtype)
    g = lib.ssm_scan_bwd(d["x"], d["delta"], d["A_log"], d["B"], d["C"], _dev(dy, dtype), disc=disc, h0=_f32(h0),
                         dfinal=_f32(dfinal))
    lib.check_device()
    hv = host_values(inp, dtype)
    ref = orc.scan_bwd(hv["x"], hv["delta"], inp["A_log"], hv["B"], hv["C"], dy, disc=disc, h0=h0, dfinal=dfinal)
    return {k: g[k].float().cpu().numpy() for k in KEYS}, ref


SHAPES = [(2, 500, 128, 16), (1, 3000, 64, 16), (1, 300, 70, 8), (3, 37, 33, 4), (1, 5, 16, 16)]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"b{s[0]}_L{s[1]}_D{s[2]}_N{s[3]}" for s in SHAPES])
@pytest.mark.parametrize("disc", ["euler", "zoh"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("with_state", [False, True], ids=["zero_state", "h0_dfinal"])
def test_bwd_parity(orc, shape, disc, dtype, with_state):
    batch, L, D, N = shape
    got, ref = _run(orc, batch, L, D, N, disc, dtype, with_state, seed=11 * L + D)
    for k in KEYS:
        e = rel_err(got[k], ref[k])
        assert e <= TOL[dtype], f"{k} rel err {e:.3g}"


@pytest.mark.parametrize("disc", ["euler", "zoh"])
def test_bwd_unstructured_A(orc, disc):
    """N = 16 with A_log drawn at random (no A_n = (n + 1) A_0 structure), one structured warp group and one
    not: the per-entry path and the decay-tree path in one launch."""
    batch, L, D, N = 2, 600, 64, 16
    a_log = np.tile(np.log(np.arange(1, N + 1, dtype=np.float32)), (D, 1))
    a_log[32:] = np.random.default_rng(3).uniform(-1.0, 1.5, (D - 32, N)).astype(np.float32)
    got, ref = _run(orc, batch, L, D, N, disc, "f32", True, seed=9, a_log=a_log)
    for k in KEYS:
        e = rel_err(got[k], ref[k])
        assert e <= TOL["f32"], f"{k} rel err {e:.3g}"


def test_bwd_long_memory(orc):
    """Small delta (softplus(N(-5, 0.5)), decays of about 0.99 per step at A = -1): the warm-up walks run
    for hundreds of steps in both directions before the carries are complete."""
    got, ref = _run(orc, 1, 4000, 64, 16, "zoh", "f32", True, seed=5, mu=-5.0)
    for k in KEYS:
        e = rel_err(got[k], ref[k])
        assert e <= TOL["f32"], f"{k} rel err {e:.3g}"


def test_bwd_empty_sequence():
    """L = 0: dh0 is dfinal, dA_log is zero, and there is nothing else."""
    import torch
    import selective_state_space_124_b300 as lib
    batch, D, N = 2, 40, 16
    z = torch.zeros((batch, 0, D), device="cuda")
    zb = torch.zeros((batch, 0, N), device="cuda")
    A = torch.zeros((D, N), device="cuda")
    df = torch.randn((batch, D, N), device="cuda")
    g = lib.ssm_scan_bwd(z, z, A, zb, zb, z, dfinal=df)
    lib.check_device()
    assert torch.equal(g["dh0"], df)
    assert torch.count_nonzero(g["dA_log"]) == 0


def test_bwd_mamba130m_sampled(orc):
    """The Mamba-130M-shaped layer (batch 2, L 2048, D 1536, N 16, fp32, Euler) in one launch; dx, ddelta,
    dh0 and dA_log checked on sampled channels (dA_log rows sum over both batch elements of a channel)."""
    import selective_state_space_124_b300 as lib
    cfg = ssm_inputs.WORKLOADS["mamba130m"]
    batch, L, D, N = cfg["batch"], cfg["L"], cfg["D"], cfg["N"]
    inp = ssm_inputs.workload_inputs("mamba130m")
    rng = np.random.default_rng(77)
    dy = _dy(rng, (batch, L, D), "f32")
    d = dev_inputs(inp, "f32")
    g = lib.ssm_scan_bwd(d["x"], d["delta"], d["A_log"], d["B"], d["C"], _dev(dy, "f32"), disc=cfg["disc"])
    lib.check_device()
    ds = [0, 31, 32, 777, 1535]
    chans = [b * D + dd for dd in ds for b in range(batch)]
    ref = orc.scan_bwd(inp["x"], inp["delta"], inp["A_log"], inp["B"], inp["C"], dy, disc=cfg["disc"],
                       channels=chans, want_bc=False)
    dx, ddt, dh0 = (g[k].cpu().numpy() for k in ("dx", "ddelta", "dh0"))
    dal = g["dA_log"].cpu().numpy()
    for i, c in enumerate(chans):
        b, dd = divmod(c, D)
        for name, got, want in (("dx", dx[b, :, dd], ref["dx"][i]), ("ddelta", ddt[b, :, dd], ref["ddelta"][i]),
                                ("dh0", dh0[b, dd], ref["dh0"][i])):
            e = rel_err(got, want)
            assert e <= TOL["f32"], f"{name} channel {c} rel err {e:.3g}"
    for j, dd in enumerate(ds):
        want = ref["dA_log"][batch * j:batch * (j + 1)].sum(axis=0)
        e = rel_err(dal[dd], want)
        assert e <= TOL["f32"], f"dA_log row {dd} rel err {e:.3g}"


def test_bwd_back_to_back_calls_reuse_outputs(orc):
    """Two backward passes back to back into the same output buffers, through the C ABI (each call zeroes
    dA_log, dB, dC in a kernel that its backward kernel follows as a programmatic dependent launch): the second
    call's sums are its own, and match the oracle."""
    import ctypes
    import torch
    from selective_state_space_124_b300 import _ffi
    batch, L, D, N = 2, 900, 128, 16
    a = ssm_inputs.make_inputs(batch, L, D, N, seed=91)
    b = ssm_inputs.make_inputs(batch, L, D, N, seed=92)
    rng = np.random.default_rng(93)
    dy = [_dy(rng, (batch, L, D), "f32") for _ in range(2)]
    out = {"dx": torch.empty((batch, L, D), device="cuda"), "ddelta": torch.empty((batch, L, D), device="cuda"),
           "dA_log": torch.empty((D, N), device="cuda"), "dB": torch.empty((batch, L, N), device="cuda"),
           "dC": torch.empty((batch, L, N), device="cuda"), "dh0": torch.empty((batch, D, N), device="cuda")}
    lib = _ffi.load()
    need = lib.ssm_scan_bwd_workspace_size(batch, L, D, N)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    v = ctypes.c_void_p
    stream = torch.cuda.current_stream()
    keep = []
    for inp, g in ((a, dy[0]), (b, dy[1])):
        d = dev_inputs(inp, "f32")
        gd = _dev(g, "f32")
        keep.append((d, gd))
        st = lib.ssm_scan_bwd(v(d["x"].data_ptr()), v(d["delta"].data_ptr()), v(d["A_log"].data_ptr()),
                              v(d["B"].data_ptr()), v(d["C"].data_ptr()), None, v(gd.data_ptr()), None,
                              *(v(out[k].data_ptr()) for k in KEYS), v(ws.data_ptr()), ws.numel(), batch, L, D, N,
                              _ffi.DTYPE["f32"], _ffi.DISC["euler"], v(stream.cuda_stream))
        _ffi.check("ssm_scan_bwd", st)
    _ffi.check("ssm_check_device", lib.ssm_check_device(v(stream.cuda_stream)))
    ref = orc.scan_bwd(b["x"], b["delta"], b["A_log"], b["B"], b["C"], dy[1], disc="euler")
    for k in KEYS:
        e = rel_err(out[k].cpu().numpy(), ref[k])
        assert e <= TOL["f32"], f"{k} rel err {e:.3g}"
