"""Parity of the Mamba-2 SSD layer (ssm_ssd_fwd, chunked, tensor-core products) with the fp64 oracle's plain
recurrence: both discretisations, with and without an initial state, sequences that end inside a chunk,
shorter than one chunk and empty, N = 64 and 128, several channel blocks per head, and the full
Mamba-2-130M-shaped layer.

Head dimension 64 with a workspace runs the chunk-parallel tcgen05 path (chunks of 128 steps, TMEM
accumulators, TMA-staged operands); other head dimensions, or no workspace, run the warp-MMA kernel (one CTA
walking each sequence, optionally in segments). Both are checked here, and against each other."""
import numpy as np
import pytest

import ssm_inputs
from tolerance import TOL, rel_err

pytestmark = pytest.mark.gpu


def _bf16(torch, a_bits, shape):
    return torch.from_numpy(a_bits.view(np.int16).copy()).view(torch.bfloat16).reshape(shape).cuda()


def _run(orc, batch, L, H, P, N, disc, with_h0, seed, workspace="auto"):
    import torch
    import selective_state_space_124_b300 as lib
    inp = ssm_inputs.make_ssd_inputs(batch, L, H, P, N, seed=seed)
    h0 = np.random.default_rng(seed + 1).standard_normal((batch, H, P, N)).astype(np.float32) if with_h0 else None
    x = _bf16(torch, inp["x_bits"], (batch, L, H, P))
    B = _bf16(torch, inp["B_bits"], (batch, L, N))
    C = _bf16(torch, inp["C_bits"], (batch, L, N))
    dt = torch.from_numpy(inp["delta"]).cuda()
    A = torch.from_numpy(inp["A_log"]).cuda()
    y, fs = lib.ssm_ssd_fwd(x, dt, A, B, C, disc=disc, h0=None if h0 is None else torch.from_numpy(h0).cuda(),
                            workspace=workspace)
    lib.check_device()
    yr, sr = orc.ssd_fwd(inp["x"], inp["delta"], inp["A_log"], inp["B"], inp["C"], disc=disc, h0=h0)
    return y.float().cpu().numpy(), fs.cpu().numpy(), yr, sr


# P = 64 shapes take the tensor-core path: a last chunk of 104 steps (L 1000), 2 steps (L 130), a sequence
# shorter than one chunk (L 64), an odd head count (the last head pair has one head), exact chunks (L 256)
SHAPES = [(2, 200, 3, 32, 64), (1, 1000, 2, 64, 128), (2, 64, 1, 16, 128), (1, 7, 2, 16, 64), (1, 130, 1, 48, 128),
          (4, 130, 24, 64, 64), (3, 300, 5, 64, 128), (1, 64, 1, 64, 64), (2, 256, 4, 64, 64), (1, 5, 3, 64, 128)]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"b{s[0]}_L{s[1]}_H{s[2]}_P{s[3]}_N{s[4]}" for s in SHAPES])
@pytest.mark.parametrize("disc", ["euler", "zoh"])
@pytest.mark.parametrize("with_h0", [False, True], ids=["zero_state", "h0"])
def test_ssd_parity(orc, shape, disc, with_h0):
    y, fs, yr, sr = _run(orc, *shape, disc, with_h0, seed=sum(shape))
    ey, es = rel_err(y, yr), rel_err(fs, sr)
    assert ey <= TOL["bf16"], f"y rel err {ey:.3g}"
    assert es <= TOL["bf16"], f"final state rel err {es:.3g}"


# with the workspace: the tensor-core path (P = 64) or segments per sequence (each scanned by its own CTAs, then
# fixed up); without it: one CTA per sequence
SEG_SHAPES = [(1, 1000, 2, 64, 128), (1, 700, 1, 16, 64), (2, 2048, 3, 32, 128), (2, 2048, 3, 64, 64)]


@pytest.mark.parametrize("shape", SEG_SHAPES, ids=[f"b{s[0]}_L{s[1]}_H{s[2]}_P{s[3]}_N{s[4]}" for s in SEG_SHAPES])
@pytest.mark.parametrize("disc", ["euler", "zoh"])
@pytest.mark.parametrize("with_h0", [False, True], ids=["zero_state", "h0"])
def test_ssd_segments_match_one_cta_per_sequence(orc, shape, disc, with_h0):
    """With and without the workspace: both against the oracle (a workspace is offered for every such shape)."""
    import selective_state_space_124_b300 as lib
    assert lib.ssd_workspace_size(shape[0], shape[1], shape[2], shape[3], shape[4]) > 0
    for ws in ("auto", None):
        y, fs, yr, sr = _run(orc, *shape, disc, with_h0, seed=sum(shape) + 1, workspace=ws)
        ey, es = rel_err(y, yr), rel_err(fs, sr)
        assert ey <= TOL["bf16"], f"workspace {ws}: y rel err {ey:.3g}"
        assert es <= TOL["bf16"], f"workspace {ws}: final state rel err {es:.3g}"


def test_ssd_empty_sequence():
    import torch
    import selective_state_space_124_b300 as lib
    batch, H, P, N = 2, 3, 16, 64
    h0 = torch.randn((batch, H, P, N), device="cuda")
    y, fs = lib.ssm_ssd_fwd(torch.zeros((batch, 0, H, P), dtype=torch.bfloat16, device="cuda"),
                            torch.zeros((batch, 0, H), device="cuda"), torch.zeros(H, device="cuda"),
                            torch.zeros((batch, 0, N), dtype=torch.bfloat16, device="cuda"),
                            torch.zeros((batch, 0, N), dtype=torch.bfloat16, device="cuda"), h0=h0)
    lib.check_device()
    assert y.numel() == 0 and torch.equal(fs, h0)


def test_ssd_mamba2_130m(orc):
    """The full Mamba-2-130M-shaped layer (batch 2, L 2048, 24 heads x 64, N 128, Euler), every output."""
    cfg = ssm_inputs.SSD_WORKLOADS["mamba2_130m"]
    y, fs, yr, sr = _run(orc, cfg["batch"], cfg["L"], cfg["H"], cfg["P"], cfg["N"], cfg["disc"], False, seed=0)
    ey, es = rel_err(y, yr), rel_err(fs, sr)
    assert ey <= TOL["bf16"], f"y rel err {ey:.3g}"
    assert es <= TOL["bf16"], f"final state rel err {es:.3g}"


def test_ssd_mamba2_2p7b_sampled_heads(orc):
    """The full Mamba-2-2.7B-shaped layer (batch 1, L 8192, 80 heads x 64, N 128) on the GPU; the oracle on
    four heads (first, last, two inside), every step and state entry of those heads. Heads are independent
    given the shared B and C, so the oracle runs on the heads' slices."""
    import torch
    import selective_state_space_124_b300 as lib
    cfg = ssm_inputs.SSD_WORKLOADS["mamba2_2p7b"]
    batch, L, H, P, N = cfg["batch"], cfg["L"], cfg["H"], cfg["P"], cfg["N"]
    inp = ssm_inputs.make_ssd_inputs(batch, L, H, P, N, seed=0)
    x = _bf16(torch, inp["x_bits"], (batch, L, H, P))
    B = _bf16(torch, inp["B_bits"], (batch, L, N))
    C = _bf16(torch, inp["C_bits"], (batch, L, N))
    y, fs = lib.ssm_ssd_fwd(x, torch.from_numpy(inp["delta"]).cuda(), torch.from_numpy(inp["A_log"]).cuda(), B, C,
                            disc=cfg["disc"])
    lib.check_device()
    heads = [0, 29, 51, H - 1]
    yr, sr = orc.ssd_fwd(np.ascontiguousarray(inp["x"][:, :, heads]), np.ascontiguousarray(inp["delta"][:, :, heads]),
                         inp["A_log"][heads], inp["B"], inp["C"], disc=cfg["disc"])
    ey = rel_err(y[:, :, heads].float().cpu().numpy(), yr)
    es = rel_err(fs[:, heads].cpu().numpy(), sr)
    assert ey <= TOL["bf16"], f"y rel err {ey:.3g}"
    assert es <= TOL["bf16"], f"final state rel err {es:.3g}"


def test_ssd_six_heads_per_cta_zoh_h0_sampled_heads(orc):
    """A layer whose three-heads-per-CTA output grid would take several waves (batch 4, L 8192, 12 heads x 64,
    N 64: 1024 CTAs), so the output kernel takes six heads per CTA, here in two full groups; ZOH with an
    initial state. The oracle on two heads, one from each group, every step and state entry."""
    import torch
    import selective_state_space_124_b300 as lib
    batch, L, H, P, N = 4, 8192, 12, 64, 64
    inp = ssm_inputs.make_ssd_inputs(batch, L, H, P, N, seed=6, mu=-3.0, sigma=1.0)
    h0 = np.random.default_rng(66).standard_normal((batch, H, P, N)).astype(np.float32)
    x = _bf16(torch, inp["x_bits"], (batch, L, H, P))
    B = _bf16(torch, inp["B_bits"], (batch, L, N))
    C = _bf16(torch, inp["C_bits"], (batch, L, N))
    y, fs = lib.ssm_ssd_fwd(x, torch.from_numpy(inp["delta"]).cuda(), torch.from_numpy(inp["A_log"]).cuda(), B, C,
                            disc="zoh", h0=torch.from_numpy(h0).cuda())
    lib.check_device()
    heads = [2, 9]
    yr, sr = orc.ssd_fwd(np.ascontiguousarray(inp["x"][:, :, heads]), np.ascontiguousarray(inp["delta"][:, :, heads]),
                         inp["A_log"][heads], inp["B"], inp["C"], disc="zoh",
                         h0=np.ascontiguousarray(h0[:, heads]))
    ey = rel_err(y[:, :, heads].float().cpu().numpy(), yr)
    es = rel_err(fs[:, heads].cpu().numpy(), sr)
    assert ey <= TOL["bf16"], f"y rel err {ey:.3g}"
    assert es <= TOL["bf16"], f"final state rel err {es:.3g}"


def test_ssd_odd_heads_several_waves_sampled_heads(orc):
    """An odd head count at a size whose chunk-state grid takes several waves (batch 1, L 8100: 64 chunks, the
    last of 36 steps; 29 heads x 64, N 128: 960 head-pair CTAs), so the last pair of every chunk has one head.
    The oracle on four heads: the first, an inner one, the last full pair's second head and the unpaired last
    head, every step and state entry."""
    import torch
    import selective_state_space_124_b300 as lib
    batch, L, H, P, N = 1, 8100, 29, 64, 128
    inp = ssm_inputs.make_ssd_inputs(batch, L, H, P, N, seed=29)
    x = _bf16(torch, inp["x_bits"], (batch, L, H, P))
    B = _bf16(torch, inp["B_bits"], (batch, L, N))
    C = _bf16(torch, inp["C_bits"], (batch, L, N))
    y, fs = lib.ssm_ssd_fwd(x, torch.from_numpy(inp["delta"]).cuda(), torch.from_numpy(inp["A_log"]).cuda(), B, C,
                            disc="euler")
    lib.check_device()
    heads = [0, 6, 27, 28]
    yr, sr = orc.ssd_fwd(np.ascontiguousarray(inp["x"][:, :, heads]), np.ascontiguousarray(inp["delta"][:, :, heads]),
                         inp["A_log"][heads], inp["B"], inp["C"], disc="euler")
    ey = rel_err(y[:, :, heads].float().cpu().numpy(), yr)
    es = rel_err(fs[:, heads].cpu().numpy(), sr)
    assert ey <= TOL["bf16"], f"y rel err {ey:.3g}"
    assert es <= TOL["bf16"], f"final state rel err {es:.3g}"


def test_ssd_rejects_unsupported_shapes():
    import torch
    import selective_state_space_124_b300 as lib
    x = torch.zeros((1, 8, 1, 16), dtype=torch.bfloat16, device="cuda")
    Bm = torch.zeros((1, 8, 32), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.SsmError, match="N = 64 or 128"):
        lib.ssm_ssd_fwd(x, torch.zeros((1, 8, 1), device="cuda"), torch.zeros(1, device="cuda"), Bm, Bm)


@pytest.mark.parametrize("disc", ["euler", "zoh"])
def test_ssd_tensor_core_path_matches_warp_mma_path(orc, disc):
    """P = 64: the tcgen05 path (with workspace) and the warp-MMA kernel (without) give the same layer within the
    bf16 tolerance of each other, on a layer of several chunks, heads and batch elements with an initial state."""
    import torch
    import selective_state_space_124_b300 as lib
    batch, L, H, P, N = 2, 700, 6, 64, 128
    inp = ssm_inputs.make_ssd_inputs(batch, L, H, P, N, seed=71)
    h0 = torch.from_numpy(np.random.default_rng(72).standard_normal((batch, H, P, N)).astype(np.float32)).cuda()
    x = _bf16(torch, inp["x_bits"], (batch, L, H, P))
    B = _bf16(torch, inp["B_bits"], (batch, L, N))
    C = _bf16(torch, inp["C_bits"], (batch, L, N))
    dt = torch.from_numpy(inp["delta"]).cuda()
    A = torch.from_numpy(inp["A_log"]).cuda()
    assert lib.ssd_workspace_size(batch, L, H, P, N) > 0
    y1, f1 = lib.ssm_ssd_fwd(x, dt, A, B, C, disc=disc, h0=h0, workspace="auto")
    y2, f2 = lib.ssm_ssd_fwd(x, dt, A, B, C, disc=disc, h0=h0, workspace=None)
    lib.check_device()
    assert rel_err(y1.float().cpu().numpy(), y2.float().cpu().numpy()) <= TOL["bf16"]
    assert rel_err(f1.cpu().numpy(), f2.cpu().numpy()) <= TOL["bf16"]
    yr, sr = orc.ssd_fwd(inp["x"], inp["delta"], inp["A_log"], inp["B"], inp["C"], disc=disc, h0=h0.cpu().numpy())
    assert rel_err(y1.float().cpu().numpy(), yr) <= TOL["bf16"]
    assert rel_err(f1.cpu().numpy(), sr) <= TOL["bf16"]


def test_ssd_back_to_back_calls_share_a_workspace(orc):
    """Two layers run back to back on one stream with one workspace (launches 2 and 3 of each call are
    programmatic dependent launches): each result equals the same call made alone."""
    import torch
    import selective_state_space_124_b300 as lib
    batch, L, H, P, N = 2, 700, 6, 64, 128
    ins = [ssm_inputs.make_ssd_inputs(batch, L, H, P, N, seed=s) for s in (81, 82)]
    dev = [dict(x=_bf16(torch, i["x_bits"], (batch, L, H, P)), B=_bf16(torch, i["B_bits"], (batch, L, N)),
                C=_bf16(torch, i["C_bits"], (batch, L, N)), dt=torch.from_numpy(i["delta"]).cuda(),
                A=torch.from_numpy(i["A_log"]).cuda()) for i in ins]
    ws = torch.empty(lib.ssd_workspace_size(batch, L, H, P, N), dtype=torch.uint8, device="cuda")
    alone = []
    for d in dev:
        alone.append(lib.ssm_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], disc="zoh", workspace=ws))
        torch.cuda.synchronize()
    both = [lib.ssm_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], disc="zoh", workspace=ws) for d in dev]
    lib.check_device()
    for (ya, fa), (yb, fb) in zip(alone, both):
        assert torch.equal(ya, yb) and torch.equal(fa, fb)
