"""Host logic of multi-GPU benchmark runs, exercised with two gloo ranks on the CPU: every rank scans its
own batch (seed = rank, weak scaling), the job time is the slowest rank's, the value counts all ranks'
units, and no collective touches the data path."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import ssm_inputs
    local = [0.5, 2.0][rank]
    t = bench.job_seconds(local, world, device="cpu")
    v = bench.job_value(1000, 10, world, t)
    inp = ssm_inputs.workload_inputs("tiny", seed=bench.rank_seed(rank))
    out[rank] = (t, v, float(inp["x"].reshape(-1)[0]))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_independent_batches():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    t0, v0, x0 = out[0]
    t1, v1, x1 = out[1]
    assert t0 == t1 == 2.0                      # slowest rank
    assert v0 == v1 == pytest.approx(2 * 1000 * 10 / 2.0)
    assert x0 != x1                             # different seeds: independent batches


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.job_seconds(1.5, 1) == 1.5
    assert bench.job_value(10, 3, 1, 1.5) == 20.0


def test_reference_arm_line(capsys):
    """--impl reference prints the contract's JSON line from the oracle alone (tiny workload)."""
    import json
    import bench
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "elems/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_bench_size_overrides_parse():
    import bench
    a = bench.parse_args(["--workload", "long", "--set", "L=16384", "--set", "batch=2", "--no-extra"])
    assert a.workload == "long" and a.set == ["L=16384", "batch=2"] and a.no_extra


def test_compulsory_byte_and_flop_counts():
    """The roofline numerators, counted by hand for small layers (fp32 and bf16 prefill, decode step,
    backward, SSD)."""
    import bench
    f32 = dict(batch=2, L=3, D=5, N=4, dtype="f32")
    # x, delta, y: 3 * 30 * 4; B, C: 2 * 6 * 4 * 4; A_log 20 * 4; final state 40 * 4
    assert bench.fwd_bytes(f32) == 360 + 192 + 80 + 160
    bf = dict(f32, dtype="bf16")
    assert bench.fwd_bytes(bf) == 180 + 96 + 80 + 160
    # x, delta, dy, dx, ddelta: 5 * 30 * 4; B, C: 2 * 24 * 4; dB, dC: 2 * 24 * 4; A_log, dA_log; dh0
    assert bench.bwd_bytes(f32) == 600 + 192 + 192 + 160 + 160
    step = dict(batch=2, D=5, N=4, dtype="f32")
    # state read + write 2 * 40 * 4; x_t, delta_t, y_t 3 * 10 * 4; B_t, C_t 2 * 8 * 4; A_log 20 * 4
    assert bench.step_bytes(step) == 320 + 120 + 64 + 80
    ssd = dict(batch=1, L=64, H=2, P=16, N=64)
    # x, y: 2 * 2048 * 2; B, C: 2 * 4096 * 2; delta 128 * 4; A_log 2 * 4; final state 2048 * 4
    assert bench.ssd_bytes(ssd) == 8192 + 16384 + 512 + 8 + 8192
    # one chunk of Q = 128 steps (full tiles): C B^T once, 2 Q^2 N; per head 2 Q^2 P + 4 Q N P
    assert bench.ssd_flops(ssd) == 2 * 128 * 128 * 64 + 2 * (2 * 128 * 128 * 16 + 4 * 128 * 64 * 16)
    # one chunk of Q = 64 (the warp-MMA kernel's chunk length)
    assert bench.ssd_flops(ssd, Q=64) == 2 * 64 * 64 * 64 + 2 * (2 * 64 * 64 * 16 + 4 * 64 * 64 * 16)


def test_committed_traffic_matches_the_current_prefill_sources():
    """profiles/ncu_traffic.json was captured on the prefill kernel as it stands (same source hash), so the
    bench line's roofline.traffic is not null; a record for another kernel is not used."""
    import bench
    for name in ("long", "mamba130m", "mamba1p4b"):
        t = bench.ncu_traffic("scan_fwd", name)
        assert t is not None and t > 0, name
    assert bench.ncu_traffic("scan_bwd", "long") is None
    assert bench.ncu_traffic("scan_fwd", "no_such_workload") is None
