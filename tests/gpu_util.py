"""Helpers for the GPU parity tests: move seeded host inputs to the device and call the library."""
import numpy as np

import ssm_inputs


def torch_mod():
    import torch
    return torch


def dev_inputs(inp, dtype):
    """Host arrays from ssm_inputs -> CUDA tensors (bf16 uploads the rounded bit patterns)."""
    torch = torch_mod()
    out = {}
    for k in ("x", "delta", "B", "C"):
        if dtype == "bf16":
            bits = inp.get(k + "_bits")
            if bits is None:
                bits = ssm_inputs.bf16_round(inp[k])
            out[k] = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(inp[k], np.float32)).cuda()
    out["A_log"] = torch.from_numpy(np.ascontiguousarray(inp["A_log"], np.float32)).cuda()
    return out


def host_values(inp, dtype):
    """The exact values the device reads (bf16 -> their float32 widening)."""
    if dtype != "bf16":
        return {k: np.ascontiguousarray(inp[k], np.float32) for k in ("x", "delta", "B", "C")}
    return {k: ssm_inputs.bf16_to_f32(ssm_inputs.bf16_round(inp[k])).reshape(inp[k].shape)
            for k in ("x", "delta", "B", "C")}


def run_fwd(inp, dtype, disc, h0=None):
    import selective_state_space_124_b300 as lib
    torch = torch_mod()
    d = dev_inputs(inp, dtype)
    h0d = None if h0 is None else torch.from_numpy(np.ascontiguousarray(h0, np.float32)).cuda()
    y, fs = lib.ssm_scan_fwd(d["x"], d["delta"], d["A_log"], d["B"], d["C"], disc=disc, h0=h0d)
    lib.check_device()
    return y.float().cpu().numpy().astype(np.float64), fs.cpu().numpy().astype(np.float64)
