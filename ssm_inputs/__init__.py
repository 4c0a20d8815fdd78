"""Seeded synthetic inputs for the selective scan.

This module only draws random numbers and converts number formats. It holds none of the scan's
arithmetic, and both the CUDA path's tests/benchmark and the CPU oracle consume exactly the arrays it
returns (bf16 inputs are rounded here once, and both sides read the rounded values).

Recipe (every workload, seed 0 unless stated; numpy PCG64 ``default_rng(seed)``; draws in this order):
  1. x      ~ N(0, 1)                          shape [batch, L, D]   (float32 draw)
  2. z      ~ N(mu, sigma), delta = softplus(z) shape [batch, L, D]   (softplus evaluated in float64, the
                                                result stored as float32 -- delta is an input of the scan)
  3. B      ~ N(0, 1)                          shape [batch, L, N]
  4. C      ~ N(0, 1)                          shape [batch, L, N]
  A_log[d, n] = log(n + 1) for every channel d (so A = -(n + 1)); not random.
  bf16 workloads: x, delta, B, C rounded float32 -> bf16 (round to nearest, ties to even).
Mamba-2 SSD layer (``make_ssd_inputs``; scalar A per head): x ~ N(0, 1) [batch, L, H, P],
  z ~ N(mu, sigma) -> delta = softplus(z) [batch, L, H] (float32), B ~ N(0, 1) [batch, L, N],
  C ~ N(0, 1) [batch, L, N], then A_log[h] = log(u), u ~ U(1, 16) [H] (A between -16 and -1, the range
  Mamba-2 initialises A in); x, B, C rounded to bf16 (the tensor-core operands), delta and A_log fp32.
Decode workload: after A_log, the state [batch, D, N] ~ N(0, 1), then per step (in step order)
  x_t ~ N(0, 1) [batch, D], z_t ~ N(mu, sigma) -> delta_t = softplus(z_t) [batch, D],
  B_t ~ N(0, 1) [batch, N], C_t ~ N(0, 1) [batch, N].
"""
from __future__ import annotations

import math

import numpy as np

# Workloads: shapes and distributions of the selective-scan layers this library is measured on.
WORKLOADS = {
    # tiny fp32 scan: batch 1, L 256, D 16, N 4
    "tiny": dict(batch=1, L=256, D=16, N=4, dtype="f32", disc="euler", mu=-1.0, sigma=0.5),
    # Mamba-130M-shaped layer: batch 2, L 2048, D 1536, N 16, fp32
    "mamba130m": dict(batch=2, L=2048, D=1536, N=16, dtype="f32", disc="euler", mu=-2.0, sigma=1.0),
    # Mamba-1.4B-shaped layer: batch 8, L 4096, D 4096, N 16, bf16 inputs/outputs, fp32 state
    "mamba1p4b": dict(batch=8, L=4096, D=4096, N=16, dtype="bf16", disc="euler", mu=-2.0, sigma=1.0),
    # long sequence, exact ZOH: batch 1, L 131072, D 1536, N 16, fp32
    "long": dict(batch=1, L=131072, D=1536, N=16, dtype="f32", disc="zoh", mu=-4.0, sigma=1.0),
    # recurrent decode: batch 128, D 5120, N 16, fp32 state, 1000 steps
    "decode": dict(batch=128, L=1, D=5120, N=16, dtype="f32", disc="euler", mu=-2.0, sigma=1.0, steps=1000),
}

# Mamba-2 SSD layers: batch, L, heads H, head dimension P, state N (one B/C group), bf16 x/B/C/y.
SSD_WORKLOADS = {
    # Mamba-2-130M-shaped layer: d_inner 1536 = 24 heads x 64, N 128
    "mamba2_130m": dict(batch=2, L=2048, H=24, P=64, N=128, disc="euler", mu=-2.0, sigma=1.0),
    # Mamba-2-2.7B-shaped layer: d_inner 5120 = 80 heads x 64, N 128, one 8192-step sequence
    "mamba2_2p7b": dict(batch=1, L=8192, H=80, P=64, N=128, disc="euler", mu=-2.0, sigma=1.0),
}

_CHUNK = 1 << 24


def bf16_round(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> the float32 values they denote (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _softplus_f32(z: np.ndarray) -> np.ndarray:
    out = np.empty(z.shape, np.float32)
    flat, of = z.reshape(-1), out.reshape(-1)
    for i in range(0, flat.size, _CHUNK):
        of[i:i + _CHUNK] = np.logaddexp(0.0, flat[i:i + _CHUNK].astype(np.float64)).astype(np.float32)
    return out


def _normal(rng, shape, mu=0.0, sigma=1.0) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        a *= np.float32(sigma)
    if mu != 0.0:
        a += np.float32(mu)
    return a


def a_log_s4d(D: int, N: int) -> np.ndarray:
    """A_log[d, n] = log(n + 1) (float32), i.e. A[d, n] = -(n + 1) for every channel."""
    row = np.array([math.log(n + 1) for n in range(N)], dtype=np.float32)
    return np.tile(row, (D, 1))


def make_inputs(batch, L, D, N, seed=0, mu=-2.0, sigma=1.0, dtype="f32", a_log=None, **_):
    """Draw x, delta, B, C per the recipe above. Returns a dict with float32 arrays x, delta, B, C,
    A_log (for bf16 also the uint16 bit patterns under x_bits, delta_bits, B_bits, C_bits, and the
    float32 arrays then hold exactly the bf16 values)."""
    rng = np.random.default_rng(seed)
    x = _normal(rng, (batch, L, D))
    delta = _softplus_f32(_normal(rng, (batch, L, D), mu, sigma))
    B = _normal(rng, (batch, L, N))
    C = _normal(rng, (batch, L, N))
    out = dict(x=x, delta=delta, B=B, C=C,
               A_log=a_log_s4d(D, N) if a_log is None else np.ascontiguousarray(a_log, np.float32))
    if dtype == "bf16":
        for k in ("x", "delta", "B", "C"):
            bits = bf16_round(out[k])
            out[k + "_bits"] = bits
            out[k] = bf16_to_f32(bits).reshape(out[k].shape)
    return out


def workload_inputs(name: str, seed: int = 0, **overrides):
    """Inputs of a named prefill workload (see WORKLOADS), with optional shape overrides."""
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    inp = make_inputs(seed=seed, **cfg)
    inp["cfg"] = cfg
    return inp


def token_inputs(batch, D, N, seed=1, mu=-2.0, sigma=1.0, **_):
    """One decode token's inputs (x_t, delta_t [batch, D]; B_t, C_t [batch, N]), same laws as above."""
    rng = np.random.default_rng(seed)
    x = _normal(rng, (batch, D))
    delta = _softplus_f32(_normal(rng, (batch, D), mu, sigma))
    B = _normal(rng, (batch, N))
    C = _normal(rng, (batch, N))
    return dict(x=x, delta=delta, B=B, C=C)


class DecodeStream:
    """Initial state and per-step inputs of the decode workload, drawn lazily in step order."""

    def __init__(self, batch=128, D=5120, N=16, seed=0, mu=-2.0, sigma=1.0, dtype="f32", **_):
        self.batch, self.D, self.N, self.mu, self.sigma = batch, D, N, mu, sigma
        self.dtype = dtype
        self.rng = np.random.default_rng(seed)
        self.A_log = a_log_s4d(D, N)
        self.state0 = _normal(self.rng, (batch, D, N))

    def next_step(self):
        x = _normal(self.rng, (self.batch, self.D))
        delta = _softplus_f32(_normal(self.rng, (self.batch, self.D), self.mu, self.sigma))
        B = _normal(self.rng, (self.batch, self.N))
        C = _normal(self.rng, (self.batch, self.N))
        return dict(x=x, delta=delta, B=B, C=C)


def make_ssd_inputs(batch, L, H, P, N, seed=0, mu=-2.0, sigma=1.0, **_):
    """Draw an SSD layer's inputs per the recipe above. Returns float32 arrays x, delta, B, C, A_log (x, B,
    C hold exactly bf16 values; their bit patterns under x_bits, B_bits, C_bits)."""
    rng = np.random.default_rng(seed)
    out = dict(x=_normal(rng, (batch, L, H, P)), delta=_softplus_f32(_normal(rng, (batch, L, H), mu, sigma)),
               B=_normal(rng, (batch, L, N)), C=_normal(rng, (batch, L, N)))
    out["A_log"] = np.log(rng.uniform(1.0, 16.0, H)).astype(np.float32)
    for k in ("x", "B", "C"):
        bits = bf16_round(out[k])
        out[k + "_bits"] = bits
        out[k] = bf16_to_f32(bits).reshape(out[k].shape)
    return out
