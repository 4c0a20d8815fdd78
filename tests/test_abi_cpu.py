"""The C-ABI library loads, exports every symbol include/ssm_scan.h declares, and rejects bad
arguments before touching the GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

from selective_state_space_124_b300 import _ffi, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ssm_scan.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssm_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _ffi.load()


def test_every_declared_symbol_is_exported(lib):
    syms = declared_symbols()
    assert "ssm_scan_fwd" in syms and "ssm_scan_step" in syms
    for s in syms:
        assert hasattr(lib, s), f"{s} declared in ssm_scan.h but not exported"
        assert s in _ffi.SIGNATURES, f"{s} has no ctypes signature in the binding"


def test_binding_loads_the_library_the_build_writes():
    assert _ffi.LIB == build.LIB


def test_version_and_status_strings(lib):
    assert lib.ssm_version() >= 100
    for code, name in enumerate(["SSM_OK", "SSM_ERR_INVALID_ARG", "SSM_ERR_UNSUPPORTED", "SSM_ERR_CUDA",
                                 "SSM_ERR_TIMEOUT"]):
        assert lib.ssm_status_string(code).decode() == name


FAKE = 1 << 40  # never dereferenced: every case below fails validation first


def fwd(lib, *, x=FAKE, delta=FAKE + (1 << 30), A_log=FAKE + (2 << 30), B=FAKE + (3 << 30), C=FAKE + (4 << 30),
        h0=None, y=FAKE + (5 << 30), fs=FAKE + (6 << 30), batch=1, L=8, D=4, N=16, dtype=0, disc=0):
    v = lambda p: None if p is None else ctypes.c_void_p(p)
    return lib.ssm_scan_fwd(v(x), v(delta), v(A_log), v(B), v(C), v(h0), v(y), v(fs), batch, L, D, N, dtype,
                            disc, None)


def test_fwd_argument_errors(lib):
    assert fwd(lib, N=17) == _ffi.SSM_ERR_UNSUPPORTED
    assert b"N = 17" in lib.ssm_last_error()
    assert fwd(lib, N=0) == _ffi.SSM_ERR_INVALID_ARG
    assert fwd(lib, L=-1) == _ffi.SSM_ERR_INVALID_ARG
    assert fwd(lib, dtype=7) == _ffi.SSM_ERR_INVALID_ARG
    assert fwd(lib, disc=2) == _ffi.SSM_ERR_INVALID_ARG
    assert fwd(lib, x=None) == _ffi.SSM_ERR_INVALID_ARG
    assert fwd(lib, B=None) == _ffi.SSM_ERR_INVALID_ARG
    assert fwd(lib, A_log=None) == _ffi.SSM_ERR_INVALID_ARG
    assert fwd(lib, y=FAKE + 16) == _ffi.SSM_ERR_INVALID_ARG            # y overlaps x
    assert b"overlap" in lib.ssm_last_error()
    assert fwd(lib, h0=FAKE + (7 << 30), fs=FAKE + (7 << 30) + 8) == _ffi.SSM_ERR_INVALID_ARG  # final overlaps h0
    assert fwd(lib, batch=1 << 40, L=1 << 20, D=1 << 20) == _ffi.SSM_ERR_INVALID_ARG  # size overflow
    assert fwd(lib, batch=0) == _ffi.SSM_OK                            # nothing to do, no GPU touched
    assert fwd(lib, D=0, x=None, y=None) == _ffi.SSM_OK


def test_step_argument_errors(lib):
    v = ctypes.c_void_p
    args = [v(FAKE), v(FAKE + (1 << 30)), v(FAKE + (2 << 30)), v(FAKE + (3 << 30)), v(FAKE + (4 << 30)),
            v(FAKE + (5 << 30)), v(FAKE + (6 << 30))]
    assert lib.ssm_scan_step(*args, 2, 8, 17, 0, 0, None) == _ffi.SSM_ERR_UNSUPPORTED
    assert lib.ssm_scan_step(*args, 2, 8, 16, 3, 0, None) == _ffi.SSM_ERR_INVALID_ARG
    bad = list(args)
    bad[6] = v(FAKE + 4)  # y_t overlaps state
    assert lib.ssm_scan_step(*bad, 2, 8, 16, 0, 0, None) == _ffi.SSM_ERR_INVALID_ARG
    bad = list(args)
    bad[1] = None
    assert lib.ssm_scan_step(*bad, 2, 8, 16, 0, 0, None) == _ffi.SSM_ERR_INVALID_ARG
    assert lib.ssm_scan_step(*args, 0, 8, 16, 0, 0, None) == _ffi.SSM_OK


def bwd(lib, *, ws=FAKE + (20 << 30), ws_bytes=1 << 30, dx=FAKE + (10 << 30), dB=FAKE + (13 << 30),
        dy=FAKE + (8 << 30), batch=2, L=64, D=32, N=16, dtype=0, disc=1, dh0=FAKE + (15 << 30)):
    v = lambda p: None if p is None else ctypes.c_void_p(p)
    ins = [v(FAKE), v(FAKE + (1 << 30)), v(FAKE + (2 << 30)), v(FAKE + (3 << 30)), v(FAKE + (4 << 30)), None, v(dy),
           None]
    outs = [v(dx), v(FAKE + (11 << 30)), v(FAKE + (12 << 30)), v(dB), v(FAKE + (14 << 30)), v(dh0)]
    return lib.ssm_scan_bwd(*ins, *outs, v(ws), ws_bytes, batch, L, D, N, dtype, disc, None)


def test_bwd_workspace_size(lib):
    # one saved state per (batch, chunk of 8 steps followed by another, entry, channel), fp32
    assert lib.ssm_scan_bwd_workspace_size(2, 500, 128, 16) == 2 * (63 - 1) * 16 * 128 * 4
    assert lib.ssm_scan_bwd_workspace_size(1, 8, 64, 16) == 0
    assert lib.ssm_scan_bwd_workspace_size(1, 9, 64, 16) == 1 * 1 * 16 * 64 * 4
    assert lib.ssm_scan_bwd_workspace_size(1, 0, 64, 16) == 0
    assert lib.ssm_scan_bwd_workspace_size(1, 64, 64, 17) == 0  # unsupported N: the call itself rejects it


def test_bwd_argument_errors(lib):
    assert bwd(lib, N=17) == _ffi.SSM_ERR_UNSUPPORTED
    assert bwd(lib, L=-1) == _ffi.SSM_ERR_INVALID_ARG
    assert bwd(lib, dtype=5) == _ffi.SSM_ERR_INVALID_ARG
    assert bwd(lib, dy=None) == _ffi.SSM_ERR_INVALID_ARG
    assert bwd(lib, dB=None) == _ffi.SSM_ERR_INVALID_ARG
    assert bwd(lib, ws=None) == _ffi.SSM_ERR_INVALID_ARG
    assert b"workspace" in lib.ssm_last_error()
    need = lib.ssm_scan_bwd_workspace_size(2, 64, 32, 16)
    assert bwd(lib, ws_bytes=need - 1) == _ffi.SSM_ERR_INVALID_ARG
    assert bwd(lib, dx=FAKE + 64) == _ffi.SSM_ERR_INVALID_ARG                 # dx overlaps x
    assert bwd(lib, dh0=FAKE + (13 << 30) + 4) == _ffi.SSM_ERR_INVALID_ARG    # dh0 overlaps dB
    assert b"each other" in lib.ssm_last_error()
    assert bwd(lib, ws=FAKE + (10 << 30) + 8) == _ffi.SSM_ERR_INVALID_ARG      # workspace overlaps dx
    assert bwd(lib, batch=1 << 40, L=1 << 20, D=1 << 20) == _ffi.SSM_ERR_INVALID_ARG


def ssd(lib, *, x=FAKE, y=FAKE + (6 << 30), ws=None, ws_bytes=0, batch=2, L=256, H=4, P=64, N=128, dtype=1, disc=0,
        final=FAKE + (7 << 30)):
    v = lambda p: None if p is None else ctypes.c_void_p(p)
    return lib.ssm_ssd_fwd(v(x), v(FAKE + (1 << 30)), v(FAKE + (2 << 30)), v(FAKE + (3 << 30)), v(FAKE + (4 << 30)),
                           None, v(y), v(final), v(ws), ws_bytes, batch, L, H, P, N, dtype, disc, None)


def test_ssd_argument_errors(lib):
    assert ssd(lib, dtype=0) == _ffi.SSM_ERR_UNSUPPORTED              # fp32 activations: bf16 only
    assert b"bf16" in lib.ssm_last_error()
    assert ssd(lib, N=96) == _ffi.SSM_ERR_UNSUPPORTED                 # N must be 64 or 128
    assert ssd(lib, P=24) == _ffi.SSM_ERR_UNSUPPORTED                 # P a multiple of 16
    assert ssd(lib, x=FAKE + 8) == _ffi.SSM_ERR_UNSUPPORTED           # 16-byte alignment
    assert ssd(lib, L=-1) == _ffi.SSM_ERR_INVALID_ARG
    assert ssd(lib, disc=3) == _ffi.SSM_ERR_INVALID_ARG
    assert ssd(lib, x=None) == _ffi.SSM_ERR_INVALID_ARG
    assert ssd(lib, y=FAKE + 64) == _ffi.SSM_ERR_INVALID_ARG          # y overlaps x
    assert ssd(lib, final=FAKE + (6 << 30) + 16) == _ffi.SSM_ERR_INVALID_ARG      # final state overlaps y
    assert ssd(lib, ws=FAKE + (1 << 30), ws_bytes=64) == _ffi.SSM_ERR_INVALID_ARG  # workspace overlaps delta
    assert ssd(lib, batch=0) == _ffi.SSM_OK                           # nothing to do, no GPU touched


def test_ssd_workspace_size(lib):
    # P = 64: the tensor-core path's chunk states (fp32), the states entering each chunk (bf16, rounded up to
    # 256 bytes) and one log decay per (batch, chunk of 128 steps, head)
    def tc_bytes(batch, L, H, N):
        nc = (L + 127) // 128
        states = batch * nc * H * 64 * N
        return 2 * ((states * 2 + 255) // 256 * 256) + batch * nc * H * 4  # E and S in bf16, decays fp32
    assert lib.ssm_ssd_fwd_workspace_size(8, 4096, 24, 64, 128) == tc_bytes(8, 4096, 24, 128)
    assert lib.ssm_ssd_fwd_workspace_size(1, 100, 2, 64, 64) == tc_bytes(1, 100, 2, 64)
    assert lib.ssm_ssd_fwd_workspace_size(1, 0, 2, 64, 128) == 0       # nothing to scan
    # other P: segments only where one CTA per sequence (batch x heads x P / 16) leaves SMs idle, each of >= 4
    # chunks of 64 steps
    assert lib.ssm_ssd_fwd_workspace_size(8, 4096, 24, 32, 128) == 0   # 384 CTAs: no split
    assert lib.ssm_ssd_fwd_workspace_size(1, 100, 2, 32, 128) == 0     # 2 chunks: too short to split
    nbytes = lib.ssm_ssd_fwd_workspace_size(1, 1000, 2, 32, 128)       # 4 CTAs, 16 chunks -> 4 segments
    assert nbytes == 1 * 2 * 4 * (32 * 128 + 1) * 4
    assert lib.ssm_ssd_fwd_workspace_size(1, 1000, 2, 64, 96) == 0     # unsupported N


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        _ffi.load(str(tmp_path / "libssm_scan.so"))


def test_wait_limit_round_trip(lib):
    """ssm_set_wait_limit_ns returns the previous bound; the default is 2 s (no GPU work)."""
    prev = lib.ssm_set_wait_limit_ns(123)
    try:
        assert prev == 2_000_000_000
        assert lib.ssm_set_wait_limit_ns(456) == 123
    finally:
        assert lib.ssm_set_wait_limit_ns(prev) == 456


def fwd_host(lib, *, x=FAKE, delta=FAKE + (1 << 30), A_log=FAKE + (2 << 30), B=FAKE + (3 << 30),
             C=FAKE + (4 << 30), h0=None, y=FAKE + (5 << 30), fs=FAKE + (6 << 30), ws=FAKE + (7 << 30),
             ws_bytes=1 << 20, seg_L=4, batch=1, L=8, D=4, N=16, dtype=0, disc=0):
    v = lambda p: None if p is None else ctypes.c_void_p(p)
    return lib.ssm_scan_fwd_host(v(x), v(delta), v(A_log), v(B), v(C), v(h0), v(y), v(fs), v(ws), ws_bytes, seg_L,
                                 batch, L, D, N, dtype, disc, None)


def test_fwd_host_argument_errors(lib):
    """The host-streaming prefill checks its arguments before any copy: sizes, pointers, segment length,
    output ranges and the workspace size."""
    assert fwd_host(lib, seg_L=0) == _ffi.SSM_ERR_INVALID_ARG
    assert b"seg_L" in lib.ssm_last_error()
    assert fwd_host(lib, N=17) == _ffi.SSM_ERR_UNSUPPORTED
    assert fwd_host(lib, x=None) == _ffi.SSM_ERR_INVALID_ARG
    assert fwd_host(lib, y=FAKE + 8) == _ffi.SSM_ERR_INVALID_ARG  # y overlaps x
    need = lib.ssm_scan_fwd_host_workspace_size(1, 4, 16, 0, 4)
    assert fwd_host(lib, ws_bytes=need - 1) == _ffi.SSM_ERR_INVALID_ARG
    assert b"needed" in lib.ssm_last_error()
    assert fwd_host(lib, ws=None) == _ffi.SSM_ERR_INVALID_ARG


def test_fwd_host_workspace_size(lib):
    """Two segment slots of x, delta, B, C and y, two states and A_log, each piece 256-byte aligned."""
    up = lambda v: (v + 255) // 256 * 256
    for batch, D, N, dtype, seg in [(1, 1536, 16, 0, 8192), (2, 100, 4, 1, 37), (3, 5, 1, 0, 1)]:
        es = 2 if dtype == 1 else 4
        sd, sn = batch * seg * D * es, batch * seg * N * es
        want = up(D * N * 4) + 2 * up(batch * D * N * 4) + 2 * (3 * up(sd) + 2 * up(sn))
        assert lib.ssm_scan_fwd_host_workspace_size(batch, D, N, dtype, seg) == want
    assert lib.ssm_scan_fwd_host_workspace_size(1, 4, 16, 0, 0) == 0
    assert lib.ssm_scan_fwd_host_workspace_size(1, 4, 17, 0, 8) == 0


def test_fwd_host_no_steps_copies_the_initial_state(lib):
    """L = 0: the final state is h0 (or zeros), written on the host, with no device work."""
    import numpy as np
    h0 = np.arange(2 * 3 * 4, dtype=np.float32).reshape(2, 3, 4) - 5.0
    fs = np.full_like(h0, 7.0)
    p = lambda a: a.ctypes.data
    assert fwd_host(lib, h0=p(h0), fs=p(fs), batch=2, L=0, D=3, N=4, ws=None, ws_bytes=0) == _ffi.SSM_OK
    assert np.array_equal(fs, h0)
    assert fwd_host(lib, h0=None, fs=p(fs), batch=2, L=0, D=3, N=4, ws=None, ws_bytes=0) == _ffi.SSM_OK
    assert not fs.any()
