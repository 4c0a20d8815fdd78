"""B300-native selective scan (Mamba): a C-ABI CUDA library for sm_103a and this thin binding.

    y, final_state = ssm_scan_fwd(x, delta, A_log, B, C, disc="euler" | "zoh", h0=None)
    y_t = ssm_scan_step(state, x_t, delta_t, A_log, B_t, C_t, disc=...)   # state updated in place
    grads = ssm_scan_bwd(x, delta, A_log, B, C, dy, disc=..., h0=None, dfinal=None)  # dict of gradients
    y, final_state = ssm_ssd_fwd(x, delta, A_log, B, C, disc=..., h0=None)   # Mamba-2 SSD layer (bf16)

Both take the layer pieces the library can fuse around the scan, each optional: ``delta_bias`` [D] and
``delta_softplus`` (the scan uses softplus(delta + bias)), ``D_skip`` [D] (adds D x to y) and ``z`` (gates
y by SiLU(z); [batch, L, D] for the prefill, ``z_t`` [batch, D] for a step).

Arguments are torch tensors: x, delta [batch, L, D] and B, C [batch, L, N] in float32 or bfloat16
(all four the same), A_log [D, N] float32, states float32. CUDA tensors run on the caller's current
stream. CPU tensors are copied to the current CUDA device (asynchronously when pinned), processed, and
the results copied back. Every arithmetic step runs in the library's kernels; this module only
marshals arguments (see include/ssm_scan.h for the contract).
"""
from __future__ import annotations

from . import _ffi
from ._ffi import SsmError

__all__ = ["ssm_scan_fwd", "ssm_scan_fwd_host", "host_workspace_size", "ssm_scan_step", "ssm_scan_bwd",
           "ssm_scan_fwd_ptr", "ssm_scan_step_ptr",
           "bwd_workspace_size", "ssm_ssd_fwd", "ssd_workspace_size", "check_device", "set_wait_limit_ns", "SsmError",
           "version"]


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return _ffi.DTYPE["f32"]
    if t.dtype == torch.bfloat16:
        return _ffi.DTYPE["bf16"]
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _stream_handle(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes_void(s.cuda_stream)


def ctypes_void(v):
    import ctypes
    return ctypes.c_void_p(v) if v else None


def _ptr(t):
    return None if t is None else ctypes_void(t.data_ptr())


def version() -> int:
    return _ffi.load().ssm_version()


def ssm_scan_fwd_ptr(x, delta, A_log, B, C, h0, y, final_state, batch, L, D, N, dtype, disc, stream):
    """Raw C-ABI call on integer device addresses (0 for NULL); dtype "f32"/"bf16", disc "euler"/"zoh"."""
    v = ctypes_void
    st = _ffi.load().ssm_scan_fwd(v(x), v(delta), v(A_log), v(B), v(C), v(h0), v(y), v(final_state),
                                  batch, L, D, N, _ffi.DTYPE[dtype], _ffi.DISC[disc], v(stream))
    _ffi.check("ssm_scan_fwd", st)


def ssm_scan_step_ptr(state, x_t, delta_t, A_log, B_t, C_t, y_t, batch, D, N, dtype, disc, stream):
    """Raw C-ABI call on integer device addresses."""
    v = ctypes_void
    st = _ffi.load().ssm_scan_step(v(state), v(x_t), v(delta_t), v(A_log), v(B_t), v(C_t), v(y_t),
                                   batch, D, N, _ffi.DTYPE[dtype], _ffi.DISC[disc], v(stream))
    _ffi.check("ssm_scan_step", st)


def _to_device(ts, device):
    return [None if t is None else t.to(device, non_blocking=True) for t in ts]


def _check_extras(name, D, x, delta_bias, D_skip, z, z_shape):
    torch = _torch()
    for nm, t in (("delta_bias", delta_bias), ("D_skip", D_skip)):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != (D,) or not t.is_contiguous()
                              or t.device != x.device):
            raise ValueError(f"{name}: {nm} must be a contiguous float32 [{D}] tensor on the inputs' device")
    if z is not None and (z.dtype != x.dtype or tuple(z.shape) != z_shape or not z.is_contiguous()
                          or z.device != x.device):
        raise ValueError(f"{name}: z must be contiguous, {x.dtype}, shape {z_shape}, on the inputs' device")


def ssm_scan_fwd(x, delta, A_log, B, C, disc: str = "euler", h0=None, *, y=None, final_state=None,
                 want_final_state: bool = True, stream=None, delta_bias=None, delta_softplus: bool = False,
                 D_skip=None, z=None):
    """Prefill selective scan. Returns (y, final_state) (final_state None if not wanted)."""
    torch = _torch()
    if x.device.type == "cpu" and delta_bias is None and D_skip is None and z is None and not delta_softplus:
        return ssm_scan_fwd_host(x, delta, A_log, B, C, disc, h0, y=y, final_state=final_state,
                                 want_final_state=want_final_state, stream=stream)
    if x.device.type == "cpu":
        dev = torch.device("cuda", torch.cuda.current_device())
        xd, dd, ad, bd, cd, hd, bb, ds, zd = _to_device([x, delta, A_log, B, C, h0, delta_bias, D_skip, z], dev)
        yd, fd = ssm_scan_fwd(xd, dd, ad, bd, cd, disc, hd, want_final_state=want_final_state, stream=stream,
                              delta_bias=bb, delta_softplus=delta_softplus, D_skip=ds, z=zd)
        torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
        return yd.cpu(), None if fd is None else fd.cpu()
    batch, L, D = x.shape
    N = A_log.shape[-1]
    code = _dtype_code(x)
    for name, t in (("delta", delta), ("B", B), ("C", C)):
        if t.dtype != x.dtype:
            raise TypeError(f"{name} has dtype {t.dtype}, x has {x.dtype}")
    if A_log.dtype != torch.float32 or (h0 is not None and h0.dtype != torch.float32):
        raise TypeError("A_log and h0 must be float32")
    if tuple(delta.shape) != (batch, L, D) or tuple(B.shape) != (batch, L, N) or tuple(C.shape) != (batch, L, N) \
            or tuple(A_log.shape) != (D, N) or (h0 is not None and tuple(h0.shape) != (batch, D, N)):
        raise ValueError("shape mismatch: x/delta [b,L,D], B/C [b,L,N], A_log [D,N], h0 [b,D,N]")
    ts = [x, delta, A_log, B, C] + ([h0] if h0 is not None else [])
    if any(not t.is_contiguous() for t in ts) or any(t.device != x.device for t in ts):
        raise ValueError("inputs must be contiguous and on one device")
    _check_extras("ssm_scan_fwd", D, x, delta_bias, D_skip, z, (batch, L, D))
    if y is None:
        y = torch.empty((batch, L, D), dtype=x.dtype, device=x.device)
    if final_state is None and want_final_state:
        final_state = torch.empty((batch, D, N), dtype=torch.float32, device=x.device)
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    st = _ffi.load().ssm_scan_fwd_ex(_ptr(x), _ptr(delta), _ptr(A_log), _ptr(B), _ptr(C), _ptr(h0),
                                     _ptr(delta_bias), int(bool(delta_softplus)), _ptr(D_skip), _ptr(z), _ptr(y),
                                     _ptr(final_state), batch, L, D, N, code, _ffi.DISC[disc],
                                     ctypes_void(s.cuda_stream))
    _ffi.check("ssm_scan_fwd", st)
    return y, final_state


HOST_SEGMENT_STEPS = 8192  # default segment of ssm_scan_fwd_host: about 100 MB of fp32 uploads at D = 1536


def host_workspace_size(batch, D, N, dtype="f32", seg_L=HOST_SEGMENT_STEPS):
    """Bytes of device workspace ssm_scan_fwd_host needs (0 for invalid sizes)."""
    return int(_ffi.load().ssm_scan_fwd_host_workspace_size(batch, D, N, _ffi.DTYPE[dtype], seg_L))


def ssm_scan_fwd_host(x, delta, A_log, B, C, disc: str = "euler", h0=None, *, y=None, final_state=None,
                      want_final_state: bool = True, stream=None, seg_L: int = HOST_SEGMENT_STEPS, workspace=None):
    """Prefill on HOST tensors (x, delta, B, C, A_log, h0, and the outputs y, final_state on the CPU), streamed
    through the device segment by segment by ssm_scan_fwd_host: uploads, the scan and downloads overlap when
    the host tensors are pinned. ``workspace``: a device uint8 tensor of host_workspace_size(...) bytes, or
    None to allocate one here. Waits for the stream before returning, so the host outputs are complete."""
    torch = _torch()
    batch, L, D = x.shape
    N = A_log.shape[-1]
    code = _dtype_code(x)
    dname = "bf16" if code == _ffi.DTYPE["bf16"] else "f32"
    for name, t in (("delta", delta), ("B", B), ("C", C)):
        if t.dtype != x.dtype:
            raise TypeError(f"{name} has dtype {t.dtype}, x has {x.dtype}")
    if A_log.dtype != torch.float32 or (h0 is not None and h0.dtype != torch.float32):
        raise TypeError("A_log and h0 must be float32")
    if tuple(delta.shape) != (batch, L, D) or tuple(B.shape) != (batch, L, N) or tuple(C.shape) != (batch, L, N) \
            or tuple(A_log.shape) != (D, N) or (h0 is not None and tuple(h0.shape) != (batch, D, N)):
        raise ValueError("shape mismatch: x/delta [b,L,D], B/C [b,L,N], A_log [D,N], h0 [b,D,N]")
    ts = [x, delta, A_log, B, C] + ([h0] if h0 is not None else [])
    if any(t.device.type != "cpu" or not t.is_contiguous() for t in ts):
        raise ValueError("ssm_scan_fwd_host: inputs must be contiguous CPU tensors")
    if y is None:
        y = torch.empty((batch, L, D), dtype=x.dtype, pin_memory=True)
    if final_state is None and want_final_state:
        final_state = torch.empty((batch, D, N), dtype=torch.float32, pin_memory=True)
    dev = torch.device("cuda", torch.cuda.current_device())
    seg_L = max(1, min(int(seg_L), max(L, 1)))
    need = host_workspace_size(batch, D, N, dname, seg_L)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    st = _ffi.load().ssm_scan_fwd_host(_ptr(x), _ptr(delta), _ptr(A_log), _ptr(B), _ptr(C), _ptr(h0), _ptr(y),
                                       _ptr(final_state), _ptr(workspace), workspace.numel(), seg_L, batch, L, D,
                                       N, code, _ffi.DISC[disc], ctypes_void(s.cuda_stream))
    _ffi.check("ssm_scan_fwd_host", st)
    s.synchronize()
    return y, final_state


def ssm_scan_step(state, x_t, delta_t, A_log, B_t, C_t, disc: str = "euler", *, y_t=None, stream=None,
                  delta_bias=None, delta_softplus: bool = False, D_skip=None, z_t=None):
    """One decode step: updates ``state`` [batch, D, N] in place and returns y_t [batch, D]."""
    torch = _torch()
    batch, D, N = state.shape
    code = _dtype_code(x_t)
    if state.dtype != torch.float32 or A_log.dtype != torch.float32:
        raise TypeError("state and A_log must be float32")
    for name, t in (("delta_t", delta_t), ("B_t", B_t), ("C_t", C_t)):
        if t.dtype != x_t.dtype:
            raise TypeError(f"{name} has dtype {t.dtype}, x_t has {x_t.dtype}")
    if tuple(x_t.shape) != (batch, D) or tuple(delta_t.shape) != (batch, D) or tuple(B_t.shape) != (batch, N) \
            or tuple(C_t.shape) != (batch, N) or tuple(A_log.shape) != (D, N):
        raise ValueError("shape mismatch: state [b,D,N], x_t/delta_t [b,D], B_t/C_t [b,N], A_log [D,N]")
    ts = [state, x_t, delta_t, A_log, B_t, C_t]
    if any(not t.is_contiguous() for t in ts) or any(t.device != state.device for t in ts):
        raise ValueError("inputs must be contiguous and on one device")
    _check_extras("ssm_scan_step", D, x_t, delta_bias, D_skip, z_t, (batch, D))
    if y_t is None:
        y_t = torch.empty((batch, D), dtype=x_t.dtype, device=state.device)
    s = stream if stream is not None else torch.cuda.current_stream(state.device)
    st = _ffi.load().ssm_scan_step_ex(_ptr(state), _ptr(x_t), _ptr(delta_t), _ptr(A_log), _ptr(B_t), _ptr(C_t),
                                      _ptr(delta_bias), int(bool(delta_softplus)), _ptr(D_skip), _ptr(z_t),
                                      _ptr(y_t), batch, D, N, code, _ffi.DISC[disc], ctypes_void(s.cuda_stream))
    _ffi.check("ssm_scan_step", st)
    return y_t


def bwd_workspace_size(batch: int, L: int, D: int, N: int) -> int:
    """Bytes of device workspace ssm_scan_bwd needs for these sizes."""
    return int(_ffi.load().ssm_scan_bwd_workspace_size(batch, L, D, N))


def ssm_scan_bwd(x, delta, A_log, B, C, dy, disc: str = "euler", h0=None, dfinal=None, *, want_dh0: bool = True,
                 workspace=None, stream=None):
    """Gradients of sum(dy * y) + sum(dfinal * final_state) for the prefill scan (CUDA tensors).

    Returns a dict: dx, ddelta [batch, L, D] in x's dtype; dA_log [D, N], dB, dC [batch, L, N] and dh0
    [batch, D, N] (None unless ``want_dh0``) in float32. ``workspace`` (a uint8 CUDA tensor of at least
    ``bwd_workspace_size(...)`` bytes) is allocated here when not given.
    """
    torch = _torch()
    batch, L, D = x.shape
    N = A_log.shape[-1]
    code = _dtype_code(x)
    for name, t in (("delta", delta), ("B", B), ("C", C), ("dy", dy)):
        if t.dtype != x.dtype:
            raise TypeError(f"{name} has dtype {t.dtype}, x has {x.dtype}")
    for name, t in (("A_log", A_log), ("h0", h0), ("dfinal", dfinal)):
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    if tuple(delta.shape) != (batch, L, D) or tuple(dy.shape) != (batch, L, D) or tuple(B.shape) != (batch, L, N) \
            or tuple(C.shape) != (batch, L, N) or tuple(A_log.shape) != (D, N) \
            or any(t is not None and tuple(t.shape) != (batch, D, N) for t in (h0, dfinal)):
        raise ValueError("shape mismatch: x/delta/dy [b,L,D], B/C [b,L,N], A_log [D,N], h0/dfinal [b,D,N]")
    ts = [t for t in (x, delta, A_log, B, C, dy, h0, dfinal) if t is not None]
    if any(not t.is_contiguous() for t in ts) or any(t.device != x.device for t in ts) or x.device.type != "cuda":
        raise ValueError("inputs must be contiguous CUDA tensors on one device")
    dev = x.device
    out = {"dx": torch.empty((batch, L, D), dtype=x.dtype, device=dev),
           "ddelta": torch.empty((batch, L, D), dtype=x.dtype, device=dev),
           "dA_log": torch.empty((D, N), dtype=torch.float32, device=dev),
           "dB": torch.empty((batch, L, N), dtype=torch.float32, device=dev),
           "dC": torch.empty((batch, L, N), dtype=torch.float32, device=dev),
           "dh0": torch.empty((batch, D, N), dtype=torch.float32, device=dev) if want_dh0 else None}
    need = bwd_workspace_size(batch, L, D, N)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    st = _ffi.load().ssm_scan_bwd(_ptr(x), _ptr(delta), _ptr(A_log), _ptr(B), _ptr(C), _ptr(h0), _ptr(dy),
                                  _ptr(dfinal), _ptr(out["dx"]), _ptr(out["ddelta"]), _ptr(out["dA_log"]),
                                  _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dh0"]), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), batch, L, D, N, code,
                                  _ffi.DISC[disc], ctypes_void(s.cuda_stream))
    _ffi.check("ssm_scan_bwd", st)
    return out


def ssd_workspace_size(batch: int, L: int, H: int, P: int, N: int) -> int:
    """Bytes of workspace that let ssm_ssd_fwd scan segments of each sequence in parallel (current device)."""
    return int(_ffi.load().ssm_ssd_fwd_workspace_size(batch, L, H, P, N))


def ssm_ssd_fwd(x, delta, A_log, B, C, disc: str = "euler", h0=None, *, want_final_state: bool = True, stream=None,
                workspace="auto"):
    """Mamba-2 SSD layer (scalar A per head), CUDA tensors: x [batch, L, H, P] bf16, delta [batch, L, H]
    float32, A_log [H] float32, B, C [batch, L, N] bf16, h0 [batch, H, P, N] float32 or None. Returns
    (y [batch, L, H, P] bf16, final_state [batch, H, P, N] float32 or None). ``workspace``: "auto" allocates
    the workspace here (head dimension 64: the chunk-parallel tensor-core path; otherwise segments of long
    sequences), None runs the warp-MMA kernel with one CTA per sequence, or a uint8 CUDA tensor."""
    torch = _torch()
    batch, L, H, P = x.shape
    N = B.shape[-1]
    if x.dtype != torch.bfloat16 or B.dtype != torch.bfloat16 or C.dtype != torch.bfloat16:
        raise TypeError("x, B and C must be bfloat16")
    if delta.dtype != torch.float32 or A_log.dtype != torch.float32 or (h0 is not None and h0.dtype != torch.float32):
        raise TypeError("delta, A_log and h0 must be float32")
    if tuple(delta.shape) != (batch, L, H) or tuple(A_log.shape) != (H,) or tuple(B.shape) != (batch, L, N) \
            or tuple(C.shape) != (batch, L, N) or (h0 is not None and tuple(h0.shape) != (batch, H, P, N)):
        raise ValueError("shape mismatch: x [b,L,H,P], delta [b,L,H], A_log [H], B/C [b,L,N], h0 [b,H,P,N]")
    ts = [t for t in (x, delta, A_log, B, C, h0) if t is not None]
    if any(not t.is_contiguous() for t in ts) or any(t.device != x.device for t in ts) or x.device.type != "cuda":
        raise ValueError("inputs must be contiguous CUDA tensors on one device")
    y = torch.empty((batch, L, H, P), dtype=torch.bfloat16, device=x.device)
    fs = torch.empty((batch, H, P, N), dtype=torch.float32, device=x.device) if want_final_state else None
    if isinstance(workspace, str):
        need = ssd_workspace_size(batch, L, H, P, N)
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device) if need > 0 else None
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    st = _ffi.load().ssm_ssd_fwd(_ptr(x), _ptr(delta), _ptr(A_log), _ptr(B), _ptr(C), _ptr(h0), _ptr(y), _ptr(fs),
                                 _ptr(workspace), wbytes, batch, L, H, P, N, _ffi.DTYPE["bf16"], _ffi.DISC[disc],
                                 ctypes_void(s.cuda_stream))
    _ffi.check("ssm_ssd_fwd", st)
    return y, fs


def set_wait_limit_ns(ns: int) -> int:
    """Bound, in nanoseconds, on one wait of the TMA prefill kernel for a staged tile (default 2 s); a wait
    that runs out makes the next check_device() raise SsmError with status SSM_ERR_TIMEOUT. Returns the
    previous bound."""
    return int(_ffi.load().ssm_set_wait_limit_ns(int(ns)))


def check_device(stream=None) -> None:
    """Synchronise the stream and raise SsmError if a kernel of this library failed on it."""
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    _ffi.check("ssm_check_device", _ffi.load().ssm_check_device(ctypes_void(s.cuda_stream)))
