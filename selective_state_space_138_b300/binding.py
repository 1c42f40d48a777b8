"""ctypes binding of ``libssscan.so`` (C ABI in include/ss_scan.h).

Argument marshalling only: shapes and dtypes are checked, outputs are
allocated with torch when the caller passes none, and the raw device pointers
plus the current CUDA stream are handed to the library. Every step of the
computation runs in the library's CUDA kernels; there is no fallback. If the
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssscan.so")

# names declared in include/ss_scan.h
EXPORTS = ("ss_scan_fwd_bf16", "ss_scan_fwd_f32", "ss_scan_fwd_ex_bf16", "ss_scan_fwd_ex_f32", "ss_state_update_bf16", "ss_state_update_f32",
           "ss_causal_conv1d_bf16", "ss_causal_conv1d_f32", "ss_conv_state_update_bf16",
           "ss_conv_state_update_f32", "ss_scan_bwd_bf16", "ss_scan_bwd_f32", "ss_scan_bwd_workspace_bytes",
           "ss_scan_bwd_noalloc_bf16", "ss_scan_bwd_noalloc_f32", "ss_ssd_fwd_bf16", "ss_ssd_workspace_bytes",
           "ss_scan_fwd_train_bf16", "ss_scan_fwd_train_f32", "ss_scan_bwd_ex_bf16", "ss_scan_bwd_ex_f32",
           "ss_device_faults", "ss_fault_probe", "ss_kernel_binary_version", "ss_last_error", "ss_abi_version")

STATUS = {0: "SS_OK", -1: "SS_ERR_NULL", -2: "SS_ERR_DIM", -3: "SS_ERR_N", -4: "SS_ERR_DEVICE_PTR",
          -5: "SS_ERR_LAUNCH", -6: "SS_ERR_INTERNAL"}
MAX_N = 64
MAX_CONV_K = 8
BWD_NOALLOC_MAX_BYTES = 64 << 20   # SS_BWD_NOALLOC_MAX_BYTES

_lib = None


class SSError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s (%d): %s" % (STATUS.get(status, "?"), status, message))
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("CUDA library %s is missing; build it with "
                           "`python -m selective_state_space_138_b300.build`" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    scan_args = [vp] * 8 + [ci, vp, vp, i64, i64, i64, i64, vp]
    upd_args = [vp] * 9 + [i64, i64, i64, vp]
    for name in ("ss_scan_fwd_bf16", "ss_scan_fwd_f32"):
        getattr(L, name).argtypes = scan_args
        getattr(L, name).restype = ci
    for name in ("ss_scan_fwd_ex_bf16", "ss_scan_fwd_ex_f32"):
        getattr(L, name).argtypes = [vp] * 8 + [ci, vp, vp, ci, vp, vp, i64, i64, i64, i64, vp]
        getattr(L, name).restype = ci
    for name in ("ss_state_update_bf16", "ss_state_update_f32"):
        getattr(L, name).argtypes = upd_args
        getattr(L, name).restype = ci
    for name in ("ss_causal_conv1d_bf16", "ss_causal_conv1d_f32"):
        getattr(L, name).argtypes = [vp, vp, vp, vp, ci, vp, vp, i64, i64, i64, i64, vp]
        getattr(L, name).restype = ci
    for name in ("ss_conv_state_update_bf16", "ss_conv_state_update_f32"):
        getattr(L, name).argtypes = [vp, vp, vp, vp, ci, vp, i64, i64, i64, vp]
        getattr(L, name).restype = ci
    for name in ("ss_scan_bwd_bf16", "ss_scan_bwd_f32"):
        getattr(L, name).argtypes = [vp] * 8 + [ci] + [vp] * 13 + [ctypes.c_size_t, ci] + [i64] * 4 + [vp]
        getattr(L, name).restype = ci
    for name in ("ss_scan_bwd_ex_bf16", "ss_scan_bwd_ex_f32"):
        getattr(L, name).argtypes = [vp] * 8 + [ci, vp, vp, ci] + [vp] * 12 + [ctypes.c_size_t] + [i64] * 4 + [vp]
        getattr(L, name).restype = ci
    for name in ("ss_scan_fwd_train_bf16", "ss_scan_fwd_train_f32"):
        getattr(L, name).argtypes = [vp] * 8 + [ci, vp, vp, vp, vp, ctypes.c_size_t] + [i64] * 4 + [vp]
        getattr(L, name).restype = ci
    for name in ("ss_scan_bwd_noalloc_bf16", "ss_scan_bwd_noalloc_f32"):
        getattr(L, name).argtypes = [vp] * 8 + [ci] + [vp] * 12 + [i64] * 4 + [vp]
        getattr(L, name).restype = ci
    L.ss_ssd_fwd_bf16.argtypes = [vp] * 8 + [ci, vp, vp, vp, vp, ctypes.c_size_t] + [i64] * 6 + [vp]
    L.ss_ssd_fwd_bf16.restype = ci
    L.ss_ssd_workspace_bytes.argtypes = [i64] * 5
    L.ss_ssd_workspace_bytes.restype = ctypes.c_size_t
    L.ss_scan_bwd_workspace_bytes.argtypes = [i64] * 4
    L.ss_scan_bwd_workspace_bytes.restype = ctypes.c_size_t
    L.ss_device_faults.argtypes = [ctypes.POINTER(ctypes.c_uint), ci]
    L.ss_device_faults.restype = ci
    L.ss_fault_probe.argtypes = [vp]
    L.ss_fault_probe.restype = ci
    L.ss_kernel_binary_version.argtypes = [ctypes.POINTER(ctypes.c_int)]
    L.ss_kernel_binary_version.restype = ci
    L.ss_last_error.argtypes = []
    L.ss_last_error.restype = ctypes.c_char_p
    L.ss_abi_version.argtypes = []
    L.ss_abi_version.restype = ci
    _lib = L
    return L


def last_error() -> str:
    return lib().ss_last_error().decode()


FAULT_WAIT_TIMEOUT = 1   # SS_FAULT_WAIT_TIMEOUT


def device_faults(clear: bool = True) -> int:
    """Bit set of device-side faults the kernels recorded (0 = none);
    synchronises the device."""
    v = ctypes.c_uint(0)
    _check(lib().ss_device_faults(ctypes.byref(v), 1 if clear else 0))
    return v.value


def fault_probe(stream=None) -> None:
    """Launch the probe whose one GPU thread waits on a barrier nothing
    completes: its bounded wait gives up after about a second and records
    FAULT_WAIT_TIMEOUT (read it with ``device_faults``); see ``ss_fault_probe``."""
    _check(lib().ss_fault_probe(_stream(stream)))


def abi_version() -> int:
    return lib().ss_abi_version()


def kernel_binary_version() -> int:
    """The architecture the library's kernels were compiled for, as the CUDA
    runtime reports it for the module loaded on the current device (103 for
    sm_103a); needs a GPU."""
    v = ctypes.c_int(0)
    _check(lib().ss_kernel_binary_version(ctypes.byref(v)))
    return v.value


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int):
    if status != 0:
        raise SSError(status, last_error())


def _need(t, name, dtype, shape):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError("%s: dtype %s, expected %s" % (name, t.dtype, dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s: shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _io_suffix(dtype):
    if dtype == torch.bfloat16:
        return "bf16"
    if dtype == torch.float32:
        return "f32"
    raise TypeError("io dtype must be bfloat16 or float32, got %s" % dtype)


def scan_fwd(x, delta, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True,
             y=None, final_state=None, return_final_state=True, stream=None):
    """Selective scan over (batch, d_inner, L) inputs; see ``ss_scan_fwd_*``.

    x, delta, z: (batch, d_inner, L); B, C: (batch, N, L) in the io dtype
    (bf16 or fp32); A: (d_inner, N), D, dt_bias: (d_inner,) fp32.
    Returns (y, final_state); final_state is None unless requested.
    """
    io = x.dtype
    sfx = _io_suffix(io)
    batch, d_inner, L = x.shape
    N = A.shape[1] if A.dim() == 2 else -1
    _need(x, "x", io, (batch, d_inner, L))
    _need(delta, "delta", io, (batch, d_inner, L))
    _need(z, "z", io, (batch, d_inner, L))
    _need(B, "B", io, (batch, N, L))
    _need(C, "C", io, (batch, N, L))
    _need(A, "A", torch.float32, (d_inner, N))
    _need(D, "D", torch.float32, (d_inner,))
    _need(dt_bias, "dt_bias", torch.float32, (d_inner,))
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", io, (batch, d_inner, L))
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, d_inner, N), dtype=torch.float32, device=x.device)
    _need(final_state, "final_state", torch.float32, (batch, d_inner, N))
    fn = getattr(lib(), "ss_scan_fwd_" + sfx)
    _check(fn(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias),
              int(bool(delta_softplus)), _ptr(y), _ptr(final_state), batch, d_inner, L, N,
              _stream(stream)))
    return y, final_state


def scan_fwd_ex(x, delta, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True, h0=None, seq_start=None,
                reverse=False, y=None, final_state=None, return_final_state=True, stream=None):
    """``scan_fwd`` with an initial state h0 (batch, d_inner, N) fp32, sequence
    starts seq_start (batch, L) bool/uint8 and/or the reverse direction; see
    ``ss_scan_fwd_ex_*``. Returns (y, final_state)."""
    io = x.dtype
    sfx = _io_suffix(io)
    batch, d_inner, L = x.shape
    N = A.shape[1] if A.dim() == 2 else -1
    for t, n, dt_, shp in ((delta, "delta", io, x.shape), (z, "z", io, x.shape), (B, "B", io, (batch, N, L)),
                           (C, "C", io, (batch, N, L)), (A, "A", torch.float32, (d_inner, N)),
                           (D, "D", torch.float32, (d_inner,)), (dt_bias, "dt_bias", torch.float32, (d_inner,)),
                           (h0, "h0", torch.float32, (batch, d_inner, N))):
        _need(t, n, dt_, shp)
    if seq_start is not None:
        if seq_start.dtype == torch.bool:
            seq_start = seq_start.to(torch.uint8)
        _need(seq_start, "seq_start", torch.uint8, (batch, L))
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", io, x.shape)
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, d_inner, N), dtype=torch.float32, device=x.device)
    _need(final_state, "final_state", torch.float32, (batch, d_inner, N))
    fn = getattr(lib(), "ss_scan_fwd_ex_" + sfx)
    _check(fn(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias),
              int(bool(delta_softplus)), _ptr(h0), _ptr(seq_start), int(bool(reverse)), _ptr(y),
              _ptr(final_state), batch, d_inner, L, N, _stream(stream)))
    return y, final_state


def state_update(state, x, delta, A, B, C, D=None, z=None, y=None, stream=None):
    """One decode step on ``state`` (batch, d_inner, N) fp32, updated in place;
    see ``ss_state_update_*``. x, delta, z: (batch, d_inner); B, C: (batch, N).
    Returns y (batch, d_inner)."""
    io = x.dtype
    sfx = _io_suffix(io)
    batch, d_inner = x.shape
    N = A.shape[1] if A.dim() == 2 else -1
    _need(state, "state", torch.float32, (batch, d_inner, N))
    _need(delta, "delta", io, (batch, d_inner))
    _need(z, "z", io, (batch, d_inner))
    _need(B, "B", io, (batch, N))
    _need(C, "C", io, (batch, N))
    _need(A, "A", torch.float32, (d_inner, N))
    _need(D, "D", torch.float32, (d_inner,))
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", io, (batch, d_inner))
    fn = getattr(lib(), "ss_state_update_" + sfx)
    _check(fn(_ptr(state), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(y),
              batch, d_inner, N, _stream(stream)))
    return y


def causal_conv1d(x, w, bias=None, state_in=None, silu=True, out=None, state_out=None, return_state=False,
                  stream=None):
    """Causal depthwise convolution (+ SiLU) of the Mamba block; see
    ``ss_causal_conv1d_*``. x: (batch, d_inner, L) bf16/fp32; w: (d_inner, k)
    fp32; bias: (d_inner,) fp32; state_in / state_out: (batch, k-1, d_inner)
    in the io dtype, oldest first. Returns (out, state_out)."""
    io = x.dtype
    sfx = _io_suffix(io)
    batch, d_inner, L = x.shape
    k = w.shape[1] if w.dim() == 2 else -1
    _need(x, "x", io, (batch, d_inner, L))
    _need(w, "w", torch.float32, (d_inner, k))
    _need(bias, "bias", torch.float32, (d_inner,))
    _need(state_in, "state_in", io, (batch, k - 1, d_inner))
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", io, (batch, d_inner, L))
    if state_out is None and return_state and k > 1:
        state_out = torch.empty((batch, k - 1, d_inner), dtype=io, device=x.device)
    _need(state_out, "state_out", io, (batch, k - 1, d_inner))
    fn = getattr(lib(), "ss_causal_conv1d_" + sfx)
    _check(fn(_ptr(x), _ptr(w), _ptr(bias), _ptr(state_in), int(bool(silu)), _ptr(out), _ptr(state_out),
              batch, d_inner, L, k, _stream(stream)))
    return out, state_out


def conv_state_update(conv_state, x, w, bias=None, silu=True, out=None, stream=None):
    """One decode step of the convolution; ``conv_state`` (batch, k-1, d_inner)
    is updated in place; see ``ss_conv_state_update_*``. Returns out
    (batch, d_inner)."""
    io = x.dtype
    sfx = _io_suffix(io)
    batch, d_inner = x.shape
    k = w.shape[1] if w.dim() == 2 else -1
    _need(w, "w", torch.float32, (d_inner, k))
    _need(bias, "bias", torch.float32, (d_inner,))
    _need(conv_state, "conv_state", io, (batch, k - 1, d_inner))
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", io, (batch, d_inner))
    fn = getattr(lib(), "ss_conv_state_update_" + sfx)
    _check(fn(_ptr(conv_state), _ptr(x), _ptr(w), _ptr(bias), int(bool(silu)), _ptr(out), batch, d_inner, k,
              _stream(stream)))
    return out


def scan_bwd_workspace_bytes(batch, d_inner, L, N) -> int:
    """Bytes of device scratch ``scan_bwd`` needs (0 for unsupported sizes)."""
    return int(lib().ss_scan_bwd_workspace_bytes(batch, d_inner, L, N))


def scan_fwd_train(x, delta, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True, h0=None, y=None,
                   final_state=None, workspace=None, stream=None):
    """``scan_fwd`` that also stores the backward pass's states in
    ``workspace`` (allocated when None); see ``ss_scan_fwd_train_*``. Returns
    (y, final_state, workspace); hand the workspace to ``scan_bwd`` with
    states_from_forward=True."""
    io = x.dtype
    sfx = _io_suffix(io)
    batch, d_inner, L = x.shape
    N = A.shape[1] if A.dim() == 2 else -1
    for t, n, dt_, shp in ((delta, "delta", io, x.shape), (z, "z", io, x.shape), (B, "B", io, (batch, N, L)),
                           (C, "C", io, (batch, N, L)), (A, "A", torch.float32, (d_inner, N)),
                           (D, "D", torch.float32, (d_inner,)), (dt_bias, "dt_bias", torch.float32, (d_inner,)),
                           (h0, "h0", torch.float32, (batch, d_inner, N))):
        _need(t, n, dt_, shp)
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", io, x.shape)
    if final_state is None:
        final_state = torch.empty((batch, d_inner, N), dtype=torch.float32, device=x.device)
    _need(final_state, "final_state", torch.float32, (batch, d_inner, N))
    if workspace is None:
        workspace = torch.empty(max(scan_bwd_workspace_bytes(batch, d_inner, L, N), 16), dtype=torch.uint8,
                                device=x.device)
    fn = getattr(lib(), "ss_scan_fwd_train_" + sfx)
    _check(fn(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias),
              int(bool(delta_softplus)), _ptr(h0), _ptr(y), _ptr(final_state), _ptr(workspace),
              workspace.numel() * workspace.element_size(), batch, d_inner, L, N, _stream(stream)))
    return y, final_state, workspace


def scan_bwd(x, delta, A, B, C, dout, D=None, z=None, dt_bias=None, delta_softplus=True, h0=None,
             dfinal_state=None, grads=None, workspace=None, stream=None, noalloc=False, states_from_forward=False,
             seq_start=None, reverse=False):
    """Gradient of ``scan_fwd`` (see ``ss_scan_bwd_*``), or with ``seq_start``
    (batch, L) bool/uint8 and/or ``reverse`` of ``scan_fwd_ex`` (see
    ``ss_scan_bwd_ex_*``; not with ``noalloc`` or ``states_from_forward``): the forward inputs,
    dout (batch, d_inner, L) in the io dtype and optionally dfinal_state
    (batch, d_inner, N) fp32. ``grads`` may hold preallocated outputs under the
    names below; missing ones are allocated. ``workspace`` is a uint8 device
    tensor of at least ``scan_bwd_workspace_bytes`` bytes (allocated when None).
    With ``noalloc`` the library's built-in scratch is used instead
    (``ss_scan_bwd_noalloc_*``; problems needing more than
    BWD_NOALLOC_MAX_BYTES are rejected).

    Returns a dict: dx, ddelta, dz (io dtype; dz None without z), dA, dB, dC,
    dD, ddt_bias, dh0 (fp32; dD / ddt_bias None without D / dt_bias, dh0 None
    without h0)."""
    io = x.dtype
    sfx = _io_suffix(io)
    batch, d_inner, L = x.shape
    N = A.shape[1] if A.dim() == 2 else -1
    for t, n, dt_, shp in ((delta, "delta", io, x.shape), (z, "z", io, x.shape), (dout, "dout", io, x.shape),
                           (B, "B", io, (batch, N, L)), (C, "C", io, (batch, N, L)),
                           (A, "A", torch.float32, (d_inner, N)), (D, "D", torch.float32, (d_inner,)),
                           (dt_bias, "dt_bias", torch.float32, (d_inner,)),
                           (h0, "h0", torch.float32, (batch, d_inner, N)),
                           (dfinal_state, "dfinal_state", torch.float32, (batch, d_inner, N))):
        _need(t, n, dt_, shp)
    g = dict(grads or {})
    dev = x.device
    shapes = {"dx": (io, x.shape), "ddelta": (io, x.shape), "dA": (torch.float32, (d_inner, N)),
              "dB": (torch.float32, (batch, N, L)), "dC": (torch.float32, (batch, N, L))}
    if z is not None:
        shapes["dz"] = (io, x.shape)
    if D is not None:
        shapes["dD"] = (torch.float32, (d_inner,))
    if dt_bias is not None:
        shapes["ddt_bias"] = (torch.float32, (d_inner,))
    if h0 is not None:
        shapes["dh0"] = (torch.float32, (batch, d_inner, N))
    for k, (dt_, shp) in shapes.items():
        if g.get(k) is None:
            g[k] = torch.empty(shp, dtype=dt_, device=dev)
        _need(g[k], k, dt_, shp)
    ex = seq_start is not None or bool(reverse)
    if ex and (noalloc or states_from_forward):
        raise ValueError("sequence starts and the reverse direction take the workspace form without "
                         "states_from_forward")
    if seq_start is not None:
        if seq_start.dtype == torch.bool:
            seq_start = seq_start.to(torch.uint8)
        _need(seq_start, "seq_start", torch.uint8, (batch, L))
    if noalloc:
        fn = getattr(lib(), "ss_scan_bwd_noalloc_" + sfx)
        _check(fn(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias),
                  int(bool(delta_softplus)), _ptr(h0), _ptr(dout), _ptr(dfinal_state), _ptr(g["dx"]),
                  _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g.get("dD")),
                  _ptr(g.get("dz")), _ptr(g.get("ddt_bias")), _ptr(g.get("dh0")), batch, d_inner, L, N,
                  _stream(stream)))
        return {k: g.get(k) for k in ("dx", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddt_bias", "dh0")}
    need = scan_bwd_workspace_bytes(batch, d_inner, L, N)
    if workspace is None:
        if states_from_forward:
            raise ValueError("states_from_forward needs the workspace that scan_fwd_train filled")
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if ex:
        fn = getattr(lib(), "ss_scan_bwd_ex_" + sfx)
        _check(fn(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias),
                  int(bool(delta_softplus)), _ptr(h0), _ptr(seq_start), int(bool(reverse)), _ptr(dout),
                  _ptr(dfinal_state), _ptr(g["dx"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]),
                  _ptr(g.get("dD")), _ptr(g.get("dz")), _ptr(g.get("ddt_bias")), _ptr(g.get("dh0")),
                  _ptr(workspace), workspace.numel() * workspace.element_size(), batch, d_inner, L, N,
                  _stream(stream)))
        return {k: g.get(k) for k in ("dx", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddt_bias", "dh0")}
    fn = getattr(lib(), "ss_scan_bwd_" + sfx)
    _check(fn(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias),
              int(bool(delta_softplus)), _ptr(h0), _ptr(dout), _ptr(dfinal_state), _ptr(g["dx"]),
              _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g.get("dD")),
              _ptr(g.get("dz")), _ptr(g.get("ddt_bias")), _ptr(g.get("dh0")), _ptr(workspace),
              workspace.numel() * workspace.element_size(), int(bool(states_from_forward)), batch, d_inner, L, N,
              _stream(stream)))
    return {k: g.get(k) for k in ("dx", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddt_bias", "dh0")}


def ssd_workspace_bytes(batch, L, nheads, ngroups, N) -> int:
    return int(lib().ss_ssd_workspace_bytes(batch, L, nheads, ngroups, N))


def ssd_fwd(x, dt, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True, h0=None, y=None, final_state=None,
            return_final_state=True, workspace=None, stream=None):
    """Mamba-2's scalar-decay scan; see ``ss_ssd_fwd_bf16``. x, z: (batch, L,
    H, P) bf16; dt (batch, L, H) bf16; B, C (batch, L, G, N) bf16; A, D,
    dt_bias (H,) fp32; h0 (batch, H, P, N) fp32. Returns (y, final_state)."""
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be bfloat16")
    batch, L, H, P = x.shape
    G, N = (B.shape[2], B.shape[3]) if B.dim() == 4 else (-1, -1)
    for t, n, dt_, shp in ((dt, "dt", torch.bfloat16, (batch, L, H)), (z, "z", torch.bfloat16, x.shape),
                           (B, "B", torch.bfloat16, (batch, L, G, N)), (C, "C", torch.bfloat16, (batch, L, G, N)),
                           (A, "A", torch.float32, (H,)), (D, "D", torch.float32, (H,)),
                           (dt_bias, "dt_bias", torch.float32, (H,)), (h0, "h0", torch.float32, (batch, H, P, N))):
        _need(t, n, dt_, shp)
    _need(x, "x", torch.bfloat16, x.shape)
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", torch.bfloat16, x.shape)
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, H, P, N), dtype=torch.float32, device=x.device)
    _need(final_state, "final_state", torch.float32, (batch, H, P, N))
    need = ssd_workspace_bytes(batch, L, H, G, N)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check(lib().ss_ssd_fwd_bf16(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias),
                                 int(bool(delta_softplus)), _ptr(h0), _ptr(y), _ptr(final_state), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), batch, L, H, P, G, N,
                                 _stream(stream)))
    return y, final_state
