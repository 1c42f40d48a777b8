"""Python entry to the float64 oracle (``ss_oracle.c``) and its small helpers.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may use this module; the product path never
does. Nothing here imports the CUDA library or its binding.

* ``scan`` / ``scan_rows`` run the plain float64 loop of ``ss_oracle.c`` over
  all rows or over a sample of rows, in parallel over rows (the C call releases
  the GIL).
* ``ssd`` is Mamba-2's scalar-decay scan (one decay per head of P channels,
  B and C shared by the heads of a group), time-major layouts.
* ``scan_ex`` is the scan with an initial state, packed-sequence starts and/or
  the reverse direction.
* ``scan_bwd`` is the gradient of the scan by the chain rule (float64; the
  states are kept, the reverse recurrence is run literally).
* ``causal_conv1d`` is the block's causal depthwise convolution (+ SiLU)
  with an optional carried history of k-1 inputs, in float64.
* ``decode_chain`` runs that same loop over consecutive single-token inputs:
  the decode update is one step of the scan, so a chain of steps equals the
  scan over the tokens ("Mamba and selective state spaces", section "Decoding
  with a constant-size cache").
* ``zoh``, ``affine_combine`` and ``affine_scan`` are the zero-order-hold
  discretisation and the affine-map composition of the pages ("Mamba,
  annotated", sections "Discretization (equation 4)" and "The scan, in one
  equation"); the tests pin them to the pages' printed numbers.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ss_oracle.c")
_LIB = os.path.join(_HERE, "libss_oracle.so")
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile ``src`` with gcc -O2 (no fast-math) into the shared library ``out``."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; returns the CDLL."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_softplus.argtypes = [ctypes.c_double]
    lib.oracle_softplus.restype = ctypes.c_double
    lib.oracle_scan_rows.argtypes = [dp] * 8 + [ctypes.c_int, dp, dp, dp] + [ctypes.c_int64] * 6
    lib.oracle_scan_rows.restype = ctypes.c_int
    if hasattr(lib, "oracle_ssd_rows"):
        lib.oracle_ssd_rows.argtypes = [dp] * 8 + [ctypes.c_int, dp, dp, dp] + [ctypes.c_int64] * 8
        lib.oracle_ssd_rows.restype = ctypes.c_int
    if hasattr(lib, "oracle_scan_ex_rows"):
        lib.oracle_scan_ex_rows.argtypes = ([dp] * 8 + [ctypes.c_int, dp, ctypes.c_void_p, ctypes.c_int, dp, dp]
                                            + [ctypes.c_int64] * 6)
        lib.oracle_scan_ex_rows.restype = ctypes.c_int
    if hasattr(lib, "oracle_scan_bwd_rows"):
        lib.oracle_scan_bwd_rows.argtypes = [dp] * 8 + [ctypes.c_int] + [dp] * 12 + [ctypes.c_int64] * 6
        lib.oracle_scan_bwd_rows.restype = ctypes.c_int
    if hasattr(lib, "oracle_scan_bwd_ex_rows"):
        lib.oracle_scan_bwd_ex_rows.argtypes = ([dp] * 8 + [ctypes.c_int, dp, ctypes.c_void_p, ctypes.c_int]
                                                + [dp] * 11 + [ctypes.c_int64] * 6)
        lib.oracle_scan_bwd_ex_rows.restype = ctypes.c_int
    if hasattr(lib, "oracle_causal_conv1d_rows"):
        lib.oracle_causal_conv1d_rows.argtypes = [dp, dp, dp, ctypes.c_int, dp, dp, dp] + [ctypes.c_int64] * 6
        lib.oracle_causal_conv1d_rows.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor (CPU): exact widening to float64
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def softplus(v: float) -> float:
    return load().oracle_softplus(float(v))


def scan(x, dt, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True, h0=None,
         threads: int | None = None, lib=None):
    """Full selective scan in float64.

    x, dt, z: (batch, d_inner, L); B, C: (batch, N, L); A: (d_inner, N);
    D, dt_bias: (d_inner,); h0: (batch, d_inner, N) or None.
    Returns (y (batch, d_inner, L), final_state (batch, d_inner, N)), float64.
    """
    lib = lib or load()
    x, dt, A, B, C = map(_f64, (x, dt, A, B, C))
    D, z, dt_bias, h0 = map(_f64, (D, z, dt_bias, h0))
    batch, d_inner, L = x.shape
    N = A.shape[1]
    assert dt.shape == x.shape and B.shape == (batch, N, L) and C.shape == (batch, N, L)
    assert A.shape == (d_inner, N)
    y = np.empty((batch, d_inner, L), dtype=np.float64)
    fs = np.empty((batch, d_inner, N), dtype=np.float64)
    rows = batch * d_inner
    nt = max(1, min(threads or default_threads(), rows)) if rows else 1
    bounds = [(rows * i) // nt for i in range(nt + 1)]

    def run(i):
        return lib.oracle_scan_rows(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                    _ptr(dt_bias), int(bool(delta_softplus)), _ptr(h0), _ptr(y),
                                    _ptr(fs), batch, d_inner, L, N, bounds[i], bounds[i + 1])

    if nt == 1:
        codes = [run(0)]
    else:
        with ThreadPoolExecutor(nt) as ex:
            codes = list(ex.map(run, range(nt)))
    if any(c != 0 for c in codes):
        raise RuntimeError("oracle_scan_rows failed: %r" % (codes,))
    return y, fs


def scan_ex(x, dt, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True, h0=None, seq_start=None,
            reverse=False, threads: int | None = None, lib=None):
    """The scan with an initial state, sequence starts (batch, L) bool/uint8
    and/or the reverse direction (``oracle_scan_ex_rows``), float64.
    Returns (y, final_state)."""
    lib = lib or load()
    x, dt, A, B, C = map(_f64, (x, dt, A, B, C))
    D, z, dt_bias, h0 = map(_f64, (D, z, dt_bias, h0))
    batch, d_inner, L = x.shape
    N = A.shape[1]
    st = None
    if seq_start is not None:
        if hasattr(seq_start, "detach"):
            seq_start = seq_start.detach().cpu().numpy()
        st = np.ascontiguousarray(np.asarray(seq_start) != 0, dtype=np.uint8)
        assert st.shape == (batch, L)
    y = np.empty((batch, d_inner, L))
    fs = np.empty((batch, d_inner, N))
    rows = batch * d_inner
    nt = max(1, min(threads or default_threads(), rows)) if rows else 1
    bounds = [(rows * i) // nt for i in range(nt + 1)]

    def run(i):
        return lib.oracle_scan_ex_rows(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                       _ptr(dt_bias), int(bool(delta_softplus)), _ptr(h0),
                                       None if st is None else st.ctypes.data_as(ctypes.c_void_p),
                                       int(bool(reverse)), _ptr(y), _ptr(fs), batch, d_inner, L, N,
                                       bounds[i], bounds[i + 1])

    if nt == 1:
        codes = [run(0)]
    else:
        with ThreadPoolExecutor(nt) as ex:
            codes = list(ex.map(run, range(nt)))
    if any(c != 0 for c in codes):
        raise RuntimeError("oracle_scan_ex_rows failed: %r" % (codes,))
    return y, fs


def ssd(x, dt, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True, h0=None, threads: int | None = None,
        lib=None):
    """Mamba-2's scalar-decay scan (``oracle_ssd_rows``) in float64.

    x, z: (batch, L, H, P); dt: (batch, L, H); B, C: (batch, L, G, N);
    A, D, dt_bias: (H,); h0: (batch, H, P, N) or None.
    Returns (y (batch, L, H, P), final_state (batch, H, P, N)).
    """
    lib = lib or load()
    x, dt, A, B, C = map(_f64, (x, dt, A, B, C))
    D, z, dt_bias, h0 = map(_f64, (D, z, dt_bias, h0))
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert dt.shape == (batch, L, H) and B.shape == (batch, L, G, N) and C.shape == B.shape and A.shape == (H,)
    y = np.empty_like(x)
    fs = np.empty((batch, H, P, N))
    rows = batch * H
    nt = max(1, min(threads or default_threads(), rows)) if rows else 1
    bounds = [(rows * i) // nt for i in range(nt + 1)]

    def run(i):
        return lib.oracle_ssd_rows(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias),
                                   int(bool(delta_softplus)), _ptr(h0), _ptr(y), _ptr(fs), batch, L, H, P, G, N,
                                   bounds[i], bounds[i + 1])

    if nt == 1:
        codes = [run(0)]
    else:
        with ThreadPoolExecutor(nt) as ex:
            codes = list(ex.map(run, range(nt)))
    if any(c != 0 for c in codes):
        raise RuntimeError("oracle_ssd_rows failed: %r" % (codes,))
    return y, fs


def scan_bwd(x, dt, A, B, C, dout, D=None, z=None, dt_bias=None, delta_softplus=True, h0=None,
             dfinal=None, seq_start=None, reverse=False, threads: int | None = None, lib=None):
    """Gradient of the selective scan in float64 (``oracle_scan_bwd_rows``;
    with sequence starts (batch, L) or the reverse direction, the gradient of
    ``scan_ex``: ``oracle_scan_bwd_ex_rows``).

    Same inputs as ``scan`` plus dout (batch, d_inner, L), the gradient of the
    (gated) output, and dfinal (batch, d_inner, N) or None, the gradient of the
    final state. Returns a dict of float64 arrays: dx, ddt (of the raw step
    input dt), dz (None without z), dA, dB, dC, dD (None without D), ddt_bias
    (None without dt_bias) and dh0 (gradient of the initial state).
    """
    lib = lib or load()
    x, dt, A, B, C, dout = map(_f64, (x, dt, A, B, C, dout))
    D, z, dt_bias, h0, dfinal = map(_f64, (D, z, dt_bias, h0, dfinal))
    batch, d_inner, L = x.shape
    N = A.shape[1]
    assert dt.shape == x.shape and dout.shape == x.shape
    assert B.shape == (batch, N, L) and C.shape == (batch, N, L) and A.shape == (d_inner, N)
    dx = np.empty_like(x)
    ddt = np.empty_like(x)
    dz = np.empty_like(x) if z is not None else None
    dh0 = np.empty((batch, d_inner, N))
    rows = batch * d_inner
    nt = max(1, min(threads or default_threads(), rows)) if rows else 1
    bounds = [(rows * i) // nt for i in range(nt + 1)]
    acc = [dict(dA=np.zeros((d_inner, N)), dB=np.zeros((batch, N, L)), dC=np.zeros((batch, N, L)),
                dD=np.zeros(d_inner), ddt_bias=np.zeros(d_inner)) for _ in range(nt)]

    st = None
    if seq_start is not None:
        if hasattr(seq_start, "detach"):
            seq_start = seq_start.detach().cpu().numpy()
        st = np.ascontiguousarray(np.asarray(seq_start) != 0, dtype=np.uint8)
        assert st.shape == (batch, L)
    ex = st is not None or bool(reverse)

    def run(i):
        a = acc[i]
        if ex:
            return lib.oracle_scan_bwd_ex_rows(
                _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias),
                int(bool(delta_softplus)), _ptr(h0), None if st is None else st.ctypes.data_as(ctypes.c_void_p),
                int(bool(reverse)), _ptr(dout), _ptr(dfinal), _ptr(dx), _ptr(ddt), _ptr(dz), _ptr(a["dA"]),
                _ptr(a["dB"]), _ptr(a["dC"]), _ptr(a["dD"]), _ptr(a["ddt_bias"]), _ptr(dh0),
                batch, d_inner, L, N, bounds[i], bounds[i + 1])
        return lib.oracle_scan_bwd_rows(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                        _ptr(dt_bias), int(bool(delta_softplus)), _ptr(h0), _ptr(dout),
                                        _ptr(dfinal), _ptr(dx), _ptr(ddt), _ptr(dz), _ptr(a["dA"]),
                                        _ptr(a["dB"]), _ptr(a["dC"]), _ptr(a["dD"]), _ptr(a["ddt_bias"]),
                                        _ptr(dh0), batch, d_inner, L, N, bounds[i], bounds[i + 1])

    if nt == 1:
        codes = [run(0)]
    else:
        with ThreadPoolExecutor(nt) as ex:
            codes = list(ex.map(run, range(nt)))
    if any(c != 0 for c in codes):
        raise RuntimeError("oracle_scan_bwd_rows failed: %r" % (codes,))
    tot = {k: sum(a[k] for a in acc) for k in acc[0]}
    return dict(dx=dx, ddt=ddt, dz=dz, dA=tot["dA"], dB=tot["dB"], dC=tot["dC"],
                dD=tot["dD"] if D is not None else None,
                ddt_bias=tot["ddt_bias"] if dt_bias is not None else None, dh0=dh0)


def scan_rows(inp: dict, rows, delta_softplus=True, use_D=True, use_z=True, use_bias=True,
              threads: int | None = None):
    """Scan only the listed rows r = b * d_inner + d of a workload.

    ``inp`` holds x, dt, z (batch, d_inner, L), B, C (batch, N, L), A, D,
    dt_bias (CPU tensors or arrays). Rows of the same batch row b are run as
    one problem over the selected channels. Returns (y (len(rows), L),
    final_state (len(rows), N)) in the order of ``rows``.
    """
    batch, d_inner, L = tuple(inp["x"].shape)
    N = inp["A"].shape[1]
    rows = [int(r) for r in rows]
    y = np.empty((len(rows), L))
    fs = np.empty((len(rows), N))
    by_b = {}
    for i, r in enumerate(rows):
        by_b.setdefault(r // d_inner, []).append(i)
    for b, idx in by_b.items():
        ds = [rows[i] % d_inner for i in idx]
        pick = lambda t: _f64(t[b][ds])[None]
        yb, fb = scan(pick(inp["x"]), pick(inp["dt"]), _f64(inp["A"][ds]),
                      _f64(inp["B"][b])[None], _f64(inp["C"][b])[None],
                      D=_f64(inp["D"][ds]) if use_D and inp.get("D") is not None else None,
                      z=pick(inp["z"]) if use_z and inp.get("z") is not None else None,
                      dt_bias=(_f64(inp["dt_bias"][ds])
                               if use_bias and inp.get("dt_bias") is not None else None),
                      delta_softplus=delta_softplus, threads=threads)
        y[idx] = yb[0]
        fs[idx] = fb[0]
    return y, fs


def decode_chain(tokens: dict, params: dict, rows, use_D=True, use_z=True, h0=None,
                 threads: int | None = None):
    """Outputs of consecutive single-token updates for the listed rows.

    tokens: x, delta, z (steps, batch, d_inner), B, C (steps, batch, N);
    params: A (d_inner, N), D (d_inner,). The step ``delta`` is final (no bias,
    no softplus). h0: None (zero state) or (len(rows), N).
    Returns (y (len(rows), steps), state after the last step (len(rows), N)).
    """
    steps, batch, d_inner = tuple(tokens["x"].shape)
    N = params["A"].shape[1]
    rows = [int(r) for r in rows]
    y = np.empty((len(rows), steps))
    fs = np.empty((len(rows), N))
    by_b = {}
    for i, r in enumerate(rows):
        by_b.setdefault(r // d_inner, []).append(i)
    for b, idx in by_b.items():
        ds = [rows[i] % d_inner for i in idx]
        col = lambda t: _f64(t[:, b][:, ds]).T[None].copy()  # (1, len(ds), steps)
        Bb = _f64(tokens["B"][:, b, :]).T[None].copy()
        Cb = _f64(tokens["C"][:, b, :]).T[None].copy()
        yb, fb = scan(col(tokens["x"]), col(tokens["delta"]), _f64(params["A"][ds]), Bb, Cb,
                      D=_f64(params["D"][ds]) if use_D else None,
                      z=col(tokens["z"]) if use_z else None, dt_bias=None, delta_softplus=False,
                      h0=None if h0 is None else _f64(np.asarray(h0)[idx])[None],
                      threads=threads)
        y[idx] = yb[0]
        fs[idx] = fb[0]
    return y, fs


def causal_conv1d(xin, w, bias=None, silu=True, state=None, threads: int | None = None, lib=None):
    """Causal depthwise convolution of the Mamba block in float64.

    xin: (batch, d_inner, L); w: (d_inner, k); bias: (d_inner,) or None;
    state: previous k-1 inputs (batch, k-1, d_inner), oldest first, or None
    (zero history). Returns (out (batch, d_inner, L), last k-1 inputs
    (batch, k-1, d_inner)).
    """
    lib = lib or load()
    xin, w, bias, state = map(_f64, (xin, w, bias, state))
    batch, d_inner, L = xin.shape
    k = w.shape[1]
    out = np.empty((batch, d_inner, L))
    st = np.empty((batch, max(k - 1, 0), d_inner))
    rows = batch * d_inner
    nt = max(1, min(threads or default_threads(), rows)) if rows else 1
    bounds = [(rows * i) // nt for i in range(nt + 1)]

    def run(i):
        return lib.oracle_causal_conv1d_rows(_ptr(xin), _ptr(w), _ptr(bias), int(bool(silu)), _ptr(state),
                                             _ptr(out), _ptr(st) if k > 1 else None, batch, d_inner, L, k,
                                             bounds[i], bounds[i + 1])

    with ThreadPoolExecutor(nt) as ex:
        codes = list(ex.map(run, range(nt)))
    if any(c != 0 for c in codes):
        raise RuntimeError("oracle_causal_conv1d_rows failed: %r" % (codes,))
    return out, st


# ---------------------------------------------------------------- helpers

def zoh(delta: float, A: float, B: float):
    """Zero-order hold of the scalar system h' = A h + B x over a step delta:
    (e^{delta A}, (e^{delta A} - 1) / A * B). Used only to pin the pages'
    printed discretisation examples; the scan itself uses delta * B."""
    a_bar = math.exp(delta * A)
    return a_bar, (a_bar - 1.0) / A * B


def affine_combine(first, then):
    """Composition of two affine maps h -> a h + b: first (a1, b1), then
    (a2, b2), gives (a1 a2, a2 b1 + b2)."""
    a1, b1 = first
    a2, b2 = then
    return a1 * a2, a2 * b1 + b2


def affine_scan(pairs, h0: float = 0.0):
    """States of h_t = a_t h_{t-1} + b_t, one after another, from h0."""
    out = []
    h = h0
    for a, b in pairs:
        h = a * h + b
        out.append(h)
    return out
