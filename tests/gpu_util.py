"""Helpers shared by the GPU parity tests: device copies, the CUDA path
through the C ABI, the oracle on the same inputs, and the tolerance check."""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as O
from selective_state_space_138_b300 import binding

# |gpu - ref| <= ATOL + RTOL * |ref|, per element (bf16 io with fp32 state, and fp32 io)
TOL = {torch.bfloat16: (2e-2, 1e-3), torch.float32: (1e-4, 1e-5)}


def dev(inp: dict, keys=("x", "dt", "z", "B", "C", "A", "D", "dt_bias")) -> dict:
    return {k: inp[k].cuda() for k in keys if inp.get(k) is not None}


def gpu_scan(inp: dict, use_D=True, use_z=True, use_bias=True, softplus=True, final_state=True):
    g = dev(inp)
    y, fs = binding.scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"],
                             D=g["D"] if use_D else None, z=g["z"] if use_z else None,
                             dt_bias=g["dt_bias"] if use_bias else None, delta_softplus=softplus,
                             return_final_state=final_state)
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64), None if fs is None else fs.cpu().numpy().astype(np.float64)


def oracle_scan(inp: dict, use_D=True, use_z=True, use_bias=True, softplus=True):
    return O.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                  D=inp["D"] if use_D else None, z=inp["z"] if use_z else None,
                  dt_bias=inp["dt_bias"] if use_bias else None, delta_softplus=softplus)


def assert_close(got, ref, dtype, what=""):
    rtol, atol = TOL[dtype]
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite GPU output" % what
    err = np.abs(got - ref) / (atol + rtol * np.abs(ref))
    worst = np.unravel_index(np.argmax(err), err.shape) if err.size else ()
    assert err.size == 0 or err.max() <= 1.0, (
        "%s: max normalised error %.3f at %s (gpu %r, oracle %r)"
        % (what, err.max(), worst, got[worst], ref[worst]))
    return float(err.max()) if err.size else 0.0


def compare_scan_all_rows(inp: dict, y, fs, dtype, block: int = 256, what: str = ""):
    """Every (batch, channel) row of a GPU scan -- y (batch, d_inner, L) and
    the final state (batch, d_inner, N), device tensors -- against the oracle,
    block by block of channels so that host memory stays bounded. Returns the
    largest normalised error of y and of the final state (1.0 = tolerance)."""
    batch, d_inner, L = tuple(inp["x"].shape)
    worst_y = worst_f = 0.0
    for b in range(batch):
        for d0 in range(0, d_inner, block):
            d1 = min(d_inner, d0 + block)
            rows = [b * d_inner + d for d in range(d0, d1)]
            yr, fr = O.scan_rows(inp, rows)
            got_y = y[b, d0:d1].float().cpu().numpy()
            got_f = fs[b, d0:d1].cpu().numpy()
            worst_y = max(worst_y, assert_close(got_y, yr, dtype, "%s y b%d d%d..%d" % (what, b, d0, d1)))
            worst_f = max(worst_f, assert_close(got_f, fr, dtype, "%s final_state b%d d%d..%d" % (what, b, d0, d1)))
    return worst_y, worst_f
