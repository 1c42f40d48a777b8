"""Seeded synthetic inputs for the selective scan and the decode state update.

This module is shared by the CUDA path's tests/bench and by the float64 oracle's
callers. It draws random numbers and applies the parameter-initialisation
recipe only; it computes none of the scan's arithmetic (no softplus of the step,
no discretisation, no recurrence, no readout, no gate).

Recipe (every workload):
  * x, z, B, C ~ N(0, 1); dt ~ N(0, 0.1) (0.1 read as the standard deviation).
  * dt_bias = softplus^-1(u) = ln(e^u - 1) with u log-uniform in [1e-3, 1e-1]
    per channel -- the step-size initialisation of "Mamba, annotated",
    section 3.6 "Additional model details", and of "Mamba and selective state
    spaces", box "How a Mamba layer is initialized".
  * A[d, n] = -(n + 1) (S4D-Real, same sources), optionally scaled per channel
    by exp(eps_d), eps_d ~ N(0, 0.1), computed in float64 then rounded to fp32.
  * D = 1.
  * Long-sequence workload: dt_bias = softplus^-1(1e-3) for every channel, and a
    fraction of time positions per batch row (shared by all channels, since the
    step is chosen per token) gets dt = softplus^-1(5) - dt_bias, so that the
    step before rounding is 5 (a state reset, "Mamba and selective state
    spaces", section "What each parameter does").
  * Decode workload: the step handed to the single-token update is drawn as
    delta = u_d * exp(dt) with dt ~ N(0, 0.1): the step size that the recipe
    above yields, to first order in u, written without a softplus.

Every tensor is drawn in blocks of ``_BLOCK`` elements of its flattened
row-major layout; block i of tensor ``tag`` comes from
``numpy.random.default_rng([seed, tag, i])`` (PCG64). Draws are float32 and are
then rounded once to the io dtype (round-to-nearest-even for bf16, by torch).
The result does not depend on the number of threads used to draw it.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

_BLOCK = 1 << 22

# tensor tags in draw order
TAG_X, TAG_Z, TAG_B, TAG_C, TAG_DT, TAG_U, TAG_EPS, TAG_RESET = 1, 2, 3, 4, 5, 6, 7, 8
# incoming gradients and initial state of the backward workloads
TAG_DOUT, TAG_DFINAL, TAG_H0 = 9, 10, 11

_POOL_THREADS = max(1, min(16, len(os.sched_getaffinity(0))))


def _inv_softplus(u: np.ndarray | float) -> np.ndarray:
    """ln(e^u - 1) in float64 (parameter initialisation only)."""
    return np.log(np.expm1(np.asarray(u, dtype=np.float64)))


def _fill_blocks(seed: int, tag: int, n: int, draw, out: torch.Tensor) -> None:
    """Fill the flat tensor ``out`` (length n) block by block.

    ``draw(rng, length) -> float32 ndarray`` produces one block.
    """
    flat = out.view(-1)
    nblk = (n + _BLOCK - 1) // _BLOCK

    def one(i: int) -> None:
        lo = i * _BLOCK
        hi = min(n, lo + _BLOCK)
        rng = np.random.default_rng([seed, tag, i])
        vals = draw(rng, hi - lo)
        flat[lo:hi].copy_(torch.from_numpy(vals))

    if nblk == 1:
        one(0)
    else:
        with ThreadPoolExecutor(_POOL_THREADS) as ex:
            list(ex.map(one, range(nblk)))


def normal(seed: int, tag: int, shape, std: float, dtype: torch.dtype) -> torch.Tensor:
    """N(0, std^2) draws of ``shape``, rounded once to ``dtype``."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(tuple(shape), dtype=dtype)
    if n == 0:
        return out

    def draw(rng, m):
        v = rng.standard_normal(m, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        return v

    _fill_blocks(seed, tag, n, draw, out)
    return out


@dataclass
class ScanSpec:
    """Shape and recipe of one scan workload."""

    batch: int
    d_inner: int
    L: int
    N: int = 16
    io: str = "bf16"          # "bf16" or "f32"
    seed: int = 0
    a_scale_eps: bool = False  # A[d, n] = -(n+1) * exp(eps_d)
    dt_bias_const: float | None = None  # step-size target shared by all channels
    reset_frac: float = 0.0    # fraction of positions per batch row with step 5
    name: str = ""

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.io == "bf16" else torch.float32

    @property
    def elem_steps(self) -> int:
        return self.batch * self.d_inner * self.L * self.N


@dataclass
class DecodeSpec:
    """Shape and recipe of the single-token decode workload."""

    batch: int
    d_inner: int
    N: int = 16
    steps: int = 1024
    seed: int = 4
    name: str = ""

    @property
    def elem_steps_per_step(self) -> int:
        return self.batch * self.d_inner * self.N


# The five workloads: a tiny fp32 scan, one Mamba-130M layer, one Mamba-1.4B
# layer with per-channel scaled A, a 131072-token scan with sparse resets, and
# the batch-256 decode. Shapes follow the layer widths of the Mamba models
# ("Mamba and selective state spaces", section "The Mamba block").
TINY = ScanSpec(batch=1, d_inner=64, L=256, N=16, io="f32", seed=0, name="tiny_fp32_b1_d64_l256_n16")
MAMBA130M = ScanSpec(batch=8, d_inner=1536, L=2048, N=16, io="bf16", seed=1,
                     name="mamba130m_layer_b8_d1536_l2048_n16")
MAMBA1P4B = ScanSpec(batch=4, d_inner=4096, L=4096, N=16, io="bf16", seed=2, a_scale_eps=True,
                     name="mamba1p4b_layer_b4_d4096_l4096_n16")
LONGSEQ = ScanSpec(batch=1, d_inner=2048, L=131072, N=16, io="bf16", seed=3, dt_bias_const=1e-3,
                   reset_frac=0.004, name="longseq_b1_d2048_l131072_n16")
DECODE = DecodeSpec(batch=256, d_inner=5120, N=16, steps=1024, seed=4,
                    name="decode_b256_d5120_n16_1024steps")

SCAN_WORKLOADS = {s.name: s for s in (TINY, MAMBA130M, MAMBA1P4B, LONGSEQ)}


def n_resets(spec: ScanSpec) -> int:
    return int(round(spec.reset_frac * spec.L))


def make_scan_inputs(spec: ScanSpec) -> dict:
    """All inputs of one scan workload as CPU tensors.

    Returns dict with x, dt, z (batch, d_inner, L) and B, C (batch, N, L) in the
    io dtype; A (d_inner, N), D (d_inner,), dt_bias (d_inner,) in float32; and
    ``reset_pos`` (batch, n_resets) int64 (possibly empty).
    """
    Bt, Dn, L, N, s = spec.batch, spec.d_inner, spec.L, spec.N, spec.seed
    io = spec.torch_dtype
    x = normal(s, TAG_X, (Bt, Dn, L), 1.0, io)
    z = normal(s, TAG_Z, (Bt, Dn, L), 1.0, io)
    B = normal(s, TAG_B, (Bt, N, L), 1.0, io)
    C = normal(s, TAG_C, (Bt, N, L), 1.0, io)
    if spec.reset_frac > 0:
        dt32 = normal(s, TAG_DT, (Bt, Dn, L), 0.1, torch.float32)
    else:
        dt = normal(s, TAG_DT, (Bt, Dn, L), 0.1, io)

    if spec.dt_bias_const is None:
        rng = np.random.default_rng([s, TAG_U, 0])
        u = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=Dn))
        dt_bias64 = _inv_softplus(u)
    else:
        dt_bias64 = np.full(Dn, _inv_softplus(spec.dt_bias_const), dtype=np.float64)
    dt_bias = torch.from_numpy(dt_bias64.astype(np.float32))

    base = -(np.arange(N, dtype=np.float64) + 1.0)
    if spec.a_scale_eps:
        rng = np.random.default_rng([s, TAG_EPS, 0])
        eps = rng.standard_normal(Dn) * 0.1
        A64 = base[None, :] * np.exp(eps)[:, None]
    else:
        A64 = np.broadcast_to(base[None, :], (Dn, N))
    A = torch.from_numpy(np.ascontiguousarray(A64.astype(np.float32)))
    D = torch.ones(Dn, dtype=torch.float32)

    k = n_resets(spec)
    reset_pos = torch.empty((Bt, k), dtype=torch.int64)
    if spec.reset_frac > 0:
        target = np.float32(_inv_softplus(5.0))
        for b in range(Bt):
            rng = np.random.default_rng([s, TAG_RESET, b])
            pos = np.sort(rng.choice(L, size=k, replace=False))
            reset_pos[b] = torch.from_numpy(pos)
            # dt + dt_bias = softplus^-1(5) at the reset positions, all channels
            dt32[b][:, pos] = torch.from_numpy(
                (target - dt_bias.numpy()[:, None]).astype(np.float32)).expand(Dn, k)
        dt = dt32.to(io)
    return dict(x=x, dt=dt, z=z, B=B, C=C, A=A, D=D, dt_bias=dt_bias, reset_pos=reset_pos)


def make_decode_params(spec: DecodeSpec) -> dict:
    """Per-channel parameters of the decode workload: A, D and the step scale u."""
    rng = np.random.default_rng([spec.seed, TAG_U, 0])
    u = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=spec.d_inner)).astype(np.float32)
    base = -(np.arange(spec.N, dtype=np.float32) + 1.0)
    A = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(base[None, :], (spec.d_inner, spec.N))))
    D = torch.ones(spec.d_inner, dtype=torch.float32)
    return dict(A=A, D=D, u=torch.from_numpy(u))


def make_decode_tokens(spec: DecodeSpec, steps: int | None = None) -> dict:
    """Token inputs of ``steps`` consecutive decode steps (default: all).

    Returns x, delta, z (steps, batch, d_inner) and B, C (steps, batch, N), bf16.
    delta = u_d * exp(dt), dt ~ N(0, 0.1), drawn blockwise like every tensor.
    """
    T = spec.steps if steps is None else steps
    Bt, Dn, N, s = spec.batch, spec.d_inner, spec.N, spec.seed
    x = normal(s, TAG_X, (T, Bt, Dn), 1.0, torch.bfloat16)
    z = normal(s, TAG_Z, (T, Bt, Dn), 1.0, torch.bfloat16)
    B = normal(s, TAG_B, (T, Bt, N), 1.0, torch.bfloat16)
    C = normal(s, TAG_C, (T, Bt, N), 1.0, torch.bfloat16)
    u = make_decode_params(spec)["u"].numpy()
    delta = torch.empty((T, Bt, Dn), dtype=torch.bfloat16)
    n = T * Bt * Dn
    if n:
        flat = delta.view(-1)
        nblk = (n + _BLOCK - 1) // _BLOCK

        def one(i: int) -> None:
            lo = i * _BLOCK
            hi = min(n, lo + _BLOCK)
            rng = np.random.default_rng([s, TAG_DT, i])
            v = rng.standard_normal(hi - lo, dtype=np.float32) * np.float32(0.1)
            ch = (np.arange(lo, hi, dtype=np.int64) % Dn)
            v = u[ch] * np.exp(v)
            flat[lo:hi].copy_(torch.from_numpy(v.astype(np.float32)))

        with ThreadPoolExecutor(_POOL_THREADS) as ex:
            list(ex.map(one, range(nblk)))
    return dict(x=x, delta=delta, z=z, B=B, C=C)


def make_bwd_inputs(spec: ScanSpec) -> dict:
    """Incoming gradients for a scan workload, all N(0, 1): dout (batch,
    d_inner, L) in the io dtype and dfinal (batch, d_inner, N) float32, plus an
    initial state h0 (batch, d_inner, N) float32 for the initial-state cases."""
    Bt, Dn, L, N, s = spec.batch, spec.d_inner, spec.L, spec.N, spec.seed
    return dict(dout=normal(s, TAG_DOUT, (Bt, Dn, L), 1.0, spec.torch_dtype),
                dfinal=normal(s, TAG_DFINAL, (Bt, Dn, N), 1.0, torch.float32),
                h0=normal(s, TAG_H0, (Bt, Dn, N), 1.0, torch.float32))


@dataclass
class SsdSpec:
    """Shape and recipe of one scalar-decay (Mamba-2) scan workload."""

    batch: int
    L: int
    nheads: int
    headdim: int = 64
    ngroups: int = 1
    N: int = 128
    seed: int = 0
    name: str = ""

    @property
    def elem_steps(self) -> int:
        return self.batch * self.L * self.nheads * self.headdim * self.N


def make_ssd_inputs(spec: SsdSpec) -> dict:
    """Inputs of a scalar-decay scan, time-major, as CPU tensors: x, z
    (batch, L, H, P), dt (batch, L, H), B, C (batch, L, G, N) in bf16; A, D,
    dt_bias (H,) fp32. x, z, B, C ~ N(0, 1), dt ~ N(0, 0.1); dt_bias =
    softplus^-1(u), u log-uniform in [1e-3, 1e-1] per head; A_h = -(1 + 15 v_h),
    v_h uniform in [0, 1) (decay rates spread over [1, 16] per head); D = 1."""
    Bt, L, H, P, G, N, s = spec.batch, spec.L, spec.nheads, spec.headdim, spec.ngroups, spec.N, spec.seed
    x = normal(s, TAG_X, (Bt, L, H, P), 1.0, torch.bfloat16)
    z = normal(s, TAG_Z, (Bt, L, H, P), 1.0, torch.bfloat16)
    B = normal(s, TAG_B, (Bt, L, G, N), 1.0, torch.bfloat16)
    C = normal(s, TAG_C, (Bt, L, G, N), 1.0, torch.bfloat16)
    dt = normal(s, TAG_DT, (Bt, L, H), 0.1, torch.bfloat16)
    rng = np.random.default_rng([s, TAG_U, 0])
    u = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=H))
    dt_bias = torch.from_numpy(_inv_softplus(u).astype(np.float32))
    rng = np.random.default_rng([s, TAG_EPS, 0])
    A = torch.from_numpy((-(1.0 + 15.0 * rng.random(H))).astype(np.float32))
    D = torch.ones(H, dtype=torch.float32)
    return dict(x=x, z=z, B=B, C=C, dt=dt, A=A, D=D, dt_bias=dt_bias)


# one Mamba-2 layer of the 2.7B width (d_model 2560, expand 2: 80 heads of 64, N = 128)
MAMBA2_LAYER = SsdSpec(batch=8, L=2048, nheads=80, headdim=64, ngroups=1, N=128, seed=7,
                       name="mamba2_layer_b8_l2048_h80_p64_n128")
