"""Mamba-2's scalar-decay scan on the tensor cores against the float64
oracle of its recurrence, every output element."""
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O
from selective_state_space_138_b300 import binding
from selective_state_space_138_b300 import inputs as I

pytestmark = pytest.mark.gpu

# The tensor-core products take bf16 operands (the masked scores C_t.B_s
# e^{..} delta_s and the step-weighted inputs are rounded once to bf16; the
# carried state enters as a bf16 pair, high part plus residual). Each rounding
# perturbs one term of a sum by at most 2^-9 of that term, so the error of an
# output is bounded by a small multiple of 2^-9 times the sum of the
# magnitudes of its terms -- which is what the same recurrence computes on the
# absolute values of its inputs (every term then positive). The bound used:
# |gpu - ref| <= 2e-2 |ref| + 1e-3 + 2^-7 * ref_abs, the first two terms the
# output's own bf16 rounding (as for the selective scan).
RTOL, ATOL, OPERAND = 2e-2, 1e-3, 2.0 ** -7


def term_scale(inp, h0, use_z, use_D, use_bias, softplus):
    """Sum of the magnitudes of the terms of every output: the recurrence on
    |x|, |B|, |C|, |D|, |h0| (the decays and steps are positive), times |silu(z)|."""
    ab = lambda t: None if t is None else t.float().abs()
    ya, fa = O.ssd(ab(inp["x"]), inp["dt"], inp["A"], ab(inp["B"]), ab(inp["C"]), D=ab(inp["D"]) if use_D else None,
                   dt_bias=inp["dt_bias"] if use_bias else None, delta_softplus=softplus, h0=ab(h0))
    if use_z:
        z = inp["z"].double().numpy()
        ya = ya * np.abs(z / (1.0 + np.exp(-z)))
    return ya, fa


def close(got, ref, scale, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref) / (RTOL * np.abs(ref) + ATOL + OPERAND * scale)
    i = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= 1.0, "%s: normalised error %.3f at %s (gpu %r, oracle %r, term scale %r)" % (
        what, err.max(), i, got[i], ref[i], scale[i])
    return float(err.max())


def run(spec, use_z=True, use_D=True, use_bias=True, softplus=True, use_h0=False):
    if spec.N == 256 and os.environ.get("SS_SCAN_TMA") == "0":
        pytest.skip("N = 256 runs on the tensor-core kernels only, which SS_SCAN_TMA=0 turns off")
    inp = I.make_ssd_inputs(spec)
    if not softplus:
        # without softplus the raw step is the step: a bias of 0.5 keeps it positive
        # (a negative step makes the recurrence grow without bound)
        inp["dt_bias"] = torch.full_like(inp["dt_bias"], 0.5)
    h0 = None
    if use_h0:
        h0 = I.normal(spec.seed, I.TAG_H0, (spec.batch, spec.nheads, spec.headdim, spec.N), 1.0, torch.float32)
    g = {k: v.cuda() for k, v in inp.items()}
    y, fs = binding.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"] if use_D else None,
                            z=g["z"] if use_z else None, dt_bias=g["dt_bias"] if use_bias else None,
                            delta_softplus=softplus, h0=None if h0 is None else h0.cuda())
    torch.cuda.synchronize()
    ry, rf = O.ssd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"] if use_D else None,
                   z=inp["z"] if use_z else None, dt_bias=inp["dt_bias"] if use_bias else None,
                   delta_softplus=softplus, h0=h0)
    ya, fa = term_scale(inp, h0, use_z, use_D, use_bias, softplus)
    return close(y.float().cpu().numpy(), ry, ya, "y"), close(fs.cpu().numpy(), rf, fa, "final_state")


SHAPES = [(1, 1, 1, 1, 64), (1, 64, 2, 1, 64), (2, 100, 4, 2, 128), (1, 257, 3, 1, 128), (2, 130, 8, 4, 64),
          (1, 1000, 2, 1, 128),
          # N = 256: two passes over the state halves
          (1, 1, 1, 1, 256), (2, 130, 4, 2, 256), (1, 700, 3, 1, 256)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b%d_l%d_h%d_g%d_n%d" % s)
def test_ssd_matches_oracle(shape):
    b, L, H, G, N = shape
    run(I.SsdSpec(b, L, H, 64, G, N, seed=L + H))


@pytest.mark.parametrize("N", [128, 256])
@pytest.mark.parametrize("opts", [dict(use_z=False, use_D=False, use_bias=False), dict(use_h0=True),
                                  dict(softplus=False), dict(use_h0=True, use_z=False)],
                         ids=["bare", "h0", "no_softplus", "h0_no_gate"])
def test_ssd_options(opts, N):
    spec = I.SsdSpec(2, 200, 4, 64, 2, N, seed=3)
    if not opts.get("softplus", True):
        spec = I.SsdSpec(2, 200, 4, 64, 2, N, seed=4)
    run(spec, **opts)


@pytest.mark.parametrize("N", [64, 128, 256])
@pytest.mark.parametrize("segments", [2, 3, 4, 8])
def test_ssd_chunk_segments(segments, N, monkeypatch):
    """Rows cut into chunk segments walked one after another, possibly by
    different CTAs, each starting from the state the one before handed over
    (forced through SS_SSD_SEGMENTS; 8 exceeds the 6 chunks of some rows)."""
    monkeypatch.setenv("SS_SSD_SEGMENTS", str(segments))
    run(I.SsdSpec(2, 1000 if N != 256 else 333, 5, 64, 1, N, seed=20 + segments), use_h0=True)


def test_ssd_more_rows_than_ctas():
    """640 (batch, head) rows with an initial state: more rows than CTAs fit at once,
    so CTAs walk several work items, each row cut into segments by the default
    choice (every item starts from h0 or from the state handed over)."""
    run(I.SsdSpec(8, 130, 80, 64, 1, 128, seed=41), use_h0=True)


@pytest.mark.parametrize("segments", [1, 2, 4])
def test_ssd_without_final_state(segments, monkeypatch):
    """No final state asked for: y is the same, bit for bit, as with it (the
    segments still hand their states over through the workspace)."""
    monkeypatch.setenv("SS_SSD_SEGMENTS", str(segments))
    spec = I.SsdSpec(2, 700, 3, 64, 1, 128, seed=31)
    inp = I.make_ssd_inputs(spec)
    g = {k: v.cuda() for k, v in inp.items()}
    y1, fs = binding.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"])
    y2, none = binding.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"],
                               return_final_state=False)
    torch.cuda.synchronize()
    assert none is None and fs is not None
    assert torch.equal(y1, y2)


def test_ssd_concurrent_calls_with_own_workspaces():
    """Two calls on two streams at once, each with its own workspace (its own work
    counters and handed-over states): each equals the same call made alone."""
    spec = I.SsdSpec(8, 130, 80, 64, 1, 128, seed=51)
    inp = I.make_ssd_inputs(spec)
    g = {k: v.cuda() for k, v in inp.items()}
    args = (g["x"], g["dt"], g["A"], g["B"], g["C"])
    kw = dict(D=g["D"], z=g["z"], dt_bias=g["dt_bias"])
    y0, f0 = binding.ssd_fwd(*args, **kw)
    torch.cuda.synchronize()
    need = binding.ssd_workspace_bytes(spec.batch, spec.L, spec.nheads, spec.ngroups, spec.N)
    ws = [torch.empty(need, dtype=torch.uint8, device="cuda") for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    outs = []
    for s, w in zip(streams, ws):
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            outs.append(binding.ssd_fwd(*args, **kw, workspace=w, stream=s))
    torch.cuda.synchronize()
    for y, f in outs:
        assert torch.equal(y, y0) and torch.equal(f, f0)


def test_ssd_continues_from_its_final_state():
    """Two halves, the second started from the first's final state, equal
    one pass (chunked prefill)."""
    spec = I.SsdSpec(1, 256, 4, 64, 1, 128, seed=12)
    inp = I.make_ssd_inputs(spec)
    g = {k: v.cuda() for k, v in inp.items()}
    y, fs = binding.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"])
    half = lambda t, a, b: t[:, a:b].contiguous()
    y1, f1 = binding.ssd_fwd(half(g["x"], 0, 128), half(g["dt"], 0, 128), g["A"], half(g["B"], 0, 128),
                             half(g["C"], 0, 128), D=g["D"], z=half(g["z"], 0, 128), dt_bias=g["dt_bias"])
    y2, f2 = binding.ssd_fwd(half(g["x"], 128, 256), half(g["dt"], 128, 256), g["A"], half(g["B"], 128, 256),
                             half(g["C"], 128, 256), D=g["D"], z=half(g["z"], 128, 256), dt_bias=g["dt_bias"], h0=f1)
    torch.cuda.synchronize()
    ya, fa = term_scale(inp, None, True, True, True, True)
    ref = torch.cat([y1, y2], dim=1).float().cpu().numpy()
    close(ref, y.float().cpu().numpy().astype(np.float64), ya, "halves")
    close(f2.cpu().numpy(), fs.cpu().numpy().astype(np.float64), fa, "final state")


def test_ssd_layer_every_head():
    """The Mamba-2 layer workload at full size, in the bench's launch
    configuration, checked against the oracle on every (batch row, head):
    every output element and every final state."""
    spec = I.MAMBA2_LAYER
    inp = I.make_ssd_inputs(spec)
    g = {k: v.cuda() for k, v in inp.items()}
    binding.device_faults(clear=True)
    y, fs = binding.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"])
    torch.cuda.synchronize()
    assert binding.device_faults() == 0
    worst_y = worst_f = 0.0
    for b in range(spec.batch):
        sl = lambda t: t[b:b + 1].contiguous()
        one = dict(x=sl(inp["x"]), dt=sl(inp["dt"]), A=inp["A"], B=sl(inp["B"]), C=sl(inp["C"]), D=inp["D"],
                   z=sl(inp["z"]), dt_bias=inp["dt_bias"])
        ry, rf = O.ssd(one["x"], one["dt"], one["A"], one["B"], one["C"], D=one["D"], z=one["z"],
                       dt_bias=one["dt_bias"])
        ya, fa = term_scale(one, None, True, True, True, True)
        worst_y = max(worst_y, close(y[b:b + 1].float().cpu().numpy(), ry, ya, "y b%d" % b))
        worst_f = max(worst_f, close(fs[b:b + 1].cpu().numpy(), rf, fa, "final state b%d" % b))
    print("%s: max normalised error y %.3f, final state %.3f (1.0 = tolerance)" % (spec.name, worst_y, worst_f))


def test_ssd_rejects_unsupported_shapes():
    x = torch.zeros(1, 8, 2, 32, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.SSError) as ei:
        binding.ssd_fwd(x, torch.zeros(1, 8, 2, dtype=torch.bfloat16, device="cuda"), -torch.ones(2, device="cuda"),
                        B, B)
    assert ei.value.status == -2 and "headdim" in str(ei.value)
