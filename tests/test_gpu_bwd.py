"""Backward pass of the scan (states recomputed on the GPU) against the
float64 oracle's chain-rule gradient on the same inputs, every output element
by element."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from selective_state_space_138_b300 import binding
from selective_state_space_138_b300 import inputs as I

pytestmark = pytest.mark.gpu

# |gpu - ref| <= RTOL |ref| + ATOL_REL rms(ref), per element. io-dtype outputs
# (dx, ddelta, dz) are rounded once to the io dtype; the fp32 sums (dA, dB,
# dC, dD, ddt_bias, dh0) carry fp32 rounding of long sums whose terms cancel,
# hence the scale term.
GTOL = {torch.bfloat16: {"io": (2e-2, 2e-3), "f32": (2e-3, 2e-4)},
        torch.float32: {"io": (1e-4, 1e-5), "f32": (1e-4, 1e-5)}}
IO_KEYS = ("dx", "ddelta", "dz")


def assert_grad_close(got, ref, io_dtype, key):
    rtol, arel = GTOL[io_dtype]["io" if key in IO_KEYS else "f32"]
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (key, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite GPU output" % key
    scale = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = np.abs(got - ref) / (rtol * np.abs(ref) + arel * scale + 1e-30)
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= 1.0, "%s: normalised error %.3f at %s (gpu %r, oracle %r, rms %g)" % (
        key, err.max(), worst, got[worst], ref[worst], scale)
    return float(err.max())


def run_case(spec, use_D=True, use_z=True, use_bias=True, softplus=True, use_h0=False, use_dfinal=True,
             seq_start=None, reverse=False):
    inp = I.make_scan_inputs(spec)
    if not softplus and not use_bias:
        # without softplus and bias the raw step is the step: keep it positive
        # (a negative step makes the recurrence grow without bound)
        inp["dt"] = (inp["dt"].float().abs() + 0.05).to(inp["dt"].dtype)
    bw = I.make_bwd_inputs(spec)
    g = {k: inp[k].cuda() for k in ("x", "dt", "z", "B", "C", "A", "D", "dt_bias")}
    h0 = bw["h0"] if use_h0 else None
    dfin = bw["dfinal"] if use_dfinal else None
    got = binding.scan_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], bw["dout"].cuda(),
                           D=g["D"] if use_D else None, z=g["z"] if use_z else None,
                           dt_bias=g["dt_bias"] if use_bias else None, delta_softplus=softplus,
                           h0=None if h0 is None else h0.cuda(),
                           dfinal_state=None if dfin is None else dfin.cuda(),
                           seq_start=None if seq_start is None else seq_start.cuda(), reverse=reverse)
    torch.cuda.synchronize()
    ref = O.scan_bwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], bw["dout"],
                     D=inp["D"] if use_D else None, z=inp["z"] if use_z else None,
                     dt_bias=inp["dt_bias"] if use_bias else None, delta_softplus=softplus, h0=h0, dfinal=dfin,
                     seq_start=seq_start, reverse=reverse)
    errs = {}
    for k, r in ref.items():
        kg = "ddelta" if k == "ddt" else k   # the oracle names it after its dt argument
        if r is None:
            assert got.get(kg) is None or kg == "dh0", kg
            continue
        if kg == "dh0" and not use_h0:
            continue
        errs[kg] = assert_grad_close(got[kg].float().cpu().numpy(), r, spec.torch_dtype, kg)
    return errs


SHAPES = [  # batch, d_inner, L, N
    (1, 1, 1, 1), (1, 3, 5, 4), (2, 5, 16, 16), (1, 32, 32, 16), (2, 33, 47, 16), (1, 40, 100, 5),
    (2, 64, 256, 16), (1, 37, 129, 8), (3, 20, 70, 20), (1, 24, 64, 32), (2, 70, 33, 1), (1, 16, 300, 12)]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b%d_d%d_l%d_n%d" % s)
def test_bwd_matches_oracle(shape, io):
    b, d, L, N = shape
    spec = I.ScanSpec(b, d, L, N, io=io, seed=1000 + L + N)
    run_case(spec)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [dict(use_D=False, use_z=False, use_bias=False, softplus=False),
                                  dict(use_h0=True), dict(use_dfinal=False), dict(use_z=False),
                                  dict(softplus=False), dict(use_h0=True, use_dfinal=False, use_D=False)],
                         ids=["bare", "h0", "no_dfinal", "no_gate", "no_softplus", "h0_only"])
def test_bwd_options(opts, io):
    spec = I.ScanSpec(2, 45, 77, 16, io=io, seed=7)
    if not opts.get("softplus", True):
        # a positive raw step without softplus: dt ~ |N(0, 0.1)| + bias > 0 is not
        # guaranteed, so shift the bias up
        spec = I.ScanSpec(2, 45, 77, 16, io=io, seed=8, dt_bias_const=5.0)
    run_case(spec, **opts)


def test_bwd_long_and_reset_steps():
    """A long row with sparse reset steps (step 5): the stored states at every
    16th step and the reverse walk over many chunks."""
    spec = I.ScanSpec(1, 64, 4096, 16, io="bf16", seed=3, dt_bias_const=1e-3, reset_frac=0.004)
    run_case(spec)


def test_bwd_headline_layer_full():
    """The headline layer shape (batch 8, d_inner 1536, L 2048, N 16, bf16),
    every gradient element against the oracle."""
    run_case(I.MAMBA130M)


SEG_SHAPES = [("bf16", (1, 64, 8192, 16)), ("bf16", (2, 40, 5000, 16)), ("bf16", (1, 33, 3000, 8)),
              ("bf16", (1, 32, 1024, 4)), ("f32", (2, 40, 5000, 16)), ("f32", (1, 33, 3000, 8)),
              ("f32", (1, 32, 1024, 4))]


@pytest.mark.parametrize("io,shape", SEG_SHAPES, ids=lambda v: v if isinstance(v, str) else "b%d_d%d_l%d_n%d" % v)
def test_bwd_segments_match_oracle(shape, io):
    """Rows long enough, with channel groups few enough, to be cut into
    cluster segments (up to 8): the folds of the states and of the adjoint
    across segments, a last segment that ends inside a chunk, an initial state
    and a final-state gradient."""
    b, d, L, N = shape
    spec = I.ScanSpec(b, d, L, N, io=io, seed=2000 + L + N)
    run_case(spec, use_h0=True)
    assert binding.device_faults() == 0


def test_bwd_long_sequence_full():
    """The long-sequence workload (batch 1, d_inner 2048, L 131072, N 16,
    bf16): one channel group per 32 channels walks 4096 chunks each way; every
    gradient element against the oracle."""
    errs = run_case(I.LONGSEQ)
    assert binding.device_faults() == 0
    print("long sequence backward: max normalised errors", errs)


def test_bwd_variant_headline_layer_full():
    """The variant the benchmark times: the backward of the reverse-direction
    scan with a sequence start every 250 steps on the headline layer shape,
    every gradient element against the oracle."""
    spec = I.MAMBA130M
    st = torch.zeros(spec.batch, spec.L, dtype=torch.uint8)
    st[:, ::250] = 1
    run_case(spec, seq_start=st, reverse=True)


def test_bwd_workspace_too_small_is_rejected():
    spec = I.ScanSpec(1, 8, 64, 16, io="f32", seed=1)
    inp = I.make_scan_inputs(spec)
    g = {k: v.cuda() for k, v in inp.items() if k != "reset_pos"}
    need = binding.scan_bwd_workspace_bytes(1, 8, 64, 16)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.SSError) as ei:
        binding.scan_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], torch.ones_like(g["x"]), workspace=ws)
    assert ei.value.status == -2


def test_bwd_repeat_is_stable():
    """Two calls on the same inputs: the io-dtype outputs are identical (the
    atomically accumulated fp32 sums may differ in their last bits)."""
    spec = I.ScanSpec(2, 64, 200, 16, io="bf16", seed=11)
    inp = I.make_scan_inputs(spec)
    bw = I.make_bwd_inputs(spec)
    g = {k: inp[k].cuda() for k in ("x", "dt", "z", "B", "C", "A", "D", "dt_bias")}
    outs = [binding.scan_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], bw["dout"].cuda(), D=g["D"], z=g["z"],
                             dt_bias=g["dt_bias"]) for _ in range(2)]
    torch.cuda.synchronize()
    for k in ("dx", "ddelta", "dz"):
        assert torch.equal(outs[0][k], outs[1][k]), k
    for k in ("dA", "dB", "dC", "dD", "ddt_bias"):
        torch.testing.assert_close(outs[0][k], outs[1][k], rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("shape", [(2, 64, 300, 16), (1, 64, 8192, 16), (2, 33, 47, 8), (8, 1536, 2048, 16)],
                         ids=lambda s: "b%d_d%d_l%d_n%d" % s)
def test_bwd_with_states_stored_by_the_training_forward(shape):
    """The training forward stores the state at every 16th step (also when it
    splits a long row into cluster segments); the backward then skips its own
    forward walk and gives the oracle's gradients."""
    b, d, L, N = shape
    spec = I.ScanSpec(b, d, L, N, io="bf16", seed=77 + L)
    inp = I.make_scan_inputs(spec)
    bw = I.make_bwd_inputs(spec)
    g = {k: inp[k].cuda() for k in ("x", "dt", "z", "B", "C", "A", "D", "dt_bias")}
    y0, f0 = binding.scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"])
    y1, f1, ws = binding.scan_fwd_train(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                                        dt_bias=g["dt_bias"])
    got = binding.scan_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], bw["dout"].cuda(), D=g["D"], z=g["z"],
                           dt_bias=g["dt_bias"], dfinal_state=bw["dfinal"].cuda(), workspace=ws,
                           states_from_forward=True)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(f0, f1)   # the stores do not change the forward's results
    ref = O.scan_bwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], bw["dout"], D=inp["D"], z=inp["z"],
                     dt_bias=inp["dt_bias"], dfinal=bw["dfinal"])
    for k, r in ref.items():
        if r is None or k == "dh0":
            continue
        kg = "ddelta" if k == "ddt" else k
        assert_grad_close(got[kg].float().cpu().numpy(), r, torch.bfloat16, kg)


def _starts(batch, L, seed, first=True, last=True):
    """Sequence starts: every row at step 0 (when `first`), a few seeded
    interior steps, and the last step (when `last`)."""
    rng = np.random.default_rng(seed)
    st = np.zeros((batch, L), dtype=np.uint8)
    for b in range(batch):
        if first:
            st[b, 0] = 1
        if L > 2:
            st[b, rng.choice(np.arange(1, L - 1), size=min(3, L - 2), replace=False)] = 1
        if last and L > 1:
            st[b, L - 1] = 1
    return torch.from_numpy(st)


EX_SHAPES = [  # batch, d_inner, L, N: a partial last chunk, a partial last 16-step block, several chunks
    (1, 1, 1, 1), (2, 5, 16, 16), (2, 33, 47, 16), (1, 40, 100, 5), (2, 64, 256, 16), (1, 37, 129, 8),
    (3, 20, 70, 20), (1, 16, 300, 12), (2, 24, 64, 32)]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("mode", ["reverse", "starts", "reverse_starts"])
@pytest.mark.parametrize("shape", EX_SHAPES, ids=lambda s: "b%d_d%d_l%d_n%d" % s)
def test_bwd_variants_match_oracle(shape, mode, io):
    """Gradient of the scan with the reverse direction and/or sequence starts
    (``ss_scan_bwd_ex_*``), with an initial state and a final-state gradient."""
    b, d, L, N = shape
    spec = I.ScanSpec(b, d, L, N, io=io, seed=2000 + L + N)
    st = _starts(b, L, seed=L) if "starts" in mode else None
    run_case(spec, use_h0=True, seq_start=st, reverse=mode.startswith("reverse"))


@pytest.mark.parametrize("mode", ["reverse", "starts", "reverse_starts"])
def test_bwd_variants_long_row(mode):
    """A 4096-step row with starts at a few hundred steps: the stored states and
    the cuts across many chunks and sub-chunks."""
    spec = I.ScanSpec(1, 64, 4096, 16, io="bf16", seed=5)
    st = None
    if "starts" in mode:
        rng = np.random.default_rng(11)
        st = torch.zeros(1, 4096, dtype=torch.uint8)
        st[0, rng.choice(4096, size=300, replace=False)] = 1
    run_case(spec, use_h0=True, seq_start=st, reverse=mode.startswith("reverse"))


def test_bwd_variants_reject_stored_forward_states():
    spec = I.ScanSpec(1, 8, 32, 4, io="f32", seed=1)
    inp = I.make_scan_inputs(spec)
    g = {k: inp[k].cuda() for k in ("x", "dt", "B", "C", "A")}
    ws = torch.zeros(binding.scan_bwd_workspace_bytes(1, 8, 32, 4), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        binding.scan_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["x"], workspace=ws, states_from_forward=True,
                         reverse=True)
