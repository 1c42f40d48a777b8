"""CUDA path (through the C ABI) against the float64 oracle, element by element.

Small problems and the full-size workloads (in the launch configuration the
benchmark uses) are compared in full, every row and every step. Tolerance: |gpu - oracle| <= atol + rtol |oracle|
with (rtol, atol) = (2e-2, 1e-3) for bf16 io and (1e-4, 1e-5) for fp32 io,
for y and for the final state.
"""
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O
from selective_state_space_138_b300 import binding
from selective_state_space_138_b300 import inputs as I
from tests.gpu_util import TOL, assert_close, compare_scan_all_rows, dev, gpu_scan, oracle_scan

pytestmark = pytest.mark.gpu

# kernel variants: the n-split kernel (whole sequence, or cut into 3 or 8
# segments joined through a thread-block cluster; "wide": its 2-stage form at
# four CTAs per SM, which 8 < N <= 16 takes), and the time-lane kernel with 1, 4,
# 16 lanes
LANES = ["nsplit", "seg3", "seg8", "wide", "1", "4", "16"]


@pytest.fixture
def lanes(request, monkeypatch):
    if request.param in ("nsplit", "wide"):
        monkeypatch.setenv("SS_SCAN_KERNEL", "nsplit")
        monkeypatch.setenv("SS_SCAN_SEGMENTS", "1")
        monkeypatch.setenv("SS_SCAN_WIDE", "1" if request.param == "wide" else "0")
        return 0
    if request.param.startswith("seg"):
        monkeypatch.setenv("SS_SCAN_KERNEL", "nsplit")
        monkeypatch.setenv("SS_SCAN_SEGMENTS", request.param[3:])
        return 0
    monkeypatch.setenv("SS_SCAN_KERNEL", "lanes")
    monkeypatch.setenv("SS_SCAN_LANES", request.param)
    return int(request.param)


@pytest.mark.parametrize("lanes", LANES, indirect=True)
def test_tiny_fp32_workload_in_full(lanes):
    inp = I.make_scan_inputs(I.TINY)
    y, fs = gpu_scan(inp)
    yr, fr = oracle_scan(inp)
    assert_close(y, yr, torch.float32, "y")
    assert_close(fs, fr, torch.float32, "final_state")


SHAPES = [
    # batch, d_inner, L, N, io
    (1, 1, 1, 1, "f32"), (1, 3, 7, 4, "f32"), (2, 37, 15, 16, "bf16"), (2, 37, 16, 16, "bf16"),
    (2, 37, 17, 16, "bf16"), (1, 130, 63, 5, "f32"), (3, 33, 64, 16, "bf16"), (1, 64, 65, 3, "bf16"),
    (2, 40, 255, 16, "f32"), (2, 40, 257, 16, "bf16"), (1, 129, 1000, 16, "bf16"),
    (1, 20, 300, 17, "f32"), (1, 12, 100, 64, "f32"), (2, 9, 77, 33, "bf16"), (1, 300, 33, 2, "bf16"),
]


@pytest.mark.parametrize("lanes", LANES, indirect=True)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b%d_d%d_l%d_n%d_%s" % s)
def test_shapes_and_ragged_tails(shape, lanes):
    batch, d, L, N, io = shape
    inp = I.make_scan_inputs(I.ScanSpec(batch=batch, d_inner=d, L=L, N=N, io=io, seed=100 + L))
    y, fs = gpu_scan(inp)
    yr, fr = oracle_scan(inp)
    dt = inp["x"].dtype
    assert_close(y, yr, dt, "y")
    assert_close(fs, fr, dt, "final_state")


OPTIONAL = [dict(use_D=False), dict(use_z=False), dict(use_bias=False), dict(softplus=False),
            dict(use_D=False, use_z=False, use_bias=False, softplus=False), dict(final_state=False)]


@pytest.mark.parametrize("lanes", ["nsplit", "seg3", "wide", "1", "16"], indirect=True)
@pytest.mark.parametrize("opt", OPTIONAL, ids=lambda o: "_".join("%s=%s" % kv for kv in o.items()))
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_optional_pointers_and_flag(opt, io, lanes):
    inp = I.make_scan_inputs(I.ScanSpec(batch=2, d_inner=24, L=200, N=16, io=io, seed=7))
    if opt.get("softplus") is False:
        # a positive step without softplus: |dt| + a positive bias
        inp["dt"] = inp["dt"].abs()
        inp["dt_bias"] = inp["dt_bias"].abs() * 0.01
    fs_on = opt.get("final_state", True)
    kw = {k: v for k, v in opt.items() if k != "final_state"}
    y, fs = gpu_scan(inp, final_state=fs_on, **kw)
    yr, fr = oracle_scan(inp, **kw)
    assert_close(y, yr, inp["x"].dtype, "y")
    if fs_on:
        assert_close(fs, fr, inp["x"].dtype, "final_state")
    else:
        assert fs is None


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("lanes", ["nsplit", "seg3", "16"], indirect=True)
def test_unaligned_pointers_take_the_scalar_path(io, lanes):
    inp = I.make_scan_inputs(I.ScanSpec(batch=2, d_inner=10, L=48, N=16, io=io, seed=8))
    g = dev(inp)
    shifted = {}
    for k in ("x", "dt", "z"):
        flat = torch.empty(g[k].numel() + 1, dtype=g[k].dtype, device="cuda")
        view = flat[1:].view(g[k].shape)
        view.copy_(g[k])
        shifted[k] = view
    assert shifted["x"].data_ptr() % 16 != 0
    y, fs = binding.scan_fwd(shifted["x"], shifted["dt"], g["A"], g["B"], g["C"], D=g["D"],
                             z=shifted["z"], dt_bias=g["dt_bias"])
    yr, fr = oracle_scan(inp)
    assert_close(y.float().cpu().numpy(), yr, inp["x"].dtype, "y")
    assert_close(fs.cpu().numpy(), fr, inp["x"].dtype, "final_state")


@pytest.mark.parametrize("lanes", ["nsplit", "seg8", "1"], indirect=True)
def test_extreme_steps_stay_finite(lanes):
    """Very large and very negative raw steps (softplus saturating both ways)."""
    inp = I.make_scan_inputs(I.ScanSpec(batch=1, d_inner=16, L=64, N=16, io="f32", seed=9))
    inp["dt"][0, :4, ::7] = 60.0
    inp["dt"][0, 4:8, ::5] = -60.0
    y, fs = gpu_scan(inp)
    yr, fr = oracle_scan(inp)
    assert_close(y, yr, torch.float32, "y")
    assert_close(fs, fr, torch.float32, "final_state")


def test_repeat_calls_are_bitwise_identical_and_stream_respected():
    inp = I.make_scan_inputs(I.ScanSpec(batch=2, d_inner=64, L=512, N=16, io="bf16", seed=10))
    g = dev(inp)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y1, f1 = binding.scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["z"], g["dt_bias"])
    s.synchronize()
    y2, f2 = binding.scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["z"], g["dt_bias"])
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(f1, f2)


def test_host_pointer_is_rejected_before_launch():
    inp = I.make_scan_inputs(I.ScanSpec(batch=1, d_inner=8, L=16, N=4, io="f32", seed=1))
    g = dev(inp)
    with pytest.raises(binding.SSError) as e:
        binding.scan_fwd(inp["x"], g["dt"], g["A"], g["B"], g["C"])
    assert e.value.status == -4
    state = torch.zeros(1, 8, 4)
    with pytest.raises(binding.SSError) as e:
        binding.state_update(state, g["x"][:, :, 0].contiguous(), g["dt"][:, :, 0].contiguous(), g["A"],
                             g["B"][:, :, 0].contiguous(), g["C"][:, :, 0].contiguous())
    assert e.value.status == -4


# ----------------------------------------------------------------- full sizes

@pytest.mark.parametrize("name", [I.MAMBA130M.name, I.MAMBA1P4B.name, I.LONGSEQ.name])
def test_full_size_workloads_every_row(name):
    """The three large workloads at full size, in the launch configuration the
    benchmark times, compared with the oracle on every (batch, channel) row:
    every step of y and every final state."""
    spec = I.SCAN_WORKLOADS[name]
    inp = I.make_scan_inputs(spec)
    g = dev(inp)
    binding.device_faults(clear=True)
    y, fs = binding.scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                             dt_bias=g["dt_bias"])
    torch.cuda.synchronize()
    assert binding.device_faults() == 0
    del g
    wy, wf = compare_scan_all_rows(inp, y, fs, torch.bfloat16, what=name)
    print("%s: max normalised error y %.3f, final state %.3f (1.0 = tolerance)" % (name, wy, wf))


# ----------------------------------------------------------------- decode

def _gpu_decode(tokens, params, state=None, use_D=True, use_z=True):
    T, Bt, Dn = tokens["x"].shape
    N = params["A"].shape[1]
    gt = {k: v.cuda() for k, v in tokens.items()}
    A = params["A"].cuda()
    D = params["D"].cuda() if use_D else None
    st = torch.zeros(Bt, Dn, N, device="cuda") if state is None else state
    ys = torch.empty_like(gt["x"])
    for t in range(T):
        binding.state_update(st, gt["x"][t], gt["delta"][t], A, gt["B"][t], gt["C"][t], D=D,
                             z=gt["z"][t] if use_z else None, y=ys[t])
    torch.cuda.synchronize()
    return ys, st


@pytest.mark.parametrize("N", [16, 5, 64, 1])
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_decode_chain_equals_oracle_scan(N, io):
    spec = I.DecodeSpec(batch=3, d_inner=50, N=N, steps=40, seed=21)
    tok = I.make_decode_tokens(spec)
    par = I.make_decode_params(spec)
    if io == "f32":
        tok = {k: v.float() for k, v in tok.items()}
    ys, st = _gpu_decode(tok, par)
    rows = list(range(spec.batch * spec.d_inner))
    yr, fr = O.decode_chain(tok, par, rows)
    dt = tok["x"].dtype
    got = ys.float().cpu().numpy().reshape(spec.steps, -1).T
    assert_close(got, yr, dt, "decode y")
    assert_close(st.cpu().numpy().reshape(-1, N), fr, dt, "decode state")


def test_decode_without_skip_and_gate():
    spec = I.DecodeSpec(batch=2, d_inner=33, N=16, steps=12, seed=22)
    tok = I.make_decode_tokens(spec)
    par = I.make_decode_params(spec)
    ys, st = _gpu_decode(tok, par, use_D=False, use_z=False)
    rows = list(range(spec.batch * spec.d_inner))
    yr, fr = O.decode_chain(tok, par, rows, use_D=False, use_z=False)
    assert_close(ys.float().cpu().numpy().reshape(spec.steps, -1).T, yr, torch.bfloat16, "y")
    assert_close(st.cpu().numpy().reshape(-1, 16), fr, torch.bfloat16, "state")


def test_prefill_scan_then_decode_continues_the_state():
    """Prefill keeps only the final state; decode continues from it."""
    spec = I.ScanSpec(batch=2, d_inner=40, L=300, N=16, io="bf16", seed=23)
    inp = I.make_scan_inputs(spec)
    g = dev(inp)
    _, fs = binding.scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                             dt_bias=g["dt_bias"])
    dspec = I.DecodeSpec(batch=2, d_inner=40, N=16, steps=25, seed=24)
    tok = I.make_decode_tokens(dspec)
    par = dict(A=inp["A"], D=inp["D"])
    ys, st = _gpu_decode(tok, par, state=fs.clone())
    rows = list(range(80))
    _, fr0 = O.scan_rows(inp, rows)
    yr, fr = O.decode_chain(tok, par, rows, h0=fr0)
    assert_close(ys.float().cpu().numpy().reshape(25, -1).T, yr, torch.bfloat16, "decode y")
    assert_close(st.cpu().numpy().reshape(-1, 16), fr, torch.bfloat16, "decode state")


def test_full_size_decode_every_row_and_step():
    """The decode workload (batch 256, d_inner 5120, N 16, 1024 tokens) against
    the oracle's scan over the same tokens, on every (batch, channel) row:
    y of every step and the state after the last one."""
    spec = I.DECODE
    tok = I.make_decode_tokens(spec)
    par = I.make_decode_params(spec)
    binding.device_faults(clear=True)
    ys, st = _gpu_decode(tok, par)
    assert binding.device_faults() == 0
    worst_y = worst_s = 0.0
    for b in range(spec.batch):
        rows = list(range(b * spec.d_inner, (b + 1) * spec.d_inner))
        yr, fr = O.decode_chain(tok, par, rows)
        got = ys[:, b, :].float().cpu().numpy().T
        worst_y = max(worst_y, assert_close(got, yr, torch.bfloat16, "decode y (every step) b%d" % b))
        worst_s = max(worst_s, assert_close(st[b].cpu().numpy(), fr, torch.bfloat16, "decode state b%d" % b))
    print("%s: max normalised error y %.3f, state %.3f (1.0 = tolerance)" % (spec.name, worst_y, worst_s))


# ----------------------------------------------------------------- device math probes

@pytest.mark.parametrize("lanes", ["nsplit", "1"], indirect=True)
def test_step_softplus_through_the_abi(lanes):
    """With L = 1, A = 0, B = C = x = 1 and no skip or gate, y = softplus(dt + bias)."""
    v = np.concatenate([np.linspace(-30, 30, 4001), [-1000.0, -88.0, -20.0, 0.0, 20.0, 88.0, 1000.0]])
    d = v.size
    bias = np.float32(0.37)
    dt = torch.tensor(v - bias, dtype=torch.float32).view(1, d, 1)
    ones = torch.ones(1, 1, 1, device="cuda")
    y, _ = binding.scan_fwd(torch.ones(1, d, 1, device="cuda"), dt.cuda(), torch.zeros(d, 1, device="cuda"),
                            ones, ones, dt_bias=torch.full((d,), float(bias), device="cuda"),
                            return_final_state=False)
    got = y.view(-1).cpu().double().numpy()
    arg = dt.view(-1).double().numpy() + np.float64(bias)
    ref = np.array([O.softplus(a) for a in arg])
    # float32 rounding of the exponent argument v*log2(e) costs up to about
    # |v| * 6e-8 relative; results below the float32 normal range flush to zero
    err = np.abs(got - ref)
    tol = (2e-6 + 1e-7 * np.abs(arg)) * ref
    ok = (err <= tol) | ((ref < 1.18e-38) & (err <= 1.18e-38))
    assert np.all(np.isfinite(got))
    assert ok.all(), (arg[~ok][:5], got[~ok][:5], ref[~ok][:5])


@pytest.mark.parametrize("lanes", ["nsplit", "1"], indirect=True)
def test_gate_silu_through_the_abi(lanes):
    """With L = 1, B = C = 0, D = 1, x = 1, y = silu(z) = z sigmoid(z)."""
    zv = np.concatenate([np.linspace(-40, 40, 4001), [-200.0, -88.0, 88.0, 200.0]])
    d = zv.size
    z = torch.tensor(zv, dtype=torch.float32).view(1, d, 1)
    zeros = torch.zeros(1, 1, 1, device="cuda")
    y, _ = binding.scan_fwd(torch.ones(1, d, 1, device="cuda"), torch.zeros(1, d, 1, device="cuda"),
                            torch.zeros(d, 1, device="cuda"), zeros, zeros, D=torch.ones(d, device="cuda"),
                            z=z.cuda(), delta_softplus=False, return_final_state=False)
    got = y.view(-1).cpu().double().numpy()
    zz = z.view(-1).double().numpy()
    ref = zz / (1.0 + np.exp(-zz))
    err = np.abs(got - ref)
    tol = (2e-6 + 1e-7 * np.abs(zz)) * np.abs(ref) + 1e-30
    assert np.all(np.isfinite(got))
    assert np.all(err <= tol), (zz[err > tol][:5], got[err > tol][:5], ref[err > tol][:5])
