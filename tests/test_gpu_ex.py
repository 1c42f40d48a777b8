"""The extended scan (initial state, packed-sequence starts, reverse
direction) against the float64 oracle's definition of the same options."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from selective_state_space_138_b300 import binding
from selective_state_space_138_b300 import inputs as I
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu


def starts_for(spec, frac, seed):
    rng = np.random.default_rng(seed)
    st = rng.random((spec.batch, spec.L)) < frac
    return torch.from_numpy(st.astype(np.uint8))


def run(spec, use_h0, use_starts, reverse, frac=0.02):
    inp = I.make_scan_inputs(spec)
    h0 = I.make_bwd_inputs(spec)["h0"] if use_h0 else None
    st = starts_for(spec, frac, spec.seed + 99) if use_starts else None
    g = {k: inp[k].cuda() for k in ("x", "dt", "z", "B", "C", "A", "D", "dt_bias")}
    y, fs = binding.scan_fwd_ex(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"],
                                h0=None if h0 is None else h0.cuda(), seq_start=None if st is None else st.cuda(),
                                reverse=reverse)
    torch.cuda.synchronize()
    ry, rfs = O.scan_ex(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"], z=inp["z"],
                        dt_bias=inp["dt_bias"], h0=h0, seq_start=st, reverse=reverse)
    assert_close(y.float().cpu().numpy(), ry, spec.torch_dtype, "y")
    assert_close(fs.cpu().numpy(), rfs, torch.float32 if spec.io == "f32" else spec.torch_dtype, "final_state")


OPTS = [(True, False, False), (False, True, False), (False, False, True), (True, True, True), (False, True, True),
        (True, False, True)]
OPT_IDS = ["h0", "starts", "reverse", "all", "starts_reverse", "h0_reverse"]
SHAPES = [(1, 1, 1, 1), (2, 5, 33, 4), (1, 40, 100, 16), (2, 33, 257, 16), (1, 64, 130, 5), (2, 24, 64, 32),
          (3, 20, 45, 8)]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("opts", OPTS, ids=OPT_IDS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b%d_d%d_l%d_n%d" % s)
def test_ex_matches_oracle(shape, opts, io):
    b, d, L, N = shape
    run(I.ScanSpec(b, d, L, N, io=io, seed=300 + L), *opts)


@pytest.mark.parametrize("opts", OPTS, ids=OPT_IDS)
def test_ex_long_rows_split_into_cluster_segments(opts):
    """Few channels and a long row: the row is cut into segments joined through
    distributed shared memory; the segment fold must honour the initial state,
    the walking direction and sequence starts inside earlier segments."""
    run(I.ScanSpec(1, 32, 8192, 16, io="bf16", seed=5), *opts, frac=0.0005)


def test_ex_without_options_equals_the_plain_entry_point():
    spec = I.ScanSpec(2, 64, 300, 16, io="bf16", seed=9)
    inp = I.make_scan_inputs(spec)
    g = {k: inp[k].cuda() for k in ("x", "dt", "z", "B", "C", "A", "D", "dt_bias")}
    y0, f0 = binding.scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"])
    y1, f1 = binding.scan_fwd_ex(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"])
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(f0, f1)


def test_ex_rejects_large_N_with_options():
    x = torch.zeros(1, 4, 8, device="cuda")
    A = -torch.ones(4, 40, device="cuda")
    B = torch.zeros(1, 40, 8, device="cuda")
    with pytest.raises(binding.SSError) as ei:
        binding.scan_fwd_ex(x, x, A, B, B, reverse=True)
    assert ei.value.status == -3
