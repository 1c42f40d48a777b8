"""The forward scan's two ways of staging a chunk in shared memory: tensor
copies (cp.async.bulk.tensor through tensor maps, the default when rows are
16-byte aligned) and per-thread 16-byte cp.async pieces (SS_SCAN_TMA=0).
Only the staging differs, so the outputs must agree bit for bit; the
tensor-copy path is also checked against the float64 oracle, the device
fault word must stay clear, and inputs whose rows are not 16-byte aligned
take the piece path and stay correct."""
import numpy as np
import pytest
import torch

from selective_state_space_138_b300 import binding
from selective_state_space_138_b300 import inputs as I
from tests.gpu_util import assert_close, dev, oracle_scan

pytestmark = pytest.mark.gpu

# L a multiple of 16 (the aligned-row condition): L below the 40-step raw row
# box, d_inner and N not multiples of the tile, every state split (N <= 4, 8,
# 16, 32), both io dtypes
SHAPES = [
    # batch, d_inner, L, N, io
    (2, 37, 16, 16, "bf16"), (1, 5, 32, 3, "f32"), (3, 33, 64, 16, "bf16"), (2, 40, 256, 8, "f32"),
    (1, 130, 1008, 16, "bf16"), (2, 64, 512, 32, "bf16"), (1, 96, 2048, 16, "f32"), (1, 32, 48, 12, "bf16"),
]


def _run(inp, monkeypatch, tma: bool, segments: int, **kw):
    monkeypatch.setenv("SS_SCAN_KERNEL", "nsplit")
    monkeypatch.setenv("SS_SCAN_SEGMENTS", str(segments))
    monkeypatch.setenv("SS_SCAN_TMA", "1" if tma else "0")
    g = dev(inp)
    fn = binding.scan_fwd_ex if kw else binding.scan_fwd
    y, fs = fn(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"], **kw)
    torch.cuda.synchronize()
    return y.float().cpu().numpy(), fs.cpu().numpy()


@pytest.mark.parametrize("segments", [1, 3])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b%d_d%d_l%d_n%d_%s" % s)
def test_tensor_copies_match_pieces_bit_for_bit(shape, segments, monkeypatch):
    batch, d, L, N, io = shape
    inp = I.make_scan_inputs(I.ScanSpec(batch=batch, d_inner=d, L=L, N=N, io=io, seed=300 + L))
    binding.device_faults(clear=True)
    y1, f1 = _run(inp, monkeypatch, True, segments)
    assert binding.device_faults() == 0
    y0, f0 = _run(inp, monkeypatch, False, segments)
    assert np.array_equal(y1, y0) and np.array_equal(f1, f0)
    yr, fr = oracle_scan(inp)
    assert_close(y1, yr, inp["x"].dtype, "y")
    assert_close(f1, fr, inp["x"].dtype, "final_state")


@pytest.mark.parametrize("variant", ["reverse", "starts", "h0"])
def test_tensor_copies_in_the_scan_variants(variant, monkeypatch):
    spec = I.ScanSpec(batch=2, d_inner=48, L=320, N=16, io="bf16", seed=41)
    inp = I.make_scan_inputs(spec)
    kw = {}
    if variant == "reverse":
        kw["reverse"] = True
    elif variant == "starts":
        st = torch.zeros(spec.batch, spec.L, dtype=torch.uint8)
        st[0, [0, 17, 160, 161]] = 1
        st[1, [5, 300]] = 1
        kw["seq_start"] = st.cuda()
    else:
        kw["h0"] = I.normal(41, 11, (spec.batch, spec.d_inner, spec.N), 0.5, torch.float32).cuda()
    binding.device_faults(clear=True)
    for seg in (1, 3):
        y1, f1 = _run(inp, monkeypatch, True, seg, **kw)
        y0, f0 = _run(inp, monkeypatch, False, seg, **kw)
        assert np.array_equal(y1, y0) and np.array_equal(f1, f0), (variant, seg)
    assert binding.device_faults() == 0


def test_unaligned_B_rows_take_the_piece_path(monkeypatch):
    """B and C one element past a 16-byte boundary: staged element by element
    (no 16-byte copies from them), still equal to the oracle."""
    monkeypatch.setenv("SS_SCAN_KERNEL", "nsplit")
    monkeypatch.setenv("SS_SCAN_SEGMENTS", "1")
    inp = I.make_scan_inputs(I.ScanSpec(batch=2, d_inner=40, L=128, N=16, io="bf16", seed=9))
    g = dev(inp)
    shifted = {}
    for k in ("B", "C"):
        buf = torch.empty(g[k].numel() + 1, dtype=g[k].dtype, device="cuda")
        shifted[k] = buf[1:].view(g[k].shape)
        shifted[k].copy_(g[k])
        assert shifted[k].data_ptr() % 16 != 0
    y, fs = binding.scan_fwd(g["x"], g["dt"], g["A"], shifted["B"], shifted["C"], D=g["D"], z=g["z"],
                             dt_bias=g["dt_bias"])
    torch.cuda.synchronize()
    yr, fr = oracle_scan(inp)
    assert_close(y.float().cpu().numpy(), yr, torch.bfloat16, "y")
    assert_close(fs.cpu().numpy(), fr, torch.bfloat16, "final_state")
