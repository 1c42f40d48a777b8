"""The backward pass through its no-allocation entry point (built-in device
scratch instead of a caller workspace) gives the results of the workspace entry
point, on two consecutive calls that reuse the same scratch."""
import pytest
import torch

from selective_state_space_138_b300 import binding
from selective_state_space_138_b300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_noalloc_matches_workspace_entry_point(io):
    spec = I.ScanSpec(2, 96, 700, 16, io=io, seed=21)
    inp = I.make_scan_inputs(spec)
    bw = I.make_bwd_inputs(spec)
    g = {k: inp[k].cuda() for k in ("x", "dt", "z", "B", "C", "A", "D", "dt_bias")}
    args = (g["x"], g["dt"], g["A"], g["B"], g["C"], bw["dout"].cuda())
    kw = dict(D=g["D"], z=g["z"], dt_bias=g["dt_bias"], h0=bw["h0"].cuda(), dfinal_state=bw["dfinal"].cuda())
    assert binding.scan_bwd_workspace_bytes(2, 96, 700, 16) <= binding.BWD_NOALLOC_MAX_BYTES
    ref = binding.scan_bwd(*args, **kw)
    for _ in range(2):   # the second call reuses the scratch the first one wrote
        got = binding.scan_bwd(*args, **kw, noalloc=True)
        torch.cuda.synchronize()
        for k in ("dx", "ddelta", "dz", "dh0"):
            assert torch.equal(got[k], ref[k]), k
        for k in ("dA", "dB", "dC", "dD", "ddt_bias"):   # fp32 atomic sums: order may differ
            torch.testing.assert_close(got[k], ref[k], rtol=1e-5, atol=1e-5)


def test_noalloc_rejects_a_problem_larger_than_its_scratch():
    spec = I.MAMBA130M
    x = torch.zeros(spec.batch, spec.d_inner, spec.L, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(spec.batch, spec.N, spec.L, dtype=torch.bfloat16, device="cuda")
    A = -torch.ones(spec.d_inner, spec.N, device="cuda")
    with pytest.raises(binding.SSError) as ei:
        binding.scan_bwd(x, x, A, B, B, x, noalloc=True)
    assert ei.value.status == -2 and "built-in scratch" in str(ei.value)
