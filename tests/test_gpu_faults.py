"""The bounded waits of the kernels: a wait that nothing completes gives up
after its limit, records the fault in the device word the host reads, and
leaves the context usable (no trap, no hang)."""
import time

import numpy as np
import pytest
import torch

from oracle import oracle as O
from selective_state_space_138_b300 import binding
from selective_state_space_138_b300 import inputs as I

pytestmark = pytest.mark.gpu


def test_bounded_wait_records_its_fault_and_the_context_survives():
    torch.cuda.set_device(0)
    assert binding.device_faults(clear=True) == 0
    t0 = time.monotonic()
    binding.fault_probe()
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    flags = binding.device_faults(clear=True)
    assert flags & binding.FAULT_WAIT_TIMEOUT, flags
    assert 0.9 <= waited < 30.0, waited   # the one-second bound, not an endless wait
    assert binding.device_faults(clear=True) == 0   # cleared

    # the context still runs kernels and gives the oracle's results
    spec = I.ScanSpec(1, 40, 100, 16, io="f32", seed=11)
    inp = I.make_scan_inputs(spec)
    g = {k: v.cuda() for k, v in inp.items() if k != "reset_pos"}
    y, fs = binding.scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"])
    torch.cuda.synchronize()
    yr, fr = O.scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"], z=inp["z"], dt_bias=inp["dt_bias"])
    assert np.all(np.abs(y.cpu().numpy() - yr) <= 1e-5 + 1e-4 * np.abs(yr))
    assert np.all(np.abs(fs.cpu().numpy() - fr) <= 1e-5 + 1e-4 * np.abs(fr))
    assert binding.device_faults() == 0
