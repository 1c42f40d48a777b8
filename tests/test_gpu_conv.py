"""Causal depthwise conv1d (+ SiLU) and its decode cache, CUDA path against the
float64 oracle, element by element (same tolerances as the scan)."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from selective_state_space_138_b300 import binding
from selective_state_space_138_b300 import inputs as I
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu


def _conv_inputs(batch, d, L, k, io, seed):
    dt = torch.bfloat16 if io == "bf16" else torch.float32
    x = I.normal(seed, 1, (batch, d, L), 1.0, dt)
    w = I.normal(seed, 2, (d, k), 0.5, torch.float32)
    bias = I.normal(seed, 3, (d,), 0.2, torch.float32)
    st = I.normal(seed, 4, (batch, max(k - 1, 0), d), 1.0, dt)
    return x, w, bias, st


CASES = [(1, 1, 1, 4), (2, 3, 3, 4), (2, 5, 7, 4), (1, 16, 8, 4), (3, 33, 9, 4), (2, 64, 100, 4),
         (1, 40, 257, 1), (2, 40, 64, 2), (2, 40, 65, 3), (2, 24, 131, 5), (1, 24, 96, 6), (1, 24, 77, 7),
         (2, 24, 200, 8), (8, 1536, 2048, 4),
         # several shared-memory tiles per row, history longer than a piece, L shorter than the history
         (2, 17, 2056, 6), (1, 12, 3072, 8), (2, 9, 4, 8), (3, 11, 1032, 4),
         # tensor-copy tiles: channels past the last group of 8, a row ending inside a segment,
         # a row of one piece, a last tile of one segment, many tiles per CTA
         (2, 13, 136, 4), (1, 5, 8, 4), (2, 20, 1088, 8), (4, 24, 3000, 3), (2, 7, 16, 2), (16, 64, 4096, 4)]


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "b%d_d%d_l%d_k%d" % c)
def test_conv_matches_oracle(case, io):
    batch, d, L, k = case
    x, w, bias, st = _conv_inputs(batch, d, L, k, io, seed=L + k)
    for silu, use_bias, use_state in ((True, True, False), (False, False, True), (True, True, True)):
        si = st.cuda() if use_state and k > 1 else None
        out, so = binding.causal_conv1d(x.cuda(), w.cuda(), bias.cuda() if use_bias else None, state_in=si,
                                        silu=silu, return_state=True)
        torch.cuda.synchronize()
        ref, ref_st = O.causal_conv1d(x, w, bias if use_bias else None, silu=silu,
                                      state=st if use_state and k > 1 else None)
        assert_close(out.float().cpu().numpy(), ref, x.dtype, "conv out")
        if k > 1:
            np.testing.assert_array_equal(so.float().cpu().numpy(), ref_st)   # the cache is copied inputs


def test_conv_unaligned_input_takes_the_scalar_path():
    x, w, bias, _ = _conv_inputs(2, 10, 48, 4, "bf16", seed=5)
    flat = torch.empty(x.numel() + 1, dtype=x.dtype, device="cuda")
    xs = flat[1:].view(x.shape)
    xs.copy_(x.cuda())
    assert xs.data_ptr() % 16 != 0
    out, _ = binding.causal_conv1d(xs, w.cuda(), bias.cuda())
    ref, _ = O.causal_conv1d(x, w, bias)
    assert_close(out.float().cpu().numpy(), ref, x.dtype, "conv out")


@pytest.mark.parametrize("d", [40, 37])
@pytest.mark.parametrize("k", [1, 2, 4, 8])
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_conv_decode_steps_equal_one_pass(k, io, d):
    """Prefill a prompt, hand its last k-1 inputs to the decode cache, then
    step token by token: every step's output equals the one-pass convolution."""
    batch, L, L1 = 3, 37, 20
    x, w, bias, _ = _conv_inputs(batch, d, L, k, io, seed=9 + k)
    g = x.cuda()
    _, cache = binding.causal_conv1d(g[:, :, :L1].contiguous(), w.cuda(), bias.cuda(), return_state=True)
    if cache is None:
        cache = torch.empty((batch, 0, d), dtype=x.dtype, device="cuda")
    outs = []
    for t in range(L1, L):
        outs.append(binding.conv_state_update(cache, g[:, :, t].contiguous(), w.cuda(), bias.cuda()))
    torch.cuda.synchronize()
    ref, ref_st = O.causal_conv1d(x, w, bias)
    got = torch.stack(outs, dim=2).float().cpu().numpy()
    assert_close(got, ref[:, :, L1:], x.dtype, "decode conv")
    if k > 1:
        np.testing.assert_array_equal(cache.float().cpu().numpy(), ref_st)


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_conv_step_decode_shape(io):
    """One decode step at the decode workload's shape (256 x 5120, k = 4) from
    a random cache."""
    batch, d, k = 256, 5120, 4
    x, w, bias, st = _conv_inputs(batch, d, 1, k, io, seed=77)
    cache = st.cuda().contiguous()
    out = binding.conv_state_update(cache, x[:, :, 0].contiguous().cuda(), w.cuda(), bias.cuda())
    torch.cuda.synchronize()
    ref, ref_st = O.causal_conv1d(x, w, bias, state=st)
    assert_close(out.float().cpu().numpy(), ref[:, :, 0], x.dtype, "decode conv")
    np.testing.assert_array_equal(cache.float().cpu().numpy(), ref_st)
