"""The oracle against the pages' printed numbers, closed forms and brute force."""
import math
import random

import numpy as np
import pytest

from oracle import oracle as O
from tests import oracle_pins as P


@pytest.fixture(scope="module")
def lib():
    return O.load()


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(lib, check):
    check(lib)


def test_zoh_fixed_points():
    g = P.GOLDEN["zoh"]
    for c in g["cases"]:
        a_bar, b_bar = O.zoh(c["delta"], g["A"], g["B"])
        assert round(a_bar, g["digits"]) == c["A_bar"]
        assert round(b_bar, g["digits"]) == c["B_bar"]
        # with A = -1 and B = 1 the keep and write shares add up to one
        assert abs(a_bar + b_bar - 1.0) < 1e-15


def test_gate_theorem_zoh():
    """Under ZOH with delta = softplus(z), A = -1, B = 1: decay 1 - sigma(z), write sigma(z)."""
    from scipy.special import expit
    for zv in np.linspace(-30, 30, 61):
        a_bar, b_bar = O.zoh(O.softplus(zv), -1.0, 1.0) if zv > -30 else (1.0, 0.0)
        assert abs(a_bar - (1.0 - expit(zv))) < 1e-12
        if zv > -30:
            assert abs(b_bar - expit(zv)) < 1e-12


def test_merge_fixed_points():
    g = P.GOLDEN["merge"]
    s = [tuple(p) for p in g["steps"]]
    m12 = O.affine_combine(s[0], s[1])
    m34 = O.affine_combine(s[2], s[3])
    assert m12 == tuple(g["steps_1_2"])
    assert m34 == tuple(g["steps_3_4"])
    assert O.affine_combine(m12, m34) == tuple(g["all_four"])
    # the final state of the loop equals the second slot of the full merge
    assert O.affine_scan(s)[-1] == g["all_four"][1]
    assert O.affine_scan(s) == P.GOLDEN["recurrence"]["y"]


def _tree_reduce(pairs, rng):
    items = list(pairs)
    while len(items) > 1:
        i = rng.randrange(len(items) - 1)
        items[i:i + 2] = [O.affine_combine(items[i], items[i + 1])]
    return items[0]


def test_combine_is_associative_in_any_tree_order():
    rng = random.Random(1)
    nprng = np.random.default_rng(2)
    for _ in range(20):
        L = int(nprng.integers(1, 40))
        pairs = list(zip(np.exp(-np.abs(nprng.normal(size=L))), nprng.normal(size=L)))
        h0 = float(nprng.normal())
        loop = O.affine_scan(pairs, h0)[-1]
        a, b = _tree_reduce(pairs, rng)
        assert abs((a * h0 + b) - loop) < 1e-12
        # every prefix, as a scan over the combine operator
        acc = (1.0, 0.0)
        for t, p in enumerate(pairs):
            acc = O.affine_combine(acc, p)
            assert abs(acc[0] * h0 + acc[1] - O.affine_scan(pairs[:t + 1], h0)[-1]) < 1e-12


def test_selective_copy_zoh_fixed_point():
    g = P.GOLDEN["selective_copy_zoh"]
    pairs = []
    for xv, dv in zip(g["x"], g["delta"]):
        if dv == 0.0:
            pairs.append((1.0, 0.0))  # the limit of ZOH at a zero step: keep all, write nothing
        else:
            a_bar, b_bar = O.zoh(dv, g["A"], g["B"])
            pairs.append((a_bar, b_bar * xv))
    h = O.affine_scan(pairs)
    assert [round(v, g["digits"]) for v in h] == g["h"]


def test_scan_rows_and_decode_chain_match_full_scan():
    import torch
    rng = np.random.default_rng(4)
    x, dt, A, B, C, D, z, dt_bias = P.random_problem(rng, bt=3, dn=5, L=17, N=4)
    y, fs = O.scan(x, dt, A, B, C, D=D, z=z, dt_bias=dt_bias, threads=3)
    inp = dict(x=x, dt=dt, z=z, B=B, C=C, A=A, D=D, dt_bias=dt_bias)
    rows = [0, 4, 7, 14]
    yr, fr = O.scan_rows(inp, rows)
    np.testing.assert_array_equal(yr, y.reshape(15, 17)[rows])
    np.testing.assert_array_equal(fr, fs.reshape(15, 4)[rows])
    # decode tokens in (steps, batch, d_inner) layout; delta already final
    delta = np.logaddexp(0.0, dt + dt_bias[None, :, None])
    tok = dict(x=np.transpose(x, (2, 0, 1)), delta=np.transpose(delta, (2, 0, 1)),
               z=np.transpose(z, (2, 0, 1)), B=np.transpose(B, (2, 0, 1)), C=np.transpose(C, (2, 0, 1)))
    yd, fd = O.decode_chain(tok, dict(A=A, D=D), rows)
    y2, fs2 = O.scan(x, delta, A, B, C, D=D, z=z, delta_softplus=False)
    np.testing.assert_array_equal(yd, y2.reshape(15, 17)[rows])
    np.testing.assert_array_equal(fd, fs2.reshape(15, 4)[rows])
    np.testing.assert_allclose(yd, y.reshape(15, 17)[rows], rtol=1e-12, atol=1e-13)


def test_oracle_rejects_bad_arguments():
    lib = O.load()
    import ctypes
    null = ctypes.POINTER(ctypes.c_double)()
    assert lib.oracle_scan_rows(null, null, null, null, null, null, null, null, 1, null, null, null,
                                1, 1, 1, 1, 0, 1) == -1
