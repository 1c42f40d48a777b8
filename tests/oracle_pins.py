"""Pins of the float64 oracle to facts outside itself.

Each ``check_*`` takes the loaded oracle library (so the same checks can be run
against deliberately broken copies of the oracle, see test_oracle_mutants.py)
and raises AssertionError when the oracle disagrees with:
  * numbers printed on the pages (tests/golden/pages_fixed_points.json),
  * closed forms derived from the pages' definitions and theorems, or
  * brute-force evaluations of the pages' unrolled (mixing-matrix) form, which
    use a different computation (exponential of summed steps, matrix product,
    numpy convolution) from the oracle's loop.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy.special import expit

from oracle import oracle as O

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_fixed_points.json")))


def _round_eq(got, want, digits):
    assert round(float(got), digits) == round(float(want), digits), (got, want, digits)


def _scan1(lib, x, delta, A=-1.0, B=1.0, C=1.0, D=None, softplus=False, dt_bias=None, z=None, h0=None):
    """One channel, one state: scalar helper around the oracle scan."""
    L = len(x)
    xs = np.asarray(x, dtype=np.float64).reshape(1, 1, L)
    dts = np.asarray(delta, dtype=np.float64).reshape(1, 1, L)
    Bs = np.broadcast_to(np.asarray(B, dtype=np.float64), (L,)).reshape(1, 1, L).copy()
    Cs = np.broadcast_to(np.asarray(C, dtype=np.float64), (L,)).reshape(1, 1, L).copy()
    y, fs = O.scan(xs, dts, np.array([[A]]), Bs, Cs,
                   D=None if D is None else np.array([D]),
                   z=None if z is None else np.asarray(z, dtype=np.float64).reshape(1, 1, L),
                   dt_bias=None if dt_bias is None else np.array([dt_bias]),
                   delta_softplus=softplus,
                   h0=None if h0 is None else np.array(h0, dtype=np.float64).reshape(1, 1, 1),
                   threads=1, lib=lib)
    return y[0, 0], fs[0, 0, 0]


# ------------------------------------------------------------ page numbers

def check_recurrence_example(lib):
    """A_bar = 0.5, B_bar = 1, C = 1, x = (1,0,0,2) gives states 1, .5, .25, 2.125.
    With the scan's Euler rule: delta = ln 2 and A = -1 give exp(delta A) = 0.5;
    B = 1/ln 2 gives delta*B = 1."""
    g = GOLDEN["recurrence"]
    y, fs = _scan1(lib, g["x"], [math.log(2.0)] * 4, A=-1.0, B=1.0 / math.log(2.0), C=g["C"])
    np.testing.assert_allclose(y, g["y"], rtol=0, atol=1e-12)
    assert abs(fs - g["y"][-1]) < 1e-12
    # the same outputs by the convolution with the printed kernel
    K = np.array(g["kernel"])
    conv = np.convolve(np.array(g["x"]), K)[:4]
    np.testing.assert_allclose(y, conv, atol=1e-12)
    assert abs(conv[3] - g["y4_by_convolution"]) < 1e-12


def check_softplus_values(lib):
    for v, want, digits in GOLDEN["softplus"]["cases"]:
        _round_eq(lib.oracle_softplus(v), want, digits)
    # extreme inputs stay finite ("Selection is a gate, numerically")
    assert lib.oracle_softplus(1000.0) == 1000.0
    assert lib.oracle_softplus(-1000.0) == 0.0
    for v, want, digits in GOLDEN["softplus_inverse"]["cases"]:
        _round_eq(math.log(math.expm1(v)), want, digits)
    u, want, digits = GOLDEN["softplus_inverse"]["roundtrip"]
    _round_eq(lib.oracle_softplus(math.log(math.expm1(u))), want, digits)


def check_gate_theorem(lib):
    """Selection is a gate: with N = 1, A = -1, B = 1 and delta = softplus(z),
    the decay is 1 - sigma(z). Under the scan's Euler rule the write is
    softplus(z) (the theorem's closing remark). Checked through the scan with
    the bias split off: dt = z - b, dt_bias = b."""
    for c in GOLDEN["gate"]["cases"]:
        z = c["z"]
        _round_eq(lib.oracle_softplus(z), c["delta"], GOLDEN["gate"]["digits"])
        _round_eq(math.exp(-lib.oracle_softplus(z)), c["A_bar"], GOLDEN["gate"]["digits"])
        _round_eq(expit(z), c["gate"], GOLDEN["gate"]["digits"])
    rng = np.random.default_rng(11)
    zs = rng.normal(0, 3, size=40)
    zs[5], zs[17] = 40.0, -40.0
    xs = rng.normal(size=40)
    b = 0.37
    y, _ = _scan1(lib, xs, zs - b, A=-1.0, B=1.0, C=1.0, softplus=True, dt_bias=b)
    h = 0.0
    for t in range(40):
        h = (1.0 - expit(zs[t])) * h + np.logaddexp(0.0, zs[t]) * xs[t]
        assert abs(y[t] - h) <= 1e-12 * max(1.0, abs(h)), (t, y[t], h)


def check_selective_copy_euler(lib):
    """The hand example's inputs x = (3,9,9,7,9), delta = (5,0,0,5,0) under the
    scan's Euler rule: h1 = 5*3 = 15, filler leaves it, h4 = e^-5 * 15 + 5*7."""
    g = GOLDEN["selective_copy_zoh"]
    y, fs = _scan1(lib, g["x"], g["delta"], A=g["A"], B=g["B"], C=g["C"])
    h4 = math.exp(-5.0) * 15.0 + 35.0
    np.testing.assert_allclose(y, [15.0, 15.0, 15.0, h4, h4], rtol=1e-14, atol=0)
    _round_eq(h4, 35.1011, 4)


# ------------------------------------------------------------ closed forms

def check_impulse_response(lib):
    """Impulse response of a 4-state channel ("State-space models & Mamba",
    section 'Discretization: making SSMs computable'): A = (-1,-.5,-.25,-.1),
    B = 1, C = (.5,.3,.15,.05), delta = .1, x = unit impulse, Euler input weight
    delta*B. Closed form: y[t] = sum_n C_n exp(t delta a_n) delta."""
    a = np.array([-1.0, -0.5, -0.25, -0.1])
    Cn = np.array([0.5, 0.3, 0.15, 0.05])
    T, dlt = 50, 0.1
    x = np.zeros((1, 1, T)); x[0, 0, 0] = 1.0
    dt = np.full((1, 1, T), dlt)
    B = np.ones((1, 4, T))
    C = np.repeat(Cn[None, :, None], T, axis=2)
    y, _ = O.scan(x, dt, a[None, :], B, C, delta_softplus=False, threads=1, lib=lib)
    t = np.arange(T)
    want = (Cn[None, :] * np.exp(np.outer(t, a) * dlt) * dlt).sum(axis=1)
    np.testing.assert_allclose(y[0, 0], want, rtol=1e-13, atol=0)
    assert abs(y[0, 0, 0] - 0.1) < 1e-15


def mixing_matrix_reference(x, dt, A, B, C, D, z, dt_bias, softplus):
    """y from the unrolled form M^(c)_{ts} = sum_n C_{t,n} exp(lambda_{cn}
    sum_{r=s+1}^{t} delta_r) delta_s B_{s,n} ("Mamba and selective state
    spaces", theorem 'The mixing matrix of a selective SSM', second form), then
    y = M x + D x, gated by z sigma(z). Also returns the final state
    h_{L,n} = sum_s exp(lambda_n sum_{r=s+1}^{L} delta_r) delta_s B_{s,n} x_s."""
    bt, dn, L = x.shape
    N = A.shape[1]
    v = dt + (0.0 if dt_bias is None else dt_bias[None, :, None])
    delta = np.logaddexp(0.0, v) if softplus else v
    y = np.zeros_like(x)
    fs = np.zeros((bt, dn, N))
    for b in range(bt):
        for c in range(dn):
            cum = np.concatenate([[0.0], np.cumsum(delta[b, c])])  # cum[k] = sum_{r<k}
            M = np.zeros((L, L))
            for t in range(L):
                for s in range(t + 1):
                    seg = cum[t + 1] - cum[s + 1]  # sum_{r=s+1}^{t} delta_r
                    M[t, s] = np.sum(C[b, :, t] * np.exp(A[c, :] * seg) * delta[b, c, s] * B[b, :, s])
            out = M @ x[b, c] + (0.0 if D is None else D[c]) * x[b, c]
            if z is not None:
                out = out * z[b, c] * expit(z[b, c])
            y[b, c] = out
            seg_end = cum[L] - cum[1:]  # sum_{r=s+1}^{L-1}
            fs[b, c] = (np.exp(A[c, :, None] * seg_end[None, :]) * delta[b, c][None, :]
                        * B[b] * x[b, c][None, :]).sum(axis=1)
    return y, fs


def random_problem(rng, bt=2, dn=3, L=12, N=4):
    x = rng.normal(size=(bt, dn, L))
    dt = rng.normal(0, 0.8, size=(bt, dn, L))
    A = -np.exp(rng.normal(0, 0.7, size=(dn, N)))
    B = rng.normal(size=(bt, N, L))
    C = rng.normal(size=(bt, N, L))
    D = rng.normal(size=dn)
    z = rng.normal(size=(bt, dn, L))
    dt_bias = rng.normal(0, 0.5, size=dn)
    return x, dt, A, B, C, D, z, dt_bias


def check_mixing_matrix(lib):
    rng = np.random.default_rng(5)
    for softplus in (True, False):
        x, dt, A, B, C, D, z, dt_bias = random_problem(rng)
        if not softplus:
            dt = np.abs(dt)
            dt_bias = np.abs(dt_bias)
        y, fs = O.scan(x, dt, A, B, C, D=D, z=z, dt_bias=dt_bias, delta_softplus=softplus,
                       threads=2, lib=lib)
        yr, fr = mixing_matrix_reference(x, dt, A, B, C, D, z, dt_bias, softplus)
        np.testing.assert_allclose(y, yr, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(fs, fr, rtol=1e-10, atol=1e-12)
    # optional parts absent: no D, no gate, no bias
    x, dt, A, B, C, D, z, dt_bias = random_problem(rng, bt=1, dn=2, L=9, N=3)
    y, fs = O.scan(x, dt, A, B, C, delta_softplus=True, threads=1, lib=lib)
    yr, fr = mixing_matrix_reference(x, dt, A, B, C, None, None, None, True)
    np.testing.assert_allclose(y, yr, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(fs, fr, rtol=1e-10, atol=1e-12)


def check_lti_convolution(lib):
    """Constant delta, B and C make the layer the convolution
    y_t = sum_j K_j x_{t-j} + D x_t with K_j = sum_n C_n exp(delta A_n)^j delta B_n."""
    rng = np.random.default_rng(7)
    L, N = 40, 5
    dlt = 0.3
    An = -np.exp(rng.normal(0, 0.5, size=N))
    Bn, Cn = rng.normal(size=N), rng.normal(size=N)
    x = rng.normal(size=L)
    Dd = 0.7
    y, _ = O.scan(x[None, None, :], np.full((1, 1, L), dlt), An[None, :],
                  np.repeat(Bn[None, :, None], L, axis=2), np.repeat(Cn[None, :, None], L, axis=2),
                  D=np.array([Dd]), delta_softplus=False, threads=1, lib=lib)
    j = np.arange(L)
    K = (Cn[None, :] * np.exp(dlt * An)[None, :] ** j[:, None] * dlt * Bn[None, :]).sum(axis=1)
    want = np.convolve(x, K)[:L] + Dd * x
    np.testing.assert_allclose(y[0, 0], want, rtol=1e-11, atol=1e-12)


def check_zero_and_huge_step(lib):
    """delta = 0 leaves the state untouched (y = C h_prev + D x); a huge step
    (delta = 50, A = -1) replaces the state by delta * B * x ("The
    discretization the code actually uses", 'What a huge step means')."""
    rng = np.random.default_rng(3)
    L, N = 6, 4
    h0 = rng.normal(size=(1, 1, N))
    x = rng.normal(size=(1, 1, L))
    B = rng.normal(size=(1, N, L)); C = rng.normal(size=(1, N, L))
    A = -np.arange(1.0, N + 1)[None, :]
    y, fs = O.scan(x, np.zeros((1, 1, L)), A, B, C, D=np.array([0.5]), delta_softplus=False,
                   h0=h0, threads=1, lib=lib)
    np.testing.assert_allclose(y[0, 0], (C[0] * h0[0, 0][:, None]).sum(0) + 0.5 * x[0, 0], atol=1e-14)
    np.testing.assert_allclose(fs, h0, atol=0)
    y, fs = O.scan(x, np.full((1, 1, L), 50.0), np.full((1, N), -1.0), B, C, delta_softplus=False,
                   h0=h0, threads=1, lib=lib)
    np.testing.assert_allclose(fs[0, 0], 50.0 * B[0, :, -1] * x[0, 0, -1], rtol=1e-12)
    np.testing.assert_allclose(y[0, 0], (C[0] * 50.0 * B[0] * x[0, 0][None, :]).sum(0), rtol=1e-9)


def check_causality_linearity_chain(lib):
    rng = np.random.default_rng(9)
    x, dt, A, B, C, D, z, dt_bias = random_problem(rng, bt=2, dn=3, L=30, N=4)
    kw = dict(D=D, z=z, dt_bias=dt_bias, delta_softplus=True, threads=2, lib=lib)
    y, fs = O.scan(x, dt, A, B, C, **kw)
    # causality: a change of x at t0 leaves every earlier output as it was
    x2 = x.copy(); x2[:, :, 17] += 3.0
    y2, _ = O.scan(x2, dt, A, B, C, **kw)
    np.testing.assert_array_equal(y2[:, :, :17], y[:, :, :17])
    assert np.all(np.abs(y2[:, :, 17] - y[:, :, 17]) > 0)
    # linearity in x with the steps, B, C and gate held fixed
    x3 = rng.normal(size=x.shape)
    ya, fa = O.scan(2.0 * x - 0.5 * x3, dt, A, B, C, **kw)
    yb, fb = O.scan(x3, dt, A, B, C, **kw)
    np.testing.assert_allclose(ya, 2.0 * y - 0.5 * yb, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(fa, 2.0 * fs - 0.5 * fb, rtol=1e-9, atol=1e-11)
    # prefill then continue from the final state == one scan over everything
    L1 = 11
    ya, fa = O.scan(x[:, :, :L1], dt[:, :, :L1], A, B[:, :, :L1], C[:, :, :L1], D=D,
                    z=z[:, :, :L1], dt_bias=dt_bias, delta_softplus=True, threads=2, lib=lib)
    yb, fb = O.scan(x[:, :, L1:], dt[:, :, L1:], A, B[:, :, L1:], C[:, :, L1:], D=D,
                    z=z[:, :, L1:], dt_bias=dt_bias, delta_softplus=True, h0=fa, threads=2, lib=lib)
    np.testing.assert_allclose(np.concatenate([ya, yb], axis=2), y, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(fb, fs, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------ causal conv1d

def check_conv_impulse_and_silu(lib):
    """The block's convolution weighs the input i steps back by w_i ("The
    Mamba block"): an impulse at t0 gives w_i at t0 + i; SiLU(v) = v sigma(v)."""
    rng = np.random.default_rng(31)
    for k in (1, 2, 4, 7):
        L, t0 = 20, 5
        w = rng.normal(size=(3, k))
        bias = rng.normal(size=3)
        x = np.zeros((2, 3, L)); x[:, :, t0] = 1.0
        out, _ = O.causal_conv1d(x, w, None, silu=False, threads=1, lib=lib)
        want = np.zeros((2, 3, L))
        want[:, :, t0:t0 + k] = w[None, :, :min(k, L - t0)]
        np.testing.assert_allclose(out, want, atol=1e-15)
        out, _ = O.causal_conv1d(x, w, bias, silu=True, threads=1, lib=lib)
        pre = want + bias[None, :, None]
        np.testing.assert_allclose(out, pre * expit(pre), rtol=1e-13, atol=1e-15)
    # printed-value-free closed form: SiLU(1) = 1/(1+e^-1), SiLU(0) = 0
    x = np.ones((1, 1, 1))
    out, _ = O.causal_conv1d(x, np.array([[1.0]]), None, silu=True, threads=1, lib=lib)
    assert abs(out[0, 0, 0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15


def check_conv_constant_input_and_zero_history(lib):
    """Constant input c with zero history: partial sums of the taps for the
    first k-1 steps, then c * sum(w)."""
    k, L, c = 4, 9, 1.5
    w = np.array([[0.5, -0.25, 0.125, 2.0]])
    out, _ = O.causal_conv1d(np.full((1, 1, L), c), w, np.array([0.1]), silu=False, threads=1, lib=lib)
    want = [c * w[0, :min(t + 1, k)].sum() + 0.1 for t in range(L)]
    np.testing.assert_allclose(out[0, 0], want, rtol=1e-14)


def check_conv_history_chain(lib):
    """The decode cache holds the last k-1 inputs, oldest first; a sequence cut
    in two with the cache carried equals one pass, and token-by-token steps
    equal it too ("Decoding with a constant-size cache")."""
    rng = np.random.default_rng(32)
    for k in (2, 4, 5):
        x = rng.normal(size=(2, 3, 23))
        w = rng.normal(size=(3, k))
        bias = rng.normal(size=3)
        full, st_full = O.causal_conv1d(x, w, bias, threads=1, lib=lib)
        for cut in (0, 1, k - 2, 11):
            a, st = O.causal_conv1d(x[:, :, :cut], w, bias, threads=1, lib=lib)
            b2, st2 = O.causal_conv1d(x[:, :, cut:], w, bias, state=st, threads=1, lib=lib)
            np.testing.assert_allclose(np.concatenate([a, b2], axis=2), full, rtol=1e-14, atol=1e-15)
            np.testing.assert_allclose(st2, st_full, atol=0)
        # the cache is the last k-1 inputs, oldest first
        np.testing.assert_array_equal(st_full, np.transpose(x[:, :, -(k - 1):], (0, 2, 1)))
        st = None
        for t in range(x.shape[2]):
            o1, st = O.causal_conv1d(x[:, :, t:t + 1], w, bias, state=st, threads=1, lib=lib)
            np.testing.assert_allclose(o1[:, :, 0], full[:, :, t], rtol=1e-14, atol=1e-15)


def _bwd_problem(rng, bt=2, dn=3, L=9, N=4):
    return dict(x=rng.normal(size=(bt, dn, L)), dt=rng.normal(size=(bt, dn, L)) * 0.5,
                A=-rng.uniform(0.2, 2.0, size=(dn, N)), B=rng.normal(size=(bt, N, L)),
                C=rng.normal(size=(bt, N, L)), D=rng.normal(size=dn), z=rng.normal(size=(bt, dn, L)),
                dt_bias=rng.normal(size=dn) * 0.3, h0=rng.normal(size=(bt, dn, N)))


def check_bwd_finite_differences(lib):
    """The gradient equals the derivative of the forward scan: central
    differences of <dout, out> + <dfinal, final_state> in every input, with
    every option on, and with softplus, gate, skip and bias off."""
    rng = np.random.default_rng(41)
    eps = 1e-6
    for full in (True, False):
        p = _bwd_problem(rng)
        if not full:
            p.update(D=None, z=None, dt_bias=None)
            p["dt"] = np.abs(p["dt"]) + 0.05   # a positive step without softplus
        dout = rng.normal(size=p["x"].shape)
        dfin = rng.normal(size=p["h0"].shape)

        def loss(**over):
            q = dict(p, **over)
            y, fs = O.scan(q["x"], q["dt"], q["A"], q["B"], q["C"], D=q["D"], z=q["z"], dt_bias=q["dt_bias"],
                           delta_softplus=full, h0=q["h0"], threads=1, lib=lib)
            return float((y * dout).sum() + (fs * dfin).sum())

        g = O.scan_bwd(p["x"], p["dt"], p["A"], p["B"], p["C"], dout, D=p["D"], z=p["z"], dt_bias=p["dt_bias"],
                       delta_softplus=full, h0=p["h0"], dfinal=dfin, threads=1, lib=lib)
        names = [("x", "dx"), ("dt", "ddt"), ("A", "dA"), ("B", "dB"), ("C", "dC"), ("h0", "dh0")]
        if full:
            names += [("D", "dD"), ("z", "dz"), ("dt_bias", "ddt_bias")]
        for name, gk in names:
            arr = p[name]
            fd = np.zeros_like(arr)
            for i in np.ndindex(arr.shape):
                hi, lo = arr.copy(), arr.copy()
                hi[i] += eps
                lo[i] -= eps
                fd[i] = (loss(**{name: hi}) - loss(**{name: lo})) / (2 * eps)
            np.testing.assert_allclose(g[gk], fd, rtol=1e-6, atol=1e-6, err_msg=name)


def check_bwd_variants_finite_differences(lib):
    """The gradient of the scan with sequence starts and/or the reverse
    direction equals the derivative of that scan: central differences of
    <dout, out> + <dfinal, final_state> in every input, with starts at the
    first step, inside the row and at the last step."""
    rng = np.random.default_rng(43)
    eps = 1e-6
    starts = np.zeros((2, 9), dtype=np.uint8)
    starts[0, [0, 4]] = 1
    starts[1, [3, 8]] = 1
    for reverse, st in ((False, starts), (True, None), (True, starts)):
        p = _bwd_problem(rng)
        dout = rng.normal(size=p["x"].shape)
        dfin = rng.normal(size=p["h0"].shape)

        def loss(**over):
            q = dict(p, **over)
            y, fs = O.scan_ex(q["x"], q["dt"], q["A"], q["B"], q["C"], D=q["D"], z=q["z"], dt_bias=q["dt_bias"],
                              h0=q["h0"], seq_start=st, reverse=reverse, threads=1, lib=lib)
            return float((y * dout).sum() + (fs * dfin).sum())

        g = O.scan_bwd(p["x"], p["dt"], p["A"], p["B"], p["C"], dout, D=p["D"], z=p["z"], dt_bias=p["dt_bias"],
                       h0=p["h0"], dfinal=dfin, seq_start=st, reverse=reverse, threads=1, lib=lib)
        for name, gk in (("x", "dx"), ("dt", "ddt"), ("A", "dA"), ("B", "dB"), ("C", "dC"), ("h0", "dh0"),
                         ("D", "dD"), ("z", "dz"), ("dt_bias", "ddt_bias")):
            arr = p[name]
            fd = np.zeros_like(arr)
            for i in np.ndindex(arr.shape):
                hi, lo = arr.copy(), arr.copy()
                hi[i] += eps
                lo[i] -= eps
                fd[i] = (loss(**{name: hi}) - loss(**{name: lo})) / (2 * eps)
            np.testing.assert_allclose(g[gk], fd, rtol=1e-6, atol=1e-6,
                                       err_msg="%s reverse=%s starts=%s" % (name, reverse, st is not None))


def check_bwd_impulse_closed_form(lib):
    """One state, constant step, an impulse x = (1, 0, ...), B = C = 1, no
    softplus, no gate: y_T = e^{A (delta_1 + ... + delta_T)} delta_0, so
    d y_T / dA = T delta^2 e^{T delta A}, d y_T / d delta_0 = e^{T delta A},
    d y_T / d delta_s = A delta e^{T delta A} (1 <= s <= T), dB_0 = dx_0 =
    delta e^{T delta A}, dC_T = y_T, and nothing reaches steps after T."""
    A, dl, L = -0.7, 0.3, 12
    for T in (0, 1, 5, 11):
        x = np.zeros((1, 1, L))
        x[0, 0, 0] = 1.0
        dt = np.full((1, 1, L), dl)
        ones = np.ones((1, 1, L))
        dout = np.zeros((1, 1, L))
        dout[0, 0, T] = 1.0
        g = O.scan_bwd(x, dt, np.array([[A]]), ones, ones, dout, delta_softplus=False, threads=1, lib=lib)
        e = math.exp(T * dl * A)
        want_ddt = np.zeros(L)
        want_ddt[0] = e
        want_ddt[1:T + 1] = A * dl * e
        np.testing.assert_allclose(g["dA"][0, 0], T * dl * dl * e, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(g["ddt"][0, 0], want_ddt, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(g["dB"][0, 0, 0], dl * e, rtol=1e-13)
        np.testing.assert_allclose(g["dx"][0, 0, 0], dl * e, rtol=1e-13)
        np.testing.assert_allclose(g["dC"][0, 0, T], dl * e, rtol=1e-13)
        assert not g["dC"][0, 0, T + 1:].any() and not g["dB"][0, 0, T + 1:].any()
        np.testing.assert_allclose(g["dh0"][0, 0, 0], math.exp((T + 1) * dl * A), rtol=1e-13)


def check_bwd_linear_in_cotangent(lib):
    """The gradient is linear in the incoming gradients (dout, dfinal)."""
    rng = np.random.default_rng(43)
    p = _bwd_problem(rng, L=7)
    d1, d2 = rng.normal(size=p["x"].shape), rng.normal(size=p["x"].shape)
    f1, f2 = rng.normal(size=p["h0"].shape), rng.normal(size=p["h0"].shape)

    def grad(do, df):
        return O.scan_bwd(p["x"], p["dt"], p["A"], p["B"], p["C"], do, D=p["D"], z=p["z"], dt_bias=p["dt_bias"],
                          h0=p["h0"], dfinal=df, threads=1, lib=lib)

    g1, g2, g12 = grad(d1, f1), grad(d2, f2), grad(2.0 * d1 - 3.0 * d2, 2.0 * f1 - 3.0 * f2)
    for k in ("dx", "ddt", "dz", "dA", "dB", "dC", "dD", "ddt_bias", "dh0"):
        np.testing.assert_allclose(g12[k], 2.0 * g1[k] - 3.0 * g2[k], rtol=1e-10, atol=1e-12, err_msg=k)


def check_reverse_is_forward_on_flipped_inputs(lib):
    """The reverse walk equals the forward walk of the time-flipped inputs,
    flipped back (the recurrence h_t = a_t h_{t+1} + delta_t B_t x_t read from
    the other end); its final state is the forward walk's final state."""
    rng = np.random.default_rng(51)
    p = _bwd_problem(rng, L=13)
    f = lambda a: np.ascontiguousarray(a[..., ::-1])
    y_r, fs_r = O.scan_ex(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], z=p["z"], dt_bias=p["dt_bias"],
                          h0=p["h0"], reverse=True, threads=1, lib=lib)
    y_f, fs_f = O.scan(f(p["x"]), f(p["dt"]), p["A"], f(p["B"]), f(p["C"]), D=p["D"], z=f(p["z"]),
                       dt_bias=p["dt_bias"], h0=p["h0"], threads=1, lib=lib)
    np.testing.assert_allclose(y_r, f(y_f), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(fs_r, fs_f, rtol=1e-14, atol=1e-15)
    # no options: the extended walk is the plain scan
    y0, fs0 = O.scan_ex(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], z=p["z"], dt_bias=p["dt_bias"],
                        threads=1, lib=lib)
    y1, fs1 = O.scan(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], z=p["z"], dt_bias=p["dt_bias"],
                     threads=1, lib=lib)
    np.testing.assert_array_equal(y0, y1)
    np.testing.assert_array_equal(fs0, fs1)


def check_reverse_gradient_is_forward_gradient_on_flipped_inputs(lib):
    """The gradient of the reverse walk equals the gradient of the forward walk
    of the time-flipped inputs, flipped back: per-step gradients (dx, ddt, dz,
    dB, dC) flipped in time, the rest (dA, dD, ddt_bias, dh0) equal. Starts
    move with the flip: a cut after reverse step t (start at t) is a cut before
    forward step L - t of the flipped row, so r'[j] = r[L - j] (no start at
    t = 0, which would zero the reverse walk's final state)."""
    rng = np.random.default_rng(53)
    L = 13
    p = _bwd_problem(rng, L=L)
    f = lambda a: np.ascontiguousarray(a[..., ::-1])
    dout = rng.normal(size=p["x"].shape)
    dfin = rng.normal(size=p["h0"].shape)
    st = np.zeros((2, L), dtype=np.uint8)
    st[0, [3, 7]] = 1
    st[1, [1, 12]] = 1
    st_f = np.zeros_like(st)
    st_f[:, 1:] = st[:, :0:-1]   # r'[j] = r[L - j], j >= 1
    for starts, starts_f in ((None, None), (st, st_f)):
        g_r = O.scan_bwd(p["x"], p["dt"], p["A"], p["B"], p["C"], dout, D=p["D"], z=p["z"], dt_bias=p["dt_bias"],
                         h0=p["h0"], dfinal=dfin, seq_start=starts, reverse=True, threads=1, lib=lib)
        g_f = O.scan_bwd(f(p["x"]), f(p["dt"]), p["A"], f(p["B"]), f(p["C"]), f(dout), D=p["D"], z=f(p["z"]),
                         dt_bias=p["dt_bias"], h0=p["h0"], dfinal=dfin, seq_start=starts_f, threads=1, lib=lib)
        for k in ("dx", "ddt", "dz", "dB", "dC"):
            np.testing.assert_allclose(g_r[k], f(g_f[k]), rtol=1e-12, atol=1e-13, err_msg=k)
        for k in ("dA", "dD", "ddt_bias", "dh0"):
            np.testing.assert_allclose(g_r[k], g_f[k], rtol=1e-12, atol=1e-13, err_msg=k)


def check_packed_gradient_is_per_sequence_gradients(lib):
    """The gradient of a row of packed sequences (starts marked) is each
    sequence's own gradient: per-step gradients side by side, per-channel sums
    (dA, dD, ddt_bias) added; the initial state and its gradient belong to the
    first sequence, the final-state gradient to the last."""
    rng = np.random.default_rng(54)
    L = 17
    p = _bwd_problem(rng, bt=1, L=L)
    dout = rng.normal(size=p["x"].shape)
    dfin = rng.normal(size=p["h0"].shape)
    st = np.zeros((1, L), dtype=np.uint8)
    st[0, [5, 11]] = 1
    g = O.scan_bwd(p["x"], p["dt"], p["A"], p["B"], p["C"], dout, D=p["D"], z=p["z"], dt_bias=p["dt_bias"],
                   h0=p["h0"], dfinal=dfin, seq_start=st, threads=1, lib=lib)
    segs = [(0, 5), (5, 11), (11, L)]
    acc = {k: 0.0 for k in ("dA", "dD", "ddt_bias")}
    for i, (a, b) in enumerate(segs):
        sl = lambda arr: np.ascontiguousarray(arr[..., a:b])
        gs = O.scan_bwd(sl(p["x"]), sl(p["dt"]), p["A"], sl(p["B"]), sl(p["C"]), sl(dout), D=p["D"], z=sl(p["z"]),
                        dt_bias=p["dt_bias"], h0=p["h0"] if i == 0 else None,
                        dfinal=dfin if i == len(segs) - 1 else None, threads=1, lib=lib)
        for k in ("dx", "ddt", "dz", "dB", "dC"):
            np.testing.assert_allclose(g[k][..., a:b], gs[k], rtol=1e-12, atol=1e-13, err_msg="%s %d" % (k, i))
        for k in acc:
            acc[k] = acc[k] + gs[k]
        if i == 0:
            np.testing.assert_allclose(g["dh0"], gs["dh0"], rtol=1e-12, atol=1e-13)
    for k, v in acc.items():
        np.testing.assert_allclose(g[k], v, rtol=1e-12, atol=1e-13, err_msg=k)


def check_sequence_starts_are_separate_sequences(lib):
    """Packed sequences with their starts marked give, in either direction,
    what scanning each sequence on its own from a zero state gives (the
    state forgets everything at a document break); the initial state reaches
    only the first sequence walked, and the final state is the last walked
    sequence's."""
    rng = np.random.default_rng(52)
    L = 17
    p = _bwd_problem(rng, bt=2, L=L)
    starts = np.zeros((2, L), dtype=bool)
    cuts = {0: [5, 6, 12], 1: [1, 9]}
    for b, cs in cuts.items():
        starts[b, cs] = True
    for reverse in (False, True):
        y, fs = O.scan_ex(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], z=p["z"], dt_bias=p["dt_bias"],
                          h0=p["h0"], seq_start=starts, reverse=reverse, threads=1, lib=lib)
        for b, cs in cuts.items():
            bounds = [0] + cs + [L]
            pieces = list(zip(bounds[:-1], bounds[1:]))
            first = pieces[-1] if reverse else pieces[0]
            for lo, hi in pieces:
                sl = lambda a: np.ascontiguousarray(a[b:b + 1, ..., lo:hi])
                h0 = p["h0"][b:b + 1] if (lo, hi) == first else None
                if reverse:
                    f = lambda a: np.ascontiguousarray(a[..., ::-1])
                    yy, ff = O.scan(f(sl(p["x"])), f(sl(p["dt"])), p["A"], f(sl(p["B"])), f(sl(p["C"])),
                                    D=p["D"], z=f(sl(p["z"])), dt_bias=p["dt_bias"], h0=h0, threads=1, lib=lib)
                    yy = f(yy)
                else:
                    yy, ff = O.scan(sl(p["x"]), sl(p["dt"]), p["A"], sl(p["B"]), sl(p["C"]), D=p["D"],
                                    z=sl(p["z"]), dt_bias=p["dt_bias"], h0=h0, threads=1, lib=lib)
                np.testing.assert_allclose(y[b:b + 1, :, lo:hi], yy, rtol=1e-13, atol=1e-14)
                last = pieces[0] if reverse else pieces[-1]
                if (lo, hi) == last:
                    np.testing.assert_allclose(fs[b:b + 1], ff, rtol=1e-13, atol=1e-14)


def _ssd_problem(rng, bt=2, L=9, H=4, P=3, G=2, N=5):
    return dict(x=rng.normal(size=(bt, L, H, P)), dt=rng.normal(size=(bt, L, H)) * 0.5,
                A=-rng.uniform(0.2, 2.0, size=H), B=rng.normal(size=(bt, L, G, N)), C=rng.normal(size=(bt, L, G, N)),
                D=rng.normal(size=H), z=rng.normal(size=(bt, L, H, P)), dt_bias=rng.normal(size=H) * 0.3,
                h0=rng.normal(size=(bt, H, P, N)))


def check_ssd_is_the_scan_with_one_decay_per_head(lib):
    """Mamba-2's scan is the selective scan whose decay rate is the same for
    all states of a head and whose B, C are shared by the heads of a group:
    channel d = (h, p) of the S6 oracle with A[d, n] = A[h], dt[d] = dt[h]."""
    rng = np.random.default_rng(61)
    p = _ssd_problem(rng)
    bt, L, H, P = p["x"].shape
    G, N = p["B"].shape[2:]
    y, fs = O.ssd(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], z=p["z"], dt_bias=p["dt_bias"], h0=p["h0"],
                  threads=1, lib=lib)
    hpg = H // G
    for g in range(G):
        hs = list(range(g * hpg, (g + 1) * hpg))
        chan = lambda a: np.ascontiguousarray(np.transpose(a[:, :, hs, :], (0, 2, 3, 1)).reshape(bt, hpg * P, L))
        per_d = lambda v: np.repeat(v[hs], P)
        y6, f6 = O.scan(chan(p["x"]), np.ascontiguousarray(np.repeat(np.transpose(p["dt"][:, :, hs], (0, 2, 1)), P,
                                                                     axis=1)),
                        np.repeat(per_d(p["A"])[:, None], N, axis=1), np.ascontiguousarray(np.transpose(
                            p["B"][:, :, g, :], (0, 2, 1))), np.ascontiguousarray(np.transpose(p["C"][:, :, g, :],
                                                                                              (0, 2, 1))),
                        D=per_d(p["D"]), z=chan(p["z"]), dt_bias=per_d(p["dt_bias"]),
                        h0=p["h0"][:, hs].reshape(bt, hpg * P, N), threads=1, lib=lib)
        np.testing.assert_allclose(chan(y), y6, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(fs[:, hs].reshape(bt, hpg * P, N), f6, rtol=1e-13, atol=1e-13)


def check_ssd_masked_matmul_form(lib):
    """The structured-matmul form of the pages ("Mamba in practice": Y is a
    mask M applied over the pairwise scores C_t . B_s): per head,
    Y = (M o C B^T) diag(delta) X + D X with M[t, s] = exp(A sum_{s<r<=t} delta_r)
    for s <= t and 0 above the diagonal, plus exp(A sum_{r<=t} delta_r) C_t h0
    from an initial state; computed with numpy matrix products."""
    rng = np.random.default_rng(62)
    p = _ssd_problem(rng, L=11)
    bt, L, H, P = p["x"].shape
    G, N = p["B"].shape[2:]
    y, fs = O.ssd(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], dt_bias=p["dt_bias"], h0=p["h0"],
                  threads=1, lib=lib)
    v = p["dt"] + p["dt_bias"]
    delta = np.maximum(v, 0) + np.log1p(np.exp(-np.abs(v)))
    for b in range(bt):
        for h in range(H):
            g = h // (H // G)
            cs = np.cumsum(delta[b, :, h])
            M = np.exp(p["A"][h] * (cs[:, None] - cs[None, :])) * np.tri(L)
            Cb, Bb = p["C"][b, :, g, :], p["B"][b, :, g, :]
            X = p["x"][b, :, h, :]
            Y = (M * (Cb @ Bb.T)) @ (delta[b, :, h][:, None] * X) + p["D"][h] * X
            Y += np.exp(p["A"][h] * cs)[:, None] * (Cb @ p["h0"][b, h].T)
            np.testing.assert_allclose(y[b, :, h, :], Y, rtol=1e-12, atol=1e-12)


ALL_CHECKS = [check_recurrence_example, check_softplus_values, check_gate_theorem,
              check_selective_copy_euler, check_impulse_response, check_mixing_matrix,
              check_lti_convolution, check_zero_and_huge_step, check_causality_linearity_chain,
              check_conv_impulse_and_silu, check_conv_constant_input_and_zero_history, check_conv_history_chain,
              check_bwd_finite_differences, check_bwd_variants_finite_differences,
              check_bwd_impulse_closed_form, check_bwd_linear_in_cotangent,
              check_reverse_is_forward_on_flipped_inputs, check_reverse_gradient_is_forward_gradient_on_flipped_inputs,
              check_sequence_starts_are_separate_sequences, check_packed_gradient_is_per_sequence_gradients,
              check_ssd_is_the_scan_with_one_decay_per_head, check_ssd_masked_matmul_form]
