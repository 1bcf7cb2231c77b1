"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: a worked
example done by hand, closed forms of special cases, the independent
quadratic (dual) form by brute force, or an invariant that the mathematics
fixes.  Together they are chosen so that a plausible slip in the recurrence
(a dropped term, a wrong sign, a transposed state, a wrong head->group map,
reading out before the update) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import ssd_fwd, ssd_quadratic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(rng, Bt, L, H, P, N, G, init=True, A_log=None):
    x = rng.standard_normal((Bt, L, H, P))
    dt_raw = 0.1 * rng.standard_normal((Bt, L, H))
    dt0 = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), H))
    dt_bias = np.log(np.expm1(dt0))
    if A_log is None:
        A_log = np.log(rng.uniform(1.0, 16.0, H))
    B = rng.standard_normal((Bt, L, G, N))
    C = rng.standard_normal((Bt, L, G, N))
    D = rng.standard_normal(H)
    h0 = 0.1 * rng.standard_normal((Bt, H, P, N)) if init else None
    return dict(x=x, dt_raw=dt_raw, dt_bias=dt_bias, A_log=np.broadcast_to(A_log, (H,)).copy(),
                B=B, C=C, D=D, init_state=h0)


def relerr(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# ---------------------------------------------------------------- softplus
@pytest.mark.parametrize("z", [-30.0, -5.0, -1.0, -1e-3, 0.0, 0.5, 3.0, 30.0])
def test_softplus_matches_definition(z):
    # log(1 + e^z) written literally, evaluated with 50 significant digits
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    ref = float(mpmath.log(1 + mpmath.exp(mpmath.mpf(z))))
    assert oracle.softplus(z) == pytest.approx(ref, rel=1e-14, abs=1e-300)


def test_softplus_extremes():
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15)
    assert oracle.softplus(800.0) == 800.0           # no overflow
    assert oracle.softplus(-800.0) == 0.0            # e^-800 underflows
    assert oracle.softplus(-50.0) == pytest.approx(math.exp(-50.0), rel=1e-12)


def test_dt_bias_recipe_inverts_softplus():
    for dt0 in (1e-3, 1e-2, 0.05, 0.1):
        assert oracle.softplus(math.log(math.expm1(dt0))) == pytest.approx(dt0, rel=1e-12)


# ---------------------------------------------------------- worked example
def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "hand_worked_example.json")) as f:
        g = json.load(f)
    dt_bias = np.array([math.log(math.e - 1.0)])
    A_log = np.array([math.log(math.log(2.0))])
    y, fin = ssd_fwd(np.array(g["x"], float), np.array(g["dt_raw"], float), dt_bias, A_log,
                     np.array(g["B"], float), np.array(g["C"], float), np.array(g["D"], float),
                     np.array(g["init_state"], float))
    np.testing.assert_allclose(y, np.array(g["expected_y"], float), rtol=0, atol=1e-12)
    np.testing.assert_allclose(fin, np.array(g["expected_final_state"], float), rtol=0, atol=1e-12)


# ------------------------------------------------------ brute-force (dual)
@pytest.mark.parametrize("shape", [
    (1, 1, 1, 1, 1, 1), (1, 7, 2, 3, 5, 1), (2, 16, 4, 8, 16, 2),
    (1, 33, 6, 4, 8, 3), (1, 64, 2, 8, 16, 1), (3, 20, 8, 2, 4, 8)])
@pytest.mark.parametrize("init", [False, True])
def test_recurrence_matches_quadratic_form(shape, init):
    rng = np.random.default_rng(hash((shape, init)) % 2**32)
    Bt, L, H, P, N, G = shape
    c = rand_case(rng, Bt, L, H, P, N, G, init=init)
    y, fin = ssd_fwd(**c)
    yq, finq = ssd_quadratic(**c)
    assert relerr(y, yq) < 1e-12
    assert relerr(fin, finq) < 1e-12


def test_quadratic_form_with_strong_decay():
    # large |A| exercises products of many small decays
    rng = np.random.default_rng(7)
    c = rand_case(rng, 1, 48, 3, 4, 8, 1, init=True, A_log=np.log([1.0, 16.0, 200.0]))
    y, fin = ssd_fwd(**c)
    yq, finq = ssd_quadratic(**c)
    assert relerr(y, yq) < 1e-12 and relerr(fin, finq) < 1e-12


# ------------------------------------------------------------ closed forms
def test_A_to_zero_is_weighted_cumsum():
    """A_log = -inf gives A = -0 and dA = 1: the state is a dt-weighted
    cumulative sum of B x^T, read out by C, plus the carried-in state."""
    rng = np.random.default_rng(1)
    Bt, L, H, P, N, G = 2, 40, 4, 3, 5, 2
    c = rand_case(rng, Bt, L, H, P, N, G, init=True, A_log=-np.inf)
    y, fin = ssd_fwd(**c)
    for b in range(Bt):
        for h in range(H):
            g = h // (H // G)
            dt = np.logaddexp(0.0, c["dt_raw"][b, :, h] + c["dt_bias"][h])
            outer = dt[:, None, None] * c["B"][b, :, g, :, None] * c["x"][b, :, h, None, :]
            S = np.cumsum(outer, axis=0) + c["init_state"][b, h].T[None]    # [L, N, P]
            yy = np.einsum("tn,tnp->tp", c["C"][b, :, g, :], S) + c["D"][h] * c["x"][b, :, h, :]
            np.testing.assert_allclose(y[b, :, h, :], yy, rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(fin[b, h], S[-1].T, rtol=1e-11, atol=1e-11)


def test_B_C_zero_gives_skip_only():
    rng = np.random.default_rng(2)
    c = rand_case(rng, 2, 30, 3, 4, 6, 1, init=True)
    c["B"][:] = 0.0
    c["C"][:] = 0.0
    y, fin = ssd_fwd(**c)
    np.testing.assert_array_equal(y, c["D"][None, None, :, None] * c["x"])
    for b in range(2):
        for h in range(3):
            dt = np.logaddexp(0.0, c["dt_raw"][b, :, h] + c["dt_bias"][h])
            decay = math.exp(-math.exp(c["A_log"][h]) * dt.sum())
            np.testing.assert_allclose(fin[b, h], decay * c["init_state"][b, h], rtol=1e-12)


def test_memoryless_limit():
    """dt*|A| >> 1 forgets everything but the current step."""
    rng = np.random.default_rng(3)
    c = rand_case(rng, 1, 25, 2, 3, 4, 1, init=True, A_log=math.log(1e6))
    y, fin = ssd_fwd(**c)
    dt = np.logaddexp(0.0, c["dt_raw"][0] + c["dt_bias"][None, :])          # [L, H]
    cb = np.einsum("tn,tn->t", c["C"][0, :, 0], c["B"][0, :, 0])            # [L]
    yy = (dt * cb[:, None])[:, :, None] * c["x"][0] + c["D"][None, :, None] * c["x"][0]
    np.testing.assert_allclose(y[0], yy, rtol=1e-12, atol=1e-12)
    last = dt[-1][:, None, None] * c["x"][0, -1][:, :, None] * c["B"][0, -1, 0][None, None, :]
    np.testing.assert_allclose(fin[0], last, rtol=1e-12, atol=1e-12)


def test_single_step_closed_form():
    """L = 1: h_0 = dA h_init + dt B x^T and y = C^T h_0 + D x, with P != N
    and an asymmetric initial state so that a transposed state layout fails."""
    rng = np.random.default_rng(4)
    H, P, N = 3, 3, 5
    c = rand_case(rng, 1, 1, H, P, N, 1, init=True)
    y, fin = ssd_fwd(**c)
    for h in range(H):
        dt = math.log1p(math.exp(c["dt_raw"][0, 0, h] + c["dt_bias"][h]))
        dA = math.exp(-math.exp(c["A_log"][h]) * dt)
        S = dA * c["init_state"][0, h].T + dt * np.outer(c["B"][0, 0, 0], c["x"][0, 0, h])   # [N,P]
        np.testing.assert_allclose(fin[0, h], S.T, rtol=1e-13)
        np.testing.assert_allclose(y[0, 0, h], c["C"][0, 0, 0] @ S + c["D"][h] * c["x"][0, 0, h],
                                   rtol=1e-13)


def test_group_mapping_contiguous_head_blocks():
    """group = head * G / H: with H = 6, G = 3 heads {0,1}->0, {2,3}->1, {4,5}->2."""
    rng = np.random.default_rng(5)
    c = rand_case(rng, 1, 12, 6, 2, 3, 3, init=False)
    c["B"][:, :, 1, :] = 0.0        # silence group 1 only
    y, _ = ssd_fwd(**c)
    skip = c["D"][None, None, :, None] * c["x"]
    for h in range(6):
        if h in (2, 3):
            np.testing.assert_array_equal(y[:, :, h], skip[:, :, h])
        else:
            assert np.max(np.abs(y[:, :, h] - skip[:, :, h])) > 1e-3


# -------------------------------------------------------------- invariants
def test_split_and_resume_is_bitwise():
    rng = np.random.default_rng(6)
    c = rand_case(rng, 2, 50, 2, 4, 6, 1, init=True)
    y, fin = ssd_fwd(**c)
    L1 = 19
    first = {k: (v[:, :L1] if k in ("x", "dt_raw", "B", "C") else v) for k, v in c.items()}
    y1, f1 = ssd_fwd(**first)
    second = {k: (v[:, L1:] if k in ("x", "dt_raw", "B", "C") else v) for k, v in c.items()}
    second["init_state"] = f1
    y2, f2 = ssd_fwd(**second)
    np.testing.assert_array_equal(np.concatenate([y1, y2], axis=1), y)
    np.testing.assert_array_equal(f2, fin)


def test_linearity_in_x_and_state():
    rng = np.random.default_rng(8)
    c = rand_case(rng, 1, 30, 2, 3, 4, 1, init=True)
    y, fin = ssd_fwd(**c)
    c3 = dict(c, x=3.0 * c["x"], init_state=3.0 * c["init_state"])
    y3, fin3 = ssd_fwd(**c3)
    np.testing.assert_allclose(y3, 3.0 * y, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(fin3, 3.0 * fin, rtol=1e-13, atol=1e-13)


def test_identical_heads_give_identical_outputs():
    rng = np.random.default_rng(9)
    c = rand_case(rng, 1, 20, 4, 3, 4, 2, init=True)
    for k in ("dt_bias", "A_log", "D"):
        c[k][1] = c[k][0]
    c["x"][:, :, 1] = c["x"][:, :, 0]
    c["dt_raw"][:, :, 1] = c["dt_raw"][:, :, 0]
    c["init_state"][:, 1] = c["init_state"][:, 0]
    y, fin = ssd_fwd(**c)
    np.testing.assert_array_equal(y[:, :, 1], y[:, :, 0])
    np.testing.assert_array_equal(fin[:, 1], fin[:, 0])


def test_threads_do_not_change_result():
    rng = np.random.default_rng(10)
    c = rand_case(rng, 3, 17, 5, 2, 3, 1, init=True)
    y1, f1 = ssd_fwd(**c, nthreads=1)
    y4, f4 = ssd_fwd(**c, nthreads=4)
    np.testing.assert_array_equal(y1, y4)
    np.testing.assert_array_equal(f1, f4)


def test_empty_sequence_returns_initial_state():
    rng = np.random.default_rng(11)
    c = rand_case(rng, 2, 0, 2, 3, 4, 1, init=True)
    y, fin = ssd_fwd(**c)
    assert y.shape == (2, 0, 2, 3)
    np.testing.assert_array_equal(fin, c["init_state"])


def test_rejects_bad_groups():
    rng = np.random.default_rng(12)
    c = rand_case(rng, 1, 4, 3, 2, 2, 2, init=False)      # 3 heads, 2 groups
    with pytest.raises(ValueError):
        ssd_fwd(**c)
