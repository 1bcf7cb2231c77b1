"""Pins of the backward oracle, on the CPU: central finite differences of the
(separately pinned) fp64 forward oracle, which shares no code with it.

The loss is sum(y * dy) + sum(final_state * d_final); each gradient of
oracle.backward.ssd_bwd must match (loss(u + e) - loss(u - e)) / 2e for the
per-head vectors (every element) and for sampled elements of the tensors.
"""
import numpy as np
import pytest

import oracle
from oracle.backward import ssd_bwd


def _case(seed, B=2, L=7, H=4, P=3, N=5, G=2, init=True):
    rng = np.random.default_rng(seed)
    inp = dict(x=rng.standard_normal((B, L, H, P)), dt_raw=0.3 * rng.standard_normal((B, L, H)),
               dt_bias=rng.uniform(-2, 0, H), A_log=np.log(rng.uniform(0.5, 3, H)),
               B=rng.standard_normal((B, L, G, N)), C=rng.standard_normal((B, L, G, N)),
               D=rng.standard_normal(H), init_state=rng.standard_normal((B, H, P, N)) if init else None)
    dy = rng.standard_normal((B, L, H, P))
    dfin = rng.standard_normal((B, H, P, N))
    return inp, dy, dfin


def _loss(inp, dy, dfin):
    y, f = oracle.ssd_fwd(**inp)
    return float(np.sum(y * dy) + np.sum(f * dfin))


def _fd(inp, dy, dfin, name, idx, eps=1e-6):
    plus = {k: (None if v is None else np.array(v, copy=True)) for k, v in inp.items()}
    minus = {k: (None if v is None else np.array(v, copy=True)) for k, v in inp.items()}
    plus[name][idx] += eps
    minus[name][idx] -= eps
    return (_loss(plus, dy, dfin) - _loss(minus, dy, dfin)) / (2 * eps)


@pytest.mark.parametrize("seed,G,init", [(1, 2, True), (2, 1, False), (3, 4, True)])
def test_backward_matches_finite_differences(seed, G, init):
    inp, dy, dfin = _case(seed, G=G, init=init)
    g = ssd_bwd(**inp, dy=dy, d_final=dfin)
    rng = np.random.default_rng(seed + 100)
    checks = [("dt_bias", "ddt_bias"), ("A_log", "dA_log"), ("D", "dD")]
    for inp_name, g_name in checks:
        for i in range(inp[inp_name].shape[0]):
            ref = _fd(inp, dy, dfin, inp_name, (i,))
            assert abs(g[g_name][i] - ref) <= 1e-6 * max(1.0, abs(ref)), (g_name, i, g[g_name][i], ref)
    tensors = [("x", "dx"), ("dt_raw", "ddt_raw"), ("B", "dB"), ("C", "dC")]
    if init:
        tensors.append(("init_state", "d_init"))
    for inp_name, g_name in tensors:
        shape = inp[inp_name].shape
        for _ in range(12):
            idx = tuple(int(rng.integers(s)) for s in shape)
            ref = _fd(inp, dy, dfin, inp_name, idx)
            assert abs(g[g_name][idx] - ref) <= 1e-6 * max(1.0, abs(ref)), (g_name, idx, g[g_name][idx], ref)


def test_backward_is_linear_in_the_output_gradients():
    inp, dy, dfin = _case(7)
    g1 = ssd_bwd(**inp, dy=dy, d_final=dfin)
    g2 = ssd_bwd(**inp, dy=2.0 * dy, d_final=2.0 * dfin)
    for k in g1:
        assert np.allclose(g2[k], 2.0 * g1[k], rtol=1e-12, atol=1e-13), k
