"""Pins of the oracle for the steps around the scan (conv1d + SiLU prologue,
gated RMSNorm epilogue), on the CPU.

conv1d_silu is tied to: numpy's own convolution (np.convolve, causal part);
single-tap weights, which make the conv a pure shift; the closed form of SiLU
at 0 and its odd part silu(v) - silu(-v) = v; splitting the sequence with the
carried conv state.  gated_rmsnorm is tied to: the unit RMS of the normalised
part; invariance under scaling y (eps = 0); a constant row's closed form.
"""
import numpy as np
import pytest
import torch

from oracle.neighbors import conv1d_silu, gated_rmsnorm, silu
from selective_state_space_04_gb300.inputs import Workload, make_conv_inputs, make_gnorm_inputs


def _w(B=2, L=9, H=2, P=4, N=3, G=1, init=True):
    return Workload("t", B, L, H, P, N, G, 1, "f32", init)


def _fused(x, Bm, Cm):
    Bt, L = x.shape[:2]
    return np.concatenate([x.reshape(Bt, L, -1), Bm.reshape(Bt, L, -1), Cm.reshape(Bt, L, -1)], axis=-1)


def test_silu_closed_forms():
    v = np.linspace(-6, 6, 25)
    assert silu(np.zeros(1))[0] == 0.0
    assert np.allclose(silu(v) - silu(-v), v, rtol=0, atol=1e-13)


@pytest.mark.parametrize("K", [2, 4])
def test_conv_matches_numpy_convolve(K):
    w = _w(init=False)
    inp = make_conv_inputs(w, K=K, seed=1)
    x, Bm, Cm, _ = conv1d_silu(**inp, H=w.nheads, P=w.headdim, G=w.ngroups, N=w.dstate)
    xbc = inp["xbc"].double().numpy()
    wt, bias = inp["weight"].double().numpy(), inp["bias"].double().numpy()
    u = _fused(x, Bm, Cm)
    for b in range(w.batch):
        for c in range(xbc.shape[2]):
            pre = np.convolve(xbc[b, :, c], wt[c])[: w.seqlen] + bias[c]
            assert np.allclose(u[b, :, c], silu(pre), rtol=1e-13, atol=1e-14)


def test_single_tap_is_a_shift():
    w = _w(L=7)
    inp = make_conv_inputs(w, K=4, seed=2)
    C = inp["xbc"].shape[2]
    for j in range(4):
        wt = torch.zeros((C, 4))
        wt[:, j] = 1.0
        x, Bm, Cm, _ = conv1d_silu(inp["xbc"], wt, None, inp["conv_state"], w.nheads, w.headdim, w.ngroups,
                                   w.dstate)
        ext = np.concatenate([inp["conv_state"].double().numpy(), inp["xbc"].double().numpy()], axis=1)
        shifted = ext[:, 3 - j: 3 - j + w.seqlen]
        assert np.allclose(_fused(x, Bm, Cm), silu(shifted), rtol=1e-14, atol=0)


def test_conv_split_and_resume():
    w = _w(L=13)
    inp = make_conv_inputs(w, K=4, seed=3)
    dims = dict(H=w.nheads, P=w.headdim, G=w.ngroups, N=w.dstate)
    x, Bm, Cm, st = conv1d_silu(**inp, **dims)
    cut = 5
    x1, B1, C1, s1 = conv1d_silu(inp["xbc"][:, :cut], inp["weight"], inp["bias"], inp["conv_state"], **dims)
    x2, B2, C2, s2 = conv1d_silu(inp["xbc"][:, cut:], inp["weight"], inp["bias"], s1, **dims)
    assert np.allclose(np.concatenate([x1, x2], 1), x, rtol=1e-14, atol=0)
    assert np.allclose(np.concatenate([B1, B2], 1), Bm, rtol=1e-14, atol=0)
    assert np.allclose(np.concatenate([C1, C2], 1), Cm, rtol=1e-14, atol=0)
    assert np.array_equal(s2, st)
    assert np.array_equal(st, inp["xbc"].double().numpy()[:, -3:])


def test_gated_rmsnorm_unit_rms_and_scale_invariance():
    w = _w(L=5, H=3, P=8)
    inp = make_gnorm_inputs(w, seed=4)
    out = gated_rmsnorm(**inp, eps=0.0)
    gate = inp["weight"].double().numpy()[None, None, :] * silu(inp["z"].double().numpy().reshape(2, 5, 24))
    normed = out.reshape(2, 5, 24) / gate
    assert np.allclose(np.sqrt(np.mean(normed ** 2, axis=-1)), 1.0, rtol=1e-12)
    out2 = gated_rmsnorm(inp["y"] * 4.0, inp["z"], inp["weight"], eps=0.0)
    assert np.allclose(out2, out, rtol=1e-12, atol=1e-14)


def test_gated_rmsnorm_constant_row():
    w = _w(B=1, L=1, H=2, P=4)
    inp = make_gnorm_inputs(w, seed=5)
    c, eps = -0.75, 1e-6
    y = torch.full((1, 1, 2, 4), c)
    out = gated_rmsnorm(y, inp["z"], inp["weight"], eps=eps)
    ref = (c / np.sqrt(c * c + eps)) * inp["weight"].double().numpy() * silu(inp["z"].double().numpy().reshape(8))
    assert np.allclose(out.reshape(8), ref, rtol=1e-13, atol=0)
