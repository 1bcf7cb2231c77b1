"""Pins of the trapezoidal (Mamba-3 SISO) scan oracle, on the CPU.

Each check ties ``oracle.trap.trap_fwd`` to something other than itself:
* brute force: the recurrence unrolled into a sum over input terms;
* trap = 1 removes the delayed term, and the scan is the Mamba-2 SSD
  recurrence, checked against the separately pinned SSD oracle;
* a = 0, trap = 1/2, constant dt: the state integrates k v^T by the
  trapezoidal rule (a textbook closed form);
* one step with trap = 0: only the carried k, v enter (closed form);
* splitting the sequence and carrying (h, k, v) gives the same result.
A swapped beta/gamma, a k_t in place of k_{t-1}, a dropped skip or decay
fails at least one of these.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.trap import trap_coefficients, trap_fwd, trap_unrolled
from selective_state_space_04_gb300.inputs import Workload, make_trap_inputs


def _w(B=2, L=7, H=4, P=3, N=5, G=2, init=True):
    return Workload("t", B, L, H, P, N, G, 16, "f32", init)


@pytest.mark.parametrize("G,init", [(1, True), (2, True), (4, False)])
def test_recurrence_matches_unrolled_sum(G, init):
    inp = make_trap_inputs(_w(G=G, init=init), seed=3)
    y1, h1, _, _ = trap_fwd(**inp)
    y2, h2 = trap_unrolled(**inp)
    assert np.max(np.abs(y1 - y2)) <= 1e-12 * max(1.0, np.max(np.abs(y2)))
    assert np.max(np.abs(h1 - h2)) <= 1e-12 * max(1.0, np.max(np.abs(h2)))


def test_trap_one_is_the_mamba2_recurrence():
    # per-head constant a = -exp(A_log), dt = softplus(dt_raw + dt_bias), trap = 1
    B, L, H, P, N = 2, 9, 4, 3, 6
    rng = np.random.default_rng(5)
    x = rng.standard_normal((B, L, H, P))
    Bm = rng.standard_normal((B, L, 1, N))
    Cm = rng.standard_normal((B, L, 1, N))
    dt_raw = 0.1 * rng.standard_normal((B, L, H))
    dt_bias = np.log(np.expm1(np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), H))))
    A_log = np.log(rng.uniform(1, 16, H))
    D = rng.standard_normal(H)
    h0 = 0.1 * rng.standard_normal((B, H, P, N))
    ref_y, ref_h = oracle.ssd_fwd(x, dt_raw, dt_bias, A_log, Bm, Cm, D, h0)
    z = dt_raw + dt_bias
    dt = np.maximum(z, 0) + np.log1p(np.exp(-np.abs(z)))
    a = np.broadcast_to(-np.exp(A_log), (B, L, H))
    y, h, _, _ = trap_fwd(x, Bm, Cm, dt, a, np.ones((B, L, H)), D, h0,
                          k0=rng.standard_normal((B, H, N)), v0=rng.standard_normal((B, H, P)))
    assert np.max(np.abs(y - ref_y)) <= 1e-12 * np.max(np.abs(ref_y))
    assert np.max(np.abs(h - ref_h)) <= 1e-12 * np.max(np.abs(ref_h))


def test_no_decay_half_trap_is_the_trapezoidal_rule():
    B, L, H, P, N = 1, 6, 2, 3, 4
    inp = make_trap_inputs(_w(B=B, L=L, H=H, P=P, N=N, G=1), seed=7)
    dt = 0.0625   # exact in fp32 and fp64
    inp.update(dt=torch.full((B, L, H), dt), a=torch.zeros((B, L, H)), trap=torch.full((B, L, H), 0.5))
    _, h, _, _ = trap_fwd(**inp)
    v, k = inp["v"].double().numpy(), inp["k"].double().numpy()
    k0, v0, h0 = inp["k0"].double().numpy(), inp["v0"].double().numpy(), inp["h0"].double().numpy()
    for hh in range(H):
        terms = [np.outer(v0[0, hh], k0[0, hh])] + [np.outer(v[0, s, hh], k[0, s, 0]) for s in range(L)]
        # trapezoid over the L + 1 samples k_{-1} v_{-1}, ..., k_{L-1} v_{L-1}
        ref = h0[0, hh] + dt * (0.5 * terms[0] + sum(terms[1:-1]) + 0.5 * terms[-1])
        assert np.allclose(h[0, hh], ref, rtol=1e-13, atol=1e-15)


def test_one_step_previous_token_only():
    inp = make_trap_inputs(_w(L=1), seed=11)
    inp["trap"] = torch.zeros_like(inp["trap"])
    y, h, kf, vf = trap_fwd(**inp)
    alpha, beta, gamma = trap_coefficients(inp["dt"], inp["a"], inp["trap"])
    assert np.all(gamma == 0)
    h0, k0, v0 = (inp[n].double().numpy() for n in ("h0", "k0", "v0"))
    al, be = alpha[:, 0, :, None, None], beta[:, 0, :, None, None]
    ref_h = al * h0 + be * v0[:, :, :, None] * k0[:, :, None, :]
    gi = np.arange(4) // 2
    q = inp["q"].double().numpy()[:, 0][:, gi]
    ref_y = np.einsum("bhpn,bhn->bhp", ref_h, q) + inp["D"].double().numpy()[None, :, None] * inp["v"].double().numpy()[:, 0]
    assert np.allclose(h, ref_h, rtol=1e-14, atol=0)
    assert np.allclose(y[:, 0], ref_y, rtol=1e-13, atol=1e-14)
    # the carried k, v are this step's
    assert np.array_equal(kf, inp["k"].double().numpy()[:, 0][:, gi])
    assert np.array_equal(vf, inp["v"].double().numpy()[:, 0])


def test_split_and_resume_with_carried_k_v():
    inp = make_trap_inputs(_w(L=11), seed=13)
    y, h, kf, vf = trap_fwd(**inp)
    cut = 4
    first = {n: (t[:, :cut] if n in ("v", "k", "q", "dt", "a", "trap") else t) for n, t in inp.items()}
    y1, h1, k1, v1 = trap_fwd(**first)
    second = {n: (t[:, cut:] if n in ("v", "k", "q", "dt", "a", "trap") else t) for n, t in inp.items()}
    second.update(h0=h1, k0=k1, v0=v1)
    y2, h2, k2, v2 = trap_fwd(**second)
    assert np.allclose(np.concatenate([y1, y2], axis=1), y, rtol=1e-13, atol=1e-13)
    assert np.allclose(h2, h, rtol=1e-13, atol=1e-15)
    assert np.array_equal(k2, kf) and np.array_equal(v2, vf)
