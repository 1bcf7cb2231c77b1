"""Pins of the complex-valued (ET) scan oracle, on the CPU, against things it
does not compute itself: an ODE solver on the continuous system the
discretisation holds exactly, the unrolled product form, the real SSD oracle
in the case arg A = pi, and the conjugation symmetry of the readout."""
import numpy as np
import pytest

import oracle
from oracle.complex_scan import complex_A, complex_fwd, complex_unrolled, to_complex


def _case(seed, Bt=2, L=6, H=3, P=4, K=3, G=1, init=True):
    rng = np.random.default_rng(seed)
    N = 2 * K
    return dict(x=rng.standard_normal((Bt, L, H, P)), dt_raw=0.5 * rng.standard_normal((Bt, L, H)),
                dt_bias=rng.uniform(-1.5, 0.5, H),
                A_polar=np.stack([np.log(rng.uniform(0.5, 4.0, H)), rng.uniform(0.6 * np.pi, 1.4 * np.pi, H)], 1),
                B=rng.standard_normal((Bt, L, G, N)), C=rng.standard_normal((Bt, L, G, N)),
                D=rng.standard_normal(H), init_state=0.3 * rng.standard_normal((Bt, H, P, N)) if init else None)


def _softplus(z):
    return np.maximum(z, 0) + np.log1p(np.exp(-np.abs(z)))


def test_each_step_is_the_exact_hold_of_the_continuous_system():
    # per step, h' = A h + B x with x and B held constant over dt: integrate it
    # numerically and compare with the oracle's state after every step
    from scipy.integrate import solve_ivp
    c = _case(3, Bt=1, L=4, H=2, P=2, K=2)
    A = complex_A(c["A_polar"])
    dt = _softplus(c["dt_raw"] + c["dt_bias"][None, None, :])
    Bc = to_complex(c["B"])
    h = np.swapaxes(to_complex(c["init_state"]), 2, 3)[0]      # [H,K,P]
    for t in range(c["x"].shape[1]):
        for hh in range(2):
            u = Bc[0, t, 0][:, None] * c["x"][0, t, hh][None, :]   # [K,P], constant over the step
            z0 = h[hh].ravel()

            def rhs(_, v, a=A[hh], u=u.ravel()):
                zc = v[: z0.size] + 1j * v[z0.size:]
                d = a * zc + u
                return np.concatenate([d.real, d.imag])
            sol = solve_ivp(rhs, (0.0, dt[0, t, hh]), np.concatenate([z0.real, z0.imag]), method="DOP853",
                            rtol=1e-12, atol=1e-14)
            v = sol.y[:, -1]
            h[hh] = (v[: z0.size] + 1j * v[z0.size:]).reshape(h[hh].shape)
        sub = {k: (v if v is None else v) for k, v in c.items()}
        sub = dict(c, x=c["x"][:, : t + 1], dt_raw=c["dt_raw"][:, : t + 1], B=c["B"][:, : t + 1],
                   C=c["C"][:, : t + 1])
        _, fin = complex_fwd(**sub)
        got = np.swapaxes(to_complex(fin), 2, 3)[0]
        assert np.allclose(got, h, rtol=1e-9, atol=1e-11), t


@pytest.mark.parametrize("seed,G,init", [(1, 1, True), (2, 3, False), (4, 1, True)])
def test_recurrence_equals_the_unrolled_products(seed, G, init):
    c = _case(seed, H=3, G=G, init=init)
    y1, f1 = complex_fwd(**c)
    y2, f2 = complex_unrolled(**c)
    assert np.allclose(y1, y2, rtol=1e-11, atol=1e-12)
    assert np.allclose(f1, f2, rtol=1e-11, atol=1e-12)


def test_real_negative_A_is_the_real_ssd_with_the_hold_weights():
    # arg A = pi: A = -|A|, A_bar = exp(-dt |A|) (the SSD's dA with A_log = log|A|),
    # B_bar = (1 - A_bar) / |A| B; with real B, C, h0 that is the real SSD whose
    # input weight dt B is replaced by (1 - A_bar) / |A| B (one group per head)
    c = _case(5, Bt=2, L=7, H=3, P=4, K=3, G=3)
    c["A_polar"][:, 1] = np.pi
    for k in ("B", "C"):
        c[k][..., 1::2] = 0.0
    c["init_state"][..., 1::2] = 0.0
    y, fin = complex_fwd(**c)
    mag = np.exp(c["A_polar"][:, 0])
    dt = _softplus(c["dt_raw"] + c["dt_bias"][None, None, :])          # [Bt,L,H]
    w = (1.0 - np.exp(-dt * mag[None, None, :])) / (mag[None, None, :] * dt)
    Bre = c["B"][..., 0::2] * w[..., None]                              # [Bt,L,G=H,K]
    yr, fr = oracle.ssd_fwd(c["x"], c["dt_raw"], c["dt_bias"], np.log(mag), Bre, c["C"][..., 0::2], c["D"],
                            c["init_state"][..., 0::2])
    assert np.allclose(y, yr, rtol=1e-10, atol=1e-12)
    assert np.allclose(fin[..., 0::2], fr, rtol=1e-10, atol=1e-12)
    assert np.max(np.abs(fin[..., 1::2])) < 1e-12 * np.max(np.abs(fr))


def test_conjugating_A_B_C_and_the_state_leaves_y_unchanged():
    c = _case(6)
    y1, f1 = complex_fwd(**c)
    cc = dict(c)
    cc["A_polar"] = c["A_polar"] * np.array([1.0, -1.0])
    for k in ("B", "C", "init_state"):
        v = c[k].copy()
        v[..., 1::2] *= -1
        cc[k] = v
    y2, f2 = complex_fwd(**cc)
    assert np.allclose(y1, y2, rtol=1e-12, atol=1e-12)
    assert np.allclose(f1[..., 0::2], f2[..., 0::2], rtol=1e-12, atol=1e-12)
    assert np.allclose(f1[..., 1::2], -f2[..., 1::2], rtol=1e-12, atol=1e-12)


def test_linear_in_the_input_and_the_state():
    c = _case(7)
    y1, f1 = complex_fwd(**c)
    y2, f2 = complex_fwd(**dict(c, x=2.5 * c["x"], init_state=2.5 * c["init_state"]))
    assert np.allclose(y2, 2.5 * y1, rtol=1e-12, atol=1e-12) and np.allclose(f2, 2.5 * f1, rtol=1e-12, atol=1e-12)
