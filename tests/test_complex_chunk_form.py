"""The chunk form of the complex-valued (ET) scan, restated on the CPU in fp64
real arithmetic over the interleaved (re, im) index, against the sequential
oracle.

The tensor-core kernel evaluates the complex recurrence chunk by chunk with real
matrix products only; this test writes those products out in the kernel's
terms (no CUDA code is used) and checks that, before any bf16 rounding, they
give the recurrence exactly:

* S_re = C^ B^T and S_im = C~ B^T with C^ = (C_r, -C_i), C~ = (C_i, C_r), so
  S_re + i S_im = C_t . B_s (no conjugate);
* M[t][s] = Re(E_ts) S_re - Im(E_ts) S_im for s <= t, E_ts = e^{A (tau_t - tau_s)} f_s,
  built per 16-step block as a row factor e^{A (tau_t - tau_e)} times a column
  factor e^{A (tau_e - tau_s)} f_s (e the block's last step);
* Y = M x + C_L H with C_L[t] = (Re(Lambda_t C_t), -Im(Lambda_t C_t));
* H' = rot(Lambda_last) H + B~^T x with B~[s] = (Re(g_s B_s), Im(g_s B_s)).

A wrong sign in C^, C~ or C_L, a conjugated product, a transposed factor or a
dropped state term each moves the result far outside the bound below.
"""
import numpy as np
import pytest

from oracle.complex_scan import complex_A, complex_fwd


def _softplus(z):
    return np.maximum(z, 0) + np.log1p(np.exp(-np.abs(z)))


def _interleave(z):
    out = np.empty(z.shape[:-1] + (2 * z.shape[-1],))
    out[..., 0::2], out[..., 1::2] = z.real, z.imag
    return out


def chunk_form(x, dt_raw, dt_bias, A_polar, B, C, D, init_state, Q, block=16, slip=None):
    """y [Bt,L,H,P] and the final state [Bt,H,P,N] by the chunk form above."""
    Bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    A = complex_A(A_polar)
    dt = _softplus(dt_raw + dt_bias[None, None, :])
    y = np.zeros((Bt, L, H, P))
    final = np.zeros((Bt, H, P, N))
    for b in range(Bt):
        for h in range(H):
            g = h // (H // G)
            a = A[h]
            Hs = np.zeros((N, P)) if init_state is None else init_state[b, h].T.copy()   # [n][p]
            for c0 in range(0, L, Q):
                st = slice(c0, min(L, c0 + Q))
                n = st.stop - st.start
                d = dt[b, st, h]
                tau = np.cumsum(d)
                f = (np.exp(a * d) - 1.0) / a
                Cr, Br = C[b, st, g], B[b, st, g]                       # [n][N] real, interleaved
                Chat = Cr.copy()
                Chat[:, 1::2] *= -1.0
                Ctil = np.empty_like(Cr)
                Ctil[:, 0::2], Ctil[:, 1::2] = Cr[:, 1::2], Cr[:, 0::2]
                if slip == "sign_in_Ctil":
                    Ctil[:, 0::2] *= -1.0
                S_re, S_im = Chat @ Br.T, Ctil @ Br.T                   # [t][s]
                M = np.zeros((n, n))
                for s0 in range(0, n, block):
                    e = min(s0 + block, n) - 1
                    cols = np.arange(s0, e + 1)
                    colf = np.exp(a * (tau[e] - tau[cols])) * f[cols]
                    for t in range(s0, n):
                        E = np.exp(a * (tau[t] - tau[e])) * colf
                        m = E.real * S_re[t, cols] - E.imag * S_im[t, cols]
                        M[t, cols] = np.where(cols <= t, m, 0.0)
                lam = np.exp(a * tau)
                Cc = Cr[:, 0::2] + 1j * Cr[:, 1::2]
                LC = lam[:, None] * Cc
                CL = np.empty_like(Cr)
                CL[:, 0::2], CL[:, 1::2] = LC.real, -LC.imag
                if slip == "sign_in_CL":
                    CL[:, 1::2] *= -1.0
                xs = x[b, st, h]
                y[b, st, h] = M @ xs + (0.0 if slip == "no_state_term" else CL @ Hs) + D[h] * xs
                gs = np.exp(a * (tau[-1] - tau)) * f
                Bt_ = _interleave(gs[:, None] * (Br[:, 0::2] + 1j * Br[:, 1::2]))   # B~ [n][N]
                Hc = (Hs[0::2] + 1j * Hs[1::2]) * (1.0 if slip == "no_rotation" else lam[-1])   # rot(Lambda_last) H
                Hs = np.empty_like(Hs)
                Hs[0::2], Hs[1::2] = Hc.real, Hc.imag
                Hs = Hs + Bt_.T @ xs
            final[b, h] = Hs.T
    return y, final


def _case(seed, Bt, L, H, P, N, G, init):
    rng = np.random.default_rng(seed)
    return dict(x=rng.standard_normal((Bt, L, H, P)), dt_raw=0.5 * rng.standard_normal((Bt, L, H)),
                dt_bias=rng.uniform(-3.0, -1.0, H),
                A_polar=np.stack([np.log(rng.uniform(0.3, 3.0, H)), rng.uniform(0.55 * np.pi, 1.45 * np.pi, H)], 1),
                B=rng.standard_normal((Bt, L, G, N)), C=rng.standard_normal((Bt, L, G, N)),
                D=rng.standard_normal(H), init_state=0.5 * rng.standard_normal((Bt, H, P, N)) if init else None)


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


@pytest.mark.parametrize("L,Q,init", [(64, 64, True), (200, 64, True), (77, 32, False), (1, 64, True),
                                      (130, 16, True)])
def test_chunk_form_equals_the_recurrence(L, Q, init):
    c = _case(11 + L + Q, Bt=2, L=L, H=3, P=5, N=8, G=1, init=init)
    y0, f0 = complex_fwd(**c)
    y1, f1 = chunk_form(**c, Q=Q)
    assert _rel(y1, y0) < 1e-10, _rel(y1, y0)
    assert _rel(f1, f0) < 1e-10, _rel(f1, f0)


def test_chunk_form_with_groups():
    c = _case(5, Bt=1, L=96, H=4, P=3, N=6, G=2, init=True)
    y0, f0 = complex_fwd(**c)
    y1, f1 = chunk_form(**c, Q=64)
    assert _rel(y1, y0) < 1e-10 and _rel(f1, f0) < 1e-10


def test_a_conjugated_product_is_caught():
    # the same form with S_im taken from conj(C) . B: the test's bound must catch it
    c = _case(7, Bt=1, L=64, H=2, P=4, N=8, G=1, init=True)
    y0, _ = complex_fwd(**c)
    bad = dict(c)
    Cb = c["C"].copy()
    Cb[..., 1::2] *= -1.0              # C_i -> -C_i everywhere: the readout of conj(C)
    y1, _ = chunk_form(**bad | {"C": Cb}, Q=64)
    assert _rel(y1, y0) > 1e-2


@pytest.mark.parametrize("slip", ["sign_in_Ctil", "sign_in_CL", "no_state_term", "no_rotation"])
def test_planted_slips_are_caught(slip):
    c = _case(13, Bt=2, L=200, H=3, P=5, N=8, G=1, init=True)
    y0, _ = complex_fwd(**c)
    y1, _ = chunk_form(**c, Q=64, slip=slip)
    assert _rel(y1, y0) > 1e-2
