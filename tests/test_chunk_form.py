"""The sub-chunk form of the forward scan that the tensor-core kernel
evaluates, restated on the CPU in fp64, against the sequential oracles.

Per head, over sub-chunks of T steps with cs the sub-chunk-local inclusive
cumsum of the log decay and u the input weight of each step:

    S      = C B^T
    M[t,s] = S[t,s] exp(cs_t - cs_s) u_s      (s <= t), per 16-step block as a
             row factor exp(cs_t - cs_e) times a column factor exp(cs_e - cs_s) u_s
    y      = M x + D x + exp(cs_t) (C P)
    P     <- exp(cs_last) P + B^T (w o x),   w_s = exp(cs_last - cs_s) u_s

For the Mamba-2 scan the log decay is dt a and u = dt. The trapezoidal mode
runs the same form on the shifted state h~_t = h_t + dt_{t+1}(1 - trap_{t+1})
k_t v_t^T: log decay a_t dt_t, u_t = gamma_t + dt_{t+1}(1 - trap_{t+1}) (gamma
alone at the last step), M's diagonal S[t,t] gamma_t, and the entering state
h0 + dt_0 (1 - trap_0) k0 v0^T.

The split evaluation cuts each sequence into units: every unit's end state
from zero and its total decay, then E_0 = the entering state, E_{k+1} =
Lambda_k E_k + S_k, then every unit again from E_k. In the trapezoidal mode
the first unit starts from the entering state and the combine from zero.

No CUDA code is used. A dropped decay factor, a row/column factor swap or a
wrong diagonal in the trapezoidal mode moves the result far outside the bound.
"""
import numpy as np
import pytest

import oracle
from oracle.trap import trap_coefficients, trap_fwd


def _softplus(z):
    return np.maximum(z, 0) + np.log1p(np.exp(-np.abs(z)))


def sub_chunk_scan(xh, Bg, Cg, logd, u, skip, Hs, T, diag=None, block=16, slip=None):
    """One head's scan over [L] steps from state Hs [N][P] by the form above.
    diag (or None): M's diagonal weight per step in place of u.  Returns (y, Hs)."""
    L = xh.shape[0]
    y = np.zeros_like(xh)
    Hs = Hs.copy()
    for t0 in range(0, L, T):
        st = slice(t0, min(L, t0 + T))
        n = st.stop - st.start
        cs = np.cumsum(logd[st])
        us, xs, Cs, Bs = u[st], xh[st], Cg[st], Bg[st]
        S = Cs @ Bs.T
        M = np.zeros((n, n))
        for s0 in range(0, n, block):
            e = min(s0 + block, n) - 1
            cols = np.arange(s0, e + 1)
            colf = np.exp(cs[e] - cs[cols]) * us[cols]
            for t in range(s0, n):
                rf = np.exp(cs[t] - cs[e])
                if slip == "swap_factors":
                    rf, cf = np.exp(cs[e] - cs[t]), np.exp(cs[cols] - cs[e]) * us[cols]
                else:
                    cf = colf
                M[t, cols] = np.where(cols <= t, S[t, cols] * rf * cf, 0.0)
        if diag is not None:
            idx = np.arange(n)
            M[idx, idx] = S[idx, idx] * diag[st]
        ecs = np.exp(cs) if slip != "no_row_decay" else np.ones(n)
        y[st] = M @ xs + skip * xs + ecs[:, None] * (Cs @ Hs)
        w = np.exp(cs[-1] - cs) * us
        Hs = np.exp(cs[-1]) * Hs + Bs.T @ (w[:, None] * xs)
    return y, Hs


def ssd_sub_chunk(x, dt_raw, dt_bias, A_log, B, C, D, init_state, T, unit=None, slip=None):
    """The Mamba-2 scan by the sub-chunk form; with unit (steps, a multiple of
    T), by the split evaluation over units of that length."""
    Bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = np.zeros_like(x)
    fin = np.zeros((Bt, H, P, N))
    for b in range(Bt):
        for h in range(H):
            g = h // (H // G)
            dt = _softplus(dt_raw[b, :, h] + dt_bias[h])
            logd = dt * -np.exp(A_log[h])
            h0 = np.zeros((N, P)) if init_state is None else init_state[b, h].T
            args = (B[b, :, g], C[b, :, g])
            if unit is None:
                yy, hs = sub_chunk_scan(x[b, :, h], *args, logd, dt, D[h], h0, T, slip=slip)
            else:
                units = [slice(s, min(L, s + unit)) for s in range(0, L, unit)]
                ends, lams = [], []
                for us_ in units:    # pass 1: every unit from zero
                    _, e = sub_chunk_scan(x[b, us_, h], args[0][us_], args[1][us_], logd[us_], dt[us_], D[h],
                                          np.zeros((N, P)), T)
                    ends.append(e)
                    lams.append(np.exp(np.sum(logd[us_])))
                E = [h0]             # the combine
                for k in range(len(units) - 1):
                    E.append(lams[k] * E[k] + ends[k])
                yy = np.zeros((L, P))
                for k, us_ in enumerate(units):    # pass 3
                    yy[us_], hs = sub_chunk_scan(x[b, us_, h], args[0][us_], args[1][us_], logd[us_], dt[us_],
                                                 D[h], E[k], T)
            y[b, :, h], fin[b, h] = yy, hs.T
    return y, fin


def trap_sub_chunk(v, k, q, dt, a, trap, D, h0, k0, v0, T, unit=None, slip=None):
    """The trapezoidal scan by the shifted-state sub-chunk form (optionally split)."""
    Bt, L, H, P = v.shape
    G, N = k.shape[2], k.shape[3]
    _, _, gamma = trap_coefficients(dt, a, trap)
    y = np.zeros_like(v)
    fin = np.zeros((Bt, H, P, N))
    for b in range(Bt):
        for h in range(H):
            g = h // (H // G)
            nxt = np.zeros(L)            # dt_{t+1} (1 - trap_{t+1}), zero past the last step
            nxt[:-1] = dt[b, 1:, h] * (1.0 - trap[b, 1:, h])
            w = gamma[b, :, h] + nxt
            logd = a[b, :, h] * dt[b, :, h]
            diag = gamma[b, :, h] if slip != "diag_w" else w
            enter = (np.zeros((N, P)) if h0 is None else h0[b, h].T.copy())
            if k0 is not None and v0 is not None:
                enter = enter + dt[b, 0, h] * (1.0 - trap[b, 0, h]) * np.outer(k0[b, h], v0[b, h])
            kk, qq, vv = k[b, :, g], q[b, :, g], v[b, :, h]
            if unit is None:
                yy, hs = sub_chunk_scan(vv, kk, qq, logd, w, D[h], enter, T, diag=diag)
            else:
                units = [slice(s, min(L, s + unit)) for s in range(0, L, unit)]
                ends, lams = [], []
                for i, us_ in enumerate(units):   # pass 1: the first unit from the entering state
                    start = enter if i == 0 else np.zeros((N, P))
                    _, e = sub_chunk_scan(vv[us_], kk[us_], qq[us_], logd[us_], w[us_], D[h], start, T,
                                          diag=diag[us_])
                    ends.append(e)
                    lams.append(np.exp(np.sum(logd[us_])))
                E = [np.zeros((N, P))]             # the combine starts from zero
                for i in range(len(units) - 1):
                    E.append(lams[i] * E[i] + ends[i])
                yy = np.zeros((L, P))
                for i, us_ in enumerate(units):
                    start = enter if i == 0 else E[i]
                    yy[us_], hs = sub_chunk_scan(vv[us_], kk[us_], qq[us_], logd[us_], w[us_], D[h], start, T,
                                                 diag=diag[us_])
            y[b, :, h], fin[b, h] = yy, hs.T
    return y, fin


def _ssd_case(seed, Bt=2, L=150, H=4, P=3, N=6, G=2, init=True):
    rng = np.random.default_rng(seed)
    return dict(x=rng.standard_normal((Bt, L, H, P)), dt_raw=0.5 * rng.standard_normal((Bt, L, H)),
                dt_bias=rng.uniform(-4.0, -2.0, H), A_log=np.log(rng.uniform(0.5, 4.0, H)),
                B=rng.standard_normal((Bt, L, G, N)), C=rng.standard_normal((Bt, L, G, N)),
                D=rng.standard_normal(H), init_state=rng.standard_normal((Bt, H, P, N)) if init else None)


def _trap_case(seed, Bt=2, L=150, H=4, P=3, N=6, G=2, carried=True):
    rng = np.random.default_rng(seed)
    return dict(v=rng.standard_normal((Bt, L, H, P)), k=rng.standard_normal((Bt, L, G, N)),
                q=rng.standard_normal((Bt, L, G, N)), dt=_softplus(rng.uniform(-4.0, -1.5, (Bt, L, H))),
                a=-rng.uniform(0.5, 4.0, (Bt, L, H)), trap=rng.uniform(0.0, 1.0, (Bt, L, H)),
                D=rng.standard_normal(H),
                h0=rng.standard_normal((Bt, H, P, N)) if carried else None,
                k0=rng.standard_normal((Bt, H, N)) if carried else None,
                v0=rng.standard_normal((Bt, H, P)) if carried else None)


def _rel(u, v):
    return float(np.max(np.abs(u - v)) / max(np.max(np.abs(v)), 1e-300))


@pytest.mark.parametrize("L,T,init", [(150, 32, True), (128, 128, False), (77, 16, True), (1, 32, True)])
def test_sub_chunk_form_equals_the_recurrence(L, T, init):
    c = _ssd_case(L + T, L=L, init=init)
    y0, f0 = oracle.ssd_fwd(**c)
    y1, f1 = ssd_sub_chunk(**c, T=T)
    assert _rel(y1, y0) < 1e-10 and _rel(f1, f0) < 1e-10, (_rel(y1, y0), _rel(f1, f0))


@pytest.mark.parametrize("L,T,unit,init", [(150, 16, 48, True), (200, 32, 32, True), (97, 16, 64, False)])
def test_split_evaluation_equals_the_recurrence(L, T, unit, init):
    c = _ssd_case(3 * L + unit, L=L, init=init)
    y0, f0 = oracle.ssd_fwd(**c)
    y1, f1 = ssd_sub_chunk(**c, T=T, unit=unit)
    assert _rel(y1, y0) < 1e-10 and _rel(f1, f0) < 1e-10, (_rel(y1, y0), _rel(f1, f0))


@pytest.mark.parametrize("L,T,unit,carried", [(150, 32, None, True), (77, 16, None, False),
                                              (150, 16, 48, True), (96, 32, 32, False)])
def test_trapezoidal_shifted_state_form(L, T, unit, carried):
    c = _trap_case(L + T, L=L, carried=carried)
    y0, f0, _, _ = trap_fwd(**c)
    y1, f1 = trap_sub_chunk(**c, T=T, unit=unit)
    assert _rel(y1, y0) < 1e-10 and _rel(f1, f0) < 1e-10, (_rel(y1, y0), _rel(f1, f0))


@pytest.mark.parametrize("slip", ["swap_factors", "no_row_decay"])
def test_planted_slips_are_caught(slip):
    c = _ssd_case(21, L=96)
    y0, _ = oracle.ssd_fwd(**c)
    y1, _ = ssd_sub_chunk(**c, T=32, slip=slip)
    assert _rel(y1, y0) > 1e-3


def test_trapezoidal_diagonal_slip_is_caught():
    c = _trap_case(22, L=64)
    y0, _, _, _ = trap_fwd(**c)
    y1, _ = trap_sub_chunk(**c, T=32, slip="diag_w")
    assert _rel(y1, y0) > 1e-3
