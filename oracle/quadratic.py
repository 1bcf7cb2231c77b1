"""Materialised quadratic (dual) form of the SSD scan, fp64 numpy -- TEST INFRASTRUCTURE.

For one (batch, head) pair with a scalar decay per step the scan output has
the closed form

    y = (Lmat o (C B^T)) (dt o X) + D X + diag(decay0) C h0,
    Lmat[t, s] = prod_{k=s+1..t} dA_k   for s <= t, else 0,
    decay0[t]  = prod_{k=0..t}   dA_k,

and the state after the last step is

    h_L = decay0[L-1] h0 + sum_s (prod_{k=s+1..L-1} dA_k) dt_s B_s x_s^T.

This is the "semiseparable matrix" view of the structured state-space
duality: the recurrence and this matrix product are two evaluations of one
linear map.  The segment products are taken as explicit products of the
per-step decays (``np.prod`` over slices), not as differences of cumulative
sums, so this routine shares no arithmetic shortcut with the recurrence in
``ssd_oracle.c``.  softplus is evaluated with ``np.logaddexp(0, z)``.

Sources: the SSD module header of @seanhogg/builderforce-memory-engine
2026.6.18 package/dist/kernels/ssd.js (scalar decay per head, state carried
between chunks) and the discretised recurrence stated there, with the
readings A = -exp(A_log), input term dt * B x^T, per-channel readout.

Cost is O(L^3) per pair; intended for L <= 64.
"""
from __future__ import annotations

import numpy as np


def ssd_quadratic(x, dt_raw, dt_bias, A_log, B, C, D, init_state=None):
    """Brute-force quadratic form.  Returns ``(y, final_state)`` float64.

    Shapes as in :func:`oracle.ssd_fwd`.
    """
    x, dt_raw, dt_bias, A_log, B, C, D = (np.asarray(v, dtype=np.float64)
                                          for v in (x, dt_raw, dt_bias, A_log, B, C, D))
    h0_all = None if init_state is None else np.asarray(init_state, dtype=np.float64)
    Bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = np.zeros((Bt, L, H, P))
    final = np.zeros((Bt, H, P, N))
    for b in range(Bt):
        for h in range(H):
            g = h * G // H
            dt = np.logaddexp(0.0, dt_raw[b, :, h] + dt_bias[h])
            A = -np.exp(A_log[h])
            dA = np.exp(dt * A)
            Lmat = np.zeros((L, L))
            for t in range(L):
                for s in range(t + 1):
                    Lmat[t, s] = np.prod(dA[s + 1:t + 1])
            Cg = C[b, :, g, :]            # [L, N]
            Bg = B[b, :, g, :]            # [L, N]
            X = x[b, :, h, :]             # [L, P]
            yy = (Lmat * (Cg @ Bg.T)) @ (dt[:, None] * X) + D[h] * X
            # state after the last step, [N, P]
            w = np.array([np.prod(dA[s + 1:]) * dt[s] for s in range(L)])
            hL = Bg.T @ (w[:, None] * X)
            if h0_all is not None:
                h0 = h0_all[b, h].T       # stored [P, N] -> [N, P]
                decay0 = np.array([np.prod(dA[:t + 1]) for t in range(L)])
                yy = yy + (decay0[:, None] * Cg) @ h0
                hL = hL + np.prod(dA) * h0
            y[b, :, h, :] = yy
            final[b, h] = hL.T
    return y, final
