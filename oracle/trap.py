"""fp64 oracle for the trapezoidal (Mamba-3 SISO) scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it; the product library never imports it.

What is computed (the Mamba-3 SISO GPU forward of the pages, mamba-rs 0.2.1
mamba3_siso/gpu/mamba3_gpu.rs: its module header states a recurrence that is
trapezoidal in three coefficients where Mamba-2's is exponential, and two
more carried states holding the last k and v; step F5b gives the
coefficients), per batch row b and head h, with v = x, k = B, q = C:

    alpha_t = exp(a_t * dt_t)
    beta_t  = alpha_t * dt_t * (1 - trap_t)
    gamma_t = trap_t * dt_t
    h_t = alpha_t * h_{t-1} + beta_t * k_{t-1} v_{t-1}^T + gamma_t * k_t v_t^T
    y_t = q_t^T h_t + D * v_t

The pages print the coefficients and the persistent k/v states but not the
recurrence itself; the form above is the reading they support (the k/v
states exist to carry k_{t-1}, v_{t-1} into the next call's first step).
k_{-1}, v_{-1} are the carried k_state, v_state (zero when not given).

Two statements of it:
* :func:`trap_fwd` -- the recurrence, one step after another.
* :func:`trap_unrolled` -- the recurrence unrolled into a sum over the input
  terms: h_t = (prod_{r<=t} alpha_r) h0 + sum_{s<=t} (prod_{s<r<=t} alpha_r)
  (beta_s k_{s-1} v_{s-1}^T + gamma_s k_s v_s^T), materialised for tiny inputs.
"""
from __future__ import annotations

import numpy as np


def _f64(v):
    if v is None:
        return None
    if hasattr(v, "detach"):
        v = v.detach().cpu()
        import torch
        if v.dtype == torch.bfloat16:
            v = v.float()
        v = v.numpy()
    return np.asarray(v, dtype=np.float64)


def trap_coefficients(dt, a, trap):
    """(alpha, beta, gamma) from dt, a and trap: step F5b of the Mamba-3 forward."""
    dt, a, trap = _f64(dt), _f64(a), _f64(trap)
    alpha = np.exp(a * dt)
    return alpha, alpha * dt * (1.0 - trap), trap * dt


def _group_index(H, G):
    return np.arange(H) // (H // G)


def trap_fwd(v, k, q, dt, a, trap, D, h0=None, k0=None, v0=None):
    """Sequential fp64 recurrence.  Returns ``(y, h_final, k_final, v_final)``.

    Shapes: ``v [Bt,L,H,P]``; ``k, q [Bt,L,G,N]``; ``dt, a, trap [Bt,L,H]``;
    ``D [H]``; ``h0 [Bt,H,P,N]``, ``k0 [Bt,H,N]``, ``v0 [Bt,H,P]`` or None
    (zero).  States are stored ``[P, N]`` (n fastest), as for the SSD scan.
    ``k_final[b,h] = k[b,L-1,g(h)]`` and ``v_final[b,h] = v[b,L-1,h]`` are the
    states a following call continues from (k0, v0 again for L = 0).
    """
    v, k, q, D = _f64(v), _f64(k), _f64(q), _f64(D)
    alpha, beta, gamma = trap_coefficients(dt, a, trap)
    Bt, L, H, P = v.shape
    G, N = k.shape[2], k.shape[3]
    gi = _group_index(H, G)
    h = np.zeros((Bt, H, P, N)) if h0 is None else _f64(h0).copy()
    kp = np.zeros((Bt, H, N)) if k0 is None else _f64(k0).copy()
    vp = np.zeros((Bt, H, P)) if v0 is None else _f64(v0).copy()
    y = np.zeros((Bt, L, H, P))
    for t in range(L):
        kt = k[:, t][:, gi]                       # [Bt,H,N]
        vt = v[:, t]                              # [Bt,H,P]
        h = (alpha[:, t, :, None, None] * h
             + beta[:, t, :, None, None] * vp[:, :, :, None] * kp[:, :, None, :]
             + gamma[:, t, :, None, None] * vt[:, :, :, None] * kt[:, :, None, :])
        y[:, t] = np.einsum("bhpn,bhn->bhp", h, q[:, t][:, gi]) + D[None, :, None] * vt
        kp, vp = kt, vt
    return y, h, kp, vp


def trap_unrolled(v, k, q, dt, a, trap, D, h0=None, k0=None, v0=None):
    """The same scan as a sum over input terms (tiny inputs only).  Returns
    ``(y, h_final)``."""
    v, k, q, D = _f64(v), _f64(k), _f64(q), _f64(D)
    alpha, beta, gamma = trap_coefficients(dt, a, trap)
    Bt, L, H, P = v.shape
    G, N = k.shape[2], k.shape[3]
    gi = _group_index(H, G)
    h0 = np.zeros((Bt, H, P, N)) if h0 is None else _f64(h0)
    k0 = np.zeros((Bt, H, N)) if k0 is None else _f64(k0)
    v0 = np.zeros((Bt, H, P)) if v0 is None else _f64(v0)
    y = np.zeros((Bt, L, H, P))
    hL = None
    for b in range(Bt):
        for hh in range(H):
            g = gi[hh]
            ks = [k0[b, hh]] + [k[b, s, g] for s in range(L)]      # ks[s+1] = k_s
            vs = [v0[b, hh]] + [v[b, s, hh] for s in range(L)]
            for t in range(L):
                ht = np.prod(alpha[b, :t + 1, hh]) * h0[b, hh]
                for s in range(t + 1):
                    decay = np.prod(alpha[b, s + 1:t + 1, hh])
                    ht = ht + decay * (beta[b, s, hh] * np.outer(vs[s], ks[s])
                                       + gamma[b, s, hh] * np.outer(vs[s + 1], ks[s + 1]))
                y[b, t, hh] = ht @ q[b, t, g] + D[hh] * v[b, t, hh]
                if t == L - 1:
                    if hL is None:
                        hL = np.zeros((Bt, H, P, N))
                    hL[b, hh] = ht
    return y, hL
