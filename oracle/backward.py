"""fp64 oracle for the backward of the SSD scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it; the product library never imports it.

The forward (the plain recurrence of :func:`oracle.ssd_fwd`), per batch row b
and head h, with dt_t = softplus(r_t + bias), a = -exp(A_log), dA_t = exp(dt_t a):
    h_t = dA_t h_{t-1} + dt_t B_t x_t^T            (state [N,P])
    y_t = C_t^T h_t + D x_t
Given dy (and d_final, the gradient of the loss with respect to the final
state), the backward runs the recurrence of the gradient of the state in
reverse, written here from differentiating the two lines above:
    G_{L-1} = d_final + C_{L-1} dy_{L-1}^T;  G_t = dA_{t+1} G_{t+1} + C_t dy_t^T
and, per step,
    dx_t   = D dy_t + dt_t G_t^T B_t
    dB_t   = dt_t G_t x_t                          (summed over the group's heads)
    dC_t   = h_t dy_t                              (summed over the group's heads)
    ddt_t  = sum_{n,p} G_t[n,p] (a dA_t h_{t-1}[n,p] + B_t[n] x_t[p])
    da    += sum_{n,p} G_t[n,p] dt_t dA_t h_{t-1}[n,p]
    dD    += dy_t . x_t
with d r_t = ddt_t sigmoid(r_t + bias), d bias = sum_{b,t} d r_t,
dA_log = da * a, and d init = dA_0 G_0.  The pages sketch a backward of their
own (the SSD module's simplified WGSL backward and the 7-step chunked
backward plan of the Mamba-3 GPU module) but print no formulas to follow;
these are the derivatives of the forward they define.
"""
from __future__ import annotations

import numpy as np


def _f64(v):
    if v is None:
        return None
    if hasattr(v, "detach"):
        import torch
        v = v.detach().cpu()
        if v.dtype == torch.bfloat16:
            v = v.float()
        v = v.numpy()
    return np.asarray(v, dtype=np.float64)


def ssd_bwd(x, dt_raw, dt_bias, A_log, B, C, D, init_state, dy, d_final=None):
    """Gradients of the SSD scan.  Shapes as :func:`oracle.ssd_fwd`, plus
    ``dy [Bt,L,H,P]`` and ``d_final [Bt,H,P,N]`` (or None).  Returns a dict
    with dx, ddt_raw, ddt_bias, dA_log, dB, dC, dD, d_init (float64; d_init
    also when init_state is None: the gradient a given initial state would get).
    """
    x, r, bias, A_log, B, C, D, dy = (_f64(v) for v in (x, dt_raw, dt_bias, A_log, B, C, D, dy))
    Bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    gi = np.arange(H) // (H // G)
    h0 = np.zeros((Bt, H, N, P)) if init_state is None else np.swapaxes(_f64(init_state), 2, 3)
    z = r + bias[None, None, :]
    dt = np.maximum(z, 0) + np.log1p(np.exp(-np.abs(z)))
    a = -np.exp(A_log)
    dA = np.exp(dt * a[None, None, :])
    Bh, Ch = B[:, :, gi], C[:, :, gi]                       # [Bt,L,H,N]
    # forward states h[t] for t = -1 .. L-1 (index t + 1), [N,P] per head
    hs = np.zeros((L + 1, Bt, H, N, P))
    hs[0] = h0
    for t in range(L):
        hs[t + 1] = dA[:, t, :, None, None] * hs[t] + dt[:, t, :, None, None] * Bh[:, t, :, :, None] * x[:, t, :, None, :]
    Gs = np.zeros((Bt, H, N, P)) if d_final is None else np.swapaxes(_f64(d_final), 2, 3).copy()
    dx = np.zeros_like(x)
    dBh = np.zeros((Bt, L, H, N))
    dCh = np.zeros((Bt, L, H, N))
    ddt = np.zeros((Bt, L, H))
    da = np.zeros(H)
    for t in range(L - 1, -1, -1):
        if t < L - 1:
            Gs = dA[:, t + 1, :, None, None] * Gs
        Gs = Gs + Ch[:, t, :, :, None] * dy[:, t, :, None, :]
        dx[:, t] = D[None, :, None] * dy[:, t] + dt[:, t, :, None] * np.einsum("bhnp,bhn->bhp", Gs, Bh[:, t])
        dBh[:, t] = dt[:, t, :, None] * np.einsum("bhnp,bhp->bhn", Gs, x[:, t])
        dCh[:, t] = np.einsum("bhnp,bhp->bhn", hs[t + 1], dy[:, t])
        gh = np.einsum("bhnp,bhnp->bh", Gs, hs[t])
        ddt[:, t] = a[None, :] * dA[:, t] * gh + np.einsum("bhnp,bhn,bhp->bh", Gs, Bh[:, t], x[:, t])
        da += np.sum(dt[:, t] * dA[:, t] * gh, axis=0)
    d_init = np.swapaxes(dA[:, 0, :, None, None] * Gs, 2, 3)
    dB = np.zeros((Bt, L, G, N))
    dC = np.zeros((Bt, L, G, N))
    for h in range(H):
        dB[:, :, gi[h]] += dBh[:, :, h]
        dC[:, :, gi[h]] += dCh[:, :, h]
    sig = 1.0 / (1.0 + np.exp(-z))
    ddt_raw = ddt * sig
    return dict(dx=dx, ddt_raw=ddt_raw, ddt_bias=ddt_raw.sum(axis=(0, 1)), dA_log=da * a,
                dB=dB, dC=dC, dD=np.einsum("blhp,blhp->h", dy, x), d_init=d_init)
