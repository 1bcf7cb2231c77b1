"""fp64 oracle for the complex-valued scan with exponential-trapezoidal (ET)
discretisation -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it; the product library never imports it.

It follows the header of the pages' Mamba-3 complex SSD kernel (the
``complex_ssd.ts`` module: complex-valued states, ET discretisation, SISO):
per head, ``A`` is complex and stored in polar form ``A_polar[h] = (log|A|,
arg A)``, so ``A = exp(log|A| + i arg A)``; with ``dt_t = softplus(dt_raw_t +
dt_bias)``,

    A_bar_t = exp(dt_t A)
    B_bar_t = (A_bar_t - 1) A^-1 B_t          (the exact zero-order hold)
    h_t     = A_bar_t h_{t-1} + B_bar_t x_t^T (state: N/2 complex rows x P)
    y_t     = Re(C_t^T h_t) + D x_t

B, C and the state hold complex numbers as interleaved (re, im) pairs along
N: component k is (v[2k], v[2k+1]).  The page's printed kernel deviates from
its header in two places. Its A_bar exponentiates dt (log|A| + i arg A)
rather than dt A. Its readout conjugates C. The header's statement is the one
taken here (it is the only one under which B_bar is the exact hold its
comment claims).
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


def complex_A(A_polar):
    """A[h] = exp(log|A| + i arg A) from the polar pairs [H, 2]."""
    ap = _f64(A_polar)
    return np.exp(ap[:, 0]) * np.exp(1j * ap[:, 1])


def to_complex(v):
    """[..., N] interleaved (re, im) -> [..., N/2] complex."""
    v = _f64(v)
    return v[..., 0::2] + 1j * v[..., 1::2]


def to_interleaved(z):
    """[..., N/2] complex -> [..., N] interleaved (re, im)."""
    out = np.empty(z.shape[:-1] + (2 * z.shape[-1],))
    out[..., 0::2] = z.real
    out[..., 1::2] = z.imag
    return out


def complex_fwd(x, dt_raw, dt_bias, A_polar, B, C, D, init_state=None):
    """The recurrence above, step by step.  Shapes: x [Bt,L,H,P]; dt_raw
    [Bt,L,H]; dt_bias, D [H]; A_polar [H,2]; B, C [Bt,L,G,N] (N even,
    interleaved); init_state [Bt,H,P,N] (interleaved) or None.  Returns
    (y [Bt,L,H,P], final_state [Bt,H,P,N]) as float64."""
    x, r, bias, D = (_f64(v) for v in (x, dt_raw, dt_bias, D))
    Bt, L, H, P = x.shape
    Bc, Cc = to_complex(B), to_complex(C)                  # [Bt,L,G,K]
    G, K = Bc.shape[2], Bc.shape[3]
    gi = np.arange(H) // (H // G)
    A = complex_A(A_polar)                                 # [H]
    z = r + bias[None, None, :]
    dt = np.maximum(z, 0) + np.log1p(np.exp(-np.abs(z)))   # softplus
    h = np.zeros((Bt, H, K, P), dtype=np.complex128)
    if init_state is not None:
        h = np.swapaxes(to_complex(init_state), 2, 3)      # [Bt,H,K,P]
    y = np.zeros((Bt, L, H, P))
    for t in range(L):
        Abar = np.exp(dt[:, t, :] * A[None, :])            # [Bt,H]
        f = (Abar - 1.0) / A[None, :]                      # (A_bar - 1) A^-1
        Bh = Bc[:, t][:, gi]                               # [Bt,H,K]
        Ch = Cc[:, t][:, gi]
        h = Abar[:, :, None, None] * h + (f[:, :, None] * Bh)[..., None] * x[:, t, :, None, :]
        y[:, t] = np.einsum("bhk,bhkp->bhp", Ch, h).real + D[None, :, None] * x[:, t]
    final = to_interleaved(np.swapaxes(h, 2, 3))           # [Bt,H,P,N]
    return y, final


def complex_unrolled(x, dt_raw, dt_bias, A_polar, B, C, D, init_state=None):
    """The same map written as sums over products of A_bar (no recurrence):
    h_t = (prod_{r<=t} A_bar_r) h0 + sum_{s<=t} (prod_{s<r<=t} A_bar_r) B_bar_s x_s^T.
    O(L^2): small inputs only."""
    x, r, bias, D = (_f64(v) for v in (x, dt_raw, dt_bias, D))
    Bt, L, H, P = x.shape
    Bc, Cc = to_complex(B), to_complex(C)
    G, K = Bc.shape[2], Bc.shape[3]
    gi = np.arange(H) // (H // G)
    A = complex_A(A_polar)
    z = r + bias[None, None, :]
    dt = np.maximum(z, 0) + np.log1p(np.exp(-np.abs(z)))
    Abar = np.exp(dt * A[None, None, :])                   # [Bt,L,H]
    h0 = np.zeros((Bt, H, K, P), dtype=np.complex128)
    if init_state is not None:
        s = _f64(init_state)
        h0 = np.swapaxes(s[..., 0::2] + 1j * s[..., 1::2], 2, 3)
    y = np.zeros((Bt, L, H, P))
    final = None
    for t in range(L):
        ht = np.prod(Abar[:, : t + 1], axis=1)[:, :, None, None] * h0
        for s_ in range(t + 1):
            decay = np.prod(Abar[:, s_ + 1: t + 1], axis=1)          # [Bt,H]
            bbar = ((Abar[:, s_] - 1.0) / A[None, :])[:, :, None] * Bc[:, s_][:, gi]
            ht = ht + decay[:, :, None, None] * bbar[..., None] * x[:, s_, :, None, :]
        y[:, t] = np.einsum("bhk,bhkp->bhp", Cc[:, t][:, gi], ht).real + D[None, :, None] * x[:, t]
        final = ht
    if final is None:
        final = h0
    fs = np.swapaxes(final, 2, 3)
    out = np.empty(fs.shape[:-1] + (2 * fs.shape[-1],))
    out[..., 0::2], out[..., 1::2] = fs.real, fs.imag
    return y, out
