"""fp64 oracle for the steps around the scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it; the product library never imports it.

* :func:`conv1d_silu` -- the causal depthwise convolution over the fused
  x | B | C channels and its SiLU (the builderforce Mamba2Block runs one
  causal conv1d over the fused x, B and C projection channels; the conv1d
  kernel page: y[b,t,d] = sum_k weight[d,k] x[b,t-k,d] + bias[d] with x = 0
  before the sequence; the mamba-rs 0.4.0 S6 forward applies SiLU in the
  conv's own kernel and carries the conv state from call to call), split into
  the scan's x [B,L,H,P], B and C [B,L,G,N].
* :func:`gated_rmsnorm` -- the gated output norm of the Mamba-3 forward (step
  F7): RMSNorm(y) * weight * SiLU(z) over the H*P channels of each token.
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


def silu(v):
    """v * sigmoid(v)."""
    return v / (1.0 + np.exp(-v))


def conv1d_silu(xbc, weight, bias, conv_state, H, P, G, N):
    """Causal depthwise conv (K taps) + SiLU over the fused channels.

    ``xbc [B,L,C]`` with C = H*P + 2*G*N (x, then B, then C channels);
    ``weight [C,K]`` (tap k multiplies the input k steps back); ``bias [C]``
    or None; ``conv_state [B,K-1,C]`` or None: the K-1 inputs before the
    sequence, oldest first (zero when None).  Returns ``(x, B, C, state_out)``
    with x [B,L,H,P], B and C [B,L,G,N] and ``state_out [B,K-1,C]``: the last
    K-1 inputs of the extended sequence (what a following call continues from).
    """
    xbc, weight = _f64(xbc), _f64(weight)
    Bt, L, Cc = xbc.shape
    K = weight.shape[1]
    assert Cc == H * P + 2 * G * N
    prev = np.zeros((Bt, K - 1, Cc)) if conv_state is None else _f64(conv_state)
    ext = np.concatenate([prev, xbc], axis=1)            # [B, K-1+L, C]; ext[:, K-1+t] = x_t
    acc = np.zeros((Bt, L, Cc))
    for t in range(L):
        for k in range(K):
            acc[:, t] += weight[None, :, k] * ext[:, K - 1 + t - k]
    if bias is not None:
        acc += _f64(bias)[None, None, :]
    u = silu(acc)
    HP, GN = H * P, G * N
    x = u[:, :, :HP].reshape(Bt, L, H, P)
    Bm = u[:, :, HP:HP + GN].reshape(Bt, L, G, N)
    Cm = u[:, :, HP + GN:].reshape(Bt, L, G, N)
    return x, Bm, Cm, ext[:, ext.shape[1] - (K - 1):]


def gated_rmsnorm(y, z, weight, eps=1e-6):
    """RMSNorm(y) * weight * SiLU(z) per token over the last two axes' H*P
    channels: ``y, z [B,L,H,P]``, ``weight [H*P]``."""
    y, z, weight = _f64(y), _f64(z), _f64(weight)
    Bt, L, H, P = y.shape
    yf = y.reshape(Bt, L, H * P)
    rms = np.sqrt(np.mean(yf * yf, axis=-1, keepdims=True) + eps)
    out = yf / rms * weight[None, None, :] * silu(z.reshape(Bt, L, H * P))
    return out.reshape(Bt, L, H, P)
