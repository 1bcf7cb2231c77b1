"""Seeded synthetic inputs for the SSD forward scan.

This module only draws random numbers and lays them out; it holds none of the
scan's arithmetic.  The same tensors (same bytes) feed the CUDA path and the
fp64 oracle.

Workloads are shaped like the Mamba layers that the source pages build
(@seanhogg/builderforce-memory-engine ``Mamba2BlockConfig``: multi-head SSM
with scalar A per head, state size N, head groups G, chunk length Q).

Distributions (one recipe for every workload):
  x ~ N(0, 1)                          [B, L, H, P]   storage dtype
  dt_raw ~ N(0, 0.1^2)                 [B, L, H]      fp32
  dt0 = exp(U[ln 1e-3, ln 1e-1]),  dt_bias = log(expm1(dt0))   [H] fp32
      (the inverse of softplus, so that softplus(dt_bias) = dt0)
  A_log = log(U[1, 16])                [H]            fp32
  B, C ~ N(0, 1)                       [B, L, G, N]   storage dtype
  D ~ N(0, 1)                          [H]            fp32
  init_state ~ N(0, 0.1^2)             [B, H, P, N]   fp32 (only where used)
Draw order is fixed: x, dt_raw, dt0, A_log, B, C, D, init_state, from one
numpy PCG64 stream seeded with ``seed``.  Values are drawn in float32 and
cast once to the storage dtype (bf16: round to nearest even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    dtype: str          # storage dtype of x, B, C, y: "bf16" or "f32"
    init_state: bool    # whether a non-zero initial state is passed
    op: str = "ssd"     # "ssd": the Mamba-2 SSD scan; "trap": the trapezoidal (Mamba-3 SISO) scan

    @property
    def token_heads(self) -> int:
        return self.batch * self.seqlen * self.nheads

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # tiny fp32 case that the oracle finishes in milliseconds
    "tiny_fp32": Workload("tiny_fp32", 1, 64, 2, 8, 16, 1, 16, "f32", False),
    # Mamba-2 130M layer: d_model 768, expand 2 -> H = 24 heads of P = 64
    "mamba2_130m_layer": Workload("mamba2_130m_layer", 4, 2048, 24, 64, 128, 1, 256, "bf16", False),
    # Mamba-2 2.7B layer: d_model 2560, expand 2 -> H = 80 heads of P = 64
    "mamba2_2p7b_layer": Workload("mamba2_2p7b_layer", 8, 4096, 80, 64, 128, 1, 256, "bf16", False),
    # one 64k-token sequence, 8 groups of 4 heads, carried-in and returned state
    "long_context_64k": Workload("long_context_64k", 1, 65536, 32, 64, 128, 8, 256, "bf16", True),
    # many 64-token sequences with per-sequence state in and out
    "many_short_seqs": Workload("many_short_seqs", 256, 64, 48, 64, 128, 1, 64, "bf16", True),
    # one decode step of the 2.7B layer's SSM for 128 sequences: one token each,
    # the carried state in and the updated state out
    "decode_2p7b_128seq": Workload("decode_2p7b_128seq", 128, 1, 80, 64, 128, 1, 256, "bf16", True),
    # trapezoidal (Mamba-3 SISO) scan: many 64-token sequences with the carried
    # state and k/v states in and out (the short-sequence regime the pages run
    # sequentially), and one decode step of 128 sequences
    "trap_many_short_seqs": Workload("trap_many_short_seqs", 256, 64, 48, 64, 128, 1, 1, "bf16", True, "trap"),
    "trap_decode_2p7b_128seq": Workload("trap_decode_2p7b_128seq", 128, 1, 80, 64, 128, 1, 1, "bf16", True,
                                        "trap"),
    # the trapezoidal scan over one 64k-token sequence (the long-context shape):
    # few chains, so the chunked kernel takes its split schedule
    "trap_long_context_64k": Workload("trap_long_context_64k", 1, 65536, 32, 64, 128, 8, 256, "bf16", True, "trap"),
    # the steps around the 2.7B layer's scan: the 4-tap conv1d + SiLU over its
    # fused x | B | C channels (with a carried conv state), and the gated RMSNorm
    "conv_silu_2p7b": Workload("conv_silu_2p7b", 8, 4096, 80, 64, 128, 1, 1, "bf16", True, "conv"),
    "gnorm_2p7b": Workload("gnorm_2p7b", 8, 4096, 80, 64, 128, 1, 1, "bf16", False, "gnorm"),
    # the conv1d + SiLU and the scan of the 2.7B layer in one call (the conv of the x
    # channels inside the chunked scan kernel), the conv state carried in and out
    "conv_scan_2p7b": Workload("conv_scan_2p7b", 8, 4096, 80, 64, 128, 1, 256, "bf16", True, "conv_scan"),
    # the backward of the scan on the 2.7B layer's heads, 2 sequences of 1024 steps
    # (dy drawn like x, N(0,1); d_final like the initial state, N(0, 0.1^2))
    "bwd_2p7b_2x1024": Workload("bwd_2p7b_2x1024", 2, 1024, 80, 64, 128, 1, 256, "bf16", True, "bwd"),
    # the complex-valued (ET) scan, N = 128 floats = 64 complex components per
    # row: many 64-token sequences with the state in and out, and one decode
    # step of 128 sequences of the 2.7B layer's heads
    "complex_many_short_seqs": Workload("complex_many_short_seqs", 256, 64, 48, 64, 128, 1, 1, "bf16", True,
                                        "complex"),
    "complex_decode_2p7b_128seq": Workload("complex_decode_2p7b_128seq", 128, 1, 80, 64, 128, 1, 1, "bf16", True,
                                           "complex"),
    # long complex sequences: 8 x 4096 tokens, 38 heads (152 pairs of batch rows and
    # heads, one per SM for the chunk form), the state in and out
    "complex_long_8x4096": Workload("complex_long_8x4096", 8, 4096, 38, 64, 128, 1, 1, "bf16", True, "complex"),
}

_TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}


def torch_dtype(dtype: str) -> torch.dtype:
    return _TORCH_DTYPE[dtype]


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Draw one seeded input set for workload ``w`` as CPU torch tensors.

    Keys: x, dt_raw, dt_bias, A_log, B, C, D, init_state (None when
    ``w.init_state`` is False).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    Bt, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    sd = _TORCH_DTYPE[w.dtype]

    def normal(shape, std=1.0):
        a = rng.standard_normal(size=shape, dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        return a

    x = torch.from_numpy(normal((Bt, L, H, P))).to(sd)
    dt_raw = torch.from_numpy(normal((Bt, L, H), 0.1))
    dt0 = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=H))
    dt_bias = torch.from_numpy(np.log(np.expm1(dt0)).astype(np.float32))
    A_log = torch.from_numpy(np.log(rng.uniform(1.0, 16.0, size=H)).astype(np.float32))
    Bm = torch.from_numpy(normal((Bt, L, G, N))).to(sd)
    Cm = torch.from_numpy(normal((Bt, L, G, N))).to(sd)
    D = torch.from_numpy(normal((H,)))
    init = torch.from_numpy(normal((Bt, H, P, N), 0.1)) if w.init_state else None
    return dict(x=x, dt_raw=dt_raw, dt_bias=dt_bias, A_log=A_log, B=Bm, C=Cm, D=D,
                init_state=init)


def make_trap_inputs(w: Workload, seed: int = 0) -> dict:
    """One seeded input set for the trapezoidal (Mamba-3 SISO) scan of
    workload ``w``, as CPU torch tensors.

    Keys (draw order): v [B,L,H,P] ~ N(0,1), k [B,L,G,N] ~ N(0,1),
    q [B,L,G,N] ~ N(0,1) (storage dtype); dt [B,L,H] = exp(U[ln 1e-3, ln 1e-1]),
    a [B,L,H] ~ -U[1, 16] (a per-token decay rate), trap [B,L,H] ~ U[0, 1]
    (a post-sigmoid mixing weight), D [H] ~ N(0,1) (fp32); when
    ``w.init_state``: h0 [B,H,P,N] ~ N(0, 0.1^2) fp32, k0 [B,H,N] and
    v0 [B,H,P] ~ N(0,1) in the storage dtype; else None.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    Bt, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    sd = _TORCH_DTYPE[w.dtype]

    def normal(shape, std=1.0):
        a = rng.standard_normal(size=shape, dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        return a

    v = torch.from_numpy(normal((Bt, L, H, P))).to(sd)
    k = torch.from_numpy(normal((Bt, L, G, N))).to(sd)
    q = torch.from_numpy(normal((Bt, L, G, N))).to(sd)
    dt = torch.from_numpy(np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=(Bt, L, H))).astype(np.float32))
    a = torch.from_numpy((-rng.uniform(1.0, 16.0, size=(Bt, L, H))).astype(np.float32))
    trap = torch.from_numpy(rng.uniform(0.0, 1.0, size=(Bt, L, H)).astype(np.float32))
    D = torch.from_numpy(normal((H,)))
    if w.init_state:
        h0 = torch.from_numpy(normal((Bt, H, P, N), 0.1))
        k0 = torch.from_numpy(normal((Bt, H, N))).to(sd)
        v0 = torch.from_numpy(normal((Bt, H, P))).to(sd)
    else:
        h0 = k0 = v0 = None
    return dict(v=v, k=k, q=q, dt=dt, a=a, trap=trap, D=D, h0=h0, k0=k0, v0=v0)


def make_complex_inputs(w: Workload, seed: int = 0) -> dict:
    """One seeded input set for the complex-valued (ET) scan of workload ``w``,
    as CPU torch tensors.

    Keys (draw order): x [B,L,H,P] ~ N(0,1); dt_raw [B,L,H] ~ N(0, 0.1^2);
    dt_bias [H] = log(expm1(dt0)), dt0 = exp(U[ln 1e-3, ln 1e-1]) (as the SSD
    inputs); A_polar [H,2] = (log U[1,16], U[0.6 pi, 1.4 pi]) (|A| as the SSD's
    decay rates, arg A with cos < 0 so every mode decays); B, C [B,L,G,N] ~
    N(0,1) (re and im parts alike); D [H] ~ N(0,1); when ``w.init_state``
    init_state [B,H,P,N] ~ N(0, 0.1^2) fp32, else None.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    Bt, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    sd = _TORCH_DTYPE[w.dtype]

    def normal(shape, std=1.0):
        a = rng.standard_normal(size=shape, dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        return a

    x = torch.from_numpy(normal((Bt, L, H, P))).to(sd)
    dt_raw = torch.from_numpy(normal((Bt, L, H), 0.1))
    dt0 = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=H))
    dt_bias = torch.from_numpy(np.log(np.expm1(dt0)).astype(np.float32))
    A_polar = torch.from_numpy(np.stack([np.log(rng.uniform(1.0, 16.0, size=H)),
                                         rng.uniform(0.6 * math.pi, 1.4 * math.pi, size=H)], 1).astype(np.float32))
    Bm = torch.from_numpy(normal((Bt, L, G, N))).to(sd)
    Cm = torch.from_numpy(normal((Bt, L, G, N))).to(sd)
    D = torch.from_numpy(normal((H,)))
    init_state = torch.from_numpy(normal((Bt, H, P, N), 0.1)) if w.init_state else None
    return dict(x=x, dt_raw=dt_raw, dt_bias=dt_bias, A_polar=A_polar, B=Bm, C=Cm, D=D, init_state=init_state)


def make_conv_inputs(w: Workload, K: int = 4, seed: int = 0) -> dict:
    """Seeded inputs of the causal conv1d + SiLU over the fused x | B | C
    channels (C = H*P + 2*G*N), as CPU torch tensors.

    Keys (draw order): xbc [B,L,C] ~ N(0,1) (storage dtype); weight [C,K] ~
    U[-0.5, 0.5], bias [C] ~ U[-0.5, 0.5] (fp32); conv_state [B,K-1,C] ~ N(0,1)
    (storage dtype) when ``w.init_state``, else None.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    sd = _TORCH_DTYPE[w.dtype]
    C = w.nheads * w.headdim + 2 * w.ngroups * w.dstate
    xbc = torch.from_numpy(rng.standard_normal(size=(w.batch, w.seqlen, C), dtype=np.float32)).to(sd)
    weight = torch.from_numpy(rng.uniform(-0.5, 0.5, size=(C, K)).astype(np.float32))
    bias = torch.from_numpy(rng.uniform(-0.5, 0.5, size=C).astype(np.float32))
    state = (torch.from_numpy(rng.standard_normal(size=(w.batch, K - 1, C), dtype=np.float32)).to(sd)
             if w.init_state else None)
    return dict(xbc=xbc, weight=weight, bias=bias, conv_state=state)


def make_gnorm_inputs(w: Workload, seed: int = 0) -> dict:
    """Seeded inputs of the gated RMSNorm over the H*P channels of a token.

    Keys (draw order): y, z [B,L,H,P] ~ N(0,1) (storage dtype); weight [H*P] ~
    1 + 0.1 N(0,1) (fp32).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    sd = _TORCH_DTYPE[w.dtype]
    shape = (w.batch, w.seqlen, w.nheads, w.headdim)
    y = torch.from_numpy(rng.standard_normal(size=shape, dtype=np.float32)).to(sd)
    z = torch.from_numpy(rng.standard_normal(size=shape, dtype=np.float32)).to(sd)
    weight = torch.from_numpy((1.0 + 0.1 * rng.standard_normal(size=w.nheads * w.headdim)).astype(np.float32))
    return dict(y=y, z=z, weight=weight)
