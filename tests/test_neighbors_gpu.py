"""GPU parity of the conv1d + SiLU prologue and the gated RMSNorm epilogue
against their fp64 oracle.  Metric: max|out - ref| / max|ref| over the whole
tensor; 1e-5 for fp32, 2e-2 for bf16.  The carried conv state is a copy of
inputs and must match exactly.
"""
import numpy as np
import pytest
import torch

from oracle.neighbors import conv1d_silu, gated_rmsnorm
from selective_state_space_04_gb300.inputs import WORKLOADS, Workload, make_conv_inputs, make_gnorm_inputs

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-5}


@pytest.fixture(scope="module")
def ssd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_04_gb300 import build
    build.build()
    from selective_state_space_04_gb300 import ssd as mod
    return mod


def relerr(a, ref):
    a = a.double().cpu().numpy()
    return float(np.max(np.abs(a - ref)) / max(np.max(np.abs(ref)), 1e-30))


def _dev(inp):
    return {n: (None if t is None else t.cuda().contiguous()) for n, t in inp.items()}


@pytest.mark.parametrize("B,L,H,P,N,G,dtype,init,K", [
    (2, 100, 4, 64, 128, 1, "bf16", True, 4),   # ragged against the 64-step tile
    (1, 130, 2, 8, 16, 1, "f32", False, 4),
    (3, 5, 2, 16, 8, 2, "f32", True, 3),
    (2, 2, 2, 8, 8, 1, "f32", True, 4),         # fewer steps than the window
    (1, 64, 2, 32, 16, 1, "bf16", True, 2),
])
def test_conv1d_silu_against_oracle(ssd, B, L, H, P, N, G, dtype, init, K):
    w = Workload("t", B, L, H, P, N, G, 1, dtype, init)
    inp = make_conv_inputs(w, K=K, seed=170 + L)
    rx, rB, rC, rs = conv1d_silu(**inp, H=H, P=P, G=G, N=N)
    d = _dev(inp)
    x, Bm, Cm, st = ssd.conv1d_silu_fwd(d["xbc"], d["weight"], d["bias"], d["conv_state"], nheads=H,
                                        headdim=P, ngroups=G, dstate=N)
    torch.cuda.synchronize()
    for got, ref in ((x, rx), (Bm, rB), (Cm, rC)):
        assert relerr(got, ref) <= TOL[dtype]
    assert np.array_equal(st.double().cpu().numpy(), rs)


def test_conv1d_silu_split_and_resume_bitwise(ssd):
    w = Workload("t", 2, 300, 4, 64, 128, 1, 1, "bf16", True)
    d = _dev(make_conv_inputs(w, K=4, seed=180))
    kw = dict(nheads=4, headdim=64, ngroups=1, dstate=128)
    x, Bm, Cm, st = ssd.conv1d_silu_fwd(d["xbc"], d["weight"], d["bias"], d["conv_state"], **kw)
    cut = 77
    x1, B1, C1, s1 = ssd.conv1d_silu_fwd(d["xbc"][:, :cut].contiguous(), d["weight"], d["bias"], d["conv_state"], **kw)
    x2, B2, C2, s2 = ssd.conv1d_silu_fwd(d["xbc"][:, cut:].contiguous(), d["weight"], d["bias"], s1, **kw)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([x1, x2], 1), x) and torch.equal(torch.cat([B1, B2], 1), Bm)
    assert torch.equal(torch.cat([C1, C2], 1), Cm) and torch.equal(s2, st)


@pytest.mark.parametrize("B,L,H,P,dtype", [(2, 64, 80, 64, "bf16"), (1, 7, 3, 8, "f32"), (3, 5, 24, 64, "f32")])
def test_gated_rmsnorm_against_oracle(ssd, B, L, H, P, dtype):
    w = Workload("t", B, L, H, P, 1, 1, 1, dtype, False)
    inp = make_gnorm_inputs(w, seed=190 + H)
    ref = gated_rmsnorm(**inp, eps=1e-6)
    d = _dev(inp)
    out = ssd.gated_rmsnorm_fwd(d["y"], d["z"], d["weight"], 1e-6)
    torch.cuda.synchronize()
    assert relerr(out, ref) <= TOL[dtype]


def test_conv_scan_norm_chain(ssd):
    # the three steps of a block's SSM part in sequence, against the oracles in sequence
    import oracle
    w = Workload("t", 2, 300, 4, 64, 128, 1, 256, "bf16", True)
    ci = make_conv_inputs(w, K=4, seed=200)
    rng = np.random.default_rng(201)
    dt_raw = torch.from_numpy((0.1 * rng.standard_normal((2, 300, 4))).astype(np.float32))
    dt_bias = torch.from_numpy(np.log(np.expm1(np.full(4, 0.01))).astype(np.float32))
    A_log = torch.from_numpy(np.log(np.full(4, 2.0)).astype(np.float32))
    D = torch.from_numpy(rng.standard_normal(4).astype(np.float32))
    gi = make_gnorm_inputs(w, seed=202)
    rx, rB, rC, _ = conv1d_silu(**ci, H=4, P=64, G=1, N=128)
    # the oracle chain starts from the GPU's bf16 conv outputs, as the GPU chain does
    d = _dev(ci)
    x, Bm, Cm, _ = ssd.conv1d_silu_fwd(d["xbc"], d["weight"], d["bias"], d["conv_state"], nheads=4, headdim=64,
                                       ngroups=1, dstate=128)
    y, _ = ssd.ssd_scan_fwd(x, dt_raw.cuda(), dt_bias.cuda(), A_log.cuda(), Bm, Cm, D.cuda(), chunk=256)
    out = ssd.gated_rmsnorm_fwd(y, gi["z"].cuda(), gi["weight"].cuda(), 1e-6)
    torch.cuda.synchronize()
    assert relerr(x, rx) <= TOL["bf16"]
    ry, _ = oracle.ssd_fwd(x.cpu(), dt_raw, dt_bias, A_log, Bm.cpu(), Cm.cpu(), D)
    ref = gated_rmsnorm(torch.from_numpy(ry).to(torch.bfloat16), gi["z"], gi["weight"], eps=1e-6)
    assert relerr(out, ref) <= TOL["bf16"]


def test_bench_workloads_sampled(ssd):
    # the bench's full conv and norm workloads in one call each; the oracle takes
    # the first two batch rows (rows and tokens run independently)
    w = WORKLOADS["conv_silu_2p7b"]
    inp = make_conv_inputs(w, K=4, seed=0)
    d = _dev(inp)
    x, Bm, Cm, st = ssd.conv1d_silu_fwd(d["xbc"], d["weight"], d["bias"], d["conv_state"], nheads=w.nheads,
                                        headdim=w.headdim, ngroups=w.ngroups, dstate=w.dstate)
    torch.cuda.synchronize()
    sub = dict(inp, xbc=inp["xbc"][:2], conv_state=None if inp["conv_state"] is None else inp["conv_state"][:2])
    rx, rB, rC, rs = conv1d_silu(**sub, H=w.nheads, P=w.headdim, G=w.ngroups, N=w.dstate)
    for got, ref in ((x, rx), (Bm, rB), (Cm, rC)):
        assert relerr(got[:2], ref) <= TOL["bf16"]
    assert np.array_equal(st[:2].double().cpu().numpy(), rs)
    w = WORKLOADS["gnorm_2p7b"]
    gi = make_gnorm_inputs(w, seed=0)
    out = ssd.gated_rmsnorm_fwd(gi["y"].cuda(), gi["z"].cuda(), gi["weight"].cuda(), 1e-6)
    torch.cuda.synchronize()
    ref = gated_rmsnorm(gi["y"][:2], gi["z"][:2], gi["weight"], eps=1e-6)
    assert relerr(out[:2], ref) <= TOL["bf16"]
