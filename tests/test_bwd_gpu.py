"""GPU parity of the SSD backward (ssd_scan_bwd), both paths (the chunk-
parallel kernels and the sequential kernel), against the fp64 backward oracle,
which is itself pinned by finite differences of the forward oracle.

Metric: max|g - g_ref| / max|g_ref| per gradient tensor.  The fp32 forms
(the chunk form's fp32 contractions, the sequential kernel) compute in fp32
from inputs that are exact in both dtypes, so the forward's fp32 bar serves
for both: 1e-4.  The chunk form's tensor-core gradient pass (bf16 inputs,
P = 64, N = 128) takes bf16 operands of the masked decay products and of the
chunk states, so its bar is the forward's bf16 bar: 2e-2.
"""
import numpy as np
import pytest
import torch

from oracle.backward import ssd_bwd
from selective_state_space_04_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu

TOL = 1e-4
TOL_TC = 2e-2


def _tol(dtype, P, N, path="auto", fp32_form=False):
    tc = dtype == "bf16" and P == 64 and N == 128 and path in ("auto", "chunked") and not fp32_form
    return TOL_TC if tc else TOL
NAMES = ("dx", "ddt_raw", "ddt_bias", "dA_log", "dB", "dC", "dD", "d_init")


@pytest.fixture(scope="module")
def ssd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_04_gb300 import build
    build.build()
    from selective_state_space_04_gb300 import ssd as mod
    return mod


def _grads_in(w, seed):
    inp = make_inputs(w, seed=seed)
    rng = np.random.default_rng(seed + 1)
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dy = torch.from_numpy(rng.standard_normal((w.batch, w.seqlen, w.nheads, w.headdim)).astype(np.float32)).to(td)
    dfin = torch.from_numpy(rng.standard_normal((w.batch, w.nheads, w.headdim, w.dstate)).astype(np.float32))
    return inp, dy, dfin


def _run(ssd, inp, dy, dfin, path="auto", fp32_form=False, split_states=False):
    d = {k: (None if v is None else v.cuda().contiguous()) for k, v in inp.items()}
    out = ssd.ssd_scan_bwd(d["x"], d["dt_raw"], d["dt_bias"], d["A_log"], d["B"], d["C"], d["D"], d["init_state"],
                           dy.cuda(), None if dfin is None else dfin.cuda(), path=path, fp32_form=fp32_form,
                           split_states=split_states)
    torch.cuda.synchronize()
    return out


def _check(out, ref, names=NAMES, tol=TOL):
    for k in names:
        r = ref[k]
        err = float(np.max(np.abs(out[k].double().cpu().numpy() - r)) / max(np.max(np.abs(r)), 1e-30))
        print(f"{k}: rel err {err:.2e}")
        assert err <= tol, f"{k}: rel err {err:.2e}"


CASES = [
    (2, 100, 4, 64, 128, 1, "f32", True, True),     # two chunks / checkpoint segments, ragged tail
    (2, 70, 4, 64, 128, 2, "bf16", True, False),
    (1, 130, 3, 17, 44, 1, "f32", False, True),     # ragged P, N; three chunks
    (1, 1, 2, 8, 16, 1, "f32", True, True),         # one step
    (3, 64, 8, 32, 64, 4, "bf16", False, False),    # exactly one chunk
    (2, 300, 6, 64, 128, 3, "bf16", True, True),    # five chunks, the last of 44 steps
    (1, 257, 2, 64, 128, 1, "f32", True, True),     # one step past four full chunks
]


@pytest.mark.parametrize("path", ["chunked", "sequential"])
@pytest.mark.parametrize("B,L,H,P,N,G,dtype,init,dfinal", CASES)
def test_backward_against_oracle(ssd, path, B, L, H, P, N, G, dtype, init, dfinal):
    w = Workload("t", B, L, H, P, N, G, 16, dtype, init)
    inp, dy, dfin = _grads_in(w, seed=210 + L)
    dfin = dfin if dfinal else None
    ref = ssd_bwd(**inp, dy=dy, d_final=dfin)
    _check(_run(ssd, inp, dy, dfin, path), ref, tol=_tol(dtype, P, N, path))


@pytest.mark.parametrize("B,L,H,G,init,dfinal", [
    (2, 70, 4, 2, True, False),      # one pair of chunks, the second of 6 steps
    (2, 300, 6, 3, True, True),      # five chunks: the last pair holds one
    (1, 128, 2, 1, False, False),    # exactly one pair, no carried states
    (1, 1000, 4, 1, True, True),     # 16 chunks, ragged tail
    (3, 64, 2, 2, True, True),       # one chunk
])
def test_backward_tensor_core_pass_against_oracle(ssd, B, L, H, G, init, dfinal):
    # the tensor-core form (bf16, P = 64, N = 128) at the bf16 bar -- its chunk states
    # as the library picks them (one walk per (b, h) up to 8 chunks here) and as two
    # launches -- and the fp32 form of the same call at the fp32 bar
    w = Workload("t", B, L, H, 64, 128, G, 16, "bf16", init)
    inp, dy, dfin = _grads_in(w, seed=260 + L + H)
    dfin = dfin if dfinal else None
    ref = ssd_bwd(**inp, dy=dy, d_final=dfin)
    _check(_run(ssd, inp, dy, dfin, "chunked"), ref, tol=TOL_TC)
    _check(_run(ssd, inp, dy, dfin, "chunked", split_states=True), ref, tol=TOL_TC)
    _check(_run(ssd, inp, dy, dfin, "chunked", fp32_form=True), ref, tol=TOL)


def test_backward_strong_decay(ssd):
    # large dt and |a|: per-step decays down to about e^-7, chunk decays to about e^-110
    w = Workload("t", 1, 200, 4, 64, 128, 1, 16, "f32", True)
    inp, dy, dfin = _grads_in(w, seed=230)
    inp["dt_raw"] = inp["dt_raw"] + 1.5
    inp["A_log"] = torch.log(torch.tensor([0.5, 2.0, 8.0, 16.0]))
    ref = ssd_bwd(**inp, dy=dy, d_final=dfin)
    for path in ("chunked", "sequential"):
        _check(_run(ssd, inp, dy, dfin, path), ref)


def test_auto_takes_the_chunked_path_up_to_p64(ssd):
    w = Workload("t", 2, 150, 4, 64, 128, 2, 16, "bf16", True)
    inp, dy, dfin = _grads_in(w, seed=240)
    a, c = _run(ssd, inp, dy, dfin, "auto"), _run(ssd, inp, dy, dfin, "chunked")
    for k in NAMES:
        assert torch.equal(a[k], c[k]), k
    # strong decay through the tensor-core pass (bf16): per-step decays to about e^-7
    w = Workload("t", 1, 300, 4, 64, 128, 1, 16, "bf16", True)
    inp, dy, dfin = _grads_in(w, seed=242)
    inp["dt_raw"] = inp["dt_raw"] + 1.5
    inp["A_log"] = torch.log(torch.tensor([0.5, 2.0, 8.0, 16.0]))
    _check(_run(ssd, inp, dy, dfin, "chunked"), ssd_bwd(**inp, dy=dy, d_final=dfin), tol=TOL_TC)
    # P = 96 is past the chunked kernels: auto takes the sequential kernel, chunked is refused
    w = Workload("t", 1, 70, 2, 96, 64, 1, 16, "f32", True)
    inp, dy, dfin = _grads_in(w, seed=241)
    _check(_run(ssd, inp, dy, dfin, "auto"), ssd_bwd(**inp, dy=dy, d_final=dfin))
    with pytest.raises(RuntimeError):
        _run(ssd, inp, dy, dfin, "chunked")


@pytest.mark.parametrize("path", ["chunked", "sequential"])
def test_backward_is_deterministic(ssd, path):
    w = Workload("t", 2, 150, 8, 64, 128, 2, 16, "bf16", True)
    inp, dy, dfin = _grads_in(w, seed=220)
    o1 = _run(ssd, inp, dy, dfin, path)
    o2 = _run(ssd, inp, dy, dfin, path)
    for k in NAMES:
        assert torch.equal(o1[k], o2[k]), k


def test_backward_full_size_sampled_heads(ssd):
    # the bench's workload (2 x 1024 steps, 80 heads, P 64, N 128, bf16, one group) in one call;
    # the oracle takes two sampled heads, whose per-head gradients do not depend on the others.
    # dB and dC sum over all heads of the group: they are checked by a call on the two heads alone.
    from selective_state_space_04_gb300.inputs import WORKLOADS
    w = WORKLOADS["bwd_2p7b_2x1024"]
    inp, dy, dfin = _grads_in(w, seed=250)
    out = _run(ssd, inp, dy, dfin)
    heads = [7, 61]
    sub = {k: (None if v is None else v) for k, v in inp.items()}
    for k in ("x", "dt_raw"):
        sub[k] = inp[k][:, :, heads].contiguous()
    for k in ("dt_bias", "A_log", "D"):
        sub[k] = inp[k][heads].contiguous()
    if inp["init_state"] is not None:
        sub["init_state"] = inp["init_state"][:, heads].contiguous()
    dy_s, dfin_s = dy[:, :, heads].contiguous(), dfin[:, heads].contiguous()
    ref = ssd_bwd(**sub, dy=dy_s, d_final=dfin_s)
    sliced = dict(dx=out["dx"][:, :, heads], ddt_raw=out["ddt_raw"][:, :, heads], ddt_bias=out["ddt_bias"][heads],
                  dA_log=out["dA_log"][heads], dD=out["dD"][heads], d_init=out["d_init"][:, heads])
    _check(sliced, ref, names=tuple(sliced), tol=TOL_TC)
    _check(_run(ssd, sub, dy_s, dfin_s), ref, names=("dB", "dC"), tol=TOL_TC)


def test_backward_state_walk_matches_the_two_launch_states(ssd):
    # 2 x 1000 steps (16 chunks, ragged tail), 80 heads: the library walks each (b, h)
    # through its chunks in one launch; forced into two launches, the chunk states
    # differ only in the order of fp32 additions, so every gradient agrees far below
    # the bf16 bar.  Both forms are bitwise repeatable.
    w = Workload("t", 2, 1000, 80, 64, 128, 1, 16, "bf16", True)
    inp, dy, dfin = _grads_in(w, seed=271)
    walk = _run(ssd, inp, dy, dfin)
    split = _run(ssd, inp, dy, dfin, split_states=True)
    for k in NAMES:
        a, b = walk[k].double(), split[k].double()
        err = float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))
        print(f"{k}: walk vs two launches {err:.2e}")
        assert err <= 1e-4, k
    again = _run(ssd, inp, dy, dfin)
    for k in NAMES:
        assert torch.equal(walk[k], again[k]), k
