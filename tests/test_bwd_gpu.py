"""GPU parity of the SSD backward (ssd_scan_bwd) against the fp64 backward
oracle, which is itself pinned by finite differences of the forward oracle.

Metric: max|g - g_ref| / max|g_ref| per gradient tensor.  The backward's
arithmetic is fp32 for bf16 and fp32 inputs alike (the inputs are exact in
both), so one bound serves: 2e-4 (sums over up to a few thousand terms).
"""
import numpy as np
import pytest
import torch

from oracle.backward import ssd_bwd
from selective_state_space_04_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-4
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


def _run(ssd, inp, dy, dfin):
    d = {k: (None if v is None else v.cuda().contiguous()) for k, v in inp.items()}
    out = ssd.ssd_scan_bwd(d["x"], d["dt_raw"], d["dt_bias"], d["A_log"], d["B"], d["C"], d["D"], d["init_state"],
                           dy.cuda(), None if dfin is None else dfin.cuda())
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("B,L,H,P,N,G,dtype,init,dfinal", [
    (2, 100, 4, 64, 128, 1, "f32", True, True),     # two checkpoint segments
    (2, 70, 4, 64, 128, 2, "bf16", True, False),
    (1, 130, 3, 17, 44, 1, "f32", False, True),     # ragged P, N; three segments
    (1, 1, 2, 8, 16, 1, "f32", True, True),         # one step
    (3, 64, 8, 32, 64, 4, "bf16", False, False),    # exactly one segment
])
def test_backward_against_oracle(ssd, B, L, H, P, N, G, dtype, init, dfinal):
    w = Workload("t", B, L, H, P, N, G, 16, dtype, init)
    inp, dy, dfin = _grads_in(w, seed=210 + L)
    dfin = dfin if dfinal else None
    ref = ssd_bwd(**inp, dy=dy, d_final=dfin)
    out = _run(ssd, inp, dy, dfin)
    for k in NAMES:
        r = ref[k]
        err = float(np.max(np.abs(out[k].double().cpu().numpy() - r)) / max(np.max(np.abs(r)), 1e-30))
        print(f"{k}: rel err {err:.2e}")
        assert err <= TOL, f"{k}: rel err {err:.2e}"


def test_backward_is_deterministic(ssd):
    w = Workload("t", 2, 150, 8, 64, 128, 2, 16, "bf16", True)
    inp, dy, dfin = _grads_in(w, seed=220)
    o1 = _run(ssd, inp, dy, dfin)
    o2 = _run(ssd, inp, dy, dfin)
    for k in NAMES:
        assert torch.equal(o1[k], o2[k]), k
