"""GPU parity of the decode step (seqlen 1) against the fp64 oracle.

The decode path applies the recurrence once to the carried state: decay, add
the input term, read out, add the skip.  The oracle is the same sequential
scan as for every other path, run for one step.  Tolerance: the whole-tensor
metric max|out - ref| / max|ref| of the scan tests (2e-2 bf16, 1e-4 fp32),
for y and for the updated state.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_04_gb300.inputs import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-4}


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
    return {k: (None if v is None else v.cuda().contiguous()) for k, v in inp.items()}


def _args(d, init=True):
    return (d["x"], d["dt_raw"], d["dt_bias"], d["A_log"], d["B"], d["C"], d["D"],
            d["init_state"] if init else None)


@pytest.mark.parametrize("batch,H,P,N,G,dtype,init", [
    (3, 4, 64, 128, 1, "bf16", True),
    (5, 6, 64, 128, 2, "bf16", False),
    (2, 4, 100, 64, 1, "f32", True),      # P not a multiple of a warp's 8 rows
    (2, 2, 8, 16, 1, "f32", True),        # N below one warp's 128 states
    (2, 4, 64, 256, 4, "bf16", True),     # two float4 per lane
    (1, 2, 32, 512, 1, "f32", True),      # four float4 per lane
    (1, 3, 17, 44, 1, "f32", False),      # ragged N (44 = 11 float4)
])
def test_decode_against_oracle(ssd, batch, H, P, N, G, dtype, init):
    w = Workload("t", batch, 1, H, P, N, G, 256, dtype, init)
    assert ssd.select_path((batch, 1, H, P), G, N, 256, dtype) == ssd.PATH_DECODE
    inp = make_inputs(w, seed=90 + N)
    ref_y, ref_f = oracle.ssd_fwd(**inp)
    d = _dev(inp)
    launches = ssd.launch_count()
    y, fin = ssd.ssd_scan_fwd(*_args(d, init), chunk=256)
    torch.cuda.synchronize()
    assert ssd.launch_count() == launches + 1
    ey, ef = relerr(y, ref_y), relerr(fin, ref_f)
    print(f"decode rel err y {ey:.3e} state {ef:.3e}")
    assert ey <= TOL[dtype] and ef <= TOL[dtype]


def test_decode_in_place_state(ssd):
    w = Workload("t", 4, 1, 8, 64, 128, 1, 256, "bf16", True)
    inp = make_inputs(w, seed=95)
    ref_y, ref_f = oracle.ssd_fwd(**inp)
    d = _dev(inp)
    state = d["init_state"].clone()
    y, fin = ssd.ssd_scan_fwd(*_args(d)[:7], state, final_state=state, chunk=256)
    torch.cuda.synchronize()
    assert fin.data_ptr() == state.data_ptr()
    assert relerr(y, ref_y) <= TOL["bf16"] and relerr(state, ref_f) <= TOL["bf16"]


def test_decode_matches_sequential_path(ssd):
    # the same fp32 recurrence on both paths; only the order of the readout sum differs
    w = Workload("t", 3, 1, 6, 64, 128, 3, 256, "f32", True)
    inp = make_inputs(w, seed=96)
    d = _dev(inp)
    y1, f1 = ssd.ssd_scan_fwd(*_args(d), chunk=256, path="decode")
    y2, f2 = ssd.ssd_scan_fwd(*_args(d), chunk=256, path="sequential")
    torch.cuda.synchronize()
    assert torch.equal(f1, f2)   # the state update is elementwise: same operations, same order
    assert float((y1 - y2).abs().max()) <= 1e-5 * float(y2.abs().max())


def test_decode_steps_equal_one_scan(ssd):
    # K decode steps with the state carried from step to step == one scan over K steps
    K = 6
    w = Workload("t", 2, K, 4, 64, 128, 1, 256, "f32", True)
    inp = make_inputs(w, seed=97)
    d = _dev(inp)
    y_scan, f_scan = ssd.ssd_scan_fwd(*_args(d), chunk=256, path="sequential")
    state = d["init_state"].clone()
    ys = []
    for t in range(K):
        sl = slice(t, t + 1)
        y, state = ssd.ssd_scan_fwd(d["x"][:, sl].contiguous(), d["dt_raw"][:, sl].contiguous(), d["dt_bias"],
                                    d["A_log"], d["B"][:, sl].contiguous(), d["C"][:, sl].contiguous(), d["D"],
                                    state, chunk=256)
        ys.append(y)
    torch.cuda.synchronize()
    y_steps = torch.cat(ys, dim=1)
    assert float((y_steps - y_scan).abs().max()) <= 1e-5 * float(y_scan.abs().max())
    assert float((state - f_scan).abs().max()) <= 1e-5 * float(f_scan.abs().max())


def test_decode_workload_full_size_sampled(ssd):
    # the benchmark's decode workload, checked on sampled (batch, head) pairs
    w = WORKLOADS["decode_2p7b_128seq"]
    inp = make_inputs(w, seed=0)
    d = _dev(inp)
    y, fin = ssd.ssd_scan_fwd(*_args(d), chunk=w.chunk)
    torch.cuda.synchronize()
    yc, fc = y.cpu(), fin.cpu()
    rng = np.random.default_rng(3)
    for _ in range(8):
        b, h = int(rng.integers(w.batch)), int(rng.integers(w.nheads))
        sl = dict(x=inp["x"][b:b + 1, :, h:h + 1], dt_raw=inp["dt_raw"][b:b + 1, :, h:h + 1],
                  dt_bias=inp["dt_bias"][h:h + 1], A_log=inp["A_log"][h:h + 1],
                  B=inp["B"][b:b + 1], C=inp["C"][b:b + 1], D=inp["D"][h:h + 1],
                  init_state=inp["init_state"][b:b + 1, h:h + 1])
        ry, rf = oracle.ssd_fwd(**sl)
        assert relerr(yc[b:b + 1, :, h:h + 1], ry) <= TOL["bf16"]
        assert relerr(fc[b:b + 1, h:h + 1], rf) <= TOL["bf16"]
