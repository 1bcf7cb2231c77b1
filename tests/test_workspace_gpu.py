"""GPU checks of ssd_scan_fwd_ws, the entry point with caller-provided scratch.

With a workspace of ssd_scan_fwd_workspace_size bytes it must equal
ssd_scan_fwd (pool scratch) bitwise, on a shape whose chains are split into
several units (so the handoff states in the workspace are used), twice in a
row on the same workspace.  One byte less is rejected before any launch.
"""
import pytest
import torch

from selective_state_space_04_gb300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 8


@pytest.fixture(scope="module")
def ssd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_04_gb300 import build
    build.build()
    from selective_state_space_04_gb300 import ssd as mod
    return mod


def _dev(seed, init):
    w = WORKLOADS["mamba2_2p7b_layer"].with_(batch=4, seqlen=2048, init_state=init)
    inp = make_inputs(w, seed)
    return w, {k: (None if v is None else v.cuda().contiguous()) for k, v in inp.items()}


def _args(d):
    return (d["x"], d["dt_raw"], d["dt_bias"], d["A_log"], d["B"], d["C"], d["D"], d["init_state"])


def test_workspace_path_matches_pool_path(ssd):
    w, _ = _dev(0, False)
    n = ssd.workspace_size((w.batch, w.seqlen, w.nheads, w.headdim), w.ngroups, w.dstate, w.chunk)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    for seed, init in ((21, False), (22, True)):
        _, d = _dev(seed, init)
        y_ref, f_ref = ssd.ssd_scan_fwd(*_args(d), chunk=w.chunk)
        y_ws, f_ws = ssd.ssd_scan_fwd_ws(*_args(d), workspace=ws, chunk=w.chunk)
        torch.cuda.synchronize()
        assert ssd.device_error() == 0
        assert torch.equal(y_ws, y_ref)
        assert torch.equal(f_ws, f_ref)


def test_too_small_workspace_rejected(ssd):
    w, d = _dev(0, False)
    n = ssd.workspace_size((w.batch, w.seqlen, w.nheads, w.headdim), w.ngroups, w.dstate, w.chunk)
    ws = torch.empty(n - 16, dtype=torch.uint8, device="cuda")
    before = ssd.launch_count()
    with pytest.raises(ssd.SsdError) as e:
        ssd.ssd_scan_fwd_ws(*_args(d), workspace=ws, chunk=w.chunk)
    assert e.value.status == SCRATCH_LIMIT
    assert ssd.launch_count() == before


def test_sequential_path_needs_no_workspace(ssd):
    w = WORKLOADS["tiny_fp32"]
    d = {k: (None if v is None else v.cuda()) for k, v in make_inputs(w, 3).items()}
    assert ssd.workspace_size((w.batch, w.seqlen, w.nheads, w.headdim), w.ngroups, w.dstate, w.chunk,
                              dtype="f32") == 0
    y_ref, f_ref = ssd.ssd_scan_fwd(*_args(d), chunk=w.chunk)
    y_ws, f_ws = ssd.ssd_scan_fwd_ws(*_args(d), workspace=None, chunk=w.chunk)
    torch.cuda.synchronize()
    assert torch.equal(y_ws, y_ref) and torch.equal(f_ws, f_ref)
