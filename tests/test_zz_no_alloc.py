"""GPU check of ssd_scan_fwd_noalloc, the allocation-free variant of the
chunked path that keeps its scratch in a fixed module-scope array.

Two consecutive calls (the second finds the first call's flags and handoff
states still in the array) must match ssd_scan_fwd, which takes its scratch
from a pool, exactly: both run the same kernel with the same schedule.  The
batch 4 x 80 heads x 2048 steps case hands states between units of a chain,
so the handoff states in the array are used.  With 640 chains the range
schedule would need more scratch than the array's 32 MiB; the call takes the
piece schedule instead (one state slot per SM), which gives the same result
bit for bit: both evaluate each chain's sub-chunks by the same arithmetic.
"""
import pytest
import torch

from selective_state_space_04_gb300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

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
    return {k: (None if v is None else v.cuda().contiguous()) for k, v in inp.items()}


def _args(d):
    return (d["x"], d["dt_raw"], d["dt_bias"], d["A_log"], d["B"], d["C"], d["D"], d["init_state"])


def test_two_consecutive_calls_match_pool_path(ssd):
    for seed, init in ((11, False), (12, True)):
        d = _dev(seed, init)
        y_ref, f_ref = ssd.ssd_scan_fwd(*_args(d), chunk=256)
        y_na, f_na = ssd.ssd_scan_fwd_noalloc(*_args(d), chunk=256)
        torch.cuda.synchronize()
        assert ssd.device_error() == 0
        assert torch.isfinite(y_na.float()).all()
        assert torch.equal(y_na, y_ref), f"seed {seed}: y differs"
        assert torch.equal(f_na, f_ref), f"seed {seed}: final state differs"


def test_many_chains_fit_the_array(ssd):
    # batch 16 x 80 heads x 4096 steps: 640 head-pair chains
    w = WORKLOADS["mamba2_2p7b_layer"].with_(batch=16)
    shape = (w.batch, w.seqlen, w.nheads, w.headdim)
    assert ssd.chunk_schedule(shape, w.ngroups, w.dstate, w.chunk) == "ranges"
    assert ssd.workspace_size(shape, w.ngroups, w.dstate, w.chunk) > 32 << 20
    assert ssd.workspace_size(shape, w.ngroups, w.dstate, w.chunk, schedule="pieces") <= 32 << 20
    inp = make_inputs(w, 13)
    d = {k: (None if v is None else v.cuda().contiguous()) for k, v in inp.items()}
    y_ref, f_ref = ssd.ssd_scan_fwd(*_args(d), chunk=w.chunk)
    y_na, f_na = ssd.ssd_scan_fwd_noalloc(*_args(d), chunk=w.chunk)
    torch.cuda.synchronize()
    assert ssd.device_error() == 0
    assert torch.equal(y_na, y_ref)
    assert torch.equal(f_na, f_ref)


def test_over_the_limit_is_refused_and_launches_nothing(ssd):
    # batch 16 x 80 heads x 4096 steps on an explicit range-schedule request
    # needs more scratch than the array holds: SSD_ERR_SCRATCH_LIMIT, with no
    # launch and nothing enqueued (the output buffer keeps its contents)
    w = WORKLOADS["mamba2_2p7b_layer"].with_(batch=16)
    inp = make_inputs(w, 14)
    d = {k: (None if v is None else v.cuda().contiguous()) for k, v in inp.items()}
    y = torch.full_like(d["x"], 7.0)
    torch.cuda.synchronize()
    before = ssd.launch_count()
    with pytest.raises(ssd.SsdError) as e:
        ssd.ssd_scan_fwd_noalloc(*_args(d), chunk=w.chunk, schedule="ranges", y=y)
    assert e.value.status == 8
    torch.cuda.synchronize()
    assert ssd.launch_count() == before
    assert bool((y == 7.0).all())
    # a request for another path is refused the same way, before any launch
    with pytest.raises(ssd.SsdError) as e:
        ssd.ssd_scan_fwd_noalloc(*_args(d), chunk=w.chunk, path="sequential", y=y)
    assert e.value.status == 4
    assert ssd.launch_count() == before
