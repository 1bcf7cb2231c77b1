"""Failure detection on the GPU without a GPU fault.

With SSD_DIAG_STALL_HANDOFF the first unit of every chain waits for a state
handoff that nothing publishes; the wait is bounded (20 ms in this mode).  The
launch must record SSD_ERR_TIMEOUT in the device error word, stop every warp,
drain its own copies and MMAs and return, leaving the context usable: the next
call on the same stream must succeed and match the oracle.
"""
import time

import pytest
import torch

import oracle
from selective_state_space_04_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu

TIMEOUT = 6


@pytest.fixture(scope="module")
def ssd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_04_gb300 import build
    build.build()
    from selective_state_space_04_gb300 import ssd as mod
    return mod


def test_stalled_handoff_times_out_and_context_survives(ssd):
    w = Workload("t", 2, 1024, 8, 64, 128, 1, 256, "bf16", True)
    inp = make_inputs(w, seed=9)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    args = (d["x"], d["dt_raw"], d["dt_bias"], d["A_log"], d["B"], d["C"], d["D"], d["init_state"])
    assert ssd.device_error() == 0
    t0 = time.perf_counter()
    # the stalled wait is a chained hand-off between units: the ranges schedule
    assert ssd.chunk_schedule((w.batch, w.seqlen, w.nheads, w.headdim), w.ngroups, w.dstate, w.chunk,
                              schedule="ranges") == "ranges"
    ssd.ssd_scan_fwd(*args, chunk=w.chunk, path="chunked", diag_stall_handoff=True, schedule="ranges")
    code = ssd.device_error()          # synchronises the stream, reads and clears the word
    elapsed = time.perf_counter() - t0
    assert code == TIMEOUT
    assert elapsed < 5.0
    # the context is still usable and the error word was cleared
    y, fin = ssd.ssd_scan_fwd(*args, chunk=w.chunk, path="chunked")
    torch.cuda.synchronize()
    assert ssd.device_error() == 0
    ref_y, ref_f = oracle.ssd_fwd(**inp)
    err = float((y.double().cpu() - torch.from_numpy(ref_y)).abs().max()) / float(abs(ref_y).max())
    assert err <= 2e-2
