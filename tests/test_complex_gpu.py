"""GPU parity of the complex-valued (ET) scan (ssd_complex_scan_fwd) against
its fp64 oracle, which the CPU tests pin to an ODE solution of the continuous
system, the unrolled product form and the real SSD oracle.  Both paths: the
sequential kernel and, for bf16 with P = 64 and N = 128, the chunk form on the
tensor cores (two batch rows per CTA, chunks of 64 steps).

Metric: max|out - ref| / max|ref| over the whole tensor, y and the final state
separately; 1e-4 for fp32 inputs, 2e-2 for bf16 (the forward's bounds).
"""
import numpy as np
import pytest
import torch

from oracle.complex_scan import complex_fwd
from selective_state_space_04_gb300.inputs import WORKLOADS, Workload, make_complex_inputs

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


def run(ssd, inp, init=None, **kw):
    d = {k: (None if v is None else v.cuda().contiguous()) for k, v in inp.items()}
    y, f = ssd.complex_scan_fwd(d["x"], d["dt_raw"], d["dt_bias"], d["A_polar"], d["B"], d["C"], d["D"],
                                d["init_state"] if init is None else init, **kw)
    torch.cuda.synchronize()
    return y, f


@pytest.mark.parametrize("B,L,H,P,N,G,dtype,init", [
    (2, 100, 4, 64, 128, 1, "f32", True),     # two time blocks, the second ragged
    (2, 70, 4, 64, 128, 2, "bf16", True),     # chunk form: two chunks, the second of 6 steps
    (1, 130, 3, 17, 44, 1, "f32", False),     # ragged P, N (11 complex components)
    (1, 1, 2, 8, 16, 1, "f32", True),         # one step: a decode step
    (3, 64, 8, 32, 256, 4, "bf16", False),    # two float4 of state per lane
    (1, 40, 2, 32, 512, 1, "f32", True),      # four float4 per lane; smaller time blocks
    (1, 20, 2, 128, 128, 1, "f32", True),     # the largest headdim: 16 warps of 8 rows
    (2, 1, 3, 64, 256, 1, "bf16", True),      # decode kernel, two float4 per lane
    (1, 1, 2, 32, 512, 2, "f32", True),       # decode kernel, four float4 per lane
])
def test_complex_scan_against_oracle(ssd, B, L, H, P, N, G, dtype, init):
    w = Workload("t", B, L, H, P, N, G, 1, dtype, init, "complex")
    inp = make_complex_inputs(w, seed=300 + L)
    ry, rf = complex_fwd(**inp)
    y, f = run(ssd, inp)
    ey, ef = relerr(y, ry), relerr(f, rf)
    print(f"y {ey:.2e} final {ef:.2e}")
    assert ey <= TOL[dtype] and ef <= TOL[dtype]


@pytest.mark.parametrize("path", ["chunked", "sequential"])
@pytest.mark.parametrize("B,L,H,G,init", [
    (3, 64, 4, 1, True),      # one chunk; an odd batch: the last CTA holds one row
    (1, 300, 2, 1, False),    # five chunks, the last of 44 steps; one row, no state in
    (2, 2, 3, 3, True),       # two steps
    (4, 200, 6, 2, True),     # four chunks, two CTAs per head
])
def test_complex_chunk_form_against_oracle(ssd, path, B, L, H, G, init):
    w = Workload("t", B, L, H, 64, 128, G, 1, "bf16", init, "complex")
    inp = make_complex_inputs(w, seed=320 + L + B)
    ry, rf = complex_fwd(**inp)
    y, f = run(ssd, inp, path=path)
    ey, ef = relerr(y, ry), relerr(f, rf)
    print(f"{path}: y {ey:.2e} final {ef:.2e}")
    assert ey <= TOL["bf16"] and ef <= TOL["bf16"]


@pytest.mark.parametrize("path,cut", [("sequential", 77), ("chunked", 64)])
def test_split_resume_and_in_place_state_are_bitwise(ssd, path, cut):
    # the sequential kernel resumes bitwise at any step; the chunk form at a chunk
    # boundary (its chunks then start at the same steps, and the state passes in fp32)
    w = Workload("t", 2, 150, 4, 64, 128, 1, 1, "bf16", True, "complex")
    inp = make_complex_inputs(w, seed=310)
    y, f = run(ssd, inp, path=path)
    first = {k: (v[:, :cut].contiguous() if k in ("x", "dt_raw", "B", "C") else v) for k, v in inp.items()}
    second = {k: (v[:, cut:].contiguous() if k in ("x", "dt_raw", "B", "C") else v) for k, v in inp.items()}
    y1, f1 = run(ssd, first, path=path)
    state = f1.clone()
    y2, _ = run(ssd, second, init=state, final_state=state, path=path)   # the state updated in place
    assert torch.equal(torch.cat([y1, y2], 1), y) and torch.equal(state, f)


def test_chunk_form_matches_the_sequential_kernel(ssd):
    # the two evaluations of the same recurrence agree far below the bf16 bar that
    # both meet against the oracle (bf16 operands in the chunk form)
    w = Workload("t", 4, 256, 8, 64, 128, 2, 1, "bf16", True, "complex")
    inp = make_complex_inputs(w, seed=330)
    yc, fc = run(ssd, inp, path="chunked")
    ys, fs = run(ssd, inp, path="sequential")
    assert relerr(yc, ys.double().cpu().numpy()) <= TOL["bf16"]
    assert relerr(fc, fs.double().cpu().numpy()) <= TOL["bf16"]


def test_no_steps_passes_the_state_through(ssd):
    w = Workload("t", 2, 0, 3, 8, 16, 1, 1, "f32", True, "complex")
    inp = make_complex_inputs(w, seed=311)
    _, f = run(ssd, inp)
    assert torch.equal(f.cpu(), inp["init_state"])


@pytest.mark.parametrize("name,rows", [("complex_many_short_seqs", 6), ("complex_decode_2p7b_128seq", 128)])
def test_bench_workloads_sampled(ssd, name, rows):
    # the bench's full workload in one call; the oracle takes the first `rows`
    # batch rows (every (b, h) runs independently of the others)
    w = WORKLOADS[name]
    inp = make_complex_inputs(w, seed=0)
    y, f = run(ssd, inp)
    sub = {k: (v[:rows] if k in ("x", "dt_raw", "B", "C", "init_state") and v is not None else v)
           for k, v in inp.items()}
    ry, rf = complex_fwd(**sub)
    assert relerr(y[:rows], ry) <= TOL[w.dtype] and relerr(f[:rows], rf) <= TOL[w.dtype]
