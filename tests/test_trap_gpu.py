"""GPU parity of the trapezoidal (Mamba-3 SISO) scan against its fp64 oracle.

Metric as for the SSD scan: max|out - ref| / max|ref| over the whole tensor,
for y and for the updated state; 1e-4 for fp32, 2e-2 for bf16.  The carried
k and v states are copies of inputs and must match exactly.
"""
import numpy as np
import pytest
import torch

from oracle.trap import trap_fwd
from selective_state_space_04_gb300.inputs import WORKLOADS, Workload, make_trap_inputs

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-4}
KEYS = ("v", "k", "q", "dt", "a", "trap", "D", "h0", "k0", "v0")


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
    return {n: (None if inp[n] is None else inp[n].cuda().contiguous()) for n in KEYS}


def _run(ssd, d, path="sequential"):
    out = ssd.ssd_trap_scan_fwd(*(d[n] for n in KEYS), path=path)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("B,L,H,P,N,G,dtype,init", [
    (1, 64, 2, 8, 16, 1, "f32", False),      # the tiny fp32 shape
    (2, 100, 4, 64, 128, 2, "f32", True),    # ragged against the 38-step time block
    (2, 77, 4, 64, 128, 1, "bf16", True),
    (1, 50, 2, 128, 64, 1, "bf16", True),    # 16 warps of 8 rows
    (2, 33, 2, 64, 256, 2, "f32", True),     # two float4 per lane
    (1, 20, 2, 32, 512, 1, "f32", False),    # four float4 per lane
    (1, 9, 3, 17, 44, 1, "f32", True),       # ragged P and N
])
def test_trap_against_oracle(ssd, B, L, H, P, N, G, dtype, init):
    w = Workload("t", B, L, H, P, N, G, 1, dtype, init)
    inp = make_trap_inputs(w, seed=120 + N + L)
    ry, rh, rk, rv = trap_fwd(**inp)
    y, h, k, v = _run(ssd, _dev(inp))
    ey, eh = relerr(y, ry), relerr(h, rh)
    print(f"trap rel err y {ey:.3e} state {eh:.3e}")
    assert ey <= TOL[dtype] and eh <= TOL[dtype]
    assert np.array_equal(k.double().cpu().numpy(), rk)
    assert np.array_equal(v.double().cpu().numpy(), rv)


def test_trap_one_step_in_place(ssd):
    w = Workload("t", 16, 1, 8, 64, 128, 1, 1, "bf16", True)
    inp = make_trap_inputs(w, seed=131)
    ry, rh, rk, rv = trap_fwd(**inp)
    d = _dev(inp)
    h, k, v = d["h0"].clone(), d["k0"].clone(), d["v0"].clone()
    y, h2, k2, v2 = ssd.ssd_trap_scan_fwd(*(d[n] for n in KEYS[:7]), h, k, v, h_final=h, k_final=k, v_final=v,
                                          path="sequential")
    torch.cuda.synchronize()
    assert h2.data_ptr() == h.data_ptr()
    assert relerr(y, ry) <= TOL["bf16"] and relerr(h, rh) <= TOL["bf16"]
    assert np.array_equal(k.double().cpu().numpy(), rk) and np.array_equal(v.double().cpu().numpy(), rv)


def test_trap_split_and_resume_bitwise(ssd):
    # the carried (h, k, v) are exact, and each step is the same arithmetic
    w = Workload("t", 2, 90, 4, 64, 128, 2, 1, "bf16", True)
    d = _dev(make_trap_inputs(w, seed=132))
    y, h, k, v = _run(ssd, d)
    cut = 41
    first = {n: (t[:, :cut].contiguous() if n in KEYS[:6] else t) for n, t in d.items()}
    y1, h1, k1, v1 = _run(ssd, first)
    second = {n: (t[:, cut:].contiguous() if n in KEYS[:6] else t) for n, t in d.items()}
    second.update(h0=h1, k0=k1, v0=v1)
    y2, h2, k2, v2 = _run(ssd, second)
    assert torch.equal(torch.cat([y1, y2], dim=1), y)
    assert torch.equal(h2, h) and torch.equal(k2, k) and torch.equal(v2, v)


def test_trap_one_equals_ssd_scan(ssd):
    # trap = 1 and a = -exp(A_log): the Mamba-2 scan on the sequential path (both fp32)
    w = WORKLOADS["tiny_fp32"].with_(batch=2, seqlen=70, nheads=4, init_state=True)
    from selective_state_space_04_gb300.inputs import make_inputs
    s = {n: (None if t is None else t.cuda()) for n, t in make_inputs(w, seed=133).items()}
    y_ref, h_ref = ssd.ssd_scan_fwd(s["x"], s["dt_raw"], s["dt_bias"], s["A_log"], s["B"], s["C"], s["D"],
                                    s["init_state"], chunk=w.chunk, path="sequential")
    dt = torch.nn.functional.softplus(s["dt_raw"] + s["dt_bias"])
    a = (-torch.exp(s["A_log"])).expand_as(dt).contiguous()
    y, h, _, _ = ssd.ssd_trap_scan_fwd(s["x"], s["B"], s["C"], dt.contiguous(), a, torch.ones_like(dt),
                                       s["D"], s["init_state"], path="sequential")
    torch.cuda.synchronize()
    assert float((y - y_ref).abs().max()) <= 1e-5 * float(y_ref.abs().max())
    assert float((h - h_ref).abs().max()) <= 1e-5 * float(h_ref.abs().max())


# ------------------------------------------------ chunked tcgen05 kernel, trapezoidal mode
def _weak(inp):
    # a = -0.05, dt = 0.01: the state carries across hundreds of steps
    inp = dict(inp)
    inp["a"] = torch.full_like(inp["a"], -0.05)
    inp["dt"] = torch.full_like(inp["dt"], 0.01)
    return inp


@pytest.mark.parametrize("B,L,H,G,init,weak", [
    (2, 1000, 4, 1, True, False),    # ragged against 128-step sub-chunks
    (1, 2048, 4, 2, False, True),
    (2, 3000, 2, 1, True, True),     # several units per chain
    (3, 1, 4, 1, True, False),       # one step
    (4, 300, 8, 4, True, False),
])
def test_trap_chunked_against_oracle(ssd, B, L, H, G, init, weak):
    w = Workload("t", B, L, H, 64, 128, G, 256, "bf16", init, "trap")
    inp = make_trap_inputs(w, seed=140 + L + H)
    if weak:
        inp = _weak(inp)
    ry, rh, rk, rv = trap_fwd(**inp)
    d = _dev(inp)
    y, h, k, v = ssd.ssd_trap_scan_fwd(*(d[n] for n in KEYS), path="chunked")
    torch.cuda.synchronize()
    assert ssd.device_error() == 0
    ey, eh = relerr(y, ry), relerr(h, rh)
    print(f"trap chunked rel err y {ey:.3e} state {eh:.3e}")
    assert ey <= TOL["bf16"] and eh <= TOL["bf16"]
    assert np.array_equal(k.double().cpu().numpy(), rk)
    assert np.array_equal(v.double().cpu().numpy(), rv)
    if weak and init:
        # the carried state matters: without it the output is far off
        d0 = dict(d, h0=None, k0=None, v0=None)
        y0, _, _, _ = ssd.ssd_trap_scan_fwd(*(d0[n] for n in KEYS), path="chunked")
        torch.cuda.synchronize()
        assert relerr(y0, ry) > 10 * TOL["bf16"]


def test_trap_auto_path_is_chunked_and_matches_sequential(ssd):
    w = Workload("t", 2, 500, 4, 64, 128, 1, 256, "bf16", True, "trap")
    d = _dev(make_trap_inputs(w, seed=150))
    launches = ssd.launch_count()
    y1, h1, k1, v1 = ssd.ssd_trap_scan_fwd(*(d[n] for n in KEYS))            # auto
    torch.cuda.synchronize()
    assert ssd.launch_count() - launches == 2                                 # chunked kernel + k/v carry
    y2, h2, k2, v2 = ssd.ssd_trap_scan_fwd(*(d[n] for n in KEYS), path="sequential")
    torch.cuda.synchronize()
    assert relerr(y1, y2.double().cpu().numpy()) <= TOL["bf16"]
    assert relerr(h1, h2.double().cpu().numpy()) <= TOL["bf16"]
    assert torch.equal(k1, k2) and torch.equal(v1, v2)


def test_trap_chunked_in_place_states(ssd):
    w = Workload("t", 2, 700, 4, 64, 128, 1, 256, "bf16", True, "trap")
    inp = make_trap_inputs(w, seed=151)
    ry, rh, rk, rv = trap_fwd(**inp)
    d = _dev(inp)
    h, k, v = d["h0"].clone(), d["k0"].clone(), d["v0"].clone()
    y, _, _, _ = ssd.ssd_trap_scan_fwd(*(d[n] for n in KEYS[:7]), h, k, v, h_final=h, k_final=k, v_final=v,
                                       path="chunked")
    torch.cuda.synchronize()
    assert relerr(y, ry) <= TOL["bf16"] and relerr(h, rh) <= TOL["bf16"]
    assert np.array_equal(k.double().cpu().numpy(), rk) and np.array_equal(v.double().cpu().numpy(), rv)


@pytest.mark.parametrize("B,H,P,N,G,dtype,init", [
    (4, 4, 64, 128, 1, "bf16", True),
    (3, 6, 64, 128, 2, "f32", False),
    (2, 4, 100, 64, 1, "f32", True),     # P not a multiple of a warp's 8 rows
    (2, 2, 8, 16, 1, "f32", True),
    (2, 4, 64, 256, 4, "bf16", True),
    (1, 2, 32, 512, 1, "f32", True),
    (1, 3, 17, 44, 1, "f32", False),
])
def test_trap_one_step_against_oracle(ssd, B, H, P, N, G, dtype, init):
    # seqlen 1 runs the decode-layout kernel
    w = Workload("t", B, 1, H, P, N, G, 256, dtype, init)
    inp = make_trap_inputs(w, seed=160 + N + P)
    ry, rh, rk, rv = trap_fwd(**inp)
    y, h, k, v = _run(ssd, _dev(inp))
    assert relerr(y, ry) <= TOL[dtype] and relerr(h, rh) <= TOL[dtype]
    assert np.array_equal(k.double().cpu().numpy(), rk) and np.array_equal(v.double().cpu().numpy(), rv)


@pytest.mark.parametrize("name,rows", [("trap_many_short_seqs", 6), ("trap_decode_2p7b_128seq", 128)])
def test_bench_workloads_sampled(ssd, name, rows):
    # the bench's full workload in one call on the auto path (as the bench runs it);
    # the oracle takes the first `rows` batch rows (every batch row runs independently)
    w = WORKLOADS[name]
    inp = make_trap_inputs(w, seed=0)
    y, h, kf, vf = _run(ssd, _dev(inp), path="auto")
    sub = {k: (None if v is None else v[:rows]) if k not in ("D",) else v for k, v in inp.items()}
    ry, rh, rk, rv = trap_fwd(**sub)
    for got, ref in ((y, ry), (h, rh)):
        assert relerr(got[:rows], ref) <= TOL[w.dtype]
    assert relerr(kf[:rows], rk) <= TOL[w.dtype] and relerr(vf[:rows], rv) <= TOL[w.dtype]


# ------------------------------------------------ split schedule of the trapezoidal mode
# The mode runs the recurrence on the shifted state h~ (linear, decay alpha), so
# the split schedule's pass 1 / combine / pass 3 apply unchanged; pass 1 starts
# each chain from h0 + dt_0 (1 - trap_0) k0 v0^T.  Weak decay makes the state
# carried between units matter; without h0, k0, v0 the combine starts from zero.
@pytest.mark.parametrize("B,L,H,G,init,weak", [
    (1, 3000, 2, 1, True, True),     # many units per chain, long-range state
    (2, 1000, 4, 2, True, False),    # ragged tail, head groups
    (1, 700, 4, 1, False, True),     # no carried states
    (1, 257, 2, 1, True, True),      # one step past a chunk: a one-step last unit
])
def test_trap_split_against_oracle(ssd, B, L, H, G, init, weak):
    w = Workload("t", B, L, H, 64, 128, G, 256, "bf16", init, "trap")
    inp = make_trap_inputs(w, seed=170 + L + H)
    if weak:
        inp = _weak(inp)
    ry, rh, rk, rv = trap_fwd(**inp)
    d = _dev(inp)
    launches = ssd.launch_count()
    y, h, k, v = ssd.ssd_trap_scan_fwd(*(d[n] for n in KEYS), path="chunked", schedule="split")
    torch.cuda.synchronize()
    assert ssd.device_error() == 0
    assert ssd.launch_count() - launches == 4          # pass 1, combine, pass 3, k/v carry
    ey, eh = relerr(y, ry), relerr(h, rh)
    print(f"trap split rel err y {ey:.3e} state {eh:.3e}")
    assert ey <= TOL["bf16"] and eh <= TOL["bf16"]
    assert np.array_equal(k.double().cpu().numpy(), rk) and np.array_equal(v.double().cpu().numpy(), rv)
    if weak and init:
        # the carried-in states matter: without them the output is far off
        d0 = dict(d, h0=None, k0=None, v0=None)
        y0, _, _, _ = ssd.ssd_trap_scan_fwd(*(d0[n] for n in KEYS), path="chunked", schedule="split")
        torch.cuda.synchronize()
        assert relerr(y0, ry) > 10 * TOL["bf16"]


def test_trap_split_agrees_with_ranges(ssd):
    # two schedules of the same scan: each within the bar of the oracle, and close
    # to each other (they differ only in where the state crosses unit boundaries)
    w = Workload("t", 2, 2000, 4, 64, 128, 1, 256, "bf16", True, "trap")
    inp = _weak(make_trap_inputs(w, seed=180))
    ry, rh, _, _ = trap_fwd(**inp)
    d = _dev(inp)
    outs = {}
    for sched in ("split", "ranges", "pieces"):
        outs[sched] = ssd.ssd_trap_scan_fwd(*(d[n] for n in KEYS), path="chunked", schedule=sched)
        torch.cuda.synchronize()
        assert ssd.device_error() == 0
        assert relerr(outs[sched][0], ry) <= TOL["bf16"] and relerr(outs[sched][1], rh) <= TOL["bf16"]
    assert relerr(outs["split"][0], outs["ranges"][0].double().cpu().numpy()) <= TOL["bf16"]


def test_trap_long_context_takes_split_sampled(ssd):
    # the 64k-token bench workload on the auto path: one sequence of 8 chains, so
    # the library chooses the split schedule (3 launches + the k/v carry); the
    # oracle takes the 4 heads of group 0
    w = WORKLOADS["trap_long_context_64k"]
    inp = make_trap_inputs(w, seed=0)
    d = _dev(inp)
    launches = ssd.launch_count()
    y, h, kf, vf = ssd.ssd_trap_scan_fwd(*(d[n] for n in KEYS))
    torch.cuda.synchronize()
    assert ssd.device_error() == 0
    assert ssd.launch_count() - launches == 4
    hp = w.nheads // w.ngroups
    sub = {"v": inp["v"][:, :, :hp], "k": inp["k"][:, :, :1], "q": inp["q"][:, :, :1], "dt": inp["dt"][:, :, :hp],
           "a": inp["a"][:, :, :hp], "trap": inp["trap"][:, :, :hp], "D": inp["D"][:hp], "h0": inp["h0"][:, :hp],
           "k0": inp["k0"][:, :hp], "v0": inp["v0"][:, :hp]}
    ry, rh, rk, rv = trap_fwd(**sub)
    assert relerr(y[:, :, :hp], ry) <= TOL["bf16"] and relerr(h[:, :hp], rh) <= TOL["bf16"]
    assert np.array_equal(kf[:, :hp].double().cpu().numpy(), rk)
    assert np.array_equal(vf[:, :hp].double().cpu().numpy(), rv)
