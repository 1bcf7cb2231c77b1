"""GPU parity: libssd (through the C ABI) against the fp64 oracle.

Metric (the method's stated bar): max|y - y_ref| / max|y_ref| over the whole
output, applied to y and to the final state separately; <= 2e-2 for bf16
inputs with fp32 accumulation, <= 1e-4 for the fp32 path.

Small cases (oracle in seconds) are compared element by element; they span
several 128-step sub-chunks, several chunks and a ragged tail.  Full-size
workloads are run in the launch configuration the benchmark times and
compared on sampled (batch, head) chains that the oracle computes one by one.
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


def to_dev(inp):
    return {k: (None if v is None else v.cuda().contiguous()) for k, v in inp.items()}


def run(ssd, inp, w, path="auto", chunk=None, init=True, schedule="auto"):
    d = to_dev(inp)
    y, fin = ssd.ssd_scan_fwd(d["x"], d["dt_raw"], d["dt_bias"], d["A_log"], d["B"], d["C"], d["D"],
                              d["init_state"] if init else None, chunk=chunk or w.chunk, path=path,
                              schedule=schedule)
    torch.cuda.synchronize()
    assert ssd.device_error() == 0
    return y, fin


def relerr(a, ref):
    a = a.double().cpu().numpy() if hasattr(a, "cpu") else a
    return float(np.max(np.abs(a - ref)) / max(np.max(np.abs(ref)), 1e-30))


def check(y, fin, ref_y, ref_fin, dtype):
    ey, ef = relerr(y, ref_y), relerr(fin, ref_fin)
    print(f"rel err y {ey:.3e}  final state {ef:.3e}")
    assert ey <= TOL[dtype], f"y rel err {ey:.3e} > {TOL[dtype]}"
    assert ef <= TOL[dtype], f"final state rel err {ef:.3e} > {TOL[dtype]}"
    return ey, ef


def small(**kw):
    base = dict(name="t", batch=2, seqlen=640, nheads=4, headdim=64, dstate=128, ngroups=1,
                chunk=256, dtype="bf16", init_state=True)
    base.update(kw)
    return Workload(**base)


# ----------------------------------------------------------- small, exact
def test_tiny_fp32_sequential(ssd):
    w = WORKLOADS["tiny_fp32"]
    inp = make_inputs(w, seed=0)
    ref = oracle.ssd_fwd(**inp)
    assert ssd.select_path((w.batch, w.seqlen, w.nheads, w.headdim), w.ngroups, w.dstate,
                           w.chunk, "f32") == ssd.PATH_SEQUENTIAL
    y, fin = run(ssd, inp, w)
    check(y, fin, *ref, "f32")


# row-layout kernel: one, two and four float4 of state per lane, and 16 warps of
# 8 rows; slice-layout kernel: N % 4 != 0, or P past the row layout's rows
@pytest.mark.parametrize("shape", [(1, 1, 2, 8, 16, 1), (2, 37, 4, 8, 16, 2), (1, 200, 3, 5, 7, 1),
                                   (2, 130, 4, 64, 128, 1), (1, 70, 2, 32, 256, 2), (1, 50, 2, 32, 512, 1),
                                   (1, 40, 2, 128, 128, 1), (1, 30, 2, 200, 64, 1)])
def test_sequential_fp32_shapes(ssd, shape):
    Bt, L, H, P, N, G = shape
    w = small(batch=Bt, seqlen=L, nheads=H, headdim=P, dstate=N, ngroups=G, chunk=16, dtype="f32")
    inp = make_inputs(w, seed=1)
    y, fin = run(ssd, inp, w, path="sequential")
    check(y, fin, *oracle.ssd_fwd(**inp), "f32")


def test_sequential_bf16(ssd):
    w = small(seqlen=300)
    inp = make_inputs(w, seed=2)
    y, fin = run(ssd, inp, w, path="sequential")
    check(y, fin, *oracle.ssd_fwd(**inp), "bf16")


@pytest.mark.parametrize("init", [False, True])
def test_chunked_small(ssd, init):
    w = small(init_state=init)
    inp = make_inputs(w, seed=3)
    assert ssd.select_path((w.batch, w.seqlen, w.nheads, w.headdim), w.ngroups, w.dstate,
                           w.chunk) == ssd.PATH_CHUNKED
    y, fin = run(ssd, inp, w, path="chunked")
    check(y, fin, *oracle.ssd_fwd(**inp), "bf16")


@pytest.mark.parametrize("chunk", [64, 128, 192, 256, 512])
def test_chunked_chunk_lengths_ragged(ssd, chunk):
    w = small(seqlen=700, chunk=chunk)
    inp = make_inputs(w, seed=4)
    y, fin = run(ssd, inp, w, path="chunked")
    check(y, fin, *oracle.ssd_fwd(**inp), "bf16")


@pytest.mark.parametrize("L", [1, 2, 63, 127, 128, 129, 255, 257])
def test_chunked_short_and_boundary_lengths(ssd, L):
    w = small(seqlen=L, batch=1, nheads=2)
    inp = make_inputs(w, seed=5)
    y, fin = run(ssd, inp, w, path="chunked")
    check(y, fin, *oracle.ssd_fwd(**inp), "bf16")


@pytest.mark.parametrize("H,G", [(8, 2), (8, 4), (16, 8), (6, 3)])
def test_chunked_groups(ssd, H, G):
    w = small(nheads=H, ngroups=G, seqlen=384)
    inp = make_inputs(w, seed=6)
    y, fin = run(ssd, inp, w, path="chunked")
    check(y, fin, *oracle.ssd_fwd(**inp), "bf16")


def test_many_short_sequences_reduced(ssd):
    w = WORKLOADS["many_short_seqs"].with_(batch=16, nheads=8)
    inp = make_inputs(w, seed=7)
    ref = oracle.ssd_fwd(**inp)
    for path in ("chunked", "sequential"):
        y, fin = run(ssd, inp, w, path=path)
        check(y, fin, *ref, "bf16")


def test_paths_agree(ssd):
    w = small(seqlen=520)
    inp = make_inputs(w, seed=8)
    y1, f1 = run(ssd, inp, w, path="chunked")
    y2, f2 = run(ssd, inp, w, path="sequential")
    ref = oracle.ssd_fwd(**inp)
    check(y1, f1, *ref, "bf16")
    check(y2, f2, *ref, "bf16")
    assert relerr(y1, y2.double().cpu().numpy()) < 2e-2


def test_chunk_length_invariance(ssd):
    w = small(seqlen=1024, init_state=True)
    inp = make_inputs(w, seed=9)
    outs = [run(ssd, inp, w, path="chunked", chunk=q) for q in (64, 128, 256, 512, 1024)]
    y0 = outs[0][0].double().cpu().numpy()
    f0 = outs[0][1].double().cpu().numpy()
    for y, f in outs[1:]:
        assert relerr(y, y0) < 1e-2
        assert relerr(f, f0) < 1e-2


def test_split_and_resume(ssd):
    w = small(seqlen=768)
    inp = make_inputs(w, seed=10)
    y, fin = run(ssd, inp, w, path="chunked")
    L1 = 256
    first = dict(inp)
    second = dict(inp)
    for k in ("x", "dt_raw", "B", "C"):
        first[k] = inp[k][:, :L1].contiguous()
        second[k] = inp[k][:, L1:].contiguous()
    y1, f1 = run(ssd, first, w.with_(seqlen=L1), path="chunked")
    second["init_state"] = f1.cpu()
    y2, f2 = run(ssd, second, w.with_(seqlen=w.seqlen - L1), path="chunked")
    ycat = torch.cat([y1, y2], dim=1)
    assert relerr(ycat, y.double().cpu().numpy()) < 1e-2
    assert relerr(f2, fin.double().cpu().numpy()) < 1e-2


def test_deterministic_bitwise(ssd):
    w = small(seqlen=900)
    inp = make_inputs(w, seed=11)
    for path in ("chunked", "sequential"):
        a = run(ssd, inp, w, path=path)
        b = run(ssd, inp, w, path=path)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_in_place_state_update(ssd):
    w = small(seqlen=400)
    inp = make_inputs(w, seed=12)
    d = to_dev(inp)
    state = d["init_state"].clone()
    y, _ = ssd.ssd_scan_fwd(d["x"], d["dt_raw"], d["dt_bias"], d["A_log"], d["B"], d["C"], d["D"],
                            state, chunk=256, path="chunked", final_state=state)
    torch.cuda.synchronize()
    ry, rf = oracle.ssd_fwd(**inp)
    check(y, state, ry, rf, "bf16")


def test_host_entry_point_matches_device(ssd):
    w = small(seqlen=333)
    inp = make_inputs(w, seed=13)
    yd, fd = run(ssd, inp, w)
    pinned = {k: (None if v is None else v.contiguous().pin_memory()) for k, v in inp.items()}
    yh, fh = ssd.ssd_scan_fwd_host(pinned["x"], pinned["dt_raw"], pinned["dt_bias"], pinned["A_log"],
                                   pinned["B"], pinned["C"], pinned["D"], pinned["init_state"],
                                   chunk=w.chunk)
    assert torch.equal(yh, yd.cpu()) and torch.equal(fh, fd.cpu())


@pytest.mark.parametrize("init", [False, True])
def test_host_entry_point_pipelined_matches_device(ssd, init):
    # 55 MB of buffers and 4 batch rows: the host path runs 4 pieces through its
    # copy-in / compute / copy-out streams; the bits must be the device path's
    w = Workload("t", 4, 2048, 24, 64, 128, 1, 256, "bf16", init)
    inp = make_inputs(w, seed=16)
    yd, fd = run(ssd, inp, w)
    pinned = {k: (None if v is None else v.contiguous().pin_memory()) for k, v in inp.items()}
    yh, fh = ssd.ssd_scan_fwd_host(pinned["x"], pinned["dt_raw"], pinned["dt_bias"], pinned["A_log"],
                                   pinned["B"], pinned["C"], pinned["D"], pinned["init_state"],
                                   chunk=w.chunk)
    assert torch.equal(yh, yd.cpu()) and torch.equal(fh, fd.cpu())


def test_empty_batch_and_sequence(ssd):
    w = small(batch=0)
    inp = make_inputs(w, seed=14)
    y, fin = run(ssd, inp, w)
    assert y.numel() == 0
    w = small(seqlen=0)
    inp = make_inputs(w, seed=15)
    y, fin = run(ssd, inp, w)
    assert torch.equal(fin.cpu(), inp["init_state"])
    y, fin = run(ssd, inp, w, init=False)
    assert torch.count_nonzero(fin).item() == 0


def test_rejects_wrong_dtype_for_chunked(ssd):
    w = small(dtype="f32")
    inp = make_inputs(w, seed=16)
    with pytest.raises(ssd.SsdError) as ei:
        run(ssd, inp, w, path="chunked")
    assert ei.value.status == 9      # SSD_ERR_UNSUPPORTED_DTYPE: the chunked path takes bf16 only


# --------------------------------------------- full size, sampled chains
def sample_pairs(w, n, seed):
    rng = np.random.default_rng(seed)
    pairs = {(0, 0), (w.batch - 1, w.nheads - 1)}
    while len(pairs) < min(n, w.batch * w.nheads):
        pairs.add((int(rng.integers(w.batch)), int(rng.integers(w.nheads))))
    return sorted(pairs)


def oracle_pair(inp, w, b, h):
    g = h // (w.nheads // w.ngroups)
    sl = dict(x=inp["x"][b:b + 1, :, h:h + 1], dt_raw=inp["dt_raw"][b:b + 1, :, h:h + 1],
              dt_bias=inp["dt_bias"][h:h + 1], A_log=inp["A_log"][h:h + 1],
              B=inp["B"][b:b + 1, :, g:g + 1], C=inp["C"][b:b + 1, :, g:g + 1], D=inp["D"][h:h + 1],
              init_state=None if inp["init_state"] is None else inp["init_state"][b:b + 1, h:h + 1])
    y, f = oracle.ssd_fwd(**sl)
    return y[0, :, 0], f[0, 0]


@pytest.mark.parametrize("name,npairs", [("mamba2_130m_layer", 6), ("mamba2_2p7b_layer", 6),
                                         ("long_context_64k", 3), ("many_short_seqs", 40)])
def test_full_size_workloads_sampled(ssd, name, npairs):
    w = WORKLOADS[name]
    inp = make_inputs(w, seed=0)
    y, fin = run(ssd, inp, w)       # auto path, as the benchmark runs it
    assert torch.isfinite(y.float()).all() and torch.isfinite(fin).all()
    yc, fc = y.cpu(), fin.cpu()
    num_y = den_y = num_f = den_f = 0.0
    for b, h in sample_pairs(w, npairs, seed=1):
        ry, rf = oracle_pair(inp, w, b, h)
        num_y = max(num_y, float(np.max(np.abs(yc[b, :, h].double().numpy() - ry))))
        den_y = max(den_y, float(np.max(np.abs(ry))))
        num_f = max(num_f, float(np.max(np.abs(fc[b, h].double().numpy() - rf))))
        den_f = max(den_f, float(np.max(np.abs(rf))))
    assert num_y / den_y <= TOL["bf16"], f"{name}: y rel err {num_y / den_y:.3e}"
    assert num_f / den_f <= TOL["bf16"], f"{name}: final rel err {num_f / den_f:.3e}"


# ----------------------------------------------------------- split schedule
# Few chains and many chunks: the chunked path runs two passes over independent
# units with a combine of the unit states in between (3 launches).
@pytest.mark.parametrize("init,H,G", [(False, 2, 1), (True, 4, 2), (True, 8, 2)])
def test_split_schedule_against_oracle(ssd, init, H, G):
    w = small(batch=1, seqlen=12000, nheads=H, ngroups=G, chunk=256, init_state=init)
    assert ssd.launches_per_call((w.batch, w.seqlen, w.nheads, w.headdim), w.ngroups, w.dstate,
                                 w.chunk) == 3
    inp = make_inputs(w, seed=30 + H)
    y, fin = run(ssd, inp, w, path="chunked")
    check(y, fin, *oracle.ssd_fwd(**inp), "bf16")


def test_split_schedule_matches_chained_schedule(ssd):
    # ssd_scan_fwd_noalloc keeps the chained schedule on the same shape
    w = small(batch=1, seqlen=8192, nheads=2, chunk=256, init_state=True)
    inp = make_inputs(w, seed=40)
    d = to_dev(inp)
    args = (d["x"], d["dt_raw"], d["dt_bias"], d["A_log"], d["B"], d["C"], d["D"], d["init_state"])
    y1, f1 = ssd.ssd_scan_fwd(*args, chunk=w.chunk)
    y2, f2 = ssd.ssd_scan_fwd_noalloc(*args, chunk=w.chunk)
    torch.cuda.synchronize()
    assert ssd.device_error() == 0
    ref_y = y2.double().cpu().numpy()
    ref_f = f2.double().cpu().numpy()
    check(y1, f1, ref_y, ref_f, "bf16")


def _weak_decay(inp, H):
    # A = -0.05 and dt = softplus(dt_raw + dt_bias) about 0.01: a decay of about
    # exp(-1.3) per 256-step chunk, so states carry across many chunks
    inp = dict(inp)
    inp["A_log"] = np.full(H, np.log(0.05), dtype=np.float32)
    inp["A_log"] = torch.from_numpy(inp["A_log"])
    inp["dt_bias"] = torch.full((H,), float(np.log(np.expm1(0.01))), dtype=torch.float32)
    return inp


@pytest.mark.parametrize("seqlen,H", [(12000, 4), (2048, 64)])
def test_weak_decay_state_passing(ssd, seqlen, H):
    # (12000, 4): few chains, split schedule; (2048, 64): many chains, chained schedule
    w = small(batch=1, seqlen=seqlen, nheads=H, chunk=256, init_state=True)
    inp = _weak_decay(make_inputs(w, seed=50), H)
    ref_y, ref_f = oracle.ssd_fwd(**inp)
    y, fin = run(ssd, inp, w, path="chunked")
    check(y, fin, ref_y, ref_f, "bf16")
    # the carried state matters here: dropping it changes the output a lot
    d = to_dev(inp)
    y0, _ = ssd.ssd_scan_fwd(d["x"], d["dt_raw"], d["dt_bias"], d["A_log"], d["B"], d["C"], d["D"],
                             None, chunk=w.chunk)
    torch.cuda.synchronize()
    assert relerr(y0, ref_y) > 10 * 2e-2


@pytest.mark.parametrize("init", [True, False])
def test_split_with_folded_combine_weak_decay(ssd, init):
    # few ranges per chain (the 130M layer's shape: 48 chains of 3 ranges): pass 3
    # forms each unit's entering state from its predecessors' end states (two
    # launches, no combine); weak decay makes those states matter
    w = WORKLOADS["mamba2_130m_layer"].with_(init_state=init)
    shape = (w.batch, w.seqlen, w.nheads, w.headdim)
    assert ssd.chunk_schedule(shape, w.ngroups, w.dstate, w.chunk) == "split"
    assert ssd.launches_per_call(shape, w.ngroups, w.dstate, w.chunk) == 2
    inp = _weak_decay(make_inputs(w, seed=90 + init), w.nheads)
    launches = ssd.launch_count()
    y, fin = run(ssd, inp, w, init=init)
    assert ssd.launch_count() - launches == 2
    yc, fc = y.cpu(), fin.cpu()
    num_y = den_y = num_f = den_f = 0.0
    for b, h in sample_pairs(w, 8, seed=3):
        ry, rf = oracle_pair(inp, w, b, h)
        num_y = max(num_y, float(np.max(np.abs(yc[b, :, h].double().numpy() - ry))))
        den_y = max(den_y, float(np.max(np.abs(ry))))
        num_f = max(num_f, float(np.max(np.abs(fc[b, h].double().numpy() - rf))))
        den_f = max(den_f, float(np.max(np.abs(rf))))
    print(f"rel err y {num_y / den_y:.3e}  final state {num_f / den_f:.3e}")
    assert num_y / den_y <= TOL["bf16"] and num_f / den_f <= TOL["bf16"]
    # the state entering the second range matters: restarting there from zero moves y far
    ry, _ = oracle_pair(inp, w, 0, 0)
    t0 = 768
    tail = dict(x=inp["x"][0:1, t0:, 0:1], dt_raw=inp["dt_raw"][0:1, t0:, 0:1], dt_bias=inp["dt_bias"][0:1],
                A_log=inp["A_log"][0:1], B=inp["B"][0:1, t0:, 0:1], C=inp["C"][0:1, t0:, 0:1], D=inp["D"][0:1],
                init_state=None)
    rt, _ = oracle.ssd_fwd(**tail)
    assert relerr(rt[0, :, 0], ry[t0:]) > 10 * TOL["bf16"]


# ----------------------------------------------------------- piece schedule
# On request: each CTA takes one run of equal length over the chains' sub-chunks
# laid end to end; with more chains than SMs some chains are cut between two
# CTAs and their state crosses the cut through a slot.  Weak decay makes that
# state matter.
def _cut_chains(nchains, nsub, sms):
    grid = min(sms, nchains)
    total = nchains * nsub
    return sum(1 for i in range(grid - 1) if ((i + 1) * total // grid) % nsub)


@pytest.mark.parametrize("batch,seqlen,H,init", [(2, 1000, 160, True), (2, 1024, 160, False),
                                                 (4, 2048, 80, True), (3, 4000, 112, True)])
def test_piece_schedule_weak_decay(ssd, batch, seqlen, H, init):
    w = small(batch=batch, seqlen=seqlen, nheads=H, chunk=256, init_state=init)
    shape = (w.batch, w.seqlen, w.nheads, w.headdim)
    assert ssd.chunk_schedule(shape, w.ngroups, w.dstate, w.chunk, schedule="pieces") == "pieces"
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert _cut_chains(batch * H // 2, -(-seqlen // 128), sms) > 0
    inp = _weak_decay(make_inputs(w, seed=70 + H), H)
    ref_y, ref_f = oracle.ssd_fwd(**inp)
    y, fin = run(ssd, inp, w, path="chunked", init=init, schedule="pieces")
    check(y, fin, ref_y, ref_f, "bf16")


@pytest.mark.parametrize("schedule", ["pieces", "ranges"])
def test_schedules_match_sliced_calls(ssd, schedule):
    # the scan over 512-step slices, one call each, the final state of one call
    # entering the next: the cuts between CTAs fall elsewhere
    w = small(batch=2, seqlen=1000, nheads=160, chunk=256, init_state=True)
    inp = _weak_decay(make_inputs(w, seed=80), w.nheads)
    y1, f1 = run(ssd, inp, w, path="chunked", schedule=schedule)
    d = to_dev(inp)
    y2 = torch.empty_like(y1)
    state = d["init_state"]
    for t0 in range(0, w.seqlen, 512):
        sl = slice(t0, min(w.seqlen, t0 + 512))
        ys, state = ssd.ssd_scan_fwd(d["x"][:, sl].contiguous(), d["dt_raw"][:, sl].contiguous(), d["dt_bias"],
                                     d["A_log"], d["B"][:, sl].contiguous(), d["C"][:, sl].contiguous(), d["D"],
                                     state, chunk=w.chunk, path="chunked", schedule=schedule)
        y2[:, sl] = ys
    torch.cuda.synchronize()
    assert ssd.device_error() == 0
    print("bitwise equal:", bool(torch.equal(y1, y2)), bool(torch.equal(f1, state)))
    check(y1, f1, y2.double().cpu().numpy(), state.double().cpu().numpy(), "bf16")
