"""GPU parity of ssd_conv_scan_fwd: the causal conv1d + SiLU over the fused
x | B | C channels, then the forward scan, with the conv of the x channels done
inside the chunked scan kernel (the builderforce Mamba2Block's conv1d -> SSD
order on one layer's buffers).

Two references:
* the fp64 oracles in sequence, oracle.neighbors.conv1d_silu then
  oracle.ssd_fwd, at the scan's bf16 bar (max|y - y_ref| / max|y_ref| <= 2e-2,
  the same for the final state; the carried conv state is a copy of inputs and
  must match exactly);
* the library's own two-call chain, ssd_conv1d_silu_fwd then ssd_scan_fwd with
  the same schedule: the fused kernel applies the same conv with the same
  operations in the same order and rounds x to bf16 as that chain does, so y,
  the final state and the conv state must match it bit for bit.

Cases span several 128-step sub-chunks and chunks, a ragged tail, kernel sizes
2 to 4, with and without a carried conv state, head groups, and every schedule
(so unit starts fall in the middle of a sequence, where the 3-step halo comes
from device memory rather than from the previous sub-chunk).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.neighbors import conv1d_silu
from selective_state_space_04_gb300.inputs import WORKLOADS, Workload, make_conv_inputs, make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def ssd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_04_gb300 import build
    build.build()
    from selective_state_space_04_gb300 import ssd as mod
    return mod


def relerr(a, ref):
    a = a.double().cpu().numpy() if hasattr(a, "cpu") else np.asarray(a, dtype=np.float64)
    return float(np.max(np.abs(a - ref)) / max(np.max(np.abs(ref)), 1e-30))


def _inputs(Bt, L, H, G, K, seed, conv_state=True, init_state=True, chunk=256):
    w = Workload("t", Bt, L, H, 64, 128, G, chunk, "bf16", conv_state)
    ci = make_conv_inputs(w, K=K, seed=seed)
    si = make_inputs(w.with_(init_state=init_state), seed + 1)   # (its x, B, C are not used)
    return w, ci, si


def _dev(t):
    return None if t is None else t.cuda().contiguous()


def _fused(ssd, w, ci, si, schedule="auto"):
    out = ssd.conv_scan_fwd(_dev(ci["xbc"]), _dev(ci["weight"]), _dev(ci["bias"]), _dev(ci["conv_state"]),
                            _dev(si["dt_raw"]), _dev(si["dt_bias"]), _dev(si["A_log"]), _dev(si["D"]),
                            _dev(si["init_state"]), nheads=w.nheads, headdim=w.headdim, ngroups=w.ngroups,
                            dstate=w.dstate, chunk=w.chunk, schedule=schedule)
    torch.cuda.synchronize()
    assert ssd.device_error() == 0
    return out


def _two_calls(ssd, w, ci, si, schedule="auto"):
    x, Bm, Cm, st = ssd.conv1d_silu_fwd(_dev(ci["xbc"]), _dev(ci["weight"]), _dev(ci["bias"]), _dev(ci["conv_state"]),
                                        nheads=w.nheads, headdim=w.headdim, ngroups=w.ngroups, dstate=w.dstate)
    y, f = ssd.ssd_scan_fwd(x, _dev(si["dt_raw"]), _dev(si["dt_bias"]), _dev(si["A_log"]), Bm, Cm, _dev(si["D"]),
                            _dev(si["init_state"]), chunk=w.chunk, path="chunked", schedule=schedule)
    torch.cuda.synchronize()
    assert ssd.device_error() == 0
    return y, f, st


@pytest.mark.parametrize("Bt,L,H,G,K,conv_state,init_state", [
    (2, 700, 4, 1, 4, True, True),     # ragged against 128-step sub-chunks and 256-step chunks
    (1, 1000, 8, 2, 3, False, False),  # head groups, no carried states
    (2, 300, 4, 1, 2, True, False),
    (3, 129, 2, 1, 4, True, True),     # one step past a sub-chunk
])
def test_conv_scan_against_oracle_chain(ssd, Bt, L, H, G, K, conv_state, init_state):
    w, ci, si = _inputs(Bt, L, H, G, K, seed=300 + L + K, conv_state=conv_state, init_state=init_state)
    y, f, st = _fused(ssd, w, ci, si)
    rx, rB, rC, rs = conv1d_silu(**ci, H=H, P=64, G=G, N=128)
    ry, rf = oracle.ssd_fwd(rx, si["dt_raw"], si["dt_bias"], si["A_log"], rB, rC, si["D"], si["init_state"])
    ey, ef = relerr(y, ry), relerr(f, rf)
    print(f"conv+scan vs oracle chain: y {ey:.3e}  final state {ef:.3e}")
    assert ey <= TOL and ef <= TOL
    assert np.array_equal(st.double().cpu().numpy(), rs)


@pytest.mark.parametrize("schedule", ["auto", "ranges", "pieces", "split"])
def test_conv_scan_matches_two_calls_bitwise(ssd, schedule):
    # 1500 steps: several units per chain on the range and split schedules, so the
    # halo of a unit start is read from device memory mid-sequence
    w, ci, si = _inputs(1, 1500, 6, 1, 4, seed=320)
    y, f, st = _fused(ssd, w, ci, si, schedule)
    y2, f2, st2 = _two_calls(ssd, w, ci, si, schedule)
    assert torch.equal(y, y2)
    assert torch.equal(f, f2)
    assert torch.equal(st, st2)


@pytest.mark.parametrize("chunk", [64, 128, 512])
def test_conv_scan_chunk_lengths(ssd, chunk):
    w, ci, si = _inputs(2, 640, 4, 1, 4, seed=330 + chunk, chunk=chunk)
    y, f, st = _fused(ssd, w, ci, si, "ranges")
    y2, f2, st2 = _two_calls(ssd, w, ci, si, "ranges")
    assert torch.equal(y, y2) and torch.equal(f, f2) and torch.equal(st, st2)


def test_conv_scan_full_size_matches_two_calls(ssd):
    # the 2.7B layer's conv and scan (the bench's conv_scan_2p7b workload), as the
    # bench runs it; its two-call chain is checked against the oracles elsewhere
    wc = WORKLOADS["conv_silu_2p7b"]
    w, ci, si = _inputs(wc.batch, wc.seqlen, wc.nheads, wc.ngroups, 4, seed=0)
    y, f, st = _fused(ssd, w, ci, si)
    y2, f2, st2 = _two_calls(ssd, w, ci, si)
    assert torch.isfinite(y.float()).all()
    assert torch.equal(y, y2) and torch.equal(f, f2) and torch.equal(st, st2)


def test_conv_scan_no_steps_and_refusals(ssd):
    w, ci, si = _inputs(2, 0, 4, 1, 4, seed=340)
    y, f, st = _fused(ssd, w, ci, si)
    assert torch.equal(f.cpu(), si["init_state"]) and torch.equal(st.cpu(), ci["conv_state"])
    # fp32 is refused (the chunked path is bf16), as is another path
    w, ci, si = _inputs(1, 64, 2, 1, 4, seed=341)
    with pytest.raises(ssd.SsdError) as e:
        ssd.conv_scan_fwd(_dev(ci["xbc"]).float(), _dev(ci["weight"]), None, None, _dev(si["dt_raw"]),
                          _dev(si["dt_bias"]), _dev(si["A_log"]), _dev(si["D"]), nheads=2, headdim=64, ngroups=1,
                          dstate=128)
    assert e.value.status == 9
    with pytest.raises(ssd.SsdError) as e:
        ssd.conv_scan_fwd(_dev(ci["xbc"]), _dev(ci["weight"]), None, None, _dev(si["dt_raw"]), _dev(si["dt_bias"]),
                          _dev(si["A_log"]), _dev(si["D"]), nheads=2, headdim=64, ngroups=1, dstate=128,
                          path="sequential")
    assert e.value.status == 4
