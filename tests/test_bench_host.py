"""Host-side logic of bench.py (CPU): byte/flop accounting and the
max-over-ranks timing used under torchrun, exercised with world size 2 on gloo."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from selective_state_space_04_gb300.inputs import WORKLOADS  # noqa: E402


def test_algorithmic_bytes_headline():
    w = WORKLOADS["mamba2_2p7b_layer"]
    x = 8 * 4096 * 80 * 64 * 2
    dt = 8 * 4096 * 80 * 4
    bc = 2 * 8 * 4096 * 1 * 128 * 2
    par = 3 * 80 * 4
    state = 8 * 80 * 64 * 128 * 4
    assert bench.algorithmic_bytes(w) == 2 * x + dt + bc + par + state
    # per token*head, about 274 B
    assert 273 < bench.algorithmic_bytes(w) / w.token_heads < 275


def test_algorithmic_bytes_counts_initial_state_when_given():
    w = WORKLOADS["many_short_seqs"]
    state = 256 * 48 * 64 * 128 * 4
    assert bench.algorithmic_bytes(w) - bench.algorithmic_bytes(w.with_(init_state=False)) == state


def test_algorithmic_flops_headline():
    w = WORKLOADS["mamba2_2p7b_layer"]
    f = bench.algorithmic_flops(w)
    assert 49.0e3 < f / w.token_heads < 50.5e3


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, lr = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    v = bench.max_over_ranks(dist, 10.0 + 5.0 * r, "cpu")
    dist.barrier()
    q.put((r, w, lr, v))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 2, 0, 15.0), (1, 2, 1, 15.0)]


def test_single_process_needs_no_process_group():
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.5, "cpu") == 3.5


def test_reference_arm_reports_the_gpu_arms_config():
    # both arms build `config` from the workload alone, so the driver can pair
    # them; the reference arm runs the fp64 oracle on the host (no GPU needed)
    import json
    import subprocess
    w = WORKLOADS["tiny_fp32"]
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny_fp32", "--steps", "2", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, check=True).stdout
    line = json.loads(out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"] == bench.workload_config(w, 0, bench.flushes_l2(bench.algorithmic_bytes(w)))
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_l2_policy():
    # the 130M layer (58.5 MB) fits in L2 and is flushed between steps; the
    # 2.7B layer (719 MB) is not
    assert bench.flushes_l2(bench.algorithmic_bytes(WORKLOADS["mamba2_130m_layer"]))
    assert not bench.flushes_l2(bench.algorithmic_bytes(WORKLOADS["mamba2_2p7b_layer"]))
    assert not bench.flushes_l2(bench.algorithmic_bytes(WORKLOADS["many_short_seqs"]))
