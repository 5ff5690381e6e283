"""The benchmark's multi-rank host logic on CPU: two gloo ranks (one process
each), as the N > 1 launch runs one replica per GPU. Each rank draws its own
replica, the step time is the slowest rank's, the whole-job value counts every
replica's work, and the reference arm runs on rank 0 only."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


_WORKER = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import importlib.util
import torch
import torch.distributed as dist
spec = importlib.util.spec_from_file_location("b", os.path.join({root!r}, "bench.py"))
b = importlib.util.module_from_spec(spec); spec.loader.exec_module(b)
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
ms = [3.0, 5.0][rank]
ms_max = b.max_over_ranks(ms, dist, "cpu")
from packed_sequence_flash_gb300 import inputs
w = inputs.config(2, b.replica_seed(0, rank))
print(json.dumps({{"rank": rank, "ms_max": ms_max, "value": b.whole_job_value(world, 1e12, ms_max),
                  "first_len": int(w.extra["lengths"][0])}}))
dist.destroy_process_group()
"""


def test_two_gloo_ranks_share_the_slowest_step_and_draw_their_own_replicas(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(_WORKER.format(root=ROOT))
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=240)
        assert p.returncode == 0, e
        outs.append(json.loads(o.strip().splitlines()[-1]))
    for o in outs:
        assert o["ms_max"] == 5.0                          # the slowest rank's time on every rank
        assert abs(o["value"] - 2 * 1e12 / 5e-3 / 1e12) < 1e-9  # both replicas' work over that time
    assert outs[0]["first_len"] != outs[1]["first_len"]    # each rank its own draws


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    b = _bench()
    monkeypatch.setenv("RANK", "1")

    class Args:
        config, seed, warmup, steps, gpus, softcap = 2, 0, 3, 1, 2, None

    assert b.reference_arm(Args()) == 0
    assert capsys.readouterr().out == ""


def test_single_rank_needs_no_process_group():
    b = _bench()
    assert b.max_over_ranks(4.25) == 4.25
    assert b.replica_seed(7, 0) == 7
    assert b.whole_job_value(1, 2e9, 1.0) == pytest.approx(2.0)


def test_captured_traffic_is_reported_only_for_its_workload_and_sources():
    b = _bench()
    for (kernel, workload), (digest, nbytes) in b.NCU_TRAFFIC.items():
        assert b.ncu_traffic(kernel, workload) == (nbytes if digest == b.kernel_source_hash(kernel) else None)
        assert b.ncu_traffic(kernel, "another_workload") is None
    assert b.ncu_traffic("attn_bwd_kernel", "cfg2_doc_causal_t8192_d128") is None


def test_dense_workload_flops_and_reference_sample():
    b = _bench()
    from packed_sequence_flash_gb300 import inputs

    assert b.dense_pairs(128, 128, True) == 128 * 129 // 2
    assert b.dense_pairs(3, 5, True) == 3 + 4 + 5  # bottom-right: query i sees keys 0..i+2
    assert b.dense_pairs(5, 3, True) == 0 + 0 + 1 + 2 + 3
    assert b.dense_pairs(4, 6, False) == 24
    w = inputs.config(1, 0)
    pairs, f, bw = b.workload_flops(w)
    assert pairs == 16512 and f == pairs * 2 * (64 + 64) and bw == pairs * (6 * 64 + 4 * 64)
    sub = b.cpu_sample_dense(w, 64)
    assert tuple(sub.q.shape) == (1, 2, 64, 64) and tuple(sub.k.shape) == (1, 1, 64, 64)
    assert b.config_dict(w, type("A", (), {"seed": 0})(), pairs, 0)["visible_pairs_x_heads"] == 16512


def test_reference_arm_times_the_oracle_on_a_dense_workload(monkeypatch, capsys):
    b = _bench()
    monkeypatch.setenv("RANK", "0")

    class Args:
        config, seed, warmup, steps, gpus, softcap = 1, 0, 0, 1, 1, None

    assert b.reference_arm(Args()) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["workload"] == "cfg1_dense_causal_n128_d64"
    assert "[b0, kv head 0, 128 rows]" in line["cpu_baseline"]["sample"]


def test_roofline_peak_is_sustained_inside_a_long_step_and_burst_otherwise():
    b = _bench()
    peaks = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0}
    # a 34 ms step: the sustained figure, whatever the number of steps
    assert b.roofline_peak(peaks, "measured", 34.0, 3)[:2] == (1800.0, 2000.0)
    # a 0.3 ms step: burst, unless the timed loop itself lasts seconds
    assert b.roofline_peak(peaks, "measured", 0.3, 300)[:2] == (2000.0, 2000.0)
    assert b.roofline_peak(peaks, "measured", 0.3, 5000)[0] == 1800.0
    peak, burst, kind = b.roofline_peak({}, "fallback", 34.0, 3)
    assert (peak, burst) == (b.FALLBACK_BF16_TFLOPS_SUSTAINED, b.FALLBACK_BF16_TFLOPS) and "of fallback" in kind


def test_document_sample_stays_within_its_budget():
    b = _bench()
    from packed_sequence_flash_gb300 import inputs

    w = inputs.config(5, 0)
    Hq, Dqk, Dv = w.q.shape[1], w.q.shape[2], w.v.shape[2]
    per_pair = Hq * (2 * (Dqk + Dv) + 6 * Dqk + 4 * Dv)
    for gflop in (2.0, 6.6, 100.0):
        for offset in (0, 5):
            sub, nd = b.cpu_sample_workload(w, gflop, offset_docs=offset)
            flops = sum(b.doc_pairs(n, w.window) for n in sub.extra["lengths"]) * per_pair
            # whole documents within the budget, or the leading tokens of one
            assert nd >= 1 and (flops <= gflop * 1e9 or len(sub.extra["lengths"]) == 1)
            _, f, bw = b.workload_flops(sub)
            assert f + bw == flops
