"""The benchmark's multi-rank path (one process per GPU, replicas with no
data-path collective) run as two gloo ranks on the CPU: rank discovery, the
per-rank batch seeds, the barrier, max-over-ranks timing, the whole-job
aggregate and the rule that rank 0 alone prints."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

import bench
from attention_sink_softmax_gb300 import inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, outdir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(ws), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    got_ws, got_rank, got_local = bench.dist_env()
    bench.init_dist(got_ws, "gloo")
    w = inputs.workload(0)
    prob = inputs.make_inputs(w, seed=bench.rank_seed(w, got_rank))
    bench.barrier(got_ws)
    # each rank's step time; the job is as slow as its slowest rank
    ms_local = 2.0 + 3.0 * got_rank
    ms = bench.max_over_ranks(ms_local, got_ws, torch.device("cpu"))
    flops = sum(bench.flops_of(w, w.window))
    value = bench.aggregate_value(flops, got_ws, ms)
    printed = bench.emit({"value": value, "rank": got_rank}, got_rank)
    torch.save({"ws": got_ws, "rank": got_rank, "local": got_local, "ms": ms, "value": value,
                "printed": printed, "q0": prob["q"].flatten()[:8].clone()},
               os.path.join(outdir, f"r{rank}.pt"))
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    ws, port = 2, _free_port()
    mp.spawn(_rank_main, args=(ws, port, str(tmp_path)), nprocs=ws, join=True)
    r = [torch.load(os.path.join(tmp_path, f"r{i}.pt")) for i in range(ws)]
    assert [x["rank"] for x in r] == [0, 1] and all(x["ws"] == 2 for x in r)
    assert [x["local"] for x in r] == [0, 1]
    # max over ranks: both see the slow rank's 5 ms
    assert r[0]["ms"] == r[1]["ms"] == 5.0
    w = inputs.workload(0)
    flops = sum(bench.flops_of(w, w.window))
    assert r[0]["value"] == pytest.approx(flops * 2 / 5e-3 / 1e12)
    # rank 0 alone prints; the line is valid JSON
    assert r[1]["printed"] is None
    assert json.loads(r[0]["printed"])["rank"] == 0
    # replicas draw different batches (weak scaling, no shared data)
    assert not torch.equal(r[0]["q0"], r[1]["q0"])


def test_reference_arm_rank_nonzero_does_no_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    def boom(*a, **k):  # the oracle must not run on rank 1
        raise AssertionError("rank 1 ran the oracle")

    monkeypatch.setattr(bench, "time_oracle", boom)
    args = type("A", (), {"gpus": 2, "steps": 1, "warmup": 0})()
    w = inputs.workload(0)
    bench.run_reference(args, w, w.window)
    assert capsys.readouterr().out == ""


def test_reference_arm_line_matches_gpu_arm_config(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    args = type("A", (), {"gpus": 1, "steps": 1, "warmup": 0})()
    w = inputs.workload(0)
    bench.run_reference(args, w, w.window)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"] == bench.config_of(w, w.window, 1)
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_algorithmic_bytes_and_flops_of_the_target_layer():
    """Per-stage algorithmic bytes and FLOPs of the causal B=2 N=8192 64/8 d=64
    layer: forward reads Q, K, V and writes O, o_lo, LSE (440 MB); the
    preprocess reads O, o_lo, dO, LSE and writes D (411 MB); 4.295e9 unmasked
    pairs."""
    w = inputs.workload(1)
    b = bench.bytes_of(w)
    assert b["fwd"] == 3 * 16384 * 64 * 64 * 2 + 2 * 16384 * 8 * 64 * 2 + 4 * 64 * 16384
    assert round(b["fwd"] / 1e6) == 440 and round(b["bwd_preprocess"] / 1e6) == 411
    assert bench.pairs_of(w, 0) == 2 * 64 * 8192 * 8193 // 2
    f_fwd, f_bwd = bench.flops_of(w, 0)
    assert f_fwd == 4 * 64 * bench.pairs_of(w, 0) and f_bwd == 10 * 64 * bench.pairs_of(w, 0)
    # the window-128 layer's backward sits below the ridge point: HBM-bound
    w2 = inputs.workload(2)
    assert bench.flops_of(w2, 128)[1] / bench.bytes_of(w2)["bwd_main"] < 1926.5e12 / 6688.8e9


_RANK_SCRIPT = """
import os, sys, json, torch
sys.path.insert(0, {root!r})
import bench
ws, rank, local = bench.dist_env()
bench.init_dist(ws, "gloo")
ms = bench.max_over_ranks(1.0 + rank, ws, torch.device("cpu"))
bench.emit({{"ws": ws, "rank": rank, "local": local, "ms": ms}}, rank)
torch.distributed.destroy_process_group()
"""


def test_spawn_ranks_runs_one_process_per_rank(tmp_path, capfd):
    """bench.py --gpus N without a launcher starts N processes itself
    (spawn_ranks): here two gloo ranks of a small script; rank 0 alone prints."""
    script = tmp_path / "rank.py"
    script.write_text(_RANK_SCRIPT.format(root=os.path.dirname(os.path.dirname(
        os.path.abspath(__file__)))))
    env = {"MASTER_ADDR": "127.0.0.1"}
    rc = bench.spawn_ranks(2, [sys.executable, str(script)], env)
    assert rc == 0
    lines = [l for l in capfd.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d == {"ws": 2, "rank": 0, "local": 0, "ms": 2.0}


def test_spawn_ranks_reports_a_failing_rank(tmp_path):
    script = tmp_path / "fail.py"
    script.write_text("import os, sys\nsys.exit(3 if os.environ['RANK'] == '1' else 0)\n")
    assert bench.spawn_ranks(2, [sys.executable, str(script)]) == 3


def test_preparation_overlaps_the_forward_only_without_a_short_window():
    """The bench issues the backward's preparation beside the forward on full
    causal layers and keeps it on the step's stream where a window of at most
    256 keys makes the forward short; --serial-prepare keeps it there always."""
    assert bench.overlaps_preparation(False, 0)
    assert bench.overlaps_preparation(False, 257)
    for window in (1, 128, 256):
        assert not bench.overlaps_preparation(False, window)
    for window in (0, 128, 4096):
        assert not bench.overlaps_preparation(True, window)
