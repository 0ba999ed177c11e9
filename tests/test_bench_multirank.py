"""Host logic of `bench.py --gpus N` on CPU: N processes on the gloo backend.

The layer shards by 128-column blocks with no exchange, so N GPUs run N
independent replicas; what the multi-rank path adds is the rank setup, the
barrier around the timed region, the max over ranks of the timed
milliseconds and the whole-job throughput (all ranks' bytes over the slowest
rank's time). These run here with world size 2 and no GPU; the reference arm's
rule that ranks other than 0 exit without work is checked too.
"""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, ws: int, port: int, ms_by_rank, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(ws), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=ws, init_method=f"tcp://127.0.0.1:{port}")
    try:
        got_ws, got_rank, got_local = bench.dist_env()
        bench.barrier(got_ws)
        ms_max, gbs = bench.whole_job(ms_by_rank[rank], 100, got_ws, torch.device("cpu"))
        bench.barrier(got_ws)
        out[rank] = (got_ws, got_rank, got_local, ms_max, gbs)
    finally:
        dist.destroy_process_group()


def test_two_replicas_time_by_the_slowest_and_sum_their_bytes():
    ws, port = 2, _free_port()
    ms_by_rank = [3.25, 4.5]  # rank 1 is the slow one
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(ws, port, ms_by_rank, out), nprocs=ws, join=True)
    want_gbs = ws * bench.STEP_WEIGHT_BYTES / (max(ms_by_rank) / 1e3 / 100) / 1e9
    for r in range(ws):
        got_ws, got_rank, got_local, ms_max, gbs = out[r]
        assert (got_ws, got_rank, got_local) == (ws, r, r)
        assert ms_max == max(ms_by_rank)  # every rank sees the slowest rank's time
        assert gbs == pytest.approx(want_gbs, rel=1e-12)


def test_one_rank_is_the_plain_single_gpu_number():
    ms_max, gbs = bench.whole_job(4.0, 100, 1, torch.device("cpu"))
    assert ms_max == 4.0
    assert gbs == pytest.approx(bench.STEP_WEIGHT_BYTES / (4.0e-3 / 100) / 1e9, rel=1e-12)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        steps, warmup = 1, 3

    assert bench.run_reference(Args()) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_reports_the_gpu_arms_workload(monkeypatch, capsys):
    # rank 0 alone, on two of the step's blocks so that the test stays short
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    blocks = bench._step_blocks()
    assert len(blocks) == sum(bench.QKV + (bench.O_N,)) // 128
    assert blocks[0] == (0, bench.QKV[0], 0) and blocks[-1] == (3, bench.O_N, bench.O_N // 128 - 1)
    monkeypatch.setattr(bench, "_step_blocks", lambda: blocks[47:49])  # last q block, first k block

    class Args:
        steps, warmup = 2, 3

    assert bench.run_reference(Args()) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    assert {k: line["config"][k] for k in bench.step_config(1)} == bench.step_config(1)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["cpu_baseline"]["value"] == line["value"] == line["e2e"]["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
