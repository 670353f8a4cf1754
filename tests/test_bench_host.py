"""Host logic of bench.py that needs no GPU: the multi-rank aggregation (two
gloo ranks on CPU), the reference arm's rank rule, the traffic lookup and the
work formulas of the scope table."""
import json
import os
import socket

import pytest

torch = pytest.importorskip("torch")

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, out_dir):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = bench.job_time_ms(local_ms[rank], world, torch.device("cpu"))
        val = bench.job_value(world, 10, ms)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": val}, f)
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank_and_value_counts_every_rank(tmp_path):
    world, port, local_ms = 2, _free_port(), [12.5, 20.0]
    torch.multiprocessing.start_processes(_rank_main, args=(world, port, local_ms, str(tmp_path)), nprocs=world,
                                          join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        assert r["ms"] == 20.0                      # max over ranks, seen by every rank
        assert r["value"] == pytest.approx(2 * 10 / 0.020)   # all ranks' steps / slowest time


def test_single_rank_needs_no_process_group():
    assert bench.job_time_ms(7.0, 1, torch.device("cpu")) == 7.0
    assert bench.job_value(1, 5, 250.0) == pytest.approx(20.0)


def test_reference_arm_runs_on_rank_0_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_traffic_lookup_follows_the_source_hash(tmp_path, monkeypatch):
    import hashlib
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    tf = tmp_path / "traffic.txt"
    tf.write_text(f"# comment\ntraffic key=linear_w4a4 50 1024 1024;source={src.name};sha={sha};bytes=1234\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tf))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_traffic(("linear_w4a4", 50, 1024, 1024)) == 1234.0
    assert bench.read_traffic(("linear_w4a4", 50, 1024, 2048)) is None   # other shape
    src.write_text("kernel v2\n")                                          # kernel changed
    assert bench.read_traffic(("linear_w4a4", 50, 1024, 1024)) is None


def test_work_formulas_match_the_scope_table():
    # one launch: ops 2MNK; bytes as in the scope table's per-call formulas:
    # int4 codes count half a byte each and int8 codes one byte, whatever the
    # storage format (the storage bytes are reported beside them)
    stack = bench.ControlStepStack.__new__(bench.ControlStepStack)
    stack.group = 128
    M, N, K = 50, 1024, 4096
    assert stack.work_of(("linear_w4a4", M, N, K)) == (2 * M * N * K, M * K // 2 + N * K // 2 + 4 * M + 4 * N + 2 * M * N)
    assert stack.work_of(("linear_w8a8", M, N, K)) == (2 * M * N * K, M * K + N * K + 4 * M + 4 * N + 2 * M * N)
    assert stack.work_of(("linear_w4a16", M, N, K)) == (2 * M * N * K, 2 * M * K + N * K // 2 + 4 * N * K // 128
                                                        + 2 * M * N)
    assert stack.work_of(("linear_w4a8", M, N, K)) == (2 * M * N * K, M * K + N * K // 2 + 4 * M + 4 * N + 2 * M * N)
    assert stack.work_of(("linear_w4a4_static", M, N, K)) == (2 * M * N * K, 2 * M * K + N * K // 2 + 4 + 4 * N
                                                              + 2 * M * N)
    assert stack.work_of(("act_quant_static", 4, M, K)) == (0, 2 * M * K + M * K // 2 + 4 * M)
    assert stack.work_of(("act_quant", 8, M, K)) == (0, 2 * M * K + M * K + 4 * M)
    # the storage format: one byte per int4 code, two per int8 code
    assert bench.storage_bytes("act_quant4", M, 0, K) == 2 * M * K + M * K + 4 * M
    assert bench.storage_bytes("linear_w8a8", M, N, K) == 2 * M * K + N * K + 4 * M + 4 * N + 2 * M * N


def test_roofline_takes_the_lower_of_the_two_ceilings():
    # 1 TFLOP over 1 GB: ridge at 6.5 TB/s x 1000 flop/B = 6500 TFLOP/s > a 2000 TFLOP/s peak -> tensor
    r = bench.roofline_of(1e12, 1e9, 1e6, 2000.0, 6500.0)   # 1 s
    assert r["bound"] == "tensor" and abs(r["frac"] - 1.0 / 2000.0) < 1e-12
    # 1 GFLOP over 1 GB: ridge 6.5 TFLOP/s -> HBM; the fraction is then the byte rate's
    r = bench.roofline_of(1e9, 1e9, 1e3, 2000.0, 6500.0)    # 1 ms: 1000 GB/s
    assert r["bound"] == "hbm" and abs(r["frac"] - 1000.0 / 6500.0) < 1e-9
    assert bench.roofline_of(0, 1e9, 1e3, 2000.0, 6500.0)["bound"] == "hbm"