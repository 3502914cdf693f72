"""bench.py host logic on the CPU: the multi-rank timing reduction with two
gloo ranks, the throughput formula, the algorithmic work per stage and the
reference arm on the tiny workload."""
import contextlib
import io
import json
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench
import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    bench.dist_init(world, "gloo")
    seconds = [0.25, 0.40][rank]            # rank 1 is the slow one
    bench.barrier(world)
    slowest = bench.max_over_ranks(seconds, world, device="cpu")
    value = bench.job_throughput(1000, world, slowest)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as fh:
        json.dump({"slowest": slowest, "value": value}, fh)
    torch.distributed.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        res = json.load(open(tmp_path / f"r{r}.json"))
        assert res["slowest"] == pytest.approx(0.40)
        assert res["value"] == pytest.approx(2 * 1000 / 0.40)


def test_single_rank_reduction_is_identity():
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.job_throughput(16384 * 100, 1, 0.778) == pytest.approx(16384 * 100 / 0.778)


def test_stage_work_of_the_1t_layer():
    cfg = workloads.get("t1")
    w = bench.stage_work(cfg)
    P = 16384 * 8
    assert w["gate_up"]["flops"] == 4 * P * 6144 * 1792 == 5_772_436_045_824
    assert w["down"]["flops"] == 2 * P * 6144 * 1792
    assert w["permute"]["bytes"] == 16384 * 6144 * 2 + P * 6144 * 2 + P * 4
    assert w["combine"]["bytes"] == P * 6144 * 2 + 16384 * 6144 * 2 + P * 8   # rows, out, dest_row, gates
    assert bench.weight_bytes_read(cfg, [1] * 384) == 384 * 3 * 6144 * 1792 * 2


def test_peaks_fall_back_when_unmeasured(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6800.0


def test_reference_arm_prints_one_json_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"])
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "tokens/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0
    assert rec["warmup"] >= 3


def test_backward_gemm_work_of_the_1t_layer():
    """Recomputed gate/up (4 P d f; the down projection is not recomputed) +
    two dgrad (6 P d f) + two wgrad (6 P d f)."""
    cfg = workloads.get("t1")
    fl = bench.backward_gemm_flops(cfg)
    P = 16384 * 8
    assert "recompute_down" not in fl
    assert sum(fl.values()) == 16 * P * 6144 * 1792
    assert fl["dgrad_gate_up"] == fl["wgrad_gate_up"] == fl["recompute_gate_up"] == 4 * P * 6144 * 1792


def test_bench_uses_only_names_the_binding_exports():
    """Every moe.<name> that bench.py calls exists in the package (caught here,
    on the CPU, rather than after a GPU run)."""
    import re
    moe = pytest.importorskip("sparse_expert_gb300")
    entry = os.path.join(os.path.dirname(bench.__file__), "__graft_entry__.py")
    names = set(re.findall(r"\bmoe\.(\w+)", open(bench.__file__).read() + open(entry).read()))
    assert names, "no binding calls found"
    missing = sorted(n for n in names if not hasattr(moe, n))
    assert not missing, missing


def _stub_arm(args):
    """Stands in for the GPU arm: the same rank environment, barrier, max over
    ranks and throughput formula, with gloo and made-up times."""
    world, rank, _ = bench.dist_env()
    bench.dist_init(world, "gloo")
    seconds = 0.1 * (rank + 1)              # the last rank is the slowest
    bench.barrier(world)
    slowest = bench.max_over_ranks(seconds, world, device="cpu")
    if rank == 0:
        print(json.dumps({"n_gpus": world, "steps": args.steps,
                          "value": bench.job_throughput(1000 * args.steps, world, slowest)}), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def test_gpus_flag_starts_one_rank_per_gpu(capfd, monkeypatch):
    for var in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    bench.main(["--gpus", "2", "--steps", "3"], arm=_stub_arm)
    lines = [json.loads(l) for l in capfd.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1, lines
    assert lines[0]["n_gpus"] == 2 and lines[0]["steps"] == 3
    assert lines[0]["value"] == pytest.approx(2 * 3000 / 0.2)


def test_gpus_flag_must_match_the_launcher(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "4")
    with pytest.raises(SystemExit, match="WORLD_SIZE=4"):
        bench.main(["--gpus", "2"], arm=_stub_arm)


def test_one_gpu_runs_in_process(capfd, monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench.main(["--steps", "2"], arm=_stub_arm)
    lines = [json.loads(l) for l in capfd.readouterr().out.splitlines() if l.startswith("{")]
    assert lines == [{"n_gpus": 1, "steps": 2, "value": pytest.approx(2000 / 0.1)}]
