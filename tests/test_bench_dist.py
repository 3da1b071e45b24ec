"""bench.py's multi-process host logic on CPU: two gloo ranks, each timing its
own replica; the job value is the units summed over ranks divided by the
slowest rank's time, and the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    d = bench.Dist()
    try:
        units = 1000.0 * (rank + 1)
        seconds = 2.0 if rank == 0 else 5.0
        value, max_s = bench.combine_ranks(d, units, seconds)
        d.barrier()
        q.put((rank, value, max_s))
    finally:
        d.close()


def test_two_rank_weak_scaling_combine():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, value, max_s in got:
        assert max_s == 5.0
        assert value == pytest.approx(3000.0 / 5.0)


def test_reference_arm_on_tiny_workload(capsys):
    import json

    import bench
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"])
    line = capsys.readouterr().out.strip().splitlines()[-1]
    res = json.loads(line)
    assert res["impl"] == "reference" and res["value"] > 0 and res["unit"] == bench.UNIT
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("workload,metric,unit", [("prefill", "PREFILL_METRIC", "tokens/s"),
                                                  ("prefill_b1", "PREFILL_METRIC", "tokens/s"),
                                                  ("prefill_attn", "PREFILL_ATTN_METRIC", "query tokens/s")])
def test_reference_arm_on_prefill_workloads(capsys, workload, metric, unit):
    """The reference arm of the append and chunked-prefill workloads times the
    oracle on that workload's own metric and unit."""
    import json

    import bench
    bench.main(["--impl", "reference", "--workload", workload, "--steps", "2", "--warmup", "3",
                "--cpu-budget", "0.5"])
    res = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert res["impl"] == "reference" and res["metric"] == getattr(bench, metric) and res["unit"] == unit
    assert res["value"] > 0 and res["cpu_baseline"]["kind"] == "oracle"
    assert res["cpu_baseline"]["value"] == res["value"] and res["e2e"]["h2d_bytes_per_step"] == 0


def test_profiled_traffic_only_for_the_captured_source(tmp_path):
    """A bench line carries a committed capture's DRAM traffic only while the
    kernel source still hashes to the one the capture was taken on."""
    import hashlib

    import bench
    src = tmp_path / "kernel.cu"
    src.write_text("// kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    prof = tmp_path / "summary.md"
    prof.write_text("# capture\n\ntraffic_bytes_per_launch: 1234\ntraffic_bytes_per_launch_nvfp4: 5678\n"
                    f"source_sha256: {sha}\n")
    assert bench.profiled_traffic(str(prof), str(src)) == 1234
    assert bench.profiled_traffic(str(prof), str(src), "traffic_bytes_per_launch_nvfp4") == 5678
    src.write_text("// kernel v2\n")
    assert bench.profiled_traffic(str(prof), str(src)) is None
    assert bench.profiled_traffic(str(tmp_path / "missing.md"), str(src)) is None


def test_committed_captures_match_the_committed_sources():
    """The committed decode, prefill and append summaries were taken on the
    committed kernel sources, so the bench lines carry their traffic."""
    import bench
    assert bench.profiled_traffic(bench.PROFILE, bench.DECODE_SRC) is not None
    assert bench.profiled_traffic(bench.PREFILL_PROFILE, bench.PREFILL_SRC) is not None
    assert bench.profiled_traffic(bench.APPEND_PROFILE, bench.APPEND_SRC) is not None
    assert bench.profiled_traffic(bench.APPEND_PROFILE, bench.APPEND_SRC, "traffic_bytes_per_launch_nvfp4") is not None
