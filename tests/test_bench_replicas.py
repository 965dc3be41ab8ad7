"""The multi-GPU form of the benchmark runs independent replicas (no data-path
collective): its only cross-rank step is the max over ranks of the timed
region. Checked here with two gloo ranks on the CPU, and the JSON line's
host-side pieces without a GPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 * (rank + 1)          # rank 1 is the slow one
    total, value = bench.whole_job(local_ms, 4096 * 5, world, device="cpu")
    out[rank] = (total, value)
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    for rank in range(world):
        total, value = res[rank]
        assert total == pytest.approx(20.0)
        # all ranks' tokens over the slowest rank's time
        assert value == pytest.approx(2 * 4096 * 5 / 0.020)


def test_single_rank_needs_no_collective():
    total, value = bench.whole_job(8.0, 1000, 1)
    assert total == 8.0 and value == pytest.approx(1000 / 0.008)


def test_workload_bytes_and_launch_counts():
    s = bench.workload_spec("prefill")
    k, h = 8, 7168
    assert s["bytes_per_token"]["dispatch"] == 2 * h + 12 * k + k * 7472
    assert s["bytes_per_token"]["combine"] == k * 2 * h + 12 * k + 2 * h
    assert bench.layout_launches(4096, 8, 256, 8) == 1
    assert bench.layout_launches(100000, 8, 256, 8) == 2  # beyond the cluster's shared memory
    # layout and dispatch as one kernel up to 2048 pairs (tiny, decode N <= 256)
    assert bench.single_kernel_layout_dispatch(128, 2, 16)
    assert bench.single_kernel_layout_dispatch(256, 8, 256)
    assert not bench.single_kernel_layout_dispatch(257, 8, 256)
    assert not bench.single_kernel_layout_dispatch(4096, 8, 256)
    sn = bench.workload_spec("prefill_norm")
    assert sn["bytes_per_token"]["combine"] == s["bytes_per_token"]["combine"] + 4 * h


def test_reference_arm_prints_a_line(capsys):
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3",
                "--cpu-seconds", "0.5"])
    import json
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["cores"] == bench.host_cores()
    assert line["cpu_baseline"]["value"] == line["value"]


@pytest.mark.parametrize("name,tokens,parts", [("prefill", 4096, 32), ("decode", 1000, 7),
                                               ("decode_ll", 5000, 16), ("prefill_bwd", 64, 4)])
def test_oracle_chunks_are_whole_rank_multiples(name, tokens, parts):
    spec = bench.workload_spec(name)
    n, r = spec["num_tokens"], spec["num_ranks"]
    chunks = bench.oracle_chunks(spec, tokens, parts)
    sizes = {t1 - t0 for t0, t1 in chunks}
    assert len(sizes) == 1 and all(s % r == 0 and 0 < s <= n for s in sizes)
    assert all(0 <= t0 < t1 <= n for t0, t1 in chunks)
    assert sum(t1 - t0 for t0, t1 in chunks) >= tokens


def test_all_cores_baseline_runs_the_oracle_in_spawned_workers():
    # two workers on a workload with a cheap oracle pass
    spec = bench.workload_spec("tiny")
    pool = bench.OraclePool(spec, 2)
    try:
        done = pool.run(bench.oracle_chunks(spec, 64, 4))
    finally:
        pool.close()
    assert done == 64


def test_routing_stats_from_layout_counts():
    """The bench line's load-balance summary of a routing: pairs per expert
    (max, mean, max/mean, empty experts) and tokens per rank."""
    import torch
    import bench
    got = bench.routing_stats(torch.tensor([0, 5, 3, 0], dtype=torch.int32),
                              torch.tensor([6, 2], dtype=torch.int32))
    assert got == {"pairs_per_expert_max": 5, "pairs_per_expert_mean": 2.0,
                   "expert_load_max_over_mean": 2.5, "empty_experts": 2,
                   "tokens_per_rank_max": 6, "tokens_per_rank_mean": 4.0}
    none = bench.routing_stats(torch.zeros(4, dtype=torch.int32), torch.zeros(2, dtype=torch.int32))
    assert none["expert_load_max_over_mean"] is None and none["empty_experts"] == 4


def test_tokens_override_is_checked():
    """--tokens takes only workloads with a free N, and a multiple of their ranks."""
    with pytest.raises(SystemExit):
        bench.main(["--workload", "tiny", "--tokens", "64"])
    with pytest.raises(SystemExit):
        bench.main(["--workload", "skewed", "--tokens", "1000"])  # R = 16
