"""Host-side logic of bench.py: byte accounting, weak-scaling reductions over
ranks (gloo, world size 2, on CPU) and the reference arm's JSON line."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from workloads import configs


def test_hbm_bytes_per_resolve_by_hand():
    k, B, m, W = 2048, 4096, 267, 1152
    reads = 4 * k + 4 * B + 2 * B            # selections, slot map, LRU order
    writes = 4 * k + 4 * k + 4 * m + 8 * m + 2 * B + m * W
    assert bench.hbm_bytes_per_resolve(k, B, m, W) == reads + writes


def test_hbm_sector_bytes_per_resolve_against_a_count_of_sectors():
    import numpy as np
    k, B, m, W = 2048, 4096, 267, 1152
    got = bench.hbm_sector_bytes_per_resolve(k, B, m, W)
    # stamp writes: the 32-byte sectors (8 slots each) of k distinct slots,
    # counted on random slot sets
    rng = np.random.default_rng(3)
    touched = np.mean([len(np.unique(rng.choice(B, k, replace=False) // 8))
                       for _ in range(200)])
    reads = 4 * k + 4 * B + 2 * B + 32 * k   # + one sector per page-table read
    writes = 4 * k + 32 * touched + 32 * m + 64 * m + 2 * B + m * W
    assert abs(got - (reads + writes)) <= 0.002 * got
    # with every slot selected the stamp array is written whole
    assert bench.hbm_sector_bytes_per_resolve(B, B, 0, W) == (
        4 * B + 4 * B + 2 * B + 32 * B + 4 * B + 4 * B + 2 * B)


def test_attention_bytes_by_hand():
    R, k, heads = 64, 2048, 16
    assert bench.attention_bytes(R, k, heads) == (
        R * k * 1152 + R * k * 4 + R * heads * 1152 + R * heads * 512 * 4)


def test_attention_heads_bytes_by_hand():
    R, k, heads = 32, 2048, 8
    assert bench.attention_heads_bytes(R, k, heads) == (
        R * k * 8 * 512 + R * k * 4 + R * heads * 128 * 2 + R * heads * 128 * 4)


def test_rank_workloads_differ_only_in_seed():
    a, b = bench.rank_workload(configs.DSA_MLA, 0), bench.rank_workload(configs.DSA_MLA, 1)
    assert a.seed != b.seed
    assert a.with_(seed=0) == b.with_(seed=0) == configs.DSA_MLA


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.reduce_max(1.5 + rank, True)      # per-rank time
    n = bench.reduce_sum(100.0 * (rank + 1), True)   # per-rank resolves
    dist.barrier()
    if rank == 0:
        q.put((t, n, n / t))
    dist.destroy_process_group()


def test_weak_scaling_reduction_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, q), nprocs=2, join=True, start_method="spawn")
    t, n, v = q.get(timeout=30)
    assert t == 2.5          # the slowest rank's time
    assert n == 300.0        # all ranks' resolves
    assert v == pytest.approx(120.0)


def test_single_rank_reductions_are_identity():
    assert bench.reduce_max(3.0, False) == 3.0
    assert bench.reduce_sum(3.0, False) == 3.0


def test_reference_arm_json(capsys):
    rc = bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "5",
                     "--warmup", "3", "--cpu-threads", "2"])
    assert rc == 0
    line = capsys.readouterr().out.strip().splitlines()[-1]
    d = json.loads(line)
    assert d["impl"] == "reference" and d["unit"] == "resolves/s" and d["value"] > 0
    # tiny has one (request, layer) pair: one of the two threads does the work
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["higher_is_better"] is True


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--impl", "reference", "--warmup", "2"])


def test_gpu_arm_refuses_without_cuda():
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(SystemExit):
        bench.main(["--steps", "3", "--warmup", "3"])


def test_gpus_flag_spawns_one_process_per_rank(capfd, monkeypatch):
    """`bench.py --gpus 2` run as a single process re-runs itself under
    torch.distributed.run with two ranks (rendezvous on 127.0.0.1); rank 0
    prints the one JSON line and both exit 0 (here through the reference
    arm, which needs no GPU)."""
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    rc = bench.main(["--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "4",
                     "--warmup", "3", "--cpu-threads", "1"])
    assert rc == 0
    out = capfd.readouterr().out
    lines = [x for x in out.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0


def test_parse_cpulist():
    assert bench.parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench.parse_cpulist("") == set()


def test_bind_without_device_reports_no_node():
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert bench.bind_to_device_numa(0) == (None, None)


def test_step_time_summary():
    st = bench.step_time_summary([1.0, 0.99, 1.5, 0.98, 2.0], 512)
    assert st["min"] == 0.98 and st["median"] == 1.0 and st["max"] == 2.0
    assert abs(st["resolves_per_s_at_median"] - 512 / 1e-3) < 1e-6
    assert st["min"] <= st["p90"] <= st["max"]
    assert bench.step_time_summary([], 512) is None
