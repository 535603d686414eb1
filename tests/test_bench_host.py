"""Host logic of bench.py: replica aggregation over torch.distributed (gloo,
world size 2, CPU) and the workload accounting."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
import synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    units, secs = bench.aggregate(100.0 * (rank + 1), 0.5 + rank)
    q.put((rank, units, secs))
    dist.destroy_process_group()


def test_aggregate_sums_units_and_takes_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, units, secs in res:
        assert units == 300.0 and secs == 1.5


def test_single_process_aggregate_is_identity():
    assert bench.aggregate(5.0, 2.0) == (5.0, 2.0)


def test_workload_accounting():
    cfg = bench.config_dict()
    assert cfg["workload"] == "gpt2_small_mlp_backward"
    wl = synth.WORKLOADS["mlp"]
    assert cfg["flops_per_step"] == sum(4 * l.BT * l.C * l.OC + l.BT * l.OC for l in wl.layers)
    assert sum(bench.layer_bytes(l) for l in wl.layers) * bench.N_SETS > 129e6 * 2


def test_traffic_is_null_for_a_changed_kernel(tmp_path, monkeypatch):
    # a summary taken on another kernel source must not be reported
    assert bench.kernel_source_sha() and len(bench.kernel_source_sha()) == 12
    prof = os.path.join(bench.ROOT, "profiles", "tc_mmbwd_kernel_mlp.md")
    if os.path.exists(prof):
        t = bench.profiled_traffic()
        assert t is None or t > 0
