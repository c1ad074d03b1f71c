"""Host-side multi-rank logic of bench.py on CPU: two gloo ranks.

Each GPU would run its own replica of the step (weak scaling, no collective on
the data path); the only cross-rank traffic is the barrier around the timed
region and the max over ranks of the measured times.  This checks that logic
with world_size 2 over gloo, rendezvous on 127.0.0.1.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        got = bench.reduce_max_over_ranks(10.0 + rank)
        results[rank] = got
        bench.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of this multi-threaded process
        results = m.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        assert dict(results) == {0: 11.0, 1: 11.0}


def test_single_process_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.reduce_max_over_ranks(3.5) == 3.5


@pytest.mark.parametrize("warmup", [0, 2])
def test_bench_rejects_short_warmup(warmup):
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--warmup", str(warmup)])


def test_traffic_entry_follows_kernel_code_not_comments(tmp_path):
    # The committed ncu traffic is used only while its kernel's code is the one
    # measured: a comment edit keeps the entry, a code edit drops it.
    import bench
    src = tmp_path / "k.cu"
    src.write_text("// kernel\n__global__ void k(int *p) { p[0] = 1; }  /* store */\n")
    h = bench.source_hash(str(src))
    src.write_text("// the kernel, reworded\n__global__ void k(int *p) {\n    p[0] = 1;\n}\n")
    assert bench.source_hash(str(src)) == h
    src.write_text("__global__ void k(int *p) { p[0] = 2; }\n")
    assert bench.source_hash(str(src)) != h
    with open(bench.TRAFFIC_PATH) as f:
        import json
        table = json.load(f)
    # entries are keyed by workload, each a whole launch's DRAM bytes
    name = "gqa_causal_4x32q8kv_4096"
    assert table[name]["bytes_per_launch"] > 0
    assert bench.traffic_for(name, str(src)) is None
    assert bench.traffic_for("no_such_workload", bench.PREFILL_KERNEL_SRC) is None
