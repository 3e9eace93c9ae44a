"""Host-side multi-rank logic of bench.py on CPU: two gloo ranks, each an
independent replica; the job time is the slowest rank's and the work sums."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    r, w, local = bench.dist_info()
    assert (r, w, local) == (rank, world, rank)
    bench.init_dist(w, "gloo")
    dev = torch.device("cpu")
    my_ms = 10.0 + 5.0 * rank  # rank 1 is the slower replica
    bench.barrier(w)
    slowest = bench.max_over_ranks(my_ms, w, dev)
    work = bench.sum_over_ranks(100.0 * (rank + 1), w, dev)
    bench.barrier(w)
    q.put((rank, slowest, work))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=5) for _ in range(2))
    for rank, slowest, work in out:
        assert slowest == 15.0
        assert work == 300.0


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.sum_over_ranks(2.0, 1, torch.device("cpu")) == 2.0


def test_workload_bytes_and_flops():
    import bench
    from speculative_decoding_draft_05_gb300 import workload

    w = workload.WORKLOADS["verify_r512_g16_v151936"]
    # U_k read (2 B) + scores write (4 B) per element, W2 (2 B per element of r x V), A_k
    assert bench.draft_tile_bytes(w) == 512 * 151936 * 6 + 256 * 151936 * 2 + 512 * 256 * 2
    assert bench.draft_tile_flops(w) == 2 * 512 * 256 * 151936


def test_reference_arm_prints_one_line_on_rank0_only(monkeypatch, capsys):
    import bench

    monkeypatch.setattr(bench, "oracle_inputs", lambda *a, **k: pytest.fail("rank 1 must not work"))
    args = bench.main.__globals__["argparse"].Namespace(steps=1, warmup=3, seed=0)
    w = bench.workload.WORKLOADS["tiny_r4_g4_v1024"]
    bench.run_reference(args, w, rank=1, world=2)
    assert capsys.readouterr().out == ""
