"""The multi-rank host logic of bench.py on the CPU: N > 1 runs independent
replicas of the layer (no collective on the data path), and the job reports
the tokens of all ranks over the slowest rank's time.  World size 2 over
gloo on 127.0.0.1, one spawned process per rank."""

import argparse
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from llama_decoder_layer_prologue_b300 import synth


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        env = bench.dist_env()
        # rank r's replica took 10 + 5 r ms for its steps
        slow = bench.max_over_ranks(dist, 10.0 + 5.0 * rank)
        dist.barrier()
        q.put((rank, env, slow, bench.job_throughput(world, 100, 8192, slow)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, slow, tput in got:
        assert env == (rank, rank, 2)
        assert slow == 15.0  # every rank sees the slowest replica's time
        assert tput == 2 * 100 * 8192 / 0.015  # both ranks' tokens


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(None, 12.5) == 12.5
    assert bench.job_throughput(1, 10, 64, 2.0) == 10 * 64 / 0.002


def test_reference_arm_runs_on_rank_zero_only():
    args = argparse.Namespace(workload="1b", steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args, rank=1, world=2) is None


def test_gpus_flag_needs_a_matching_world():
    """`--gpus N` with N > 1 must come from torchrun (one process per GPU):
    a single process asked for 2 GPUs refuses instead of timing one replica
    and reporting it as two."""
    import pytest

    bench.check_world(1, 1)
    bench.check_world(2, 2)
    with pytest.raises(SystemExit, match="WORLD_SIZE=1"):
        bench.check_world(2, 1)
    with pytest.raises(SystemExit):
        bench.check_world(1, 4)


def test_headline_also_runs_the_other_layer_workloads():
    ns = lambda **kw: argparse.Namespace(**{"workload": bench.HEADLINE, "also": "auto",
                                           **kw})
    assert bench.also_list(ns()) == list(bench.ALSO_AUTO)
    assert "bwd_8b" in bench.ALSO_AUTO and "decode" in bench.ALSO_AUTO
    assert bench.also_list(ns(workload="1b")) == []
    assert bench.also_list(ns(also="none")) == []
    assert bench.also_list(ns(also="8b,varlen")) == ["8b"]


def test_split_kv_route_follows_the_library():
    """The bench's label of the chunked attention follows the library's
    route: split-KV while a sequence's new tokens form at most two groups of
    16 / n_rep, else the tensor-core attention over the cache."""
    s8 = synth.WORKLOADS["8b"].shape  # 4 query heads per kv head: groups of 4
    assert [bench.split_kv_attention(s8, S) for S in (1, 4, 8, 9, 12, 15)] == \
        [True, True, True, False, False, False]
    mha = synth.custom_workload("m", synth.WORKLOADS["tiny"].shape, "decode").shape
    assert mha.n_heads // mha.n_kv_heads == 2  # groups of 8
    assert bench.split_kv_attention(mha, 15) and not bench.split_kv_attention(mha, 17)
