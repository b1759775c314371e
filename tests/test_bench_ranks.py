"""The benchmark's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

bench.py runs one independent replica per GPU (the decode step shards by
sequence and has no collective); the job's time is the slowest rank's and its
throughput counts every rank's work. Both rules are checked here without a GPU.
"""
import os
import socket

import pytest

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's own total step time; the job takes the slowest
        q.put((rank, bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert got == [(0, 15.0), (1, 15.0)]
    assert all(p.exitcode == 0 for p in procs)


def test_max_over_ranks_is_identity_on_one_rank():
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25


@pytest.mark.parametrize("world", [1, 2, 4, 8])
def test_job_rate_counts_every_rank(world):
    # 1000 units per rank in a 2 ms step: world * 500,000 units/s
    assert bench.job_rate(world, 1000, 2.0) == pytest.approx(world * 5.0e5)


def test_algorithmic_bytes_by_hand():
    """The roofline numerators, counted by hand for the DeepSeek-V3 shape."""
    import bench
    from mla_latent_kv_16_gb300 import workloads as W
    w = W.preset("dsv3_bf16")
    # decode: 32 x 4096 rows of 1152 B, q (576 bf16 per head), u (512 bf16) + lse (fp32) per head
    assert bench.decode_bytes(w) == 32 * 4096 * 1152 + 32 * 128 * 576 * 2 + 32 * 128 * (512 * 2 + 4)
    # fused output projection: W~ 7168 x 65536, u 32 x 65536, y 32 x 7168, all bf16
    assert bench.fused_bytes(32, 7168, 128) == 2 * (7168 * 65536 + 32 * 65536 + 32 * 7168)
    assert bench.fused_bytes(32, 7168, 128) == 944_177_152
    # whole layer: W_DQKV, W_UQR, W_UK, W~ once, the cache rows, and the step's activations
    weights = 2 * (2112 * 7168 + 24576 * 1536 + 128 * 128 * 512 + 7168 * 65536)
    acts = 2 * 32 * (7168 + 128 * (128 + 64 + 512 + 512) + 576 + 7168)
    assert bench.layer_bytes(w, 7168, 1536) == weights + 32 * 4096 * 1152 + acts
    # E4M3 rows carry 576 B of codes and 20 B of scales
    assert W.preset("fp8_lq2").row_bytes() == 596
