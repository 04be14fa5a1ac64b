"""Host-side logic of bench.py (CPU only): algorithmic byte/flop counts and the
max-over-ranks / sum-over-ranks aggregation, run as two gloo ranks."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_algorithmic_counts():
    # decode: packed + scales + x + fp32 logits (N=128256, K=4096)
    assert bench.decode_bytes(1) == 128256 * 2048 + 128256 * 256 + 2 * 4096 + 4 * 128256
    assert abs(bench.decode_bytes(1) / 1e6 - 296.0) < 0.5
    assert abs(bench.decode_bytes(64) / 1e6 - 328.9) < 0.5
    # quantizer: two reads of W plus codes, scales and the global scale
    assert bench.quant_bytes(151936, 5120) == 3549224964
    assert abs(bench.prefill_flops() / 1e12 - 2.152) < 0.001


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t, u = bench.aggregate(elapsed_s=1.0 + rank, units=10.0 * (rank + 1), world=world)
        out[rank] = (t, u)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: (2.0, 30.0), 1: (2.0, 30.0)}


def test_single_rank_passthrough():
    assert bench.aggregate(1.5, 7.0, world=1) == (1.5, 7.0)
