"""The N > 1 path on CPU: two gloo ranks on 127.0.0.1.

bench.py runs one replica per GPU (weak scaling): a barrier on each side of
the timed region, the maximum time over ranks, and no collective on the data
path.  These tests run its distributed helpers with world size 2, and check
the property that makes token sharding free ("Efficient Quantization Training
with Stochastic Rounding via Structured Subspace Randomness" §III-B: the
per-token threshold is keyed by the token's global index): each rank
quantizes its own token shard with global indices, and the gathered shards
equal the quantization of the whole tensor on one process.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    import sys
    sys.path.insert(0, ROOT)
    # CPU ranks even on a machine with GPUs (before anything initializes CUDA): gloo, not nccl
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import torch.distributed as dist
    import bench
    import oracle
    w, r, _ = bench.dist_setup(world)
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.0 + rank, w)
    # token shard of a [256, 384] gradient: rows 128 r .. 128 r + 127, thresholds by global token index
    rng = np.random.default_rng(17)
    G = (rng.standard_t(3, size=(256, 384)) * 1e-3).astype(np.float32)
    rows = slice(128 * rank, 128 * (rank + 1))
    out = {}
    for mode in (oracle.S3R, oracle.INDEP, oracle.S3R7):
        Q, delta, _, st = oracle.quantize(G[rows], mode=mode, seed=5, tensor_id=1, window=(128 * rank, 0, 384))
        assert st == 0
        parts = [torch.zeros(128, 384, dtype=torch.int8) for _ in range(world)]
        dist.all_gather(parts, torch.from_numpy(Q))
        out[mode] = torch.cat(parts).numpy()
    bench.barrier(w)
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), slowest=slowest, **{f"m{k}": v for k, v in out.items()})
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_max_time_and_token_sharding(tmp_path):
    import oracle
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True, start_method="spawn")
    rng = np.random.default_rng(17)
    G = (rng.standard_t(3, size=(256, 384)) * 1e-3).astype(np.float32)
    for rank in range(world):
        res = np.load(tmp_path / f"rank{rank}.npz")
        assert float(res["slowest"]) == 2.0   # max over ranks of 1 + rank
        for mode in (oracle.S3R, oracle.INDEP, oracle.S3R7):
            whole, _, _, st = oracle.quantize(G, mode=mode, seed=5, tensor_id=1)
            assert st == 0
            assert np.array_equal(res[f"m{mode}"], whole)
    # the shards really differ from a shard quantized as if it started at token 0
    local, _, _, _ = oracle.quantize(G[128:], mode=oracle.S3R, seed=5, tensor_id=1)
    assert not np.array_equal(local, np.load(tmp_path / "rank1.npz")[f"m{oracle.S3R}"][128:])
