"""Host logic of bench.py's multi-GPU line (replicas only): the barrier and
the max over ranks, run as two gloo ranks on the CPU."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    # each replica times its own work; the line reports the slowest rank
    out[rank] = bench.max_over_ranks(10.0 + rank, w)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        assert dict(out) == {0: 11.0, 1: 11.0}


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_round_bytes_matches_the_analytic_count():
    """3.43 GB per bs1 round at ctx 4096 with 4 held rows (weights 3.34 GB,
    context K/V 84 MB, logits and features the rest)."""
    import bench
    import synthetic as S
    rb = bench.round_bytes(S.CONFIGS["qwen3_8b_bf16"], 4096, 4)
    assert 3.40e9 < rb < 3.46e9
