"""Host logic of bench.py: the max-over-ranks time and summed work of N replicas
(gloo, world size 2, CPU only), Eq. 7-10 arithmetic of a bench step."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), DG_BENCH_BACKEND="gloo")
    w, r, local, pg = bench.dist_setup()
    t = bench.reduce_over_ranks(pg, 10.0 + 5 * rank, "max")     # per-rank times 10, 15
    s = bench.reduce_over_ranks(pg, 100 * (rank + 1), "sum")    # per-rank steps 100, 200
    q.put((r, w, t, s))
    dist.destroy_process_group()


def test_two_replicas_reduce_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for r, w, t, s in res:
        assert w == 2 and t == 15.0 and s == 300.0


def test_single_rank_is_identity():
    assert bench.reduce_over_ranks(None, 3.5, "max") == 3.5


def test_expert_bytes_formula():
    import discrete_diffusion_block_gb300 as dgp
    b = bench.expert_bytes(dgp.full_config(), 128, 2048)
    weights = 128 * (1408 * 2816 + 2816 * 704) * 2          # gate/up and down of 128 experts
    rows = 2048 * 2816 * 2 + 2 * 2048 * 704 * 2 + 2048 * 2816 * 2  # x in, act out and in, y out (bf16)
    assert b == {"expert_ffn": weights + rows}
