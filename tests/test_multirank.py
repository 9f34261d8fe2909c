"""Multi-rank host logic on CPU with gloo (world_size 2): the bench's
max-over-ranks timing and whole-job throughput, and batch-row sharding of the
commit step (each rank computes its shard; the gathered result equals the
unsharded one).  No GPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _timing_worker(rank, world, port, q):
    import bench

    _init(rank, world, port)
    local_ms = [12.0, 20.0][rank]
    m = bench.max_over_ranks(local_ms, torch.device("cpu"), world)
    v = bench.whole_job_gbs(1_000_000_000, 10, world, m)
    q.put((rank, m, v))
    dist.destroy_process_group()


def _shard_worker(rank, world, port, q):
    import oracle
    from commit_step_gb300.shard import shard_batch_rows

    _init(rank, world, port)
    rng = np.random.default_rng(5)
    B, L, V = 5, 6, 300
    z = (rng.standard_normal((B * L, V)) * 3).astype(np.float32)
    cand = (rng.random((B, L)) < 0.6).astype(np.uint8)
    b0, b1 = shard_batch_rows(B, rank, world)
    x0, p, h = oracle.token_stats(z[b0 * L:b1 * L], suppress_ids=[0])
    commit = oracle.threshold_transfer(p.astype(np.float32).reshape(b1 - b0, L), cand[b0:b1], 0.5)
    local = torch.from_numpy(np.concatenate([x0.astype(np.float64), p, commit.reshape(-1).astype(np.float64)]))
    sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(sizes, torch.tensor([local.numel()]))
    parts = [torch.zeros(int(n.item()), dtype=torch.float64) for n in sizes]
    padded = max(int(n.item()) for n in sizes)
    buf = [torch.zeros(padded, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(buf, torch.nn.functional.pad(local, (0, padded - local.numel())))
    if rank == 0:
        full_x0, full_p, full_h = oracle.token_stats(z, suppress_ids=[0])
        full_c = oracle.threshold_transfer(full_p.astype(np.float32).reshape(B, L), cand, 0.5)
        got_x0, got_p, got_c = [], [], []
        for r in range(world):
            c0, c1 = shard_batch_rows(B, r, world)
            n = (c1 - c0) * L
            v = buf[r][: int(sizes[r].item())].numpy()
            got_x0.append(v[:n]), got_p.append(v[n:2 * n]), got_c.append(v[2 * n:3 * n])
        ok = (np.array_equal(np.concatenate(got_x0), full_x0) and np.array_equal(np.concatenate(got_p), full_p)
              and np.array_equal(np.concatenate(got_c), full_c.reshape(-1)))
        q.put(ok)
    dist.destroy_process_group()


def _spawn(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=fn, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    out = []
    while not q.empty():
        out.append(q.get())
    return out


def test_bench_timing_takes_the_slowest_rank():
    res = sorted(_spawn(_timing_worker))
    assert [r[1] for r in res] == [20.0, 20.0]
    # 2 ranks x 10 steps x 1 GB over 20 ms
    assert res[0][2] == pytest.approx(2 * 10 * 1.0 / 0.020)


def test_batch_row_sharding_matches_unsharded():
    assert _spawn(_shard_worker) == [True]


def test_shard_bounds_cover_every_row_once():
    from commit_step_gb300.shard import shard_batch_rows

    for B in range(0, 40):
        for world in range(1, 9):
            rows = []
            for r in range(world):
                b0, b1 = shard_batch_rows(B, r, world)
                rows.extend(range(b0, b1))
            assert rows == list(range(B))
    with pytest.raises(ValueError):
        shard_batch_rows(4, 2, 2)
