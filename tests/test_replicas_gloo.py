"""World-size-2 gloo run of the replica path on CPU: each rank takes its
slice of the requests, works on it alone, and the job time is the maximum
over ranks.  The union of the per-rank results equals the single-process
result, which holds because requests never interact."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from block_speculative_decoding_ctx_gb300 import replicas


def test_partition_covers_every_request_once():
    for n in (0, 1, 7, 16, 33):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                a, b = replicas.partition(n, world, r)
                seen.extend(range(a, b))
                assert b - a in (n // world, n // world + 1)
            assert seen == list(range(n))
    with pytest.raises(ValueError):
        replicas.partition(4, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import verify as over
    rng = np.random.default_rng(0)
    B, gamma, V = 9, 6, 50
    t = rng.normal(size=(B, gamma, V)).astype(np.float32)
    y = t[:, :gamma - 1].argmax(-1)
    y[::2, 2] = (y[::2, 2] + 1) % V
    a, b = replicas.partition(B, world, rank)
    n, tok = over.greedy(t[a:b], y[a:b])
    np.save(os.path.join(out_dir, f"n{rank}.npy"), n)
    np.save(os.path.join(out_dir, f"t{rank}.npy"), tok)
    slow = replicas.max_over_ranks(1.0 + rank)
    np.save(os.path.join(out_dir, f"m{rank}.npy"), np.array([slow]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_match_single_process(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    from oracle import verify as over
    rng = np.random.default_rng(0)
    B, gamma, V = 9, 6, 50
    t = rng.normal(size=(B, gamma, V)).astype(np.float32)
    y = t[:, :gamma - 1].argmax(-1)
    y[::2, 2] = (y[::2, 2] + 1) % V
    n_all, tok_all = over.greedy(t, y)
    n = np.concatenate([np.load(tmp_path / f"n{r}.npy") for r in range(2)])
    tok = np.concatenate([np.load(tmp_path / f"t{r}.npy") for r in range(2)])
    np.testing.assert_array_equal(n, n_all)
    np.testing.assert_array_equal(tok, tok_all)
    assert all(float(np.load(tmp_path / f"m{r}.npy")[0]) == 2.0 for r in range(2))
    assert replicas.job_throughput([5, 4], [1.0, 2.0]) == 4.5


def _bench_worker(rank, world, port, out_dir):
    """One replica rank driven through bench.py's own helpers: its slice of
    the job's requests, its own (oracle) verification of them, and the job
    figure from the slowest rank's time."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from oracle import verify as over
    r, ws = bench.dist_setup(backend="gloo")
    assert (r, ws) == (rank, world)
    B, gamma, V = 5, 6, 50                       # requests per rank (weak scaling)
    rng = np.random.default_rng(1)
    t = rng.normal(size=(B * world, gamma, V)).astype(np.float32)
    y = t[:, :gamma - 1].argmax(-1)
    y[1::3, 1] = (y[1::3, 1] + 1) % V
    a, b = bench.replica_requests(B, rank, ws)
    n, tok = over.greedy(t[a:b], y[a:b])
    ms = 2.0 + 3.0 * rank                         # this rank's step time
    ms_max = bench.max_over_ranks(ms, ws)
    bench.barrier(ws)
    np.save(os.path.join(out_dir, f"bn{rank}.npy"), n)
    np.save(os.path.join(out_dir, f"bt{rank}.npy"), tok)
    np.save(os.path.join(out_dir, f"bv{rank}.npy"), np.array([a, b, ms_max, bench.job_value(B, ws, ms_max)]))
    dist.destroy_process_group()


def test_bench_replica_path_on_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_bench_worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    from oracle import verify as over
    B, gamma, V = 5, 6, 50
    rng = np.random.default_rng(1)
    t = rng.normal(size=(2 * B, gamma, V)).astype(np.float32)
    y = t[:, :gamma - 1].argmax(-1)
    y[1::3, 1] = (y[1::3, 1] + 1) % V
    n_all, tok_all = over.greedy(t, y)
    v = [np.load(tmp_path / f"bv{r}.npy") for r in range(2)]
    assert [(int(x[0]), int(x[1])) for x in v] == [(0, B), (B, 2 * B)]
    np.testing.assert_array_equal(np.concatenate([np.load(tmp_path / f"bn{r}.npy") for r in range(2)]), n_all)
    np.testing.assert_array_equal(np.concatenate([np.load(tmp_path / f"bt{r}.npy") for r in range(2)]), tok_all)
    for x in v:
        assert x[2] == 5.0                        # the slowest rank's time on every rank
        assert x[3] == pytest.approx(2 * B / 5.0e-3)  # all requests over the slowest time


def test_bench_gpus_flag_against_world_size(monkeypatch):
    import argparse
    import bench
    monkeypatch.setenv("WORLD_SIZE", "1")
    assert bench.spawn_replicas(argparse.Namespace(gpus=2)) == 2   # mismatch is an error
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.spawn_replicas(argparse.Namespace(gpus=2)) is None
    monkeypatch.delenv("WORLD_SIZE")
    assert bench.spawn_replicas(argparse.Namespace(gpus=1)) is None
