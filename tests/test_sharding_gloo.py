"""Data-parallel sharding by request, checked with two gloo ranks on the CPU.

Each rank runs the oracle's step on its request shard; rank 0 gathers the
shards' outputs and checks that, concatenated, they equal the step on the
whole batch.  Nothing is exchanged on the data path: the only collective is
the gather the test uses to compare results.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _caches(w):
    from paged_sparse_kv_gb300 import synthetic
    return {name: (None if getattr(w, name) is None else
                   synthetic.random_cache_bytes(70 + i, getattr(w, name)))
            for i, name in enumerate(("swa_cache", "comp_cache", "index_cache"))}


def _worker(rank, world, port, name, result_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle.pipeline import run_step
        from paged_sparse_kv_gb300 import synthetic
        from paged_sparse_kv_gb300.sharding import shard_requests
        w = synthetic.make(name)
        sub, t0, t1 = shard_requests(w, rank, world)
        c = _caches(w)  # same initial caches on every rank
        res = run_step(sub, c["swa_cache"], c["comp_cache"], c["index_cache"])
        payload = {k: v for k, v in res.items() if isinstance(v, np.ndarray)}
        payload["span"] = np.array([t0, t1])
        gathered = [None] * world if rank == 0 else None
        dist.gather_object(payload, gathered, dst=0)
        if rank == 0:
            full = run_step(w, *(_caches(w)[k] for k in ("swa_cache", "comp_cache", "index_cache")))
            ok = True
            for key in ("sparse_indices", "lens", "gathered", "global_topk", "global_lens",
                        "gathered_index"):
                if key not in full:
                    continue
                parts = [g[key] for g in gathered]
                cat = np.concatenate(parts, axis=0)
                ok &= bool(np.array_equal(cat, full[key]))
            spans = [tuple(g["span"]) for g in gathered]
            ok &= spans[0][0] == 0 and spans[-1][1] == w.num_tokens and \
                all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            with open(os.path.join(result_dir, "result.txt"), "w") as f:
                f.write("ok" if ok else "mismatch")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_two_rank_request_shards_reproduce_the_batch(tmp_path, name, oracle_mod):
    world = 2
    port = _free_port()
    mp.start_processes(_worker, args=(world, port, name, str(tmp_path)), nprocs=world,
                       start_method="spawn")
    assert (tmp_path / "result.txt").read_text() == "ok"


def test_request_ranges_partition():
    from paged_sparse_kv_gb300.sharding import request_range
    for R in (1, 2, 7, 64, 258):
        for world in (1, 2, 3, 8):
            spans = [request_range(R, k, world) for k in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == R
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
