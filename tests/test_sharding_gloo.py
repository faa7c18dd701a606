"""Data-parallel sharding by request, checked with two gloo ranks on the CPU.

Each rank holds only its requests' pages (rank-local caches cut from the whole
batch's, tables and slot mappings rewritten to local page ids) and runs the
oracle's step on its request shard; rank 0 gathers the shards' outputs and
checks that, with local slot ids mapped back, they equal the step on the whole
batch, that every rank's pages end up as the whole batch's do, and that no page
is held by two ranks.  Nothing is exchanged on the data path: the only
collective is the gather the test uses to compare results.
"""
import hashlib
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


# gathered rows are compared on every SAMPLE-th token of the batch (index
# matrices, lens and caches on every token)
SAMPLE = {"tiny": 1, "decode": 1, "mixed": 64}


def _sample(name, t0, t1):
    step = SAMPLE[name]
    return np.array([t for t in range(t0, t1) if t % step == 0], dtype=np.int64)


def _local_step(w, name, rank, world):
    """The oracle's step on the rank's shard, with the rank-local caches cut from
    the whole batch's initial caches; slot outputs mapped back to global ids."""
    from oracle.pipeline import run_step
    from paged_sparse_kv_gb300.sharding import shard_requests
    sh = shard_requests(w, rank, world)
    whole = _caches(w)
    local = {k: (None if sh.maps[k] is None or whole[k] is None else
                 sh.maps[k].local_cache(whole[k])) for k in whole}
    toks = _sample(name, sh.first_token, sh.end_token) - sh.first_token
    res = run_step(sh.w, local["swa_cache"], local["comp_cache"], local["index_cache"], toks)
    out = {k: v for k, v in res.items() if isinstance(v, np.ndarray)}
    if "sparse_indices" in out:
        W = w.window
        si = out["sparse_indices"].copy()
        si[:, :W] = sh.maps["swa_cache"].global_slots(si[:, :W], w.swa_cache.block_size)
        si[:, W:] = sh.maps["comp_cache"].global_slots(si[:, W:], w.comp_cache.block_size)
        out["sparse_indices"] = si
    out["global_topk"] = sh.maps["index_cache"].global_slots(out["global_topk"],
                                                             w.index_cache.block_size)
    out["span"] = np.array([sh.first_token, sh.end_token])
    for k, c in local.items():
        if c is not None:
            out[f"cache:{k}"] = hashlib.sha1(c.tobytes()).hexdigest()
            out[f"pages:{k}"] = sh.maps[k].pages
    return out


def _worker(rank, world, port, name, result_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle.pipeline import run_step
        from paged_sparse_kv_gb300 import synthetic
        w = synthetic.make(name)
        payload = _local_step(w, name, rank, world)
        gathered = [None] * world if rank == 0 else None
        dist.gather_object(payload, gathered, dst=0)
        if rank == 0:
            whole = _caches(w)
            full = run_step(w, whole["swa_cache"], whole["comp_cache"], whole["index_cache"],
                            _sample(name, 0, w.num_tokens))
            bad = []
            for key in ("sparse_indices", "lens", "gathered", "global_topk", "global_lens",
                        "gathered_index"):
                if key not in full:
                    continue
                cat = np.concatenate([g[key] for g in gathered], axis=0)
                if not np.array_equal(cat, full[key]):
                    bad.append(key)
            spans = [tuple(g["span"]) for g in gathered]
            if not (spans[0][0] == 0 and spans[-1][1] == w.num_tokens and
                    all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))):
                bad.append("spans")
            for k, c in whole.items():
                if c is None:
                    continue
                # every rank's pages after its step equal the whole batch's
                for g in gathered:
                    want = hashlib.sha1(np.ascontiguousarray(c[g[f"pages:{k}"]]).tobytes())
                    if g[f"cache:{k}"] != want.hexdigest():
                        bad.append(f"cache {k}")
                # no rank holds a page of another rank's requests (no page is
                # shared between requests in these batches)
                owned = np.concatenate([g[f"pages:{k}"] for g in gathered])
                if np.unique(owned).size != owned.size:
                    bad.append(f"pages {k} held twice")
            with open(os.path.join(result_dir, "result.txt"), "w") as f:
                f.write("ok" if not bad else "mismatch: " + ", ".join(bad))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name", ["tiny", "decode", "mixed"])
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
