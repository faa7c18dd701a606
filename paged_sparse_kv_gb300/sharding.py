"""Split a batch across data-parallel ranks by request (host-side bookkeeping).

Every step of the pipeline works per token, and a token touches only its own
request's block-table rows and pages; requests are independent.  A batch
therefore shards by contiguous request ranges with no exchange between ranks:
rank k takes requests [R*k/N, R*(k+1)/N) with their query tokens, and its
metadata is rebased (query_start_loc starts at 0, token_to_req counts from the
rank's first request).  Slot ids and page ids are left unchanged: each rank's
caches hold the pages of its own requests (data-parallel attention keeps a
request and its KV on one rank).
"""
from __future__ import annotations

import dataclasses

import numpy as np

from .synthetic import Workload


def request_range(num_reqs: int, rank: int, world: int) -> tuple[int, int]:
    return num_reqs * rank // world, num_reqs * (rank + 1) // world


def shard_requests(w: Workload, rank: int, world: int) -> tuple[Workload, int, int]:
    """The rank's share of a batch; returns (workload, first_token, end_token)
    where [first_token, end_token) are the batch's token indices it covers."""
    r0, r1 = request_range(w.num_reqs, rank, world)
    qsl = w.query_start_loc
    t0, t1 = int(qsl[r0]), int(qsl[r1])

    def rows(a, lo, hi):
        return None if a is None else np.ascontiguousarray(a[lo:hi])

    sub = dataclasses.replace(
        w,
        name=f"{w.name}[rank {rank}/{world}]",
        k=rows(w.k, t0, t1),
        insert_slots=rows(w.insert_slots, t0, t1),
        index_k=rows(w.index_k, t0, t1) if w.index_k is not None and
        w.index_k.shape[0] == w.num_tokens else w.index_k,
        index_insert_slots=rows(w.index_insert_slots, t0, t1)
        if w.index_insert_slots is not None and w.index_insert_slots.shape[0] == w.num_tokens
        else w.index_insert_slots,
        query_start_loc=np.ascontiguousarray(qsl[r0:r1 + 1] - qsl[r0]).astype(np.int32),
        seq_lens=rows(w.seq_lens, r0, r1),
        token_to_req=np.ascontiguousarray(w.token_to_req[t0:t1] - r0).astype(np.int32),
        replay_start=rows(w.replay_start, r0, r1),
        is_valid_token=rows(w.is_valid_token, t0, t1),
        swa_block_table=rows(w.swa_block_table, r0, r1),
        comp_block_table=rows(w.comp_block_table, r0, r1),
        topk_local=rows(w.topk_local, t0, t1),
    )
    return sub, t0, t1
