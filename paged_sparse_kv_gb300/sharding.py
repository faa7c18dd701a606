"""Split a batch across data-parallel ranks by request (host-side bookkeeping).

Every step of the pipeline works per token, and a token touches only its own
request's block-table rows and pages; requests are independent.  A batch
therefore shards by contiguous request ranges with no exchange between ranks:
rank k takes requests [R*k/N, R*(k+1)/N) with their query tokens, and its
metadata is rebased (query_start_loc starts at 0, token_to_req counts from the
rank's first request).

Each rank also holds only the pages its requests use (data-parallel attention
keeps a request and its KV on one rank).  For every cache, the pages the
rank's block-table rows name are numbered 0..L-1 in ascending global order
(a ``PageMap``); the rank's tables and slot mappings are rewritten to those
local ids and its caches are [L, page_stride].  A page two ranks' requests
share (prefix sharing) is held by both.  Entries keep their meaning:
-1 stays -1, a slot in a page the rank does not hold is skipped (-1), and a
page beyond the whole cache stays beyond the local one by the same distance,
so a local step's outputs map back to the whole batch's slot for slot.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

from .synthetic import CacheGeom, Workload


def request_range(num_reqs: int, rank: int, world: int) -> tuple[int, int]:
    return num_reqs * rank // world, num_reqs * (rank + 1) // world


@dataclasses.dataclass
class PageMap:
    """Rank-local page ids of one cache: local page i is global page pages[i]."""
    pages: np.ndarray   # int64 [L], ascending global page ids
    num_global: int     # pages in the whole cache

    @property
    def num_local(self) -> int:
        return int(self.pages.size)

    def local_pages(self, table: np.ndarray) -> np.ndarray:
        """A block table in local page ids (int32)."""
        t = np.asarray(table, dtype=np.int64)
        out = np.full(t.shape, -1, dtype=np.int64)
        held = (t >= 0) & (t < self.num_global)
        out[held] = np.searchsorted(self.pages, t[held])
        beyond = t >= self.num_global
        out[beyond] = self.num_local + (t[beyond] - self.num_global)
        return out.astype(np.int32)

    def local_slots(self, slots: np.ndarray, block_size: int) -> np.ndarray:
        """Global slot ids as local ones (int64); -1 where negative or where the
        rank does not hold the page."""
        s = np.asarray(slots, dtype=np.int64)
        page, off = np.divmod(np.maximum(s, 0), block_size)
        out = np.full(s.shape, -1, dtype=np.int64)
        inside = (s >= 0) & (page < self.num_global)
        pos = np.searchsorted(self.pages, page[inside])
        pos_c = np.minimum(pos, max(self.num_local - 1, 0))
        held = np.zeros(inside.sum(), dtype=bool)
        if self.num_local:
            held = self.pages[pos_c] == page[inside]
        vals = np.full(held.shape, -1, dtype=np.int64)
        vals[held] = pos[held] * block_size + off[inside][held]
        out[inside] = vals
        beyond = (s >= 0) & (page >= self.num_global)
        out[beyond] = (self.num_local + page[beyond] - self.num_global) * block_size + off[beyond]
        return out

    def global_slots(self, slots: np.ndarray, block_size: int) -> np.ndarray:
        """Local slot ids (an index matrix of a local step) as the whole batch's."""
        s = np.asarray(slots, dtype=np.int64)
        page, off = np.divmod(np.maximum(s, 0), block_size)
        out = np.full(s.shape, -1, dtype=np.int64)
        held = (s >= 0) & (page < self.num_local)
        out[held] = self.pages[page[held]] * block_size + off[held]
        beyond = (s >= 0) & (page >= self.num_local)
        out[beyond] = (self.num_global + page[beyond] - self.num_local) * block_size + off[beyond]
        return out.astype(slots.dtype)

    def local_cache(self, cache: np.ndarray) -> np.ndarray:
        """The rank's copy of a whole cache's pages ([L, page_stride])."""
        return np.ascontiguousarray(cache[self.pages])


def _pages_named(*tables) -> np.ndarray:
    ids = [np.asarray(t, dtype=np.int64).reshape(-1) for t in tables if t is not None]
    if not ids:
        return np.zeros(0, dtype=np.int64)
    allp = np.concatenate(ids)
    return np.unique(allp[allp >= 0])


@dataclasses.dataclass
class Shard:
    """One rank's share of a batch."""
    w: Workload                  # its requests, tokens, local tables and slots
    first_token: int             # [first_token, end_token): the batch tokens it covers
    end_token: int
    maps: dict                   # cache name -> PageMap (None where the batch has no cache)


def shard_requests(w: Workload, rank: int, world: int) -> Shard:
    """The rank's requests with rank-local page ids and cache geometries."""
    r0, r1 = request_range(w.num_reqs, rank, world)
    qsl = w.query_start_loc
    t0, t1 = int(qsl[r0]), int(qsl[r1])

    def rows(a, lo, hi):
        return None if a is None else np.ascontiguousarray(a[lo:hi])

    swa_rows = rows(w.swa_block_table, r0, r1)
    comp_rows = rows(w.comp_block_table, r0, r1)

    def page_map(table, *caches) -> Optional[PageMap]:
        """One map per table: the caches a table addresses share its page ids."""
        geoms = [g for g in caches if g is not None]
        if table is None or not geoms:
            return None
        n = geoms[0].num_pages
        if any(g.num_pages != n for g in geoms):
            raise ValueError("caches addressed through one block table must have as many pages")
        named = _pages_named(table)
        return PageMap(named[named < n], n)

    if comp_rows is None:  # one table for the SWA and the compressed caches
        swa_map = comp_map = page_map(swa_rows, w.swa_cache, w.comp_cache, w.index_cache)
    else:
        swa_map = page_map(swa_rows, w.swa_cache)
        comp_map = page_map(comp_rows, w.comp_cache, w.index_cache)
    maps: dict[str, Optional[PageMap]] = {
        "swa_cache": swa_map if w.swa_cache is not None else None,
        "comp_cache": comp_map if w.comp_cache is not None else None,
        "index_cache": comp_map if w.index_cache is not None else None}

    def geom(name):
        g = getattr(w, name)
        return None if g is None else CacheGeom(maps[name].num_local, g.block_size, g.page_stride)

    def local_table(table, m):
        return None if table is None or m is None else m.local_pages(table)

    # per-token inserts follow the tokens; a whole-cache fill (more rows than
    # tokens) goes to every rank, each writing the pages it holds
    per_token_index = w.index_k is not None and w.index_k.shape[0] == w.num_tokens
    ins = rows(w.insert_slots, t0, t1)
    iins = rows(w.index_insert_slots, t0, t1) if per_token_index else w.index_insert_slots
    sub = dataclasses.replace(
        w,
        name=f"{w.name}[rank {rank}/{world}]",
        k=rows(w.k, t0, t1),
        insert_slots=None if ins is None else maps["swa_cache"].local_slots(
            ins, w.swa_cache.block_size),
        index_k=rows(w.index_k, t0, t1) if per_token_index else w.index_k,
        index_insert_slots=None if iins is None else maps["index_cache"].local_slots(
            iins, w.index_cache.block_size),
        query_start_loc=np.ascontiguousarray(qsl[r0:r1 + 1] - qsl[r0]).astype(np.int32),
        seq_lens=rows(w.seq_lens, r0, r1),
        token_to_req=np.ascontiguousarray(w.token_to_req[t0:t1] - r0).astype(np.int32),
        replay_start=rows(w.replay_start, r0, r1),
        is_valid_token=rows(w.is_valid_token, t0, t1),
        swa_block_table=local_table(swa_rows, swa_map),
        comp_block_table=local_table(comp_rows, comp_map),
        topk_local=rows(w.topk_local, t0, t1),
        positions=rows(w.positions, t0, t1),
        swa_cache=geom("swa_cache"),
        comp_cache=geom("comp_cache"),
        index_cache=geom("index_cache"),
    )
    return Shard(sub, t0, t1, maps)
