"""Seeded synthetic workloads for the paged sparse K-cache pipeline.

This module only draws inputs: K rows, request metadata, block tables, cache
slots and local top-k indices, with the shapes, sizes and value distributions
of the five workloads below.  It computes none of the pipeline's arithmetic
(no quantisation, no index mapping, no dequantisation); where it needs the
slot that a token's position occupies in a cache, it enumerates the slots of
the request's pages in order, the way a serving runtime hands out its
``slot_mapping``.

The pages (TokenSpeed's DeepSeek-V4 runtime and vLLM's DeepSeek-V4.1 ops)
measure on no public dataset, so every input here is synthetic:

* ``tiny``    2 requests (37 and 100 new tokens), page 16, head_dim 128 with no
              rope tail, window 8, top-k 8, ratio 4.
* ``decode``  64 requests x 1 token, context U[1024, 8192], head_dim 512
              (448 fp8 + 64 bf16 rope), page 64, window 128, top-k 512 with
              ~5% trailing -1.
* ``prefill`` 4 requests x 4096 new tokens, K ~ N(0,1) with 1% of elements
              x20, 65536-slot caches, window 128, top-k 512.
* ``mixed``   256 decode tokens (context U[2048, 32768]) then 2 prefill
              requests of 2048 tokens with replay_start U[0, 1024]; separate
              SWA and compressed tables; top-k 1024, window 128.
* ``mxfp4``   1,048,576 indexer-key rows [*, 128] into a 1,048,576-slot MXFP4
              cache (random-permutation slot mapping); 128 decode tokens at
              context 131072, top-k 2048 over 32768 compressed entries.
* ``decode_hca`` the decode batch of a layer with heavily compressed attention
              (compress ratio 128, no indexer): 64 requests x 1 token, context
              U[1024, 8192], window 128, every visible compressed entry
              (dense width 64 = 8192 / 128).

Seeds are ``20261202 + index`` in the order above (``prefill_small`` +5,
``decode_hca`` +6).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

CONFIG_NAMES = ("tiny", "decode", "prefill", "mixed", "mxfp4")
BASE_SEED = 20261202


@dataclasses.dataclass
class CacheGeom:
    """Geometry of one paged cache: ``num_pages`` pages of ``page_stride`` bytes,
    ``block_size`` token slots per page."""
    num_pages: int
    block_size: int
    page_stride: int


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    # record geometry
    head_dim: int
    rope_dim: int
    index_head_dim: int
    window: int
    compress_ratio: int
    topk: int
    # new rows inserted this step (bf16 bit patterns) and where they go
    k: Optional[np.ndarray]            # uint16 [T, head_dim]
    insert_slots: Optional[np.ndarray]  # int64 [T] (SWA cache)
    index_k: Optional[np.ndarray]      # uint16 [Ni, index_head_dim]
    index_insert_slots: Optional[np.ndarray]  # int64 [Ni] (indexer cache)
    # request metadata
    query_start_loc: np.ndarray        # int32 [R+1]
    seq_lens: np.ndarray               # int32 [R]
    token_to_req: np.ndarray           # int32 [T]
    replay_start: np.ndarray           # int32 [R]
    is_valid_token: Optional[np.ndarray]
    # block tables (int32, -1 = no page)
    swa_block_table: Optional[np.ndarray]
    comp_block_table: Optional[np.ndarray]  # None -> the SWA table is reused
    topk_local: np.ndarray             # int32 [T, topk]
    # caches
    swa_cache: Optional[CacheGeom]
    comp_cache: Optional[CacheGeom]
    index_cache: Optional[CacheGeom]
    # which steps the workload runs
    has_fp8: bool = True
    # dense builders: token positions and the dense compressed width (0: none)
    positions: Optional[np.ndarray] = None  # int64 [T]
    dense_width: int = 0

    @property
    def num_tokens(self) -> int:
        return int(self.token_to_req.shape[0])

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def padded_topk(self) -> int:
        return (self.topk + 3) // 4 * 4


# ---- record sizes (layout facts, stated by the insert/read docs) -------------

def fp8_record_bytes(head_dim: int, rope_dim: int, ue8m0: bool = True) -> int:
    """Bytes one token occupies in an fp8_ds_mla page: nope e4m3 bytes, rope
    bf16 bytes, and one scale slot per 64 dims (1 byte UE8M0 or 4 bytes fp32)."""
    nope = head_dim - rope_dim
    return nope + 2 * rope_dim + (head_dim // 64) * (1 if ue8m0 else 4)


def mxfp4_record_bytes(head_dim: int) -> int:
    """Bytes one token occupies in an MXFP4 page: two E2M1 per byte plus one
    E8M0 byte per 32 dims."""
    return head_dim // 2 + head_dim // 32


# ---- drawing helpers ---------------------------------------------------------

def _randn_bf16(gen: torch.Generator, rows: int, cols: int,
                outlier_frac: float = 0.0, outlier_scale: float = 1.0) -> np.ndarray:
    x = torch.randn(rows, cols, generator=gen, dtype=torch.float32)
    if outlier_frac > 0.0:
        mask = torch.rand(rows, cols, generator=gen) < outlier_frac
        x = torch.where(mask, x * outlier_scale, x)
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _page_slots(pages: np.ndarray, block_size: int) -> np.ndarray:
    """Slots of the listed pages in order (-1 pages contribute -1 slots)."""
    pages = np.asarray(pages, dtype=np.int64)
    offs = np.arange(block_size, dtype=np.int64)
    slots = pages[:, None] * block_size + offs[None, :]
    slots[pages < 0, :] = -1
    return slots.reshape(-1)


def _distinct_topk(rng: np.random.Generator, count: int, upper: int,
                   width: int) -> np.ndarray:
    """``count`` distinct uniform ints in [0, upper), then -1 up to ``width``."""
    row = np.full(width, -1, dtype=np.int32)
    count = min(count, upper, width)
    if count > 0:
        row[:count] = rng.choice(upper, size=count, replace=False).astype(np.int32)
    return row


def _tables_from_page_counts(rng: np.random.Generator, counts, total_pages: int,
                             width: int) -> np.ndarray:
    """One block-table row per request: consecutive slices of a random page
    permutation, padded with -1 to ``width``."""
    perm = rng.permutation(total_pages).astype(np.int32)
    table = np.full((len(counts), width), -1, dtype=np.int32)
    at = 0
    for r, c in enumerate(counts):
        table[r, :c] = perm[at:at + c]
        at += c
    assert at <= total_pages
    return table


# ---- workloads ---------------------------------------------------------------

def make_tiny(seed: int = BASE_SEED + 0) -> Workload:
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    bs, D, W, K, ratio = 16, 128, 8, 8, 4
    lens = np.array([37, 100], dtype=np.int32)
    R, T = 2, int(lens.sum())
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    t2r = np.repeat(np.arange(R, dtype=np.int32), lens)
    pos = np.concatenate([np.arange(L) for L in lens]).astype(np.int64)
    counts = [(int(L) + bs - 1) // bs for L in lens]       # 3 and 7 pages
    table = _tables_from_page_counts(rng, counts, 32, max(counts))
    # slot of each new token: its position's slot in the request's page list
    insert = np.empty(T, dtype=np.int64)
    for t in range(T):
        insert[t] = _page_slots(table[t2r[t]], bs)[pos[t]]
    topk = np.stack([_distinct_topk(rng, min(K, int(p) // ratio + 1), int(p) // ratio + 1, K)
                     for p in pos])
    fp8 = CacheGeom(32, bs, bs * fp8_record_bytes(D, 0))
    mx = CacheGeom(32, bs, bs * mxfp4_record_bytes(128))
    return Workload(
        name="tiny", seed=seed, head_dim=D, rope_dim=0, index_head_dim=128,
        window=W, compress_ratio=ratio, topk=K,
        k=_randn_bf16(gen, T, D), insert_slots=insert,
        index_k=_randn_bf16(gen, T, 128), index_insert_slots=insert.copy(),
        query_start_loc=qsl, seq_lens=lens, token_to_req=t2r,
        replay_start=np.zeros(R, dtype=np.int32), is_valid_token=None,
        swa_block_table=table, comp_block_table=None, topk_local=topk,
        swa_cache=fp8, comp_cache=dataclasses.replace(fp8), index_cache=mx)


def make_decode(seed: int = BASE_SEED + 1) -> Workload:
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    R, bs, D, rope, W, K, ratio = 64, 64, 512, 64, 128, 512, 4
    L = rng.integers(1024, 8192, size=R, endpoint=True).astype(np.int32)
    qsl = np.arange(R + 1, dtype=np.int32)
    t2r = np.arange(R, dtype=np.int32)
    pos = L.astype(np.int64) - 1
    swa_counts = [(int(x) + bs - 1) // bs for x in L]
    swa_pages = int(sum(swa_counts))
    swa_table = _tables_from_page_counts(rng, swa_counts, swa_pages, max(swa_counts))
    Lc = (pos + 1) // ratio
    comp_counts = [max(1, (int(c) + bs - 1) // bs) for c in Lc]
    comp_pages = int(sum(comp_counts))
    comp_table = _tables_from_page_counts(rng, comp_counts, comp_pages, max(comp_counts))
    insert = np.array([_page_slots(swa_table[r], bs)[pos[r]] for r in range(R)], dtype=np.int64)
    # the newest complete compressed entry of each request takes an indexer key
    idx_insert = np.array([_page_slots(comp_table[r], bs)[Lc[r] - 1] for r in range(R)],
                          dtype=np.int64)
    topk = np.stack([_distinct_topk(rng, min(int(c), 486), int(c), K) for c in Lc])
    return Workload(
        name="decode", seed=seed, head_dim=D, rope_dim=rope, index_head_dim=128,
        window=W, compress_ratio=ratio, topk=K,
        k=_randn_bf16(gen, R, D), insert_slots=insert,
        index_k=_randn_bf16(gen, R, 128), index_insert_slots=idx_insert,
        query_start_loc=qsl, seq_lens=L, token_to_req=t2r,
        replay_start=np.zeros(R, dtype=np.int32), is_valid_token=None,
        swa_block_table=swa_table, comp_block_table=comp_table, topk_local=topk,
        swa_cache=CacheGeom(swa_pages, bs, bs * fp8_record_bytes(D, rope)),
        comp_cache=CacheGeom(comp_pages, bs, bs * fp8_record_bytes(D, rope)),
        index_cache=CacheGeom(comp_pages, bs, bs * mxfp4_record_bytes(128)))


def make_prefill(seed: int = BASE_SEED + 2, num_reqs: int = 4) -> Workload:
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    R, Q, bs, D, rope, W, K, ratio = num_reqs, 4096, 64, 512, 64, 128, 512, 4
    T = R * Q
    lens = np.full(R, Q, dtype=np.int32)
    qsl = (np.arange(R + 1) * Q).astype(np.int32)
    t2r = np.repeat(np.arange(R, dtype=np.int32), Q)
    pos = np.tile(np.arange(Q, dtype=np.int64), R)
    table = _tables_from_page_counts(rng, [64] * R, 1024, 64)
    slot_lists = [_page_slots(table[r], bs) for r in range(R)]
    insert = np.array([slot_lists[t2r[t]][pos[t]] for t in range(T)], dtype=np.int64)
    # indexer keys land at compressed-entry boundaries only; other tokens skip (-1)
    idx_insert = np.full(T, -1, dtype=np.int64)
    for t in range(T):
        if (pos[t] + 1) % ratio == 0:
            idx_insert[t] = slot_lists[t2r[t]][(pos[t] + 1) // ratio - 1]
    topk = np.stack([_distinct_topk(rng, K, int(p + 1) // ratio, K) for p in pos])
    geom = CacheGeom(1024, bs, bs * fp8_record_bytes(D, rope))
    return Workload(
        name="prefill" if num_reqs == 4 else f"prefill_{num_reqs}req", seed=seed, head_dim=D, rope_dim=rope, index_head_dim=128,
        window=W, compress_ratio=ratio, topk=K,
        k=_randn_bf16(gen, T, D, outlier_frac=0.01, outlier_scale=20.0),
        insert_slots=insert,
        index_k=_randn_bf16(gen, T, 128), index_insert_slots=idx_insert,
        query_start_loc=qsl, seq_lens=lens, token_to_req=t2r,
        replay_start=np.zeros(R, dtype=np.int32), is_valid_token=None,
        swa_block_table=table, comp_block_table=None, topk_local=topk,
        swa_cache=geom, comp_cache=dataclasses.replace(geom),
        index_cache=CacheGeom(1024, bs, bs * mxfp4_record_bytes(128)))


def make_mixed(seed: int = BASE_SEED + 3) -> Workload:
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    Rd, Rp, Q, bs, D, rope, W, K, ratio = 256, 2, 2048, 64, 512, 64, 128, 1024, 4
    R = Rd + Rp
    Ld = rng.integers(2048, 32768, size=Rd, endpoint=True)
    rho = rng.integers(0, 1024, size=Rp, endpoint=True)
    seq = np.concatenate([Ld, rho + Q]).astype(np.int32)
    qlens = np.concatenate([np.ones(Rd, np.int64), np.full(Rp, Q, np.int64)])
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    T = int(qsl[-1])
    t2r = np.repeat(np.arange(R, dtype=np.int32), qlens)
    pos = np.concatenate([[int(Ld[r]) - 1] for r in range(Rd)] +
                         [np.arange(int(rho[i]), int(rho[i]) + Q) for i in range(Rp)]
                         ).astype(np.int64)
    replay = np.concatenate([np.zeros(Rd, np.int64), rho]).astype(np.int32)
    # SWA table: real pages only for logical pages some window reaches
    swa_width = (int(seq.max()) + bs - 1) // bs
    reach = []
    for r in range(R):
        first_pos = int(seq[r] - qlens[r])
        lo = max(int(replay[r]), first_pos - W + 1, 0)
        reach.append(np.arange(lo // bs, (int(seq[r]) - 1) // bs + 1))
    swa_pages = 1024
    perm = rng.permutation(swa_pages).astype(np.int32)
    swa_table = np.full((R, swa_width), -1, dtype=np.int32)
    at = 0
    for r in range(R):
        n = len(reach[r])
        swa_table[r, reach[r]] = perm[at:at + n]
        at += n
    assert at <= swa_pages
    Lc_req = seq.astype(np.int64) // ratio
    comp_counts = [max(1, (int(c) + bs - 1) // bs) for c in Lc_req]
    comp_pages = int(sum(comp_counts))
    comp_table = _tables_from_page_counts(rng, comp_counts, comp_pages, max(comp_counts))
    swa_lists = [_page_slots(swa_table[r], bs) for r in range(R)]
    comp_lists = [_page_slots(comp_table[r], bs) for r in range(R)]
    insert = np.array([swa_lists[t2r[t]][pos[t]] for t in range(T)], dtype=np.int64)
    idx_insert = np.full(T, -1, dtype=np.int64)
    for t in range(T):
        if (pos[t] + 1) % ratio == 0:
            idx_insert[t] = comp_lists[t2r[t]][(pos[t] + 1) // ratio - 1]
    topk = np.stack([_distinct_topk(rng, K, int(p + 1) // ratio, K) for p in pos])
    return Workload(
        name="mixed", seed=seed, head_dim=D, rope_dim=rope, index_head_dim=128,
        window=W, compress_ratio=ratio, topk=K,
        k=_randn_bf16(gen, T, D), insert_slots=insert,
        index_k=_randn_bf16(gen, T, 128), index_insert_slots=idx_insert,
        query_start_loc=qsl, seq_lens=seq, token_to_req=t2r,
        replay_start=replay, is_valid_token=None,
        swa_block_table=swa_table, comp_block_table=comp_table, topk_local=topk,
        swa_cache=CacheGeom(swa_pages, bs, bs * fp8_record_bytes(D, rope)),
        comp_cache=CacheGeom(comp_pages, bs, bs * fp8_record_bytes(D, rope)),
        index_cache=CacheGeom(comp_pages, bs, bs * mxfp4_record_bytes(128)))


def make_mxfp4(seed: int = BASE_SEED + 4) -> Workload:
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    N, pages, bs, D, R, K, ratio = 1 << 20, 16384, 64, 128, 128, 2048, 4
    ctx = 131072
    Lc = ctx // ratio                      # 32768 compressed entries
    width = Lc // bs                       # 512 pages per request
    table = np.stack([rng.choice(pages, size=width, replace=False).astype(np.int32)
                      for _ in range(R)])
    topk = np.stack([_distinct_topk(rng, K, Lc, K) for _ in range(R)])
    return Workload(
        name="mxfp4", seed=seed, head_dim=D, rope_dim=0, index_head_dim=D,
        window=0, compress_ratio=ratio, topk=K,
        k=None, insert_slots=None,
        index_k=_randn_bf16(gen, N, D),
        index_insert_slots=rng.permutation(N).astype(np.int64),
        query_start_loc=np.arange(R + 1, dtype=np.int32),
        seq_lens=np.full(R, ctx, dtype=np.int32),
        token_to_req=np.arange(R, dtype=np.int32),
        replay_start=np.zeros(R, dtype=np.int32), is_valid_token=None,
        swa_block_table=None, comp_block_table=table, topk_local=topk,
        swa_cache=None, comp_cache=None,
        index_cache=CacheGeom(pages, bs, bs * mxfp4_record_bytes(D)),
        has_fp8=False)


def make_prefill_small(seed: int = BASE_SEED + 5) -> Workload:
    """One request of the prefill workload (4096 new tokens): the same kernels
    at a quarter of the size, small enough for a full profiler capture."""
    return make_prefill(seed, num_reqs=1)


def make_decode_hca(seed: int = BASE_SEED + 6) -> Workload:
    """Decode batch of a heavily compressed (ratio 128) attention layer: no
    top-k and no indexer; each token attends to its window and to every
    compressed entry its position has completed."""
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    R, bs, D, rope, W, ratio, ctx = 64, 64, 512, 64, 128, 128, 8192
    L = rng.integers(1024, ctx, size=R, endpoint=True).astype(np.int32)
    pos = L.astype(np.int64) - 1
    swa_counts = [(int(x) + bs - 1) // bs for x in L]
    swa_pages = int(sum(swa_counts))
    swa_table = _tables_from_page_counts(rng, swa_counts, swa_pages, max(swa_counts))
    Lc = (pos + 1) // ratio
    comp_counts = [max(1, (int(c) + bs - 1) // bs) for c in Lc]
    comp_pages = int(sum(comp_counts))
    comp_table = _tables_from_page_counts(rng, comp_counts, comp_pages, max(comp_counts))
    insert = np.array([_page_slots(swa_table[r], bs)[pos[r]] for r in range(R)], dtype=np.int64)
    width = (ctx + ratio - 1) // ratio
    return Workload(
        name="decode_hca", seed=seed, head_dim=D, rope_dim=rope, index_head_dim=128,
        window=W, compress_ratio=ratio, topk=0,
        k=_randn_bf16(gen, R, D), insert_slots=insert,
        index_k=None, index_insert_slots=None,
        query_start_loc=np.arange(R + 1, dtype=np.int32), seq_lens=L,
        token_to_req=np.arange(R, dtype=np.int32),
        replay_start=np.zeros(R, dtype=np.int32), is_valid_token=None,
        swa_block_table=swa_table, comp_block_table=comp_table,
        topk_local=np.zeros((R, 0), dtype=np.int32),
        swa_cache=CacheGeom(swa_pages, bs, bs * fp8_record_bytes(D, rope)),
        comp_cache=CacheGeom(comp_pages, bs, bs * fp8_record_bytes(D, rope)),
        index_cache=None, positions=pos, dense_width=width)


MAKERS = {"tiny": make_tiny, "decode": make_decode, "prefill": make_prefill,
          "mixed": make_mixed, "mxfp4": make_mxfp4, "prefill_small": make_prefill_small,
          "decode_hca": make_decode_hca}
DEFAULT_SEEDS = {"tiny": BASE_SEED + 0, "decode": BASE_SEED + 1, "prefill": BASE_SEED + 2,
                 "mixed": BASE_SEED + 3, "mxfp4": BASE_SEED + 4, "prefill_small": BASE_SEED + 5,
                 "decode_hca": BASE_SEED + 6}


def make(name: str, seed_offset: int = 0) -> Workload:
    """The named workload, drawn from its seed (plus seed_offset, e.g. one
    independent batch per GPU)."""
    return MAKERS[name](DEFAULT_SEEDS[name] + seed_offset)


def gptj_cos_sin(max_pos: int, rope_dim: int = 64, base: float = 10000.0) -> np.ndarray:
    """A RoPE table [max_pos, rope_dim] in binary32, GPT-J layout (rope_dim/2
    cosines, then rope_dim/2 sines) with the usual inverse-frequency ladder:
    the input a model's RoPE instance would hand the indexer-key store."""
    half = rope_dim // 2
    theta = base ** (-np.arange(half, dtype=np.float64) / half)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * theta[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def norm_weight(seed: int, dim: int = 128) -> np.ndarray:
    """A k_norm weight vector [dim] in binary32, U[0.5, 2]."""
    return np.random.default_rng(seed).uniform(0.5, 2.0, size=dim).astype(np.float32)


def compressor_inputs(w: Workload, ratio: int, seed: int) -> dict:
    """Inputs of one compressor layer for a batch (compress ratio 4 with the
    overlapping window -- state width 1024 -- or 128 without -- 512): the
    binary32 kv and score projections N(0,1) and N(0,3), the APE rows
    N(0, 0.5) and the norm weight.  The state cache is paged by position like
    the SWA cache, so its table and each token's state slot are the SWA ones;
    ratio 4 writes its rows at the compressed-entry slots the indexer keys use
    (floor(pos / 4) through the compressed table), ratio 128 at slots of its
    own small cache (entry floor(pos / 128), one page per 64 entries)."""
    overlap = ratio == 4
    sw = (2 if overlap else 1) * 512
    T = w.num_tokens
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    kv = torch.randn(T, sw, generator=gen).numpy()
    score = (torch.randn(T, sw, generator=gen) * 3.0).numpy()
    ape = (torch.randn(ratio, sw, generator=gen) * 0.5).numpy()
    qlen = np.diff(w.query_start_loc).astype(np.int64)
    pos = np.concatenate([np.arange(s - q, s) for s, q in zip(w.seq_lens.astype(np.int64), qlen)])
    if overlap:
        kv_slots = np.asarray(w.index_insert_slots, np.int64)
        kv_table = w.comp_block_table if w.comp_block_table is not None else w.swa_block_table
        kv_geom = w.comp_cache
    else:
        n_ent = (w.seq_lens.astype(np.int64) + ratio - 1) // ratio
        per = int((n_ent.max() + 63) // 64)
        pages = w.num_reqs * per
        kv_table = rng.permutation(pages).astype(np.int32).reshape(w.num_reqs, per)
        kv_slots = np.full(T, -1, np.int64)
        for t in range(T):
            if (pos[t] + 1) % ratio == 0:
                e = pos[t] // ratio
                r = w.token_to_req[t]
                kv_slots[t] = int(kv_table[r, e // 64]) * 64 + e % 64
        kv_geom = CacheGeom(pages, 64, 64 * fp8_record_bytes(512, 64))
    return {"ratio": ratio, "overlap": overlap, "state_width": sw, "kv": kv, "score": score,
            "ape": ape, "positions": pos.astype(np.int64), "state_slots": w.insert_slots,
            "state_table": w.swa_block_table, "state_bs": w.swa_cache.block_size,
            "state_pages": w.swa_cache.num_pages, "kv_slots": kv_slots, "kv_table": kv_table,
            "kv_geom": kv_geom, "weight": norm_weight(seed, 512),
            "cos_sin": gptj_cos_sin(int(w.seq_lens.max()))}


def random_cache_bytes(seed: int, geom: CacheGeom) -> np.ndarray:
    """A cache filled with seeded random bytes, none of them 0x7F or 0xFF (the
    E4M3 NaN codes), so that every record decodes to finite or infinite
    values and both implementations see identical bytes."""
    rng = np.random.default_rng(seed)
    n = geom.num_pages * geom.page_stride
    b = np.frombuffer(rng.bytes(n), dtype=np.uint8).reshape(geom.num_pages, geom.page_stride)
    b = b.copy()
    b[(b & 0x7F) == 0x7F] ^= 1  # 0x7F -> 0x7E, 0xFF -> 0xFE
    return b
