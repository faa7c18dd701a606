"""Pins for the oracle's prefill-workspace path: range-form gather, workspace
indices and raw MXFP4 gather.

* Hand-worked golden cases (tests/golden/workspace_golden.json).
* Brute force: every range-gathered row equals the index-form gather of the
  slot found by walking the request's pages; every raw MXFP4 row equals the
  record bytes found the same way.
* Cross-consistency: a workspace filled by the two range gathers, read through
  the workspace indices, gives exactly the rows the global-slot builder and the
  index-form gather give (the two prefill paths agree entry by entry).
"""
import json
import os

import numpy as np
import pytest

from conftest import GOLDEN
from paged_sparse_kv_gb300 import synthetic


def _golden():
    return json.load(open(os.path.join(GOLDEN, "workspace_golden.json")))


def test_workspace_indices_golden(oracle_mod):
    g = _golden()["indices"]
    out, lens = oracle_mod.combine_topk_swa_workspace_indices(
        np.array(g["query_start_loc"], np.int32), np.array(g["seq_lens"], np.int32),
        np.array(g["gather_lens"], np.int32), np.array(g["token_to_req"], np.int32),
        g["window"], g["compress_ratio"], np.array(g["topk_local"], np.int32),
        g["workspace_width"], g["compressed_base"])
    assert out.tolist() == g["expected_indices"]
    assert lens.tolist() == g["expected_lens"]


def test_range_gather_golden(oracle_mod):
    g = _golden()["range_gather"]
    rng = np.random.default_rng(0)
    bs, D = g["block_size"], 128
    cache = rng.integers(0, 254, size=(4, bs * 130 + 12), dtype=np.uint8)
    cache[cache >= 0x7F] += 1
    out = np.full((1, g["out_rows"], D), 0x1234, np.uint16)
    oracle_mod.dequantize_and_gather_k_cache_ranges(
        out, cache, bs, 0, D, 0, np.array(g["seq_lens"], np.int32),
        np.array(g["gather_lens"], np.int32), np.array(g["block_table"], np.int32),
        g["offset"])
    for row, s in enumerate(g["expected_slots"]):
        if s is None:
            assert np.all(out[0, row] == 0x1234)
            continue
        want = oracle_mod.dequantize_and_gather_k_cache(cache, bs, 0, D, 0,
                                                        np.array([[s]], np.int32))[0, 0]
        assert np.array_equal(out[0, row], want), row


def test_mxfp4_raw_gather_golden(oracle_mod):
    g = _golden()["mxfp4_raw"]
    rng = np.random.default_rng(1)
    bs, D = g["block_size"], 128
    cache = rng.integers(0, 256, size=(3, bs * 68), dtype=np.uint8)
    vals, scl = oracle_mod.indexer_mxfp4_paged_gather(
        cache, bs, D, np.array(g["block_table"], np.int32), np.array(g["cu_seq_lens"], np.int32))
    for row, s in enumerate(g["expected_slots"]):
        page, off = divmod(s, bs)
        assert np.array_equal(vals[row], cache[page, off * 64:(off + 1) * 64])
        assert np.array_equal(scl[row], cache[page, bs * 64 + off * 4: bs * 64 + off * 4 + 4])


def _slot_dict(row, base, bs):
    d = {}
    for lp, page in enumerate(row):
        if page >= 0:
            for o in range(bs):
                d[(lp + base) * bs + o] = page * bs + o
    return d


@pytest.mark.parametrize("seed", range(12))
def test_range_gather_vs_enumeration(oracle_mod, seed):
    rng = np.random.default_rng(300 + seed)
    bs = int(rng.choice([1, 2, 4, 16]))
    R, width, pages, D, rope = int(rng.integers(1, 4)), 6, 12, 128, 0
    table = rng.integers(-1, pages, size=(R, width)).astype(np.int32)
    base = None if rng.random() < 0.5 else rng.integers(0, 2, size=R).astype(np.int32)
    seq = rng.integers(0, (width + 1) * bs, size=R).astype(np.int32)
    glen = None if rng.random() < 0.3 else np.minimum(seq, rng.integers(0, 9, size=R)).astype(np.int32)
    rows, offset = 12, int(rng.integers(0, 4))
    cache = synthetic.random_cache_bytes(seed, synthetic.CacheGeom(pages, bs, bs * 130 + 14))
    out = np.full((R, rows, D), 0xBEEF, np.uint16)
    oracle_mod.dequantize_and_gather_k_cache_ranges(out, cache, bs, 0, D, rope, seq, glen,
                                                    table, offset, base_offsets=base)
    for r in range(R):
        d = _slot_dict(table[r], int(base[r]) if base is not None else 0, bs)
        g = int(glen[r]) if glen is not None else int(seq[r])
        written = set()
        for i in range(g):
            if not 0 <= offset + i < rows:
                continue
            p = int(seq[r]) - g + i
            s = d.get(p, -1)
            want = oracle_mod.dequantize_and_gather_k_cache(cache, bs, 0, D, rope,
                                                            np.array([[s]], np.int32))[0, 0]
            assert np.array_equal(out[r, offset + i], want)
            written.add(offset + i)
        for k in set(range(rows)) - written:
            assert np.all(out[r, k] == 0xBEEF)


@pytest.mark.parametrize("name", ["tiny", "prefill_small"])
def test_workspace_path_agrees_with_global_slot_path(oracle_mod, name):
    """The prefill workspace path names the same rows as the global-slot path."""
    w = synthetic.make(name)
    W, ratio = w.window, w.compress_ratio
    seq = w.seq_lens.astype(np.int64)
    qlen = np.diff(w.query_start_loc).astype(np.int64)
    prefix = seq - qlen
    glen = (qlen + np.minimum(prefix, max(W - 1, 0))).astype(np.int32)
    lc = (seq // ratio).astype(np.int32)
    cb = int(lc.max())
    ww = cb + int(glen.max())
    swa = synthetic.random_cache_bytes(5, w.swa_cache)
    comp = synthetic.random_cache_bytes(6, w.comp_cache)
    ws = np.zeros((w.num_reqs, ww, w.head_dim), np.uint16)
    comp_table = w.comp_block_table if w.comp_block_table is not None else w.swa_block_table
    oracle_mod.dequantize_and_gather_k_cache_ranges(
        ws, comp, w.comp_cache.block_size, 0, w.head_dim, w.rope_dim, lc, None, comp_table, 0)
    oracle_mod.dequantize_and_gather_k_cache_ranges(
        ws, swa, w.swa_cache.block_size, 0, w.head_dim, w.rope_dim, w.seq_lens, glen,
        w.swa_block_table, cb)
    wsi, wlens = oracle_mod.combine_topk_swa_workspace_indices(
        w.query_start_loc, w.seq_lens, glen, w.token_to_req, W, ratio, w.topk_local, ww, cb)
    gsi, glens = oracle_mod.combine_topk_swa_indices(
        w.query_start_loc, w.seq_lens, w.token_to_req, w.replay_start, w.swa_block_table,
        w.swa_cache.block_size, w.comp_block_table, w.comp_cache.block_size, W, ratio,
        w.topk_local)
    # The workspace holds seq // ratio compressed entries per request; a top-k
    # index at or beyond that (a not-yet-complete entry, which only the tiny
    # recipe draws) is -1 there but may have a page in the global path.
    beyond = np.zeros_like(gsi, dtype=bool)
    beyond[:, W:W + w.topk] = w.topk_local >= lc[w.token_to_req][:, None]
    assert np.array_equal(wsi >= 0, (gsi >= 0) & ~beyond)
    assert np.array_equal(wlens, ((gsi >= 0) & ~beyond).sum(axis=1))
    flat = ws.reshape(-1, w.head_dim)
    toks = np.linspace(0, w.num_tokens - 1, min(w.num_tokens, 40)).astype(int)
    for t in toks:
        g_swa = oracle_mod.dequantize_and_gather_k_cache(
            swa, w.swa_cache.block_size, 0, w.head_dim, w.rope_dim, gsi[t:t + 1, :W])[0]
        g_top = oracle_mod.dequantize_and_gather_k_cache(
            comp, w.comp_cache.block_size, 0, w.head_dim, w.rope_dim, gsi[t:t + 1, W:])[0]
        g = np.concatenate([g_swa, g_top])
        for c in np.nonzero(wsi[t] >= 0)[0]:
            assert np.array_equal(flat[wsi[t, c]], g[c]), (t, c)
