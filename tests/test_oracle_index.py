"""Pins for the oracle's index builders.

* The hand-worked golden case (tests/golden/index_golden.json).
* A brute-force enumeration written here from the definitions, not from the
  oracle's formulas: each request's pages are walked to build a dictionary
  position -> slot, the window is the sorted set of positions that satisfy the
  three window predicates, and top-k entries are dictionary look-ups.
  Randomised over page sizes, windows, top-k widths, -1 entries in the tables
  and in the top-k rows, base offsets, replay_start, invalid tokens and
  request indices out of range.
* Invariants on the five workloads: lens equals the count of entries >= 0,
  padding columns are -1, the window columns are consecutive slots inside a
  page, and every top-k entry lands in the request's own pages.
"""
import json
import os

import numpy as np
import pytest

from conftest import GOLDEN
from paged_sparse_kv_gb300 import synthetic


def _slot_dict(row, base, bs):
    """position -> slot by walking the request's pages in order."""
    d = {}
    for lp, page in enumerate(row):
        if page < 0:
            continue
        for o in range(bs):
            p = (lp + base) * bs + o
            s = page * bs + o
            if s <= 2**31 - 1:
                d[p] = s
    return d


def _brute_combine(qsl, seq, t2r, replay, swa_bt, swa_base, swa_bs, comp_bt,
                   comp_base, comp_bs, W, topk, valid):
    T, K = topk.shape
    P = (K + 3) // 4 * 4
    R = len(seq)
    if comp_bt is None:
        comp_bt = swa_bt
    out = np.full((T, W + P), -1, np.int64)
    lens = np.zeros(T, np.int64)
    for t in range(T):
        r = int(t2r[t])
        if (valid is not None and not valid[t]) or r < 0 or r >= R:
            continue
        # position by counting: the token is the (t - start)-th of the
        # request's query tokens, which are its last qlen positions
        start, end = int(qsl[r]), int(qsl[r + 1])
        positions = list(range(int(seq[r]) - (end - start), int(seq[r])))
        pos = positions[t - start]
        sd = _slot_dict(swa_bt[r], int(swa_base[r]) if swa_base is not None else 0, swa_bs)
        rs = int(replay[r]) if replay is not None else 0
        win = sorted(p for p in range(0, pos + 1) if p >= rs and p > pos - W)
        for c, p in enumerate(win):
            out[t, c] = sd.get(p, -1)
        cd = _slot_dict(comp_bt[r], int(comp_base[r]) if comp_base is not None else 0, comp_bs)
        for j in range(K):
            l = int(topk[t, j])
            if l >= 0:
                out[t, W + j] = cd.get(l, -1)
        lens[t] = int((out[t] >= 0).sum())
    return out, lens


def test_index_golden(oracle_mod):
    spec = json.load(open(os.path.join(GOLDEN, "index_golden.json")))
    for case in spec["cases"]:
        bt = np.array(case["block_table"], np.int32)
        topk = np.array(case["topk_local"], np.int32)
        valid = None if case["is_valid_token"] is None else np.array(case["is_valid_token"], np.uint8)
        swa_base = None if case["swa_base_offsets"] is None else np.array(case["swa_base_offsets"], np.int32)
        out, lens = oracle_mod.combine_topk_swa_indices(
            np.array(case["query_start_loc"], np.int32), np.array(case["seq_lens"], np.int32),
            np.array(case["token_to_req"], np.int32), np.array(case["replay_start"], np.int32),
            bt, case["block_size"], None, case["block_size"], case["window"],
            case["compress_ratio"], topk, swa_base_offsets=swa_base, is_valid_token=valid)
        assert out.tolist() == case["expected_indices"], case["name"]
        assert lens.tolist() == case["expected_lens"], case["name"]
        if "expected_global_topk" in case:
            g, gl = oracle_mod.compute_global_topk_indices_and_lens(
                topk, np.array(case["token_to_req"], np.int32), bt, case["block_size"],
                is_valid_token=valid)
            assert g.tolist() == case["expected_global_topk"]
            assert gl.tolist() == case["expected_global_lens"]


def _random_case(rng):
    bs = int(rng.choice([1, 2, 4, 16, 64]))
    W = int(rng.choice([1, 3, 4, 8, 128]))
    K = int(rng.choice([1, 5, 8, 13, 64]))
    R = int(rng.integers(1, 5))
    qlens = rng.integers(0, 6, size=R)
    seq = np.array([int(q) + int(rng.integers(0, 300)) for q in qlens], np.int32)
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    T = int(qsl[-1])
    t2r = np.repeat(np.arange(R, dtype=np.int32), qlens)
    if T and rng.random() < 0.3:
        t2r[rng.integers(0, T)] = int(rng.choice([-1, R, R + 3]))
    width = int(rng.integers(1, 12))
    pages = 40
    swa_bt = rng.integers(-1, pages, size=(R, width)).astype(np.int32)
    comp_bt = None if rng.random() < 0.3 else rng.integers(-1, pages, size=(R, width + 2)).astype(np.int32)
    swa_base = None if rng.random() < 0.5 else rng.integers(0, 4, size=R).astype(np.int32)
    comp_base = None if rng.random() < 0.5 else rng.integers(0, 3, size=R).astype(np.int32)
    replay = None if rng.random() < 0.3 else rng.integers(0, 310, size=R).astype(np.int32)
    topk = rng.integers(-1, max(1, 80), size=(T, K)).astype(np.int32)
    topk[rng.random(topk.shape) < 0.2] = -1
    valid = None if rng.random() < 0.5 else (rng.random(T) < 0.8).astype(np.uint8)
    return dict(bs=bs, W=W, K=K, qsl=qsl, seq=seq, t2r=t2r, swa_bt=swa_bt, comp_bt=comp_bt,
                swa_base=swa_base, comp_base=comp_base, replay=replay, topk=topk, valid=valid)


@pytest.mark.parametrize("seed", range(60))
def test_combine_vs_bruteforce_fuzz(oracle_mod, seed):
    rng = np.random.default_rng(1000 + seed)
    c = _random_case(rng)
    comp_bs = c["bs"] if rng.random() < 0.5 else int(rng.choice([1, 4, 16]))
    want, want_lens = _brute_combine(c["qsl"], c["seq"], c["t2r"], c["replay"], c["swa_bt"],
                                     c["swa_base"], c["bs"], c["comp_bt"], c["comp_base"],
                                     comp_bs, c["W"], c["topk"], c["valid"])
    replay = c["replay"] if c["replay"] is not None else np.zeros(len(c["seq"]), np.int32)
    got, lens = oracle_mod.combine_topk_swa_indices(
        c["qsl"], c["seq"], c["t2r"], replay, c["swa_bt"], c["bs"], c["comp_bt"], comp_bs,
        c["W"], 4, c["topk"], swa_base_offsets=c["swa_base"], comp_base_offsets=c["comp_base"],
        is_valid_token=c["valid"])
    assert np.array_equal(got, want)
    assert np.array_equal(lens, want_lens)


@pytest.mark.parametrize("seed", range(40))
def test_global_topk_vs_bruteforce_fuzz(oracle_mod, seed):
    rng = np.random.default_rng(2000 + seed)
    c = _random_case(rng)
    bt = c["comp_bt"] if c["comp_bt"] is not None else c["swa_bt"]
    T, K = c["topk"].shape
    want = np.full((T, K), -1, np.int64)
    R = bt.shape[0]
    for t in range(T):
        r = int(c["t2r"][t])
        if (c["valid"] is not None and not c["valid"][t]) or r < 0 or r >= R:
            continue
        d = _slot_dict(bt[r], int(c["comp_base"][r]) if c["comp_base"] is not None else 0, c["bs"])
        for j in range(K):
            l = int(c["topk"][t, j])
            if l >= 0:
                want[t, j] = d.get(l, -1)
    got, lens = oracle_mod.compute_global_topk_indices_and_lens(
        c["topk"], c["t2r"], bt, c["bs"], base_offsets=c["comp_base"], is_valid_token=c["valid"])
    assert np.array_equal(got, want)
    assert np.array_equal(lens, (want >= 0).sum(axis=1))


def test_slot_beyond_int32_is_invalid(oracle_mod):
    bt = np.array([[2**31 // 64 + 5, 1]], np.int32)
    topk = np.array([[0, 64, 65]], np.int32)
    g, gl = oracle_mod.compute_global_topk_indices_and_lens(
        topk, np.array([0], np.int32), bt, 64)
    assert g.tolist() == [[-1, 64, 65]] and gl.tolist() == [2]


@pytest.mark.parametrize("name", ["tiny", "decode", "mixed"])
def test_combine_invariants_on_workloads(oracle_mod, name):
    w = synthetic.make(name)
    out, lens = oracle_mod.combine_topk_swa_indices(
        w.query_start_loc, w.seq_lens, w.token_to_req, w.replay_start, w.swa_block_table,
        w.swa_cache.block_size, w.comp_block_table, w.comp_cache.block_size, w.window,
        w.compress_ratio, w.topk_local)
    W, K, P = w.window, w.topk, w.padded_topk
    assert out.shape == (w.num_tokens, W + P)
    assert np.array_equal(lens, (out >= 0).sum(axis=1))
    assert np.all(out[:, W + K:] == -1)
    assert np.all(lens <= W + K)
    # window columns: valid entries are a left-aligned run of consecutive
    # positions, so their slots step by one inside a page
    sw = out[:, :W]
    nvalid = (sw >= 0).sum(axis=1)
    for t in range(w.num_tokens):
        n = int(nvalid[t])
        assert np.all(sw[t, :n] >= 0) and np.all(sw[t, n:] == -1)
        bs = w.swa_cache.block_size
        for a, b in zip(sw[t, :n - 1], sw[t, 1:n]):
            assert b == a + 1 or (b % bs == 0 and (a + 1) % bs == 0)
    # the newest window entry is the token's own insert slot
    has = nvalid > 0
    last = sw[np.arange(w.num_tokens), np.maximum(nvalid - 1, 0)]
    assert np.array_equal(last[has], w.insert_slots[has])
    # every top-k slot is in one of the request's compressed pages
    bt = w.comp_block_table if w.comp_block_table is not None else w.swa_block_table
    cbs = w.comp_cache.block_size
    for t in range(0, w.num_tokens, max(1, w.num_tokens // 64)):
        pages = set(bt[w.token_to_req[t]].tolist()) - {-1}
        tk = out[t, W:W + K]
        assert all((s // cbs) in pages for s in tk[tk >= 0])
        # a top-k entry is -1 exactly where the local index is -1
        assert np.array_equal(tk >= 0, w.topk_local[t] >= 0)


def test_prefill_window_counts(oracle_mod):
    """Prefill with all tokens new: token at position p sees min(p+1, W)
    window entries and min(512, (p+1)//4) top-k entries."""
    w = synthetic.make("prefill")
    out, lens = oracle_mod.combine_topk_swa_indices(
        w.query_start_loc, w.seq_lens, w.token_to_req, w.replay_start, w.swa_block_table,
        w.swa_cache.block_size, w.comp_block_table, w.comp_cache.block_size, w.window,
        w.compress_ratio, w.topk_local)
    pos = np.tile(np.arange(4096), 4)
    want = np.minimum(pos + 1, w.window) + np.minimum(512, (pos + 1) // 4)
    assert np.array_equal(lens, want)


def test_mixed_replay_start_bounds_window(oracle_mod):
    w = synthetic.make("mixed")
    out, lens = oracle_mod.combine_topk_swa_indices(
        w.query_start_loc, w.seq_lens, w.token_to_req, w.replay_start, w.swa_block_table,
        w.swa_cache.block_size, w.comp_block_table, w.comp_cache.block_size, w.window,
        w.compress_ratio, w.topk_local)
    # prefill request r: token i sits at replay_start + i and sees min(i+1, W)
    for r in (256, 257):
        a, b = w.query_start_loc[r], w.query_start_loc[r + 1]
        i = np.arange(b - a)
        nwin = (out[a:b, :w.window] >= 0).sum(axis=1)
        assert np.array_equal(nwin, np.minimum(i + 1, w.window))
