"""Pins for the oracle's dense index builders (decode SWA indices, HCA dense
compressed indices, dense prefill local indices, SWA-only workspace combine).

* Hand-worked golden cases (tests/golden/dense_golden.json).
* Brute-force enumeration written from the definitions: a request's pages are
  walked to build a dictionary position -> slot; the window is the sorted set
  of positions satisfying the window predicates; dense entries are look-ups of
  0..n-1 with n counted by repeated subtraction, not by a division.
* The decode SWA indices equal the window part of the fused builder with no
  top-k and no replay_start (a second, independently written oracle function).
"""
import json
import os

import numpy as np
import pytest

from conftest import GOLDEN


def _slot_dict(row, base, bs):
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


def _visible(pos, ratio, width):
    """floor((pos+1)/ratio) clamped to [0, width], by counting whole groups."""
    n, rest = 0, pos + 1
    while rest >= ratio and n < width:
        rest -= ratio
        n += 1
    return n


@pytest.fixture(scope="module")
def gold():
    with open(os.path.join(GOLDEN, "dense_golden.json")) as f:
        return json.load(f)


def test_decode_swa_golden(oracle_mod, gold):
    g = gold["decode_swa"]
    a = [np.array(g[k], np.int32) for k in ("query_start_loc", "seq_lens", "token_to_req")]
    bt = np.array(g["block_table"], np.int32)
    out, lens = oracle_mod.decode_swa_indices_and_lens(*a, bt, g["block_size"], g["window"])
    assert out.tolist() == g["expected"] and lens.tolist() == g["expected_lens"]
    out, lens = oracle_mod.decode_swa_indices_and_lens(
        *a, bt, g["block_size"], g["window"], base_offsets=np.array(g["base_offsets"], np.int32))
    assert out.tolist() == g["expected_base"] and lens.tolist() == g["expected_base_lens"]
    out, lens = oracle_mod.decode_swa_indices_and_lens(
        *a, bt, g["block_size"], g["window"], is_valid_token=np.array(g["is_valid_token"]))
    assert out.tolist() == g["expected_valid"] and lens.tolist() == g["expected_valid_lens"]


def test_dense_compressed_golden(oracle_mod, gold):
    g = gold["dense_compressed"]
    pos = np.array(g["positions"], np.int64)
    t2r = np.array(g["token_to_req"], np.int32)
    bt = np.array(g["block_table"], np.int32)
    args = (pos, t2r, bt, g["block_size"], g["compress_ratio"], g["width"])
    out, lens = oracle_mod.compute_dense_compressed_indices_and_lens(*args)
    assert out.tolist() == g["expected"] and lens.tolist() == g["expected_lens"]
    out, lens = oracle_mod.compute_dense_compressed_indices_and_lens(
        *args, base_offsets=np.array(g["base_offsets"], np.int32))
    assert out.tolist() == g["expected_base"] and lens.tolist() == g["expected_base_lens"]
    out, lens = oracle_mod.compute_dense_compressed_indices_and_lens(
        *args, is_valid_token=np.array(g["is_valid_token"]))
    assert out.tolist() == g["expected_valid"] and lens.tolist() == g["expected_valid_lens"]


def test_dense_local_golden(oracle_mod, gold):
    g = gold["dense_local"]
    out = oracle_mod.build_dense_prefill_local_compressed_indices(
        np.array(g["positions"], np.int64), g["compress_ratio"], g["width"])
    assert out.tolist() == g["expected"]


def test_dense_swa_golden(oracle_mod, gold):
    g = gold["dense_swa"]
    pos = np.array(g["positions"], np.int64)
    t2r = np.array(g["token_to_req"], np.int32)
    seq = np.array(g["seq_lens"], np.int32)
    out, lens = oracle_mod.combine_dense_swa_indices(
        pos, t2r, seq, np.array(g["gather_lens"], np.int32), g["window"], g["workspace_width"],
        g["compressed_base"])
    assert out.tolist() == g["expected"] and lens.tolist() == g["expected_lens"]
    out, _ = oracle_mod.combine_dense_swa_indices(
        pos, t2r, seq, np.array(g["gather_lens"], np.int32), g["window"],
        g["workspace_width_2"], g["compressed_base_2"])
    assert out.tolist() == g["expected_2"]
    out, lens = oracle_mod.combine_dense_swa_indices(
        pos, t2r, seq, np.array(g["gather_lens_3"], np.int32), g["window"],
        g["workspace_width"], g["compressed_base"])
    assert out.tolist() == g["expected_3"] and lens.tolist() == g["expected_3_lens"]


def _random_tables(rng, R, width, pages, base_max):
    bt = rng.integers(-1, pages, size=(R, width)).astype(np.int32)
    base = None if rng.random() < 0.4 else rng.integers(0, base_max + 1, size=R).astype(np.int32)
    return bt, base


@pytest.mark.parametrize("seed", range(40))
def test_decode_swa_vs_enumeration(oracle_mod, seed):
    rng = np.random.default_rng(900 + seed)
    R = int(rng.integers(1, 5))
    bs = int(rng.choice([1, 2, 3, 4, 8]))
    W = int(rng.integers(1, 12))
    qlen = rng.integers(0, 4, size=R)
    seq = (qlen + rng.integers(0, 20, size=R)).astype(np.int32)
    qsl = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    T = int(qsl[-1])
    t2r = np.repeat(np.arange(R), qlen).astype(np.int32)
    if T and rng.random() < 0.3:
        t2r[rng.integers(0, T)] = R  # a request index out of range
    valid = None if rng.random() < 0.5 else rng.random(T) < 0.8
    bt, base = _random_tables(rng, R, int(rng.integers(1, 8)), 12, 2)
    out, lens = oracle_mod.decode_swa_indices_and_lens(qsl, seq, t2r, bt, bs, W,
                                                       base_offsets=base, is_valid_token=valid)
    for t in range(T):
        r = int(t2r[t])
        if r >= R or (valid is not None and not valid[t]):
            assert np.all(out[t] == -1) and lens[t] == 0
            continue
        pos = int(seq[r]) - int(qlen[r]) + (t - int(qsl[r]))
        d = _slot_dict(bt[r], int(base[r]) if base is not None else 0, bs)
        win = sorted(p for p in range(0, pos + 1) if p > pos - W)
        want = [d.get(p, -1) for p in win] + [-1] * (W - len(win))
        assert out[t].tolist() == want
        assert lens[t] == sum(v >= 0 for v in want)


@pytest.mark.parametrize("seed", range(40))
def test_dense_compressed_vs_enumeration(oracle_mod, seed):
    rng = np.random.default_rng(1900 + seed)
    R = int(rng.integers(1, 5))
    T = int(rng.integers(0, 12))
    bs = int(rng.choice([1, 2, 3, 4, 16]))
    ratio = int(rng.choice([1, 2, 3, 4, 128]))
    width = int(rng.integers(0, 24))
    pos = rng.integers(-3, 400, size=T).astype(np.int64)
    t2r = rng.integers(0, R + 1, size=T).astype(np.int32)  # R = out of range
    valid = None if rng.random() < 0.5 else rng.random(T) < 0.8
    bt, base = _random_tables(rng, R, int(rng.integers(1, 8)), 12, 1)
    out, lens = oracle_mod.compute_dense_compressed_indices_and_lens(
        pos, t2r, bt, bs, ratio, width, base_offsets=base, is_valid_token=valid)
    assert out.shape == (T, width)
    for t in range(T):
        r = int(t2r[t])
        if r >= R or (valid is not None and not valid[t]):
            assert np.all(out[t] == -1) and lens[t] == 0
            continue
        n = _visible(int(pos[t]), ratio, width)
        d = _slot_dict(bt[r], int(base[r]) if base is not None else 0, bs)
        assert out[t].tolist() == [d.get(j, -1) if j < n else -1 for j in range(width)]
        assert lens[t] == n


@pytest.mark.parametrize("seed", range(20))
def test_dense_local_vs_counting(oracle_mod, seed):
    rng = np.random.default_rng(2900 + seed)
    ratio = int(rng.choice([1, 2, 4, 128]))
    width = int(rng.integers(0, 40))
    pos = rng.integers(-5, 6000, size=int(rng.integers(0, 30))).astype(np.int64)
    out = oracle_mod.build_dense_prefill_local_compressed_indices(pos, ratio, width)
    for t, p in enumerate(pos):
        n = _visible(int(p), ratio, width)
        assert out[t].tolist() == list(range(n)) + [-1] * (width - n)


@pytest.mark.parametrize("seed", range(30))
def test_dense_swa_vs_enumeration(oracle_mod, seed):
    rng = np.random.default_rng(3900 + seed)
    R = int(rng.integers(1, 5))
    W = int(rng.integers(1, 10))
    qlen = rng.integers(0, 5, size=R)
    seq = (qlen + rng.integers(0, 20, size=R)).astype(np.int32)
    glen = np.minimum(seq, qlen + rng.integers(0, W + 2, size=R)).astype(np.int32)
    qsl = np.concatenate([[0], np.cumsum(qlen)])
    T = int(qsl[-1])
    t2r = np.repeat(np.arange(R), qlen).astype(np.int32)
    if T and rng.random() < 0.3:
        t2r[rng.integers(0, T)] = -1
    pos = np.array([int(seq[t2r[t]]) - int(qlen[t2r[t]]) + t - int(qsl[t2r[t]])
                    if t2r[t] >= 0 else 0 for t in range(T)], np.int64)
    cb = int(rng.integers(0, 5))
    ww = cb + int(glen.max()) + int(rng.integers(0, 3))
    out, lens = oracle_mod.combine_dense_swa_indices(pos, t2r, seq, glen, W, ww, cb)
    for t in range(T):
        r = int(t2r[t])
        if r < 0:
            assert np.all(out[t] == -1) and lens[t] == 0
            continue
        g0 = int(seq[r]) - int(glen[r])
        # the workspace rows of request r: position g0 + i at row r*ww + cb + i
        rows = {g0 + i: r * ww + cb + i for i in range(int(glen[r]))}
        win = sorted(p for p in range(0, int(pos[t]) + 1) if p > int(pos[t]) - W)
        want = [rows.get(p, -1) for p in win] + [-1] * (W - len(win))
        assert out[t].tolist() == want and lens[t] == sum(v >= 0 for v in want)


@pytest.mark.parametrize("name", ["tiny", "decode", "mixed"])
def test_decode_swa_matches_fused_window_part(oracle_mod, name):
    from paged_sparse_kv_gb300 import synthetic
    w = synthetic.make(name)
    bs = w.swa_cache.block_size
    out, lens = oracle_mod.decode_swa_indices_and_lens(
        w.query_start_loc, w.seq_lens, w.token_to_req, w.swa_block_table, bs, w.window,
        is_valid_token=w.is_valid_token)
    empty = np.zeros((w.num_tokens, 0), np.int32)
    si, sl = oracle_mod.combine_topk_swa_indices(
        w.query_start_loc, w.seq_lens, w.token_to_req, None, w.swa_block_table, bs,
        w.comp_block_table, w.comp_cache.block_size, w.window, w.compress_ratio, empty,
        is_valid_token=w.is_valid_token)
    assert np.array_equal(out, si[:, :w.window]) and np.array_equal(lens, sl)
