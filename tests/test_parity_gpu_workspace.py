"""GPU parity for the prefill-workspace path: range-form gather, workspace
indices and raw MXFP4 gather, bit for bit against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_sparse_kv_gb300 import ops, synthetic

pytestmark = pytest.mark.gpu


def _i32(a, dev):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _workspace_geometry(w):
    W, ratio = w.window, w.compress_ratio
    seq = w.seq_lens.astype(np.int64)
    qlen = np.diff(w.query_start_loc).astype(np.int64)
    glen = (qlen + np.minimum(seq - qlen, max(W - 1, 0))).astype(np.int32)
    lc = (seq // ratio).astype(np.int32)
    cb = int(lc.max())
    return glen, lc, cb, cb + int(glen.max())


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.empty_cache()


@pytest.mark.parametrize("seed", range(16))
def test_range_gather_fuzz(cuda_device, seed):
    rng = np.random.default_rng(500 + seed)
    bs = int(rng.choice([1, 2, 3, 4, 5, 16, 64]))
    D, rope = [(128, 0), (512, 64), (256, 64)][seed % 3]
    ue8m0 = bool(seed % 4)
    R, width, pages = int(rng.integers(1, 5)), 7, 13
    table = rng.integers(-1, pages, size=(R, width)).astype(np.int32)
    base = None if rng.random() < 0.5 else rng.integers(0, 2, size=R).astype(np.int32)
    seq = rng.integers(0, (width + 1) * bs, size=R).astype(np.int32)
    glen = None if rng.random() < 0.3 else np.minimum(seq, rng.integers(0, 40, size=R)).astype(np.int32)
    rows, offset = int(rng.integers(8, 60)), int(rng.integers(0, 5))
    rec = oracle.fp8_record_bytes(D, rope, ue8m0)
    geom = synthetic.CacheGeom(pages, bs, (bs * rec + 15) // 16 * 16)
    if ue8m0:
        cache = synthetic.random_cache_bytes(seed, geom)
    else:
        cache = np.zeros((pages, geom.page_stride), np.uint8)
        k = torch.from_numpy(rng.standard_normal((pages * bs, D)).astype(np.float32)).to(
            torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        oracle.quantize_and_insert_k_cache(k, np.arange(pages * bs, dtype=np.int64), cache, bs,
                                           D, rope, False)
    want = np.full((R, rows, D), 0x1357, np.uint16)
    oracle.dequantize_and_gather_k_cache_ranges(want, cache, bs, 0, D, rope, seq, glen, table,
                                                offset, base_offsets=base, is_ue8m0=ue8m0)
    # the output is a strided view (extra rows and a gap between requests)
    big = torch.full((R, rows + 3, D), 0, dtype=torch.int16, device=cuda_device)
    big[:] = 0x1357
    out = big.view(torch.bfloat16)[:, :rows, :]
    ops.dequantize_and_gather_k_cache_ranges(out, torch.from_numpy(cache).to(cuda_device),
                                             _i32(seq, cuda_device), _i32(glen, cuda_device),
                                             _i32(table, cuda_device), bs, offset, rope_dim=rope,
                                             is_ue8m0=ue8m0, base_offsets=_i32(base, cuda_device))
    got = _u16(big)
    assert np.array_equal(got[:, :rows], want)
    assert np.all(got[:, rows:] == 0x1357)


@pytest.mark.parametrize("name", ["tiny", "prefill_small", "prefill", "mixed"])
def test_workspace_indices_match_oracle(cuda_device, name):
    w = synthetic.make(name)
    glen, lc, cb, ww = _workspace_geometry(w)
    d = cuda_device
    got, glens = ops.combine_topk_swa_workspace_indices(
        _i32(w.topk_local, d), _i32(w.query_start_loc, d), _i32(w.seq_lens, d), _i32(glen, d),
        _i32(w.token_to_req, d), w.window, w.compress_ratio, ww, cb)
    want, wlens = oracle.combine_topk_swa_workspace_indices(
        w.query_start_loc, w.seq_lens, glen, w.token_to_req, w.window, w.compress_ratio,
        w.topk_local, ww, cb)
    assert np.array_equal(got.cpu().numpy(), want)
    assert np.array_equal(glens.cpu().numpy(), wlens)


@pytest.mark.parametrize("seed", range(8))
def test_workspace_indices_fuzz(cuda_device, seed):
    """Odd windows and top-k widths (per-column path), padding tokens,
    request indices out of range."""
    rng = np.random.default_rng(700 + seed)
    R = int(rng.integers(1, 5))
    qlens = rng.integers(0, 7, size=R)
    seq = np.array([int(q) + int(rng.integers(0, 200)) for q in qlens], np.int32)
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    T = int(qsl[-1])
    t2r = np.repeat(np.arange(R, dtype=np.int32), qlens)
    if T:
        t2r[rng.integers(0, T)] = R + 1
    W = int(rng.choice([1, 3, 4, 8, 128]))
    K = int(rng.choice([1, 5, 8, 16]))
    ratio = int(rng.choice([1, 4, 128]))
    prefix = seq - qlens
    glen = (qlens + np.minimum(prefix, max(W - 1, 0))).astype(np.int32)
    lc = seq // ratio
    cb = int(lc.max()) if R else 0
    ww = cb + int(glen.max()) if R else 1
    topk = rng.integers(-1, 80, size=(T, K)).astype(np.int32)
    valid = (rng.random(T) < 0.8).astype(np.uint8)
    d = cuda_device
    got, gl = ops.combine_topk_swa_workspace_indices(
        _i32(topk, d), _i32(qsl, d), _i32(seq, d), _i32(glen, d), _i32(t2r, d), W, ratio, ww, cb,
        is_valid_token=torch.from_numpy(valid).to(d))
    want, wl = oracle.combine_topk_swa_workspace_indices(qsl, seq, glen, t2r, W, ratio, topk, ww,
                                                         cb, is_valid_token=valid)
    if T:
        assert np.array_equal(got.cpu().numpy(), want)
        assert np.array_equal(gl.cpu().numpy(), wl)


@pytest.mark.parametrize("case", ["window_rows_cross", "topk_rows_cross"])
def test_workspace_indices_int32_edges(cuda_device, case):
    """Workspace rows near INT32_MAX: request r's rows start at r * width, so a
    wide workspace puts one request's window rows (or top-k rows) across
    INT32_MAX -- those become -1, the rows below stay -- and the last request
    past it entirely (all -1, not counted in lens)."""
    rng = np.random.default_rng(31 if case == "window_rows_cross" else 32)
    R, W, ratio, K = 3, 128, 4, 64
    qlens = np.array([40, 50, 30])
    seq = np.array([900, 16000, 700], np.int32)
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    T = int(qsl[-1])
    t2r = np.repeat(np.arange(R, dtype=np.int32), qlens)
    glen = (qlens + np.minimum(seq - qlens, W - 1)).astype(np.int32)
    lc = seq // ratio
    if case == "window_rows_cross":
        ww = 1_100_000_000               # request 1 at 1.1e9, request 2 past INT32_MAX
        cb = 2_147_483_600 - ww          # request 1's window rows cross INT32_MAX
    else:
        ww = 2_147_480_000               # request 1's top-k rows cross at l = 3648
        cb = 8
    topk = np.where(rng.random((T, K)) < 0.1, -1,
                    rng.integers(0, np.repeat(lc, qlens)[:, None] + 1, size=(T, K))).astype(np.int32)
    topk[qsl[1]:qsl[2], :8] = np.arange(3640, 3648 + 8, 2, dtype=np.int32)[None, :8]
    d = cuda_device
    got, gl = ops.combine_topk_swa_workspace_indices(
        _i32(topk, d), _i32(qsl, d), _i32(seq, d), _i32(glen, d), _i32(t2r, d), W, ratio, ww, cb)
    want, wl = oracle.combine_topk_swa_workspace_indices(qsl, seq, glen, t2r, W, ratio, topk, ww,
                                                         cb)
    g = got.cpu().numpy()
    assert np.array_equal(g, want)
    assert np.array_equal(gl.cpu().numpy(), wl)
    # the case is what it says: request 1 has both kept and dropped rows, request 2 none
    r1 = want[qsl[1]:qsl[2]]
    part = r1[:, :W] if case == "window_rows_cross" else r1[:, W:]
    assert (part >= 0).any() and (part > 2_000_000_000).any()
    assert np.all(want[qsl[2]:qsl[3]] == -1) and np.all(wl[qsl[2]:qsl[3]] == 0)


def test_prefill_workspace_full_size(cuda_device):
    """Both range gathers into one workspace at the prefill workload's size."""
    w = synthetic.make("prefill")
    glen, lc, cb, ww = _workspace_geometry(w)
    d = cuda_device
    swa = synthetic.random_cache_bytes(31, w.swa_cache)
    comp = synthetic.random_cache_bytes(32, w.comp_cache)
    ws = torch.zeros((w.num_reqs, ww, w.head_dim), dtype=torch.bfloat16, device=d)
    table = _i32(w.swa_block_table, d)
    ops.dequantize_and_gather_k_cache_ranges(ws[:, :cb], torch.from_numpy(comp).to(d),
                                             _i32(lc, d), None, table, w.comp_cache.block_size, 0,
                                             rope_dim=w.rope_dim)
    ops.dequantize_and_gather_k_cache_ranges(ws, torch.from_numpy(swa).to(d),
                                             _i32(w.seq_lens, d), _i32(glen, d), table,
                                             w.swa_cache.block_size, cb, rope_dim=w.rope_dim)
    want = np.zeros((w.num_reqs, ww, w.head_dim), np.uint16)
    want_c = np.zeros((w.num_reqs, cb, w.head_dim), np.uint16)
    oracle.dequantize_and_gather_k_cache_ranges(want_c, comp, w.comp_cache.block_size, 0,
                                                w.head_dim, w.rope_dim, lc, None,
                                                w.swa_block_table, 0)
    want[:, :cb] = want_c
    oracle.dequantize_and_gather_k_cache_ranges(want, swa, w.swa_cache.block_size, 0, w.head_dim,
                                                w.rope_dim, w.seq_lens, glen, w.swa_block_table,
                                                cb)
    assert np.array_equal(_u16(ws), want)


@pytest.mark.parametrize("bs", [8, 6])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_mxfp4_raw_gather_fuzz(cuda_device, D, bs):
    rng = np.random.default_rng(D)
    pages, R = 17, 5
    rec = D // 2 + D // 32
    geom = synthetic.CacheGeom(pages, bs, (bs * rec + 15) // 16 * 16)
    cache = rng.integers(0, 256, size=(pages, geom.page_stride), dtype=np.uint8)
    table = rng.integers(-1, pages, size=(R, 6)).astype(np.int32)
    lens = rng.integers(0, 60, size=R)
    lens[1] = 0
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    d = cuda_device
    v, s = ops.indexer_mxfp4_paged_gather(torch.from_numpy(cache).to(d), _i32(table, d),
                                          _i32(cu, d), bs, D, int(cu[-1]))
    wv, ws = oracle.indexer_mxfp4_paged_gather(cache, bs, D, table, cu)
    assert np.array_equal(v.cpu().numpy(), wv)
    assert np.array_equal(s.cpu().numpy(), ws)


def test_mxfp4_raw_gather_indexer_workload(cuda_device):
    """Every compressed key of 16 of the 128 indexer requests (32768 each)."""
    w = synthetic.make("mxfp4")
    R = 16
    table = w.comp_block_table[:R]
    lens = np.full(R, w.seq_lens[0] // w.compress_ratio)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cache = synthetic.random_cache_bytes(33, w.index_cache)
    d = cuda_device
    v, s = ops.indexer_mxfp4_paged_gather(torch.from_numpy(cache).to(d), _i32(table, d),
                                          _i32(cu, d), w.index_cache.block_size, 128, int(cu[-1]))
    wv, ws = oracle.indexer_mxfp4_paged_gather(cache, w.index_cache.block_size, 128, table, cu)
    assert np.array_equal(v.cpu().numpy(), wv)
    assert np.array_equal(s.cpu().numpy(), ws)


@pytest.mark.parametrize("name,mode", [("tiny", "serial"), ("prefill_small", "concurrent"),
                                       ("prefill", "graph")])
def test_workspace_step_matches_oracle(cuda_device, name, mode):
    """The whole prefill workspace step as the benchmark launches it."""
    from oracle.pipeline import run_workspace_step
    from paged_sparse_kv_gb300.pipeline import Pipeline, workspace_geometry
    w = synthetic.make(name)
    geom = workspace_geometry(w)
    host = {c: synthetic.random_cache_bytes(60 + i, getattr(w, c))
            for i, c in enumerate(("swa_cache", "comp_cache", "index_cache"))}
    p = Pipeline(w, cuda_device)
    for c, arr in host.items():
        getattr(p, c).copy_(torch.from_numpy(arr))
    p.alloc_workspace()
    if mode == "graph":
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(cuda_device)
        side.wait_stream(torch.cuda.current_stream(cuda_device))
        with torch.cuda.graph(g, stream=side):
            p.step(concurrent=True, path="workspace")
        g.replay()
    else:
        p.step(concurrent=(mode == "concurrent"), path="workspace")
    torch.cuda.synchronize()
    ref = run_workspace_step(w, geom, host["swa_cache"], host["comp_cache"], host["index_cache"])
    for c, arr in host.items():
        assert np.array_equal(getattr(p, c).cpu().numpy(), arr), c
    cb = geom["compressed_base"]
    ws = _u16(p.ws)
    for r in range(w.num_reqs):
        lc, gl = int(geom["compressed_lens"][r]), int(geom["gather_lens"][r])
        assert np.array_equal(ws[r, :lc], ref["workspace_compressed"][r, :lc])
        assert np.array_equal(ws[r, cb:cb + gl], ref["workspace_window"][r, :gl])
    assert np.array_equal(p.ws_indices.cpu().numpy(), ref["ws_indices"])
    assert np.array_equal(p.ws_lens.cpu().numpy(), ref["ws_lens"])
    assert np.array_equal(p.raw_values.cpu().numpy(), ref["raw_values"])
    assert np.array_equal(p.raw_scales.cpu().numpy(), ref["raw_scales"])
    assert int(p.err.item()) == ref["err"]
