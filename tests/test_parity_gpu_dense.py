"""GPU parity for the dense index builders (decode SWA indices, HCA dense
compressed indices, dense prefill local indices, SWA-only workspace combine)
and the dense decode step, bit for bit against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle.pipeline import run_dense_step
from paged_sparse_kv_gb300 import ops, synthetic
from paged_sparse_kv_gb300.pipeline import Pipeline

pytestmark = pytest.mark.gpu


def _i32(a, dev):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def _i64(a, dev):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).to(dev)


def _u8(a, dev):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(dev)


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _out(T, cols, extra, dev, fill=-7):
    """An output [T, cols] as a view of a wider buffer (row stride cols + extra,
    shifted by one column when extra is odd so rows are not 16-byte aligned)."""
    shift = extra % 2
    big = torch.full((T, cols + extra), fill, dtype=torch.int32, device=dev)
    return big, big[:, shift:shift + cols]


@pytest.mark.parametrize("seed", range(24))
def test_decode_swa_fuzz(cuda_device, seed):
    rng = np.random.default_rng(100 + seed)
    d = cuda_device
    R = int(rng.integers(1, 6))
    bs = int(rng.choice([1, 2, 3, 4, 16, 64]))
    W = int(rng.choice([1, 3, 4, 8, 12, 128]))
    qlen = rng.integers(0, 5, size=R)
    seq = (qlen + rng.integers(0, 300, size=R)).astype(np.int32)
    qsl = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    T = int(qsl[-1])
    t2r = np.repeat(np.arange(R), qlen).astype(np.int32)
    if T and rng.random() < 0.3:
        t2r[rng.integers(0, T)] = R
    valid = None if rng.random() < 0.5 else (rng.random(T) < 0.8)
    width = int(rng.integers(1, 300 // bs + 3))
    bt = rng.integers(-1, 40, size=(R, width)).astype(np.int32)
    base = None if rng.random() < 0.5 else rng.integers(0, 2, size=R).astype(np.int32)
    want, wl = oracle.decode_swa_indices_and_lens(qsl, seq, t2r, bt, bs, W, base_offsets=base,
                                                  is_valid_token=valid)
    extra = int(rng.choice([0, 1, 4]))
    big, out = _out(T, W, extra, d)
    lens = torch.full((T,), -9, dtype=torch.int32, device=d)
    ops.decode_swa_indices_and_lens(_i32(qsl, d), _i32(seq, d), _i32(t2r, d), _i32(bt, d), bs, W,
                                    base_offsets=_i32(base, d), is_valid_token=_u8(valid, d),
                                    out=out, lens=lens)
    assert np.array_equal(out.cpu().numpy(), want)
    assert np.array_equal(lens.cpu().numpy(), wl)
    g = big.cpu().numpy()
    if extra:  # columns outside the view are untouched
        rest = np.concatenate([g[:, :extra % 2], g[:, extra % 2 + W:]], axis=1)
        assert np.all(rest == -7)


@pytest.mark.parametrize("seed", range(24))
def test_dense_compressed_fuzz(cuda_device, seed):
    rng = np.random.default_rng(200 + seed)
    d = cuda_device
    R = int(rng.integers(1, 6))
    T = int(rng.integers(0, 200))
    bs = int(rng.choice([1, 2, 3, 4, 16, 64]))
    ratio = int(rng.choice([1, 2, 4, 7, 128]))
    width = int(rng.choice([0, 1, 5, 8, 64, 130]))
    pos = rng.integers(-3, 20000, size=T).astype(np.int64)
    if T:
        pos[0] = 2**40  # clamps to width
    t2r = rng.integers(0, R + 1, size=T).astype(np.int32)
    valid = None if rng.random() < 0.5 else (rng.random(T) < 0.8)
    bt = rng.integers(-1, 50, size=(R, int(rng.integers(1, 40)))).astype(np.int32)
    base = None if rng.random() < 0.5 else rng.integers(0, 3, size=R).astype(np.int32)
    want, wl = oracle.compute_dense_compressed_indices_and_lens(
        pos, t2r, bt, bs, ratio, width, base_offsets=base, is_valid_token=valid)
    extra = int(rng.choice([0, 1, 4]))
    big, out = _out(T, width, extra, d)
    lens = torch.full((T,), -9, dtype=torch.int32, device=d)
    ops.compute_dense_compressed_indices_and_lens(
        _i64(pos, d), _i32(t2r, d), _i32(bt, d), bs, ratio, width, base_offsets=_i32(base, d),
        is_valid_token=_u8(valid, d), out=out, lens=lens)
    assert np.array_equal(out.cpu().numpy(), want)
    assert np.array_equal(lens.cpu().numpy(), wl)


def test_dense_compressed_int32_extremes(cuda_device):
    """Pages whose slots straddle INT32_MAX, for a power-of-two and an odd page size."""
    d = cuda_device
    for bs in (64, 3):
        imax = 2**31 - 1
        maxp = imax // bs
        bt = np.array([[maxp - 1, maxp, maxp + 1, -1, 0, 2**31 - 1]], np.int32)
        T, width = 3, 6 * bs
        pos = np.array([width * 1 - 1, 3 * bs, 10**9], np.int64)
        t2r = np.zeros(T, np.int32)
        want, wl = oracle.compute_dense_compressed_indices_and_lens(pos, t2r, bt, bs, 1, width)
        out, lens = ops.compute_dense_compressed_indices_and_lens(_i64(pos, d), _i32(t2r, d),
                                                                  _i32(bt, d), bs, 1, width)
        assert np.array_equal(out.cpu().numpy(), want)
        assert np.array_equal(lens.cpu().numpy(), wl)


@pytest.mark.parametrize("seed", range(12))
def test_dense_local_fuzz(cuda_device, seed):
    rng = np.random.default_rng(300 + seed)
    d = cuda_device
    T = int(rng.integers(0, 500))
    ratio = int(rng.choice([1, 2, 4, 128]))
    width = int(rng.choice([1, 3, 4, 33, 64, 1024]))
    pos = rng.integers(-5, 140000, size=T).astype(np.int64)
    want = oracle.build_dense_prefill_local_compressed_indices(pos, ratio, width)
    extra = int(rng.choice([0, 1, 4]))
    big, out = _out(T, width, extra, d)
    ops.build_dense_prefill_local_compressed_indices(_i64(pos, d), ratio, width, out=out)
    assert np.array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("seed", range(16))
def test_dense_swa_fuzz(cuda_device, seed):
    rng = np.random.default_rng(400 + seed)
    d = cuda_device
    R = int(rng.integers(1, 6))
    W = int(rng.choice([1, 4, 7, 8, 128]))
    qlen = rng.integers(0, 40, size=R)
    seq = (qlen + rng.integers(0, 300, size=R)).astype(np.int32)
    glen = np.minimum(seq, qlen + rng.integers(0, W + 3, size=R)).astype(np.int32)
    qsl = np.concatenate([[0], np.cumsum(qlen)])
    T = int(qsl[-1])
    t2r = np.repeat(np.arange(R), qlen).astype(np.int32)
    if T and rng.random() < 0.3:
        t2r[rng.integers(0, T)] = -1
    pos = np.array([int(seq[t2r[t]]) - int(qlen[t2r[t]]) + t - int(qsl[t2r[t]])
                    if t2r[t] >= 0 else 5 for t in range(T)], np.int64)
    cb = int(rng.integers(0, 50))
    ww = cb + int(glen.max()) + int(rng.integers(0, 3))
    want, wl = oracle.combine_dense_swa_indices(pos, t2r, seq, glen, W, ww, cb)
    extra = int(rng.choice([0, 1, 4]))
    big, out = _out(T, W, extra, d)
    lens = torch.full((T,), -9, dtype=torch.int32, device=d)
    ops.combine_dense_swa_indices(_i64(pos, d), _i32(t2r, d), _i32(seq, d), _i32(glen, d), W, ww,
                                  cb, out=out, lens=lens)
    assert np.array_equal(out.cpu().numpy(), want)
    assert np.array_equal(lens.cpu().numpy(), wl)


@pytest.mark.parametrize("name", ["prefill", "mixed"])
def test_dense_prefill_builders_at_workload_size(cuda_device, name):
    """The HCA prefill route (dense local indices -> workspace combine) and the
    SWA-only combine on every token of the prefill and mixed batches."""
    d = cuda_device
    w = synthetic.make(name)
    qlen = np.diff(w.query_start_loc).astype(np.int64)
    seq = w.seq_lens.astype(np.int64)
    pos = np.concatenate([np.arange(s - q, s) for s, q in zip(seq, qlen)]).astype(np.int64)
    ratio, width = 128, 256
    local = oracle.build_dense_prefill_local_compressed_indices(pos, ratio, width)
    got = ops.build_dense_prefill_local_compressed_indices(_i64(pos, d), ratio, width)
    assert np.array_equal(got.cpu().numpy(), local)
    glen = (qlen + np.minimum(seq - qlen, w.window - 1)).astype(np.int32)
    lc = (seq // ratio).astype(np.int32)
    cb = int(lc.max())
    ww = cb + int(glen.max())
    want, wl = oracle.combine_topk_swa_workspace_indices(
        w.query_start_loc, w.seq_lens, glen, w.token_to_req, w.window, ratio, local, ww, cb)
    gi, gl = ops.combine_topk_swa_workspace_indices(
        got, _i32(w.query_start_loc, d), _i32(w.seq_lens, d), _i32(glen, d),
        _i32(w.token_to_req, d), w.window, ratio, ww, cb)
    assert np.array_equal(gi.cpu().numpy(), want) and np.array_equal(gl.cpu().numpy(), wl)
    # SWA-only layer: no compressed part, compressed_base 0
    ww0 = int(glen.max())
    want, wl = oracle.combine_dense_swa_indices(pos, w.token_to_req, w.seq_lens, glen, w.window,
                                                ww0, 0)
    gi, gl = ops.combine_dense_swa_indices(_i64(pos, d), _i32(w.token_to_req, d),
                                           _i32(w.seq_lens, d), _i32(glen, d), w.window, ww0, 0)
    assert np.array_equal(gi.cpu().numpy(), want) and np.array_equal(gl.cpu().numpy(), wl)


@pytest.mark.parametrize("name", ["decode", "mixed"])
def test_decode_swa_at_workload_size(cuda_device, name):
    d = cuda_device
    w = synthetic.make(name)
    want, wl = oracle.decode_swa_indices_and_lens(
        w.query_start_loc, w.seq_lens, w.token_to_req, w.swa_block_table,
        w.swa_cache.block_size, w.window, is_valid_token=w.is_valid_token)
    valid = None if w.is_valid_token is None else _u8(w.is_valid_token, d)
    out, lens = ops.decode_swa_indices_and_lens(
        _i32(w.query_start_loc, d), _i32(w.seq_lens, d), _i32(w.token_to_req, d),
        _i32(w.swa_block_table, d), w.swa_cache.block_size, w.window, is_valid_token=valid)
    assert np.array_equal(out.cpu().numpy(), want) and np.array_equal(lens.cpu().numpy(), wl)


@pytest.mark.parametrize("path", ["dense", "dense_fused"])
@pytest.mark.parametrize("mode", ["serial", "concurrent", "graph"])
def test_dense_step_matches_oracle(cuda_device, mode, path):
    """The whole dense decode step as the benchmark launches it (builders then
    gathers, or gathers that compute their own slots beside the builders)."""
    w = synthetic.make("decode_hca")
    p = Pipeline(w, cuda_device)
    swa = synthetic.random_cache_bytes(61, w.swa_cache)
    comp = synthetic.random_cache_bytes(62, w.comp_cache)
    p.swa_cache.copy_(torch.from_numpy(swa))
    p.comp_cache.copy_(torch.from_numpy(comp))
    p.alloc_dense()
    if mode == "graph":
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(cuda_device)
        side.wait_stream(torch.cuda.current_stream(cuda_device))
        with torch.cuda.graph(g, stream=side):
            p.step(concurrent=True, path=path)
        torch.cuda.synchronize()
        assert np.array_equal(p.swa_cache.cpu().numpy(), swa)  # capture launched nothing
        g.replay()
    else:
        p.step(concurrent=(mode == "concurrent"), path=path)
    torch.cuda.synchronize(cuda_device)
    want = run_dense_step(w, swa, comp)
    assert np.array_equal(p.swa_indices.cpu().numpy(), want["swa_indices"])
    assert np.array_equal(p.swa_lens.cpu().numpy(), want["swa_lens"])
    assert np.array_equal(p.dense_indices.cpu().numpy(), want["dense_indices"])
    assert np.array_equal(p.dense_lens.cpu().numpy(), want["dense_lens"])
    assert np.array_equal(_u16(p.dense_gathered), want["gathered"])
    assert np.array_equal(p.swa_cache.cpu().numpy(), swa)
    assert int(p.err.item()) == want["err"]


@pytest.mark.parametrize("bs,ratio,width", [(64, 128, 40), (5, 3, 12), (16, 4, 64)])
def test_dense_gather_matches_builder_then_gather(cuda_device, bs, ratio, width):
    """dequantize_and_gather_k_cache_dense == compute_dense_compressed_indices_and_lens
    + dequantize_and_gather_k_cache: negative and large positions, padding and
    out-of-range requests, base offsets, -1 pages and pages past the int32 slot
    range, visible counts below and above the width."""
    rng = np.random.default_rng(bs * 7 + ratio + width)
    d = cuda_device
    R, T, bt_w, pages, D, rope = 5, 97, 30, 40, 512, 64
    table = rng.integers(-1, pages, size=(R, bt_w)).astype(np.int32)
    table[0, 3] = (2**31 - 1) // bs + 1  # slots past INT32_MAX
    base = rng.integers(0, 3, size=R).astype(np.int32)
    t2r = rng.integers(0, R, size=T).astype(np.int32)
    t2r[::13] = R  # out of range
    pos = rng.integers(-5, (bt_w + 3) * bs * ratio // max(ratio, 1), size=T).astype(np.int64)
    pos[1] = 2**40
    valid = (rng.random(T) < 0.9).astype(np.uint8)
    rec = oracle.fp8_record_bytes(D, rope, True)
    geom = synthetic.CacheGeom(pages, bs, (bs * rec + 15) // 16 * 16)
    host = synthetic.random_cache_bytes(77, geom)
    idx, _ = oracle.compute_dense_compressed_indices_and_lens(
        pos, t2r, table, bs, ratio, width, base_offsets=base, is_valid_token=valid)
    want = oracle.dequantize_and_gather_k_cache(host, bs, 0, D, rope, idx)
    out = torch.full((T, width + 1, D), 9, dtype=torch.bfloat16, device=d)
    ops.dequantize_and_gather_k_cache_dense(
        out[:, :width], torch.from_numpy(host).to(d), torch.from_numpy(pos).to(d),
        torch.from_numpy(t2r).to(d), torch.from_numpy(table).to(d), bs, ratio, rope_dim=rope,
        num_reqs=R, base_offsets=torch.from_numpy(base).to(d),
        is_valid_token=torch.from_numpy(valid).to(d))
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got[:, :width], want)
    nine = np.uint16(torch.tensor(9.0, dtype=torch.bfloat16).view(torch.int16).item())
    assert np.all(got[:, width] == nine)
    assert (idx >= 0).any() and (idx < 0).any()
