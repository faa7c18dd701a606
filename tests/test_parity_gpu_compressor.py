"""GPU parity for the compressed-KV producer: the compressor-state writer and
the window-pooled compressed-row insert, byte for byte (and float bit for
float bit) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_sparse_kv_gb300 import ops, synthetic
from test_parity_gpu import _assert_same

pytestmark = pytest.mark.gpu


def _t(a, dev, dtype=None):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a).to(dev) if dtype is None else torch.from_numpy(a).to(dev, dtype)


@pytest.mark.parametrize("sw,pad", [(512, 0), (1024, 8)])
def test_save_state_fuzz(cuda_device, sw, pad):
    rng = np.random.default_rng(sw + pad)
    d = cuda_device
    T, ratio, bs, pages = 300, 4 if sw == 1024 else 128, 16, 30
    kv = rng.standard_normal((T, sw + pad)).astype(np.float32)
    score = rng.standard_normal((T, sw + pad)).astype(np.float32) * 3
    ape = rng.standard_normal((ratio, sw)).astype(np.float32)
    pos = rng.integers(-5, 5000, size=T).astype(np.int64)
    slots = rng.permutation(pages * bs)[:T].astype(np.int64)
    slots[::7] = -1
    slots[3] = pages * bs + 2
    host = rng.standard_normal((pages, bs, 2 * sw)).astype(np.float32)
    dev_state = _t(host, d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    ops.save_compressor_state(_t(kv, d)[:, :sw], _t(score, d)[:, :sw], _t(ape, d), dev_state,
                              _t(slots, d), _t(pos, d), bs, ratio, err_count=err)
    n = oracle.save_compressor_state(np.ascontiguousarray(kv[:, :sw]),
                                     np.ascontiguousarray(score[:, :sw]), ape, slots, pos, ratio,
                                     host, bs)
    got = dev_state.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), host.view(np.uint32))
    assert int(err.item()) == n == 1


def _gptj(max_pos):
    return synthetic.gptj_cos_sin(max_pos)


def _compress_case(rng, ratio, overlap, bs_state, kv_bs, R=3, T=260):
    sw = (2 if overlap else 1) * 512
    width = 12
    spages = R * width + 3
    state = rng.standard_normal((spages, bs_state, 2 * sw)).astype(np.float32)
    state[:, :, sw:] *= 4.0  # scores
    table = rng.permutation(spages)[: R * width].reshape(R, width).astype(np.int32)
    table[rng.random(table.shape) < 0.1] = -1
    base = None if rng.random() < 0.5 else rng.integers(0, 2, size=R).astype(np.int32)
    t2r = rng.integers(0, R, size=T).astype(np.int32)
    hi = (width + 1) * bs_state
    pos = rng.integers(-4, hi, size=T).astype(np.int64)
    # most tokens close a group so that many rows are written
    pos[: T // 2] = (pos[: T // 2] // ratio) * ratio + ratio - 1
    sslots = rng.integers(0, 5, size=T).astype(np.int64)
    sslots[::11] = -1
    kv_pages = (T + kv_bs - 1) // kv_bs + 2
    kv_slots = rng.permutation(kv_pages * kv_bs)[:T].astype(np.int64)
    kv_slots[::13] = -1
    kv_slots[5] = kv_pages * kv_bs + 1
    return sw, state, table, base, t2r, pos, sslots, kv_pages, kv_slots


@pytest.mark.parametrize("kv_bs", [64, 5])
@pytest.mark.parametrize("ratio,overlap,bs_state", [(4, True, 8), (4, True, 3), (128, False, 64),
                                                    (128, False, 7), (2, False, 4), (8, True, 16),
                                                    (1, False, 4), (3, True, 5)])
def test_compress_fuzz(cuda_device, ratio, overlap, bs_state, kv_bs):
    rng = np.random.default_rng(ratio * 100 + bs_state + kv_bs)
    d = cuda_device
    sw, state, table, base, t2r, pos, sslots, kv_pages, kv_slots = _compress_case(
        rng, ratio, overlap, bs_state, kv_bs)
    max_pos = int(pos.max()) - 3  # a few RoPE rows out of range
    cs = _gptj(max(max_pos, 1))
    w = rng.uniform(0.5, 2.0, size=512).astype(np.float32)
    eps = 1e-6
    stride = (kv_bs * 584 + 15) // 16 * 16
    host = synthetic.random_cache_bytes(3, synthetic.CacheGeom(kv_pages, kv_bs, stride))
    dev_cache = _t(host, d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    ops.compress_kv_cache_insert(_t(state, d), _t(t2r, d), _t(pos, d), _t(sslots, d),
                                 _t(table, d), bs_state, _t(w, d), eps, _t(cs, d), dev_cache,
                                 _t(kv_slots, d), kv_bs, ratio, overlap=overlap,
                                 block_table_base_offsets=None if base is None else _t(base, d),
                                 err_count=err)
    n = oracle.compress_kv_cache_insert(state, t2r, pos, sslots, table, bs_state, w, eps, cs,
                                        host, kv_slots, kv_bs, ratio, overlap,
                                        base_offsets=base)
    _assert_same(dev_cache.cpu().numpy(), host, f"compress ratio={ratio} overlap={overlap}")
    assert int(err.item()) == n and n >= 1


@pytest.mark.parametrize("ratio,overlap", [(4, True), (128, False)])
def test_compress_rsqrt_reading(cuda_device, ratio, overlap):
    """The pooled row on which a binary32 square root followed by a division and
    a correctly rounded reciprocal square root round the first RoPE dim to
    different bfloat16 values (every state row c = (3, 3, 3, 3, 1, ..., 1),
    equal scores, eps = 2^-7, v + eps = 137/128, weight 0x3F8006D5 there): the
    kernel stores the oracle's bytes, bfloat16 0x3F77, for the short-window
    kernel (window 8) and the clustered one (window 128)."""
    d, D, bs = cuda_device, 512, 8
    sw = (2 if overlap else 1) * D
    pos = 2 * ratio - 1 if overlap else ratio - 1
    c = np.ones(D, np.float32)
    c[:4] = 3.0
    npages = (pos + bs) // bs + 1
    state = np.zeros((npages, bs, 2 * sw), np.float32)
    state[:, :, :sw] = np.tile(c, sw // D)
    table = np.arange(npages, dtype=np.int32)[None, :]
    w = np.ones(D, np.float32)
    w[D - 64] = np.array([0x3F8006D5], np.uint32).view(np.float32)[0]
    cs = np.zeros((pos + 1, 64), np.float32)
    cs[:, :32] = 1.0
    t2r, p64 = np.zeros(1, np.int32), np.array([pos], np.int64)
    kv_slots = np.array([0], np.int64)
    host = np.zeros((1, 592), np.uint8)
    dev_cache = _t(host, d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    ops.compress_kv_cache_insert(_t(state, d), _t(t2r, d), _t(p64, d), _t(p64, d), _t(table, d),
                                 bs, _t(w, d), 2.0 ** -7, _t(cs, d), dev_cache, _t(kv_slots, d),
                                 1, ratio, overlap=overlap, err_count=err)
    n = oracle.compress_kv_cache_insert(state, t2r, p64, p64, table, bs, w, 2.0 ** -7, cs, host,
                                        kv_slots, 1, ratio, overlap)
    got = dev_cache.cpu().numpy()
    _assert_same(got, host, f"compress rsqrt reading row, ratio={ratio}")
    assert int(err.item()) == n == 0
    assert got[0, D - 64:D - 62].view(np.uint16)[0] == 0x3F77


@pytest.mark.parametrize("mode", ["serial", "concurrent"])
def test_compressor_step_matches_oracle(cuda_device, mode):
    """The compressor step of the prefill batch (16384 tokens) for the ratio-4
    and ratio-128 layers, as the benchmark launches it: every state float and
    every compressed record byte against the oracle."""
    from oracle.pipeline import run_compressor_step
    from paged_sparse_kv_gb300.pipeline import Pipeline
    w = synthetic.make("prefill")
    p = Pipeline(w, cuda_device)
    p.alloc_compressor()
    host_kv = []
    for c in p.comp_layers:
        g = c["host"]["kv_geom"]
        h = synthetic.random_cache_bytes(8 + c["ratio"], g)
        c["kv_cache"].copy_(torch.from_numpy(h))
        host_kv.append(h)
    p.step(concurrent=(mode == "concurrent"), path="compressor")
    torch.cuda.synchronize(cuda_device)
    layers = [c["host"] for c in p.comp_layers]
    states = [np.zeros(c["state"].shape, np.float32) for c in p.comp_layers]
    want = run_compressor_step(w, layers, states, host_kv)
    for c, st, kvc in zip(p.comp_layers, states, host_kv):
        assert np.array_equal(c["state"].cpu().numpy().view(np.uint32), st.view(np.uint32))
        _assert_same(c["kv_cache"].cpu().numpy(), kvc, f"compressed cache ratio {c['ratio']}")
    assert int(p.err.item()) == want["err"] == 0
