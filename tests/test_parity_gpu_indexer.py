"""GPU parity for the indexer-key variants: the FP8 indexer record (writer and
reader through dequantize_and_gather_k_cache) and indexer_k_norm_rope_store,
byte for byte against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_sparse_kv_gb300 import ops, synthetic
from test_parity_gpu import _assert_same, _bf16_dev, _exhaustive_rows

pytestmark = pytest.mark.gpu


def _i64(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).to(dev)


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_fp8_indexer_insert_exhaustive_codes(cuda_device):
    """Every finite bf16 value under every scale exponent from below the
    1e-10 quotient floor (2^-40) to 2^120, one 32-dim row per lead."""
    rows = _exhaustive_rows(448.0, -40, 120, 32, 1)
    N, bs = rows.shape[0], 64
    pages = (N + bs - 1) // bs
    host = np.zeros((pages, bs * 36), np.uint8)
    slots = np.arange(N, dtype=np.int64)
    dev_cache = torch.from_numpy(host).to(cuda_device)
    ops.write_indexer_fp8_cache(_bf16_dev(rows, cuda_device), dev_cache, _i64(slots, cuda_device),
                                bs)
    oracle.write_indexer_fp8_cache(rows, slots, host, bs, 32)
    assert N > 100000
    _assert_same(dev_cache.cpu().numpy(), host, "exhaustive fp8 indexer codes")


def test_fp8_indexer_insert_non_finite_inputs(cuda_device):
    """+-inf, NaN of both signs, all-NaN and all-zero stretches in 128-dim keys:
    the row amax passes over NaN, +-inf saturates to +-448, NaN of either sign
    encodes as 0x7F; every byte (codes and binary32 scales) must match."""
    from test_parity_gpu import _fp8_code_positions, _rows_with_specials
    rng = np.random.default_rng(13)
    D, N, bs = 128, 200, 16
    k = _rows_with_specials(rng, N, D, 32, D // 32)
    pages = N // bs + 3
    host = np.full((pages, bs * (D + 4)), 0x5A, np.uint8)
    slots = rng.permutation(pages * bs)[:N].astype(np.int64)
    dev_cache = torch.from_numpy(host).to(cuda_device)
    ops.write_indexer_fp8_cache(_bf16_dev(k, cuda_device), dev_cache, _i64(slots, cuda_device), bs)
    oracle.write_indexer_fp8_cache(k, slots, host, bs, D)
    got = dev_cache.cpu().numpy().reshape(-1).copy()
    want = host.reshape(-1)
    codes = _fp8_code_positions(slots, pages, bs * (D + 4), bs, D, D)
    assert np.any(want[codes] == 0x7F)  # NaN inputs reached the codes
    _assert_same(got, want, "non-finite fp8 indexer insert")


@pytest.mark.parametrize("bs", [64, 7])
@pytest.mark.parametrize("D", [32, 64, 128, 256, 512, 1024])
def test_fp8_indexer_insert_shapes_and_skips(cuda_device, D, bs):
    rng = np.random.default_rng(D + bs)
    N, pages = 97, 20
    x = (rng.standard_normal((N, D + 8)) * np.exp(rng.uniform(-8, 8, size=(N, 1)))).astype(
        np.float32)
    x[4] = 0.0
    k = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    slots = rng.permutation(pages * bs)[:N].astype(np.int64)
    slots[::6] = -1
    slots[5] = pages * bs + 3
    stride = (bs * (D + 4) + 15) // 16 * 16
    host = synthetic.random_cache_bytes(9, synthetic.CacheGeom(pages, bs, stride))
    dev_cache = torch.from_numpy(host).to(cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    kd = _bf16_dev(k, cuda_device)
    ops.write_indexer_fp8_cache(kd[:, :D], dev_cache, _i64(slots, cuda_device), bs, err_count=err)
    n_err = oracle.write_indexer_fp8_cache(np.ascontiguousarray(k[:, :D]), slots, host, bs, D)
    _assert_same(dev_cache.cpu().numpy(), host, f"fp8 indexer insert D={D}")
    assert int(err.item()) == n_err == 1


@pytest.mark.parametrize("bs", [8, 5])
@pytest.mark.parametrize("D", [32, 128, 512])
def test_fp8_indexer_gather_random_records(cuda_device, D, bs):
    """Arbitrary e4m3 bytes (no NaN codes) with power-of-two and arbitrary
    finite binary32 scales; -1 and out-of-range indices give zero rows."""
    rng = np.random.default_rng(3 * D + bs)
    pages = 9
    stride = (bs * (D + 4) + 15) // 16 * 16
    host = synthetic.random_cache_bytes(31, synthetic.CacheGeom(pages, bs, stride))
    for s in range(pages * bs):
        page, off = divmod(s, bs)
        e = int(rng.integers(-60, 60))
        v = np.float32(np.ldexp(1.0, e)) * (np.float32(rng.uniform(0.5, 2)) if s % 2 else 1)
        host[page, bs * D + off * 4: bs * D + off * 4 + 4] = np.frombuffer(
            np.float32(v).tobytes(), np.uint8)
    R, C = 21, 17
    idx = rng.integers(-1, pages * bs + 2, size=(R, C)).astype(np.int32)
    out = torch.full((R, C, D), 3, dtype=torch.bfloat16, device=cuda_device)
    ops.dequantize_and_gather_k_cache(out, torch.from_numpy(host).to(cuda_device),
                                      torch.from_numpy(idx).to(cuda_device), bs,
                                      record=ops.PSK_REC_FP8_INDEXER)
    want = oracle.dequantize_and_gather_k_cache(host, bs, 2, D, 0, idx)
    _assert_same(_u16(out), want, f"fp8 indexer gather D={D}")


def _gptj_table(max_pos, dtype=np.float32):
    theta = 10000.0 ** (-np.arange(32) / 32.0)
    ang = np.arange(max_pos)[:, None] * theta[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(dtype)


@pytest.mark.parametrize("cs_pad", [0, 3])
@pytest.mark.parametrize("fp4", [True, False])
@pytest.mark.parametrize("ratio", [1, 2, 3, 4])
@pytest.mark.parametrize("bs", [64, 3])
def test_norm_rope_store_fuzz(cuda_device, fp4, ratio, bs, cs_pad):
    rng = np.random.default_rng(100 * ratio + bs + fp4)
    N, pages, max_pos = 1500, 40, 4096
    x = rng.standard_normal((N, 136)).astype(np.float32)
    out = rng.random((N, 136)) < 0.01
    x[out] *= 20.0
    x *= np.exp(rng.uniform(-6, 6, size=(N, 1))).astype(np.float32)
    x[7] = 0.0
    k = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    pos = rng.integers(-3, max_pos + 40, size=N).astype(np.int64)
    slots = rng.permutation(pages * bs)[:N].astype(np.int64) if pages * bs >= N else \
        rng.integers(0, pages * bs, size=N).astype(np.int64)
    slots[::9] = -1
    if pages * bs < N:  # distinct slots among the tokens that write
        emit = np.nonzero(slots >= 0)[0]
        slots[emit] = -1
        keep = emit[: pages * bs]
        slots[keep] = rng.permutation(pages * bs)[: keep.size]
    # two counted skips: a slot beyond the cache and a RoPE row beyond max_pos,
    # both on group boundaries
    pos[11], slots[11] = 5 * ratio - 1, pages * bs + 1
    # the first group-closing position whose RoPE row floor(p / ratio) * ratio >= max_pos
    pos[13], slots[13] = (-(-max_pos // ratio) + 1) * ratio - 1, pages * bs + 2
    cs = _gptj_table(max_pos)
    cs_dev = np.zeros((max_pos, 64 + cs_pad), np.float32)  # stride 67: scalar cos/sin loads
    cs_dev[:, :64] = cs
    w = rng.uniform(0.25, 4.0, size=128).astype(np.float32)
    eps = 1e-6
    rec = 68 if fp4 else 132
    stride = (bs * rec + 15) // 16 * 16
    host = synthetic.random_cache_bytes(5, synthetic.CacheGeom(pages, bs, stride))
    d = cuda_device
    dev_cache = torch.from_numpy(host).to(d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    kd = _bf16_dev(k, d)
    ops.indexer_k_norm_rope_store(kd[:, :128], _i64(pos, d), torch.from_numpy(cs_dev).to(d),
                                  torch.from_numpy(w).to(d), eps, dev_cache, _i64(slots, d), ratio,
                                  fp4, bs, err_count=err)
    n_err = oracle.indexer_k_norm_rope_store(np.ascontiguousarray(k[:, :128]), pos, cs, w, eps,
                                             slots, ratio, 1 if fp4 else 2, host, bs)
    _assert_same(dev_cache.cpu().numpy(), host, f"norm rope store fp4={fp4} ratio={ratio}")
    assert int(err.item()) == n_err and n_err >= 2


@pytest.mark.parametrize("fp4", [True, False])
def test_norm_rope_store_overflowing_weights(cuda_device, fp4):
    """Norm weights near the binary32 maximum push some normalised values to
    +-inf: the FP8 row scale 2^ceil(log2(amax / 448)) then rounds to +inf and
    the codes are e4m3(y / inf) (+-0, NaN for +-inf); MXFP4 codes are
    e2m1(y * 2^-128) (+-6 for +-inf).  E4M3 NaN is 0x7F on both sides."""
    from test_parity_gpu import _fp8_code_positions
    rng = np.random.default_rng(31 + fp4)
    N, bs, max_pos = 300, 16, 1024
    pages = N // bs + 2
    x = rng.standard_normal((N, 128)).astype(np.float32)
    k = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    pos = rng.integers(0, max_pos, size=N).astype(np.int64)
    slots = rng.permutation(pages * bs)[:N].astype(np.int64)
    cs = _gptj_table(max_pos)
    w = rng.uniform(0.25, 4.0, size=128).astype(np.float32)
    w[[3, 40, 70, 101]] = [3.0e38, -3.0e38, 3.0e38, 3.0e38]
    rec = 68 if fp4 else 132
    stride = bs * rec
    host = np.full((pages, stride), 0x5A, np.uint8)
    d = cuda_device
    dev_cache = torch.from_numpy(host).to(d)
    ops.indexer_k_norm_rope_store(_bf16_dev(k, d), _i64(pos, d), torch.from_numpy(cs).to(d),
                                  torch.from_numpy(w).to(d), 1e-6, dev_cache, _i64(slots, d), 1,
                                  fp4, bs)
    oracle.indexer_k_norm_rope_store(k, pos, cs, w, 1e-6, slots, 1, 1 if fp4 else 2, host, bs)
    got = dev_cache.cpu().numpy().reshape(-1).copy()
    want = host.reshape(-1)
    if not fp4:
        codes = _fp8_code_positions(slots, pages, stride, bs, 128, 128)
        assert np.any(want[codes] == 0x7F)  # NaN inputs reached the codes
    _assert_same(got, want, f"norm rope store, overflowing weights, fp4={fp4}")


def test_norm_rope_store_rsqrt_reading(cuda_device):
    """The row on which a binary32 square root followed by a division and a
    correctly rounded reciprocal square root store different FP8 codes
    (x = (3, 1, ..., 1), eps = 2^-7, v + eps = 137/128, weight 0x3F80490B on
    dim 1): the kernel stores the oracle's bytes, code 0x6F at dim 1."""
    d, bs = cuda_device, 4  # page strides of 528 and 272 bytes (multiples of 16)
    x = np.ones((1, 128), np.float32)
    x[0, 0] = 3.0
    k = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    w = np.ones(128, np.float32)
    w[1] = np.array([0x3F80490B], np.uint32).view(np.float32)[0]
    cs = np.zeros((4, 64), np.float32)
    cs[:, :32] = 1.0
    pos, slots = np.array([0], np.int64), np.array([1], np.int64)
    for fp4 in (False, True):
        host = np.zeros((1, bs * (68 if fp4 else 132)), np.uint8)
        dev_cache = torch.from_numpy(host).to(d)
        ops.indexer_k_norm_rope_store(_bf16_dev(k, d), _i64(pos, d), torch.from_numpy(cs).to(d),
                                      torch.from_numpy(w).to(d), 2.0 ** -7, dev_cache,
                                      _i64(slots, d), 1, fp4, bs)
        oracle.indexer_k_norm_rope_store(k, pos, cs, w, 2.0 ** -7, slots, 1, 1 if fp4 else 2,
                                         host, bs)
        got = dev_cache.cpu().numpy()
        _assert_same(got, host, f"norm rope store, rsqrt reading row, fp4={fp4}")
        if not fp4:
            assert got[0, 128:131].tolist() == [0x7C, 0x6F, 0x6F]


def test_norm_rope_store_prefill_size(cuda_device):
    """The prefill batch's 16384 tokens at ratio 4 (a key per 4 tokens) into the
    MXFP4 and FP8 indexer caches, strided k_pre and a padded cos_sin table."""
    w_ = synthetic.make("prefill")
    d = cuda_device
    qlen = np.diff(w_.query_start_loc)
    pos = np.concatenate([np.arange(s - q, s) for s, q in zip(w_.seq_lens, qlen)]).astype(np.int64)
    rng = np.random.default_rng(77)
    k = torch.from_numpy(rng.standard_normal((pos.size, 256)).astype(np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    cs = np.zeros((4096, 72), np.float32)
    cs[:, :64] = _gptj_table(4096)
    wt = rng.uniform(0.5, 2.0, size=128).astype(np.float32)
    for fp4 in (True, False):
        bs, rec = 64, (68 if fp4 else 132)
        pages = w_.index_cache.num_pages
        host = np.zeros((pages, bs * rec), np.uint8)
        slots = w_.index_insert_slots
        dev_cache = torch.from_numpy(host).to(d)
        kd = _bf16_dev(k, d)
        ops.indexer_k_norm_rope_store(kd[:, 64:192], _i64(pos, d), torch.from_numpy(cs).to(d),
                                      torch.from_numpy(wt).to(d), 1e-6, dev_cache, _i64(slots, d),
                                      4, fp4, bs)
        oracle.indexer_k_norm_rope_store(np.ascontiguousarray(k[:, 64:192]), pos, cs[:, :64], wt,
                                         1e-6, slots, 4, 1 if fp4 else 2, host, bs)
        _assert_same(dev_cache.cpu().numpy(), host, f"prefill norm rope store fp4={fp4}")


@pytest.mark.parametrize("path", ["indexer_fp8", "indexer_store"])
def test_indexer_steps_match_oracle(cuda_device, path):
    """The indexer steps of the 1,048,576-key workload as the benchmark launches
    them (concurrent streams): every cache byte, the global top-k and lens, and
    the gathered keys of a sample of tokens, against the oracle."""
    from oracle.pipeline import run_indexer_step
    from paged_sparse_kv_gb300.pipeline import Pipeline
    w = synthetic.make("mxfp4")
    p = Pipeline(w, cuda_device)
    variant = path.split("_")[1]
    p.indexer_launches(variant)
    g = w.index_cache
    if variant == "fp8":
        host = np.zeros((g.num_pages, g.block_size * 132), np.uint8)
        dev_cache = p.fp8i_cache
    else:
        host = synthetic.random_cache_bytes(44, g)
        dev_cache = p.index_cache
    dev_cache.copy_(torch.from_numpy(host))
    p.step(concurrent=True, path=path)
    torch.cuda.synchronize(cuda_device)
    n = w.index_k.shape[0]
    inputs = {"positions": np.arange(n, dtype=np.int64) % Pipeline.INDEXER_MAX_POS,
              "cos_sin": synthetic.gptj_cos_sin(Pipeline.INDEXER_MAX_POS),
              "weight": synthetic.norm_weight(w.seed), "eps": 1e-6}
    toks = np.arange(0, w.num_tokens, 9)
    want = run_indexer_step(w, variant, host, inputs, toks)
    _assert_same(dev_cache.cpu().numpy(), host, f"{path} cache")
    assert np.array_equal(p.global_topk.cpu().numpy(), want["global_topk"])
    assert np.array_equal(p.global_lens.cpu().numpy(), want["global_lens"])
    _assert_same(_u16(p.gathered_index)[toks], want["gathered_index"], f"{path} gathered")
    assert int(p.err.item()) == want["err"] == 0
