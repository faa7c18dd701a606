"""GPU parity: every CUDA entry point against the CPU oracle, bit for bit.

Integer outputs (slots, lens) and packed bytes (FP8/FP4 codes, scale bytes,
untouched cache bytes) must be identical; the dequantized bf16 rows must be
identical too (tolerance 0: the products are exact in bf16 for UE8M0 scales,
and both sides round binary32 products the same way for fp32 scales).

Sizes: the five workloads at full size through the benchmark's pipeline
(large gathers compared on a seeded sample of tokens), exhaustive code tables,
and randomised small cases with ragged shapes and edge cases.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.pipeline import run_step
from paged_sparse_kv_gb300 import ops, synthetic
from paged_sparse_kv_gb300.pipeline import Pipeline
from test_oracle_index import _random_case

pytestmark = pytest.mark.gpu


def _bf16_dev(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def _u16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _assert_same(got: np.ndarray, want: np.ndarray, what: str):
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.nonzero(got.reshape(-1) != want.reshape(-1))[0]
    assert bad.size == 0, f"{what}: {bad.size} mismatches, first at flat {bad[:5].tolist()}: " \
                          f"got {got.reshape(-1)[bad[:5]].tolist()} want {want.reshape(-1)[bad[:5]].tolist()}"


@pytest.fixture(autouse=True)
def _free_gpu_memory():
    yield
    torch.cuda.empty_cache()


def test_smoke(cuda_device):
    import __graft_entry__
    __graft_entry__.smoke()


# ---- inserts ---------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "mixed"])
@pytest.mark.parametrize("ue8m0", [True, False])
def test_fp8_insert_matches_oracle(cuda_device, name, ue8m0):
    w = synthetic.make(name)
    g = w.swa_cache
    rec = oracle.fp8_record_bytes(w.head_dim, w.rope_dim, ue8m0)
    stride = (g.block_size * rec + 15) // 16 * 16
    geom = synthetic.CacheGeom(g.num_pages, g.block_size, stride)
    host = synthetic.random_cache_bytes(7, geom)
    dev_cache = torch.from_numpy(host).to(cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ops.quantize_and_insert_k_cache(_bf16_dev(w.k, cuda_device), dev_cache,
                                    torch.from_numpy(w.insert_slots).to(cuda_device),
                                    g.block_size, rope_dim=w.rope_dim, is_ue8m0=ue8m0,
                                    err_count=err)
    n_err = oracle.quantize_and_insert_k_cache(w.k, w.insert_slots, host, g.block_size,
                                               w.head_dim, w.rope_dim, ue8m0)
    _assert_same(dev_cache.cpu().numpy(), host, f"{name} fp8 cache (ue8m0={ue8m0})")
    assert int(err.item()) == n_err == 0


def _exhaustive_rows(max_code: float, e_lo: int, e_hi: int, block: int, blocks_per_row: int):
    """bf16 rows whose blocks reach every scale exponent in [e_lo, e_hi]: each
    block starts with an element fixing its amax at max_code * 2^e and is
    filled with every finite bf16 value of magnitude <= that amax."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    fin = np.isfinite(vals)
    bf_max = np.float32((np.uint32(0x7F7F) << 16).view(np.float32))
    blocks = []
    for e in range(e_lo, e_hi + 1):
        lead = np.float32(max_code * 2.0 ** e) if max_code * 2.0 ** e <= bf_max else bf_max
        pick = bits[fin & (np.abs(vals) <= lead)].astype(np.uint16)
        per = block - 1
        pad = (-pick.size) % per
        pick = np.concatenate([pick, np.zeros(pad, np.uint16)]).reshape(-1, per)
        lead_bits = np.uint16(np.array([lead], np.float32).view(np.uint32)[0] >> 16)
        blk = np.concatenate([np.full((pick.shape[0], 1), lead_bits, np.uint16), pick], axis=1)
        blocks.append(blk)
    blocks = np.concatenate(blocks)
    pad = (-blocks.shape[0]) % blocks_per_row
    blocks = np.concatenate([blocks, np.zeros((pad, block), np.uint16)])
    return blocks.reshape(-1, blocks_per_row * block)


def test_fp8_insert_exhaustive_codes(cuda_device):
    """Every finite bf16 value under every reachable UE8M0 exponent
    (e in [-22, 120]) through the GPU insert, against the oracle."""
    nope = _exhaustive_rows(448.0, -22, 120, 64, 7)
    k = np.concatenate([nope, np.zeros((nope.shape[0], 64), np.uint16)], axis=1)
    N, bs = k.shape[0], 64
    pages = (N + bs - 1) // bs
    geom = synthetic.CacheGeom(pages, bs, bs * 584)
    host = np.zeros((geom.num_pages, geom.page_stride), np.uint8)
    slots = np.arange(N, dtype=np.int64)
    dev_cache = torch.from_numpy(host).to(cuda_device)
    ops.quantize_and_insert_k_cache(_bf16_dev(k, cuda_device), dev_cache,
                                    torch.from_numpy(slots).to(cuda_device), bs, rope_dim=64)
    oracle.quantize_and_insert_k_cache(k, slots, host, bs, 512, 64)
    assert N > 10000
    _assert_same(dev_cache.cpu().numpy(), host, "exhaustive fp8 codes")


_SPECIALS = np.array([0x7F80, 0xFF80, 0x7FC0, 0xFFC0, 0x7F81, 0xFF81, 0x8000, 0x7F7F, 0xFF7F],
                     np.uint16)   # +-inf, +-qNaN, +-sNaN, -0, +-largest finite


def _rows_with_specials(rng, N, D, block, nblk):
    """bf16 rows ~ 3 N(0,1) with, in the first nblk blocks of `block` elements:
    a few scattered specials, whole blocks of NaN, whole blocks of +-0."""
    vals = rng.standard_normal((N, D)).astype(np.float32) * 3
    k = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for t in range(N):
        for b in range(nblk):
            kind = (t * 7 + b) % 5
            if kind == 0:
                pos = rng.choice(block, size=3, replace=False)
                k[t, b * block + pos] = rng.choice(_SPECIALS, size=3)
            elif kind == 1 and t % 3 == 0:
                k[t, b * block:(b + 1) * block] = rng.choice(_SPECIALS[2:6], size=block)
            elif kind == 2 and t % 4 == 1:
                k[t, b * block:(b + 1) * block] = rng.choice(np.array([0, 0x8000], np.uint16),
                                                             size=block)
    return k


def _fp8_code_positions(slots, num_pages, page_stride, bs, ts, nope):
    """Flat byte offsets of the e4m3 codes of each inserted token."""
    page, off = slots // bs, slots % bs
    start = page * page_stride + off * ts
    return (start[:, None] + np.arange(nope)[None, :]).reshape(-1)


@pytest.mark.parametrize("ue8m0", [True, False])
def test_fp8_insert_non_finite_inputs(cuda_device, ue8m0):
    """+-inf, NaN of both signs (quiet and signalling payloads), all-NaN and
    all-zero blocks, -0 and the largest finite bf16, planted in random rows.
    amax passes over NaN; +-inf saturates to +-448.  NaN of either sign
    encodes as 0x7F, the one NaN code both sides write; every byte must
    match."""
    rng = np.random.default_rng(11)
    D, rope, N, bs = 512, 64, 96, 16
    nope = D - rope
    k = _rows_with_specials(rng, N, D, 64, nope // 64)
    rec = oracle.fp8_record_bytes(D, rope, ue8m0)
    pages = N // bs + 2
    geom = synthetic.CacheGeom(pages, bs, (bs * rec + 15) // 16 * 16)
    host = np.full((geom.num_pages, geom.page_stride), 0x5A, np.uint8)
    slots = rng.permutation(pages * bs)[:N].astype(np.int64)
    dev_cache = torch.from_numpy(host).to(cuda_device)
    ops.quantize_and_insert_k_cache(_bf16_dev(k, cuda_device), dev_cache,
                                    torch.from_numpy(slots).to(cuda_device), bs,
                                    rope_dim=rope, is_ue8m0=ue8m0)
    oracle.quantize_and_insert_k_cache(k, slots, host, bs, D, rope, ue8m0)
    got = dev_cache.cpu().numpy().reshape(-1).copy()
    want = host.reshape(-1)
    codes = _fp8_code_positions(slots, pages, geom.page_stride, bs, nope + 2 * rope, nope)
    assert np.any(want[codes] == 0x7F)  # NaN inputs reached the codes
    assert np.any(want[codes] == 0x7E) and np.any(want[codes] == 0xFE)
    _assert_same(got, want, f"non-finite fp8 insert ue8m0={ue8m0}")


def test_mxfp4_insert_exhaustive_codes(cuda_device):
    rows = _exhaustive_rows(6.0, -15, 126, 32, 4)
    N, bs = rows.shape[0], 64
    pages = (N + bs - 1) // bs
    host = np.zeros((pages, bs * 68), np.uint8)
    slots = np.arange(N, dtype=np.int64)
    dev_cache = torch.from_numpy(host).to(cuda_device)
    ops.write_indexer_mxfp4_cache(_bf16_dev(rows, cuda_device), dev_cache,
                                  torch.from_numpy(slots).to(cuda_device), bs)
    oracle.write_indexer_mxfp4_cache(rows, slots, host, bs, 128)
    _assert_same(dev_cache.cpu().numpy(), host, "exhaustive mxfp4 codes")


def test_mxfp4_insert_non_finite_inputs(cuda_device):
    """+-inf, NaN of both signs, all-NaN and all-zero blocks in 128-dim keys:
    amax passes over NaN, +-inf and NaN saturate to the E2M1 codes the oracle
    gives (E2M1 has neither), every byte must match."""
    rng = np.random.default_rng(12)
    D, N, bs = 128, 200, 16
    k = _rows_with_specials(rng, N, D, 32, D // 32)
    pages = N // bs + 3
    host = np.full((pages, bs * (D // 2 + D // 32)), 0x5A, np.uint8)
    slots = rng.permutation(pages * bs)[:N].astype(np.int64)
    dev_cache = torch.from_numpy(host).to(cuda_device)
    ops.write_indexer_mxfp4_cache(_bf16_dev(k, cuda_device), dev_cache,
                                  torch.from_numpy(slots).to(cuda_device), bs)
    oracle.write_indexer_mxfp4_cache(k, slots, host, bs, D)
    _assert_same(dev_cache.cpu().numpy(), host, "non-finite mxfp4 insert")


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "mxfp4"])
def test_mxfp4_insert_matches_oracle(cuda_device, name):
    w = synthetic.make(name)
    host = synthetic.random_cache_bytes(11, w.index_cache)
    dev_cache = torch.from_numpy(host).to(cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ops.write_indexer_mxfp4_cache(_bf16_dev(w.index_k, cuda_device), dev_cache,
                                  torch.from_numpy(w.index_insert_slots).to(cuda_device),
                                  w.index_cache.block_size, err_count=err)
    n_err = oracle.write_indexer_mxfp4_cache(w.index_k, w.index_insert_slots, host,
                                             w.index_cache.block_size, w.index_head_dim)
    _assert_same(dev_cache.cpu().numpy(), host, f"{name} mxfp4 cache")
    assert int(err.item()) == n_err


@pytest.mark.parametrize("bs", [16, 12])
@pytest.mark.parametrize("D,rope,ue8m0", [(64, 0, True), (128, 0, True), (256, 128, True),
                                          (512, 64, False), (1024, 64, True)])
def test_fp8_insert_shapes_strides_and_skips(cuda_device, D, rope, ue8m0, bs):
    """Ragged token count, a k with extra rows and a wider row stride,
    negative and out-of-range slots (counted), all head_dim variants; a
    power-of-two and an odd block size."""
    rng = np.random.default_rng(D + rope)
    N, pages = 203, 20
    rows = rng.standard_normal((N + 5, D + 24)).astype(np.float32) * 3
    k = torch.from_numpy(rows).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    slots = rng.permutation(pages * bs)[:N].astype(np.int64)
    slots[::7] = -1
    slots[3] = pages * bs + 5
    slots[11] = 1 << 40
    rec = oracle.fp8_record_bytes(D, rope, ue8m0)
    geom = synthetic.CacheGeom(pages, bs, (bs * rec + 31) // 16 * 16)
    host = synthetic.random_cache_bytes(3, geom)
    dev_cache = torch.from_numpy(host).to(cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    kd = _bf16_dev(k, cuda_device)
    ops.quantize_and_insert_k_cache(kd[:, :D], dev_cache, torch.from_numpy(slots).to(cuda_device),
                                    bs, rope_dim=rope, is_ue8m0=ue8m0, err_count=err)
    n_err = oracle.quantize_and_insert_k_cache(np.ascontiguousarray(k[:N, :D]), slots, host, bs,
                                               D, rope, ue8m0)
    _assert_same(dev_cache.cpu().numpy(), host, f"fp8 insert D={D} rope={rope}")
    assert int(err.item()) == n_err == 2


@pytest.mark.parametrize("bs", [8, 7])
@pytest.mark.parametrize("D", [32, 64, 128, 256, 512, 1024])
def test_mxfp4_insert_shapes_and_skips(cuda_device, D, bs):
    rng = np.random.default_rng(D)
    N, pages = 77, 12
    rows = rng.standard_normal((N, D)).astype(np.float32)
    rows[5] = 0.0
    k = torch.from_numpy(rows).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    slots = rng.permutation(pages * bs)[:N].astype(np.int64)
    slots[::5] = -1
    slots[2] = pages * bs
    rec = D // 2 + D // 32
    geom = synthetic.CacheGeom(pages, bs, (bs * rec + 15) // 16 * 16)
    host = synthetic.random_cache_bytes(4, geom)
    dev_cache = torch.from_numpy(host).to(cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ops.write_indexer_mxfp4_cache(_bf16_dev(k, cuda_device), dev_cache,
                                  torch.from_numpy(slots).to(cuda_device), bs, err_count=err)
    n_err = oracle.write_indexer_mxfp4_cache(k, slots, host, bs, D)
    _assert_same(dev_cache.cpu().numpy(), host, f"mxfp4 insert D={D}")
    assert int(err.item()) == n_err == 1


def test_insert_zero_tokens_touches_nothing(cuda_device):
    cache = torch.full((4, 64 * 584), 0xA5, dtype=torch.uint8, device=cuda_device)
    k = torch.zeros((3, 512), dtype=torch.bfloat16, device=cuda_device)
    ops.quantize_and_insert_k_cache(k, cache, torch.empty(0, dtype=torch.int64, device=cuda_device), 64)
    ops.quantize_and_insert_k_cache(k, cache, torch.full((3,), -1, dtype=torch.int64, device=cuda_device), 64)
    torch.cuda.synchronize()
    assert bool((cache == 0xA5).all())


# ---- index builders ------------------------------------------------------------------

def _dev_i32(a, dev):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "mixed"])
def test_combine_matches_oracle(cuda_device, name):
    w = synthetic.make(name)
    d = cuda_device
    si, lens = ops.combine_topk_swa_indices(
        _dev_i32(w.query_start_loc, d), _dev_i32(w.seq_lens, d), _dev_i32(w.token_to_req, d),
        _dev_i32(w.replay_start, d), _dev_i32(w.swa_block_table, d), w.swa_cache.block_size,
        _dev_i32(w.comp_block_table, d), w.comp_cache.block_size, w.window, w.compress_ratio,
        _dev_i32(w.topk_local, d))
    want, want_lens = oracle.combine_topk_swa_indices(
        w.query_start_loc, w.seq_lens, w.token_to_req, w.replay_start, w.swa_block_table,
        w.swa_cache.block_size, w.comp_block_table, w.comp_cache.block_size, w.window,
        w.compress_ratio, w.topk_local)
    _assert_same(si.cpu().numpy(), want, f"{name} sparse_indices")
    _assert_same(lens.cpu().numpy(), want_lens, f"{name} lens")


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "mixed", "mxfp4"])
def test_global_topk_matches_oracle(cuda_device, name):
    w = synthetic.make(name)
    d = cuda_device
    table = w.comp_block_table if w.comp_block_table is not None else w.swa_block_table
    out, lens = ops.compute_global_topk_indices_and_lens(
        _dev_i32(w.topk_local, d), _dev_i32(w.token_to_req, d), _dev_i32(table, d),
        w.index_cache.block_size)
    want, want_lens = oracle.compute_global_topk_indices_and_lens(
        w.topk_local, w.token_to_req, table, w.index_cache.block_size)
    _assert_same(out.cpu().numpy(), want, f"{name} global top-k")
    _assert_same(lens.cpu().numpy(), want_lens, f"{name} global lens")


@pytest.mark.parametrize("seed", range(40))
def test_index_builders_fuzz(cuda_device, seed):
    """Random small cases: page sizes 1..64, odd windows and top-k widths (the
    unvectorised path), -1 table and top-k entries, base offsets, replay_start,
    invalid tokens, out-of-range request indices, shared-memory staging."""
    rng = np.random.default_rng(1000 + seed)
    c = _random_case(rng)
    comp_bs = c["bs"] if rng.random() < 0.5 else int(rng.choice([1, 4, 16]))
    d = cuda_device
    T = c["topk"].shape[0]
    replay = c["replay"] if c["replay"] is not None else np.zeros(len(c["seq"]), np.int32)
    valid = None if c["valid"] is None else torch.from_numpy(c["valid"]).to(d)
    si, lens = ops.combine_topk_swa_indices(
        _dev_i32(c["qsl"], d), _dev_i32(c["seq"], d), _dev_i32(c["t2r"], d), _dev_i32(replay, d),
        _dev_i32(c["swa_bt"], d), c["bs"], _dev_i32(c["comp_bt"], d), comp_bs, c["W"], 4,
        _dev_i32(c["topk"], d), swa_base_offsets=_dev_i32(c["swa_base"], d),
        compressed_base_offsets=_dev_i32(c["comp_base"], d), is_valid_token=valid, num_tokens=T)
    want, want_lens = oracle.combine_topk_swa_indices(
        c["qsl"], c["seq"], c["t2r"], replay, c["swa_bt"], c["bs"], c["comp_bt"], comp_bs,
        c["W"], 4, c["topk"], swa_base_offsets=c["swa_base"], comp_base_offsets=c["comp_base"],
        is_valid_token=c["valid"])
    if T:
        _assert_same(si.cpu().numpy(), want, "fuzz sparse_indices")
        _assert_same(lens.cpu().numpy(), want_lens, "fuzz lens")
    bt = c["comp_bt"] if c["comp_bt"] is not None else c["swa_bt"]
    out, gl = ops.compute_global_topk_indices_and_lens(
        _dev_i32(c["topk"], d), _dev_i32(c["t2r"], d), _dev_i32(bt, d), comp_bs, valid,
        base_offsets=_dev_i32(c["comp_base"], d))
    want_g, want_gl = oracle.compute_global_topk_indices_and_lens(
        c["topk"], c["t2r"], bt, comp_bs, base_offsets=c["comp_base"], is_valid_token=c["valid"])
    if T:
        _assert_same(out.cpu().numpy(), want_g, "fuzz global top-k")
        _assert_same(gl.cpu().numpy(), want_gl, "fuzz global lens")


def test_index_build_strided_views(cuda_device):
    """Top-k and output rows that are column views of wider matrices (row
    strides not multiples of 4 -> per-column path)."""
    w = synthetic.make("tiny")
    d = cuda_device
    T, K = w.topk_local.shape
    wide = np.full((T, K + 3), 99, np.int32)
    wide[:, 1:K + 1] = w.topk_local
    wide_d = _dev_i32(wide, d)
    out_wide = torch.full((T, w.window + 8 + 5), -7, dtype=torch.int32, device=d)
    lens = torch.empty(T, dtype=torch.int32, device=d)
    ops.combine_topk_swa_indices(
        _dev_i32(w.query_start_loc, d), _dev_i32(w.seq_lens, d), _dev_i32(w.token_to_req, d),
        _dev_i32(w.replay_start, d), _dev_i32(w.swa_block_table, d), w.swa_cache.block_size,
        None, w.comp_cache.block_size, w.window, 4, wide_d[:, 1:K + 1],
        out=out_wide[:, 2:2 + w.window + 8], lens=lens)
    want, want_lens = oracle.combine_topk_swa_indices(
        w.query_start_loc, w.seq_lens, w.token_to_req, w.replay_start, w.swa_block_table,
        w.swa_cache.block_size, None, w.comp_cache.block_size, w.window, 4, w.topk_local)
    got = out_wide.cpu().numpy()
    _assert_same(got[:, 2:2 + w.window + 8], want, "strided sparse_indices")
    assert np.all(got[:, :2] == -7) and np.all(got[:, 2 + w.window + 8:] == -7)
    _assert_same(lens.cpu().numpy(), want_lens, "strided lens")


# ---- gathers -------------------------------------------------------------------------

@pytest.mark.parametrize("bs", [16, 5])
@pytest.mark.parametrize("D,rope,ue8m0", [(512, 64, True), (128, 0, True), (512, 64, False),
                                          (256, 128, True), (64, 0, False)])
def test_fp8_gather_random_records(cuda_device, D, rope, ue8m0, bs):
    """Arbitrary record bytes (UE8M0: no NaN codes; scales 2^-127..2^127, so
    products hit bf16 subnormals and infinities); indices with -1 and
    out-of-range slots; ragged rows x columns; output as a strided view."""
    rng = np.random.default_rng(D * 3 + rope)
    pages = 9
    rec = oracle.fp8_record_bytes(D, rope, ue8m0)
    geom = synthetic.CacheGeom(pages, bs, (bs * rec + 15) // 16 * 16)
    if ue8m0:
        host = synthetic.random_cache_bytes(21, geom)
    else:  # fp32 scales: fill through the oracle insert so scales are finite
        host = np.zeros((geom.num_pages, geom.page_stride), np.uint8)
        rows = torch.from_numpy(rng.standard_normal((pages * bs, D)).astype(np.float32) * 4).to(
            torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        oracle.quantize_and_insert_k_cache(rows, np.arange(pages * bs, dtype=np.int64), host,
                                           bs, D, rope, False)
    R, Cc = 37, 19
    idx = rng.integers(-1, pages * bs, size=(R, Cc)).astype(np.int32)
    idx[0, :] = -1
    idx[1, 3] = pages * bs
    idx[2, 4] = 2**31 - 1
    out = torch.full((R, Cc + 2, D), 7, dtype=torch.bfloat16, device=cuda_device)
    ops.dequantize_and_gather_k_cache(out[:, 1:Cc + 1, :], torch.from_numpy(host).to(cuda_device),
                                      _dev_i32(idx, cuda_device), bs, rope_dim=rope,
                                      is_ue8m0=ue8m0)
    want = oracle.dequantize_and_gather_k_cache(host, bs, 0, D, rope, idx, is_ue8m0=ue8m0)
    got = _u16(out)
    _assert_same(got[:, 1:Cc + 1], want, f"fp8 gather D={D}")
    seven = np.uint16(torch.tensor(7.0, dtype=torch.bfloat16).view(torch.int16).item())
    assert np.all(got[:, 0] == seven) and np.all(got[:, Cc + 1] == seven)


@pytest.mark.parametrize("record", ["fp8_ds_mla", "mxfp4", "fp8_indexer"])
@pytest.mark.parametrize("shift", [8, 72])
def test_gather_output_16_byte_aligned_only(cuda_device, record, shift):
    """Outputs whose rows start on 16-byte but not 32-byte boundaries (a base
    offset of 16 bytes, or a row stride of an odd number of 16-byte units) take
    the gathers' two-16-byte-store path: same bytes as the oracle, and nothing
    outside the rows is written."""
    rng = np.random.default_rng(17 + shift)
    D, rope, bs, pages = (512, 64, 16, 8) if record == "fp8_ds_mla" else (128, 0, 16, 8)
    if record == "fp8_ds_mla":
        rec, code = oracle.fp8_record_bytes(D, rope), 0
    elif record == "mxfp4":
        rec, code = D // 2 + D // 32, ops.PSK_REC_MXFP4
    else:
        rec, code = D + 4, ops.PSK_REC_FP8_INDEXER
    geom = synthetic.CacheGeom(pages, bs, (bs * rec + 15) // 16 * 16)
    host = synthetic.random_cache_bytes(23, geom)
    if record == "fp8_indexer":  # finite binary32 row scales
        sc = rng.integers(0, 1 << 32, size=(pages, bs), dtype=np.uint64).astype(np.uint32)
        sc[((sc >> 23) & 0xFF) == 0xFF] &= ~np.uint32(0x40000000)
        host[:, bs * D: bs * D + 4 * bs] = sc.view(np.uint8).reshape(pages, 4 * bs)
    R, Cc = 13, 9
    idx = rng.integers(-1, pages * bs, size=(R, Cc)).astype(np.int32)
    # shift 8: rows of D values from element 8 (16 bytes past a 32-byte boundary);
    # shift 72: a row stride of D + 72 values ((2 D + 144) bytes, 16- but not 32-aligned)
    stride_j = D if shift == 8 else D + shift
    base = torch.full((R * Cc * stride_j + 64,), 7, dtype=torch.bfloat16, device=cuda_device)
    off = 8 if shift == 8 else 0
    out = base[off:off + R * Cc * stride_j].view(R, Cc, stride_j)[:, :, :D]
    assert (out.data_ptr() % 32 != 0) or ((stride_j * 2) % 32 != 0)
    ops.dequantize_and_gather_k_cache(out, torch.from_numpy(host).to(cuda_device),
                                      _dev_i32(idx, cuda_device), bs, rope_dim=rope, record=code)
    want = oracle.dequantize_and_gather_k_cache(host, bs, code, D, rope, idx)
    _assert_same(_u16(out), want, f"16-byte-aligned output, {record}, shift {shift}")
    seven = np.uint16(torch.tensor(7.0, dtype=torch.bfloat16).view(torch.int16).item())
    flat = _u16(base)
    mask = np.ones(flat.size, bool)
    for t in range(R):
        for j in range(Cc):
            st = off + (t * Cc + j) * stride_j
            mask[st:st + D] = False
    assert np.all(flat[mask] == seven), "bytes outside the rows were written"


@pytest.mark.parametrize("ue8m0", [True, False])
def test_fp8_gather_every_scale(cuda_device, ue8m0):
    """Every scale a record can hold: UE8M0 bytes cycling through 0..254 (127,
    the scale 2^0, included), or binary32 scale words of random finite bit
    patterns (normals of every exponent, subnormals, +-0), so the binary32
    products round, overflow to +-inf and go subnormal; random non-NaN codes."""
    rng = np.random.default_rng(31 + ue8m0)
    D, rope, bs, pages = 512, 64, 16, 20
    nope, ts, nb = D - rope, D - rope + 2 * rope, D // 64
    rec = oracle.fp8_record_bytes(D, rope, ue8m0)
    geom = synthetic.CacheGeom(pages, bs, bs * rec)
    host = synthetic.random_cache_bytes(41 + ue8m0, geom)
    n = pages * bs
    if ue8m0:
        scl = (np.arange(n * nb) % 255).astype(np.uint8).reshape(n, nb)
        scl[:, nb - 1] = 0  # the pad slot
        for s_ in range(n):
            page, off = divmod(s_, bs)
            host[page, bs * ts + off * nb: bs * ts + (off + 1) * nb] = scl[s_]
        assert set(np.unique(scl[:, :nb - 1])) == set(range(255))
    else:
        w = rng.integers(0, 1 << 32, size=(n, nb), dtype=np.uint64).astype(np.uint32)
        w[((w >> 23) & 0xFF) == 0xFF] &= ~np.uint32(0x40000000)
        w[0] = np.array([0, 0x80000000, 1, 0x807FFFFF, 0x7F7FFFFF, 0x00800000, 0x3F800000, 0],
                        np.uint32)
        for s_ in range(n):
            page, off = divmod(s_, bs)
            host[page, bs * ts + off * 4 * nb: bs * ts + (off + 1) * 4 * nb] = w[s_].view(np.uint8)
    idx = rng.permutation(n).astype(np.int32).reshape(20, 16)
    idx[3, 5] = -1
    out = torch.empty((20, 16, D), dtype=torch.bfloat16, device=cuda_device)
    ops.dequantize_and_gather_k_cache(out, torch.from_numpy(host).to(cuda_device),
                                      _dev_i32(idx, cuda_device), bs, rope_dim=rope,
                                      is_ue8m0=ue8m0)
    want = oracle.dequantize_and_gather_k_cache(host, bs, 0, D, rope, idx, is_ue8m0=ue8m0)
    got = _u16(out)
    _assert_same(got, want, f"every scale, ue8m0={ue8m0}")
    flat = want[:, :, :nope].reshape(-1)
    assert np.any((flat & 0x7FFF) == 0x7F80), "no product reached +-inf"
    assert np.any(((flat & 0x7F80) == 0) & ((flat & 0x7FFF) != 0)), "no subnormal result"


@pytest.mark.parametrize("bs", [8, 3])
@pytest.mark.parametrize("D", [32, 64, 128, 256, 512, 1024])
def test_mxfp4_gather_random_records(cuda_device, D, bs):
    rng = np.random.default_rng(D + 5)
    pages = 11
    rec = D // 2 + D // 32
    geom = synthetic.CacheGeom(pages, bs, (bs * rec + 15) // 16 * 16)
    host = rng.integers(0, 256, size=(geom.num_pages, geom.page_stride), dtype=np.uint8)
    R, Cc = 23, 31
    idx = rng.integers(-1, pages * bs + 3, size=(R, Cc)).astype(np.int32)
    out = torch.empty((R, Cc, D), dtype=torch.bfloat16, device=cuda_device)
    ops.dequantize_and_gather_k_cache(out, torch.from_numpy(host).to(cuda_device),
                                      _dev_i32(idx, cuda_device), bs, record=ops.PSK_REC_MXFP4)
    want = oracle.dequantize_and_gather_k_cache(host, bs, 1, D, 0, idx)
    _assert_same(_u16(out), want, f"mxfp4 gather D={D}")


# ---- the whole step, at full size, as the benchmark launches it -----------------------

SAMPLE = {"tiny": None, "decode": None, "prefill": 48, "mixed": 48, "mxfp4": None}


@pytest.mark.parametrize("name,mode", [("tiny", "serial"), ("decode", "serial"),
                                       ("prefill", "serial"), ("mixed", "serial"),
                                       ("mxfp4", "serial"), ("tiny", "graph"),
                                       ("decode", "graph"), ("mixed", "concurrent"),
                                       ("prefill", "graph"), ("mixed", "graph"),
                                       ("mxfp4", "graph")])
def test_pipeline_step_matches_oracle(cuda_device, name, mode):
    """The whole step at full size, launched the way the benchmark launches it
    (serial, three concurrent streams, or a CUDA graph of the concurrent step)."""
    w = synthetic.make(name)
    host = {}
    for i, cname in enumerate(("swa_cache", "comp_cache", "index_cache")):
        g = getattr(w, cname)
        host[cname] = None if g is None else synthetic.random_cache_bytes(50 + i, g)
    p = Pipeline(w, cuda_device)
    for cname, arr in host.items():
        if arr is not None:
            getattr(p, cname).copy_(torch.from_numpy(arr))
    if mode == "serial":
        p.step()
    elif mode == "concurrent":
        p.step(concurrent=True)
    else:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(cuda_device)
        side.wait_stream(torch.cuda.current_stream(cuda_device))
        with torch.cuda.graph(g, stream=side):
            p.step(concurrent=True)
        torch.cuda.synchronize()
        # capture launched nothing: the caches still hold the initial bytes
        for cname, arr in host.items():
            if arr is not None:
                _assert_same(getattr(p, cname).cpu().numpy(), arr, f"{name} {cname} untouched")
        g.replay()
    torch.cuda.synchronize()
    toks = None
    if SAMPLE[name]:
        rng = np.random.default_rng(99)
        toks = np.unique(np.concatenate([[0, w.num_tokens - 1],
                                         rng.integers(0, w.num_tokens, SAMPLE[name])]))
    ref = run_step(w, host["swa_cache"], host["comp_cache"], host["index_cache"], toks)
    for cname, arr in host.items():
        if arr is not None:
            _assert_same(getattr(p, cname).cpu().numpy(), arr, f"{name} {cname}")
    if w.has_fp8:
        _assert_same(p.sparse_indices.cpu().numpy(), ref["sparse_indices"], f"{name} indices")
        _assert_same(p.lens.cpu().numpy(), ref["lens"], f"{name} lens")
        g = p.gathered if toks is None else p.gathered[torch.from_numpy(toks).to(cuda_device)]
        _assert_same(_u16(g), ref["gathered"], f"{name} gathered rows")
    _assert_same(p.global_topk.cpu().numpy(), ref["global_topk"], f"{name} global top-k")
    _assert_same(p.global_lens.cpu().numpy(), ref["global_lens"], f"{name} global lens")
    gi = p.gathered_index if toks is None else p.gathered_index[torch.from_numpy(toks).to(cuda_device)]
    _assert_same(_u16(gi), ref["gathered_index"], f"{name} gathered mxfp4 rows")
    assert int(p.err.item()) == ref["err"] == 0
    del p


@pytest.mark.parametrize("bs", [1, 3, 64])
def test_index_build_int32_extremes(cuda_device, bs):
    """Base offsets at the int32 limits, pages whose slots straddle INT32_MAX,
    local indices near INT32_MAX: the 32-bit device arithmetic must agree with
    the oracle's 64-bit arithmetic."""
    rng = np.random.default_rng(bs)
    imax = 2**31 - 1
    maxp = imax // bs
    R, width, T, K = 3, 6, 24, 12
    table = rng.choice(np.array([maxp, maxp - 1, maxp + 1 if maxp + 1 <= imax else maxp, 0, 5, -1,
                                 imax], np.int64), size=(R, width)).astype(np.int32)
    base = np.array([-2**31, imax, 0], np.int32)
    t2r = rng.integers(0, R, size=T).astype(np.int32)
    cand = np.array([0, bs - 1, bs, imax, imax - 1, imax - bs, -1, 7], np.int64)
    topk = rng.choice(cand, size=(T, K)).astype(np.int32)
    # positions that reach logical pages 0.. of each base: p = (lp + base) * bs + o
    for r in range(R):
        lo = (int(base[r]) * bs) if base[r] >= 0 else 0
        for j in range(0, K, 3):
            rows = np.nonzero(t2r == r)[0]
            if rows.size and 0 <= lo <= imax - width * bs:
                topk[rows, j] = lo + int(rng.integers(0, width * bs))
    d = cuda_device
    out, lens = ops.compute_global_topk_indices_and_lens(
        _dev_i32(topk, d), _dev_i32(t2r, d), _dev_i32(table, d), bs,
        base_offsets=_dev_i32(base, d))
    want, wl = oracle.compute_global_topk_indices_and_lens(topk, t2r, table, bs, base_offsets=base)
    _assert_same(out.cpu().numpy(), want, "extreme global top-k")
    _assert_same(lens.cpu().numpy(), wl, "extreme lens")
    assert (want >= 0).any()


@pytest.mark.parametrize("bs", [1, 16, 64])
@pytest.mark.parametrize("base", [-3, 0, 2])
def test_index_build_staged_tables_large_batch(cuda_device, bs, base):
    """Batches large enough for one warp per token and 8 tokens per CTA, one
    request per CTA (tables staged in shared memory): negative and positive
    base offsets, -1 pages and pages whose slots pass INT32_MAX, top-k entries
    below, inside and past each table's range, replay_start, invalid tokens;
    one request with positions near INT32_MAX."""
    rng = np.random.default_rng(100 * bs + base + 7)
    imax = 2**31 - 1
    maxp = imax // bs
    R, width, K, W = 3, 24, 16, 8
    qlen = np.array([1500, 1200, 40], np.int64)
    seq = np.array([1500 + 300, 1200 + 5, imax - 3], np.int64)
    qsl = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    T = int(qsl[-1])
    t2r = np.repeat(np.arange(R), qlen).astype(np.int32)
    valid = (rng.random(T) < 0.9).astype(np.uint8)
    replay = np.array([0, 600, 0], np.int32)
    pages = rng.integers(-1, 50, size=(R, width)).astype(np.int64)
    pages[rng.random(pages.shape) < 0.1] = maxp
    if maxp + 1 <= imax:
        pages[rng.random(pages.shape) < 0.05] = maxp + 1
    table = pages.astype(np.int32)
    swa_table = rng.integers(-1, 50, size=(R, width)).astype(np.int32)
    bases = np.array([base, base + 1, 0], np.int32)
    # the third request's window lives at logical pages near imax // bs
    swa_base = np.array([base, base, (imax - 3 - 2 * W) // bs], np.int32)
    lo = np.maximum(bases.astype(np.int64) * bs, 0)
    topk = np.empty((T, K), np.int64)
    for r in range(R):
        rows = t2r == r
        span = width * bs
        topk[rows] = rng.integers(lo[r] - bs, lo[r] + span + bs, size=(int(rows.sum()), K))
    topk[rng.random(topk.shape) < 0.1] = -1
    topk[rng.random(topk.shape) < 0.02] = imax
    topk = np.clip(topk, -1, imax).astype(np.int32)
    d = cuda_device
    si, lens = ops.combine_topk_swa_indices(
        _dev_i32(qsl, d), _dev_i32(seq.astype(np.int32), d), _dev_i32(t2r, d), _dev_i32(replay, d),
        _dev_i32(swa_table, d), bs, _dev_i32(table, d), bs, W, 4, _dev_i32(topk, d),
        swa_base_offsets=_dev_i32(swa_base, d), compressed_base_offsets=_dev_i32(bases, d),
        is_valid_token=torch.from_numpy(valid).to(d), num_tokens=T)
    want, want_lens = oracle.combine_topk_swa_indices(
        qsl, seq.astype(np.int32), t2r, replay, swa_table, bs, table, bs, W, 4, topk,
        swa_base_offsets=swa_base, comp_base_offsets=bases, is_valid_token=valid)
    _assert_same(si.cpu().numpy(), want, "staged combine")
    _assert_same(lens.cpu().numpy(), want_lens, "staged combine lens")
    assert (want[:, :W] >= 0).any() and (want[:, W:] >= 0).any()
    out, gl = ops.compute_global_topk_indices_and_lens(
        _dev_i32(topk, d), _dev_i32(t2r, d), _dev_i32(table, d), bs,
        torch.from_numpy(valid).to(d), base_offsets=_dev_i32(bases, d))
    want_g, want_gl = oracle.compute_global_topk_indices_and_lens(
        topk, t2r, table, bs, base_offsets=bases, is_valid_token=valid)
    _assert_same(out.cpu().numpy(), want_g, "staged global top-k")
    _assert_same(gl.cpu().numpy(), want_gl, "staged global lens")


@pytest.mark.parametrize("split_kind", ["zero", "mid", "all"])
@pytest.mark.parametrize("D,rope", [(512, 64), (128, 0)])
def test_pair_gather_matches_two_range_gathers(cuda_device, split_kind, D, rope):
    """One index matrix over two caches (different pages, strides and page
    sizes): columns < split from cache A, the rest from cache B; slots past
    either cache's capacity give zero rows; strided output."""
    rng = np.random.default_rng(D + {"zero": 0, "mid": 1, "all": 2}[split_kind])
    rec = oracle.fp8_record_bytes(D, rope, True)
    ga = synthetic.CacheGeom(9, 16, (16 * rec + 15) // 16 * 16 + 32)
    gb = synthetic.CacheGeom(13, 5, (5 * rec + 15) // 16 * 16)
    ha = synthetic.random_cache_bytes(31, ga)
    hb = synthetic.random_cache_bytes(32, gb)
    R, Cc = 37, 21
    split = {"zero": 0, "mid": 8, "all": Cc}[split_kind]
    cap_a, cap_b = 9 * 16, 13 * 5
    idx = rng.integers(-1, max(cap_a, cap_b) + 4, size=(R, Cc)).astype(np.int32)
    idx[0, :] = -1
    idx[1, :] = cap_b  # valid in A, past B
    idx[2, :] = cap_a  # past A (and B)
    d = cuda_device
    out = torch.full((R, Cc + 2, D), 3, dtype=torch.bfloat16, device=d)
    ops.dequantize_and_gather_k_cache_pair(out[:, 1:Cc + 1], torch.from_numpy(ha).to(d), 16,
                                           torch.from_numpy(hb).to(d), 5,
                                           _dev_i32(idx, d), split, rope_dim=rope)
    got = _u16(out)
    want_a = oracle.dequantize_and_gather_k_cache(ha, 16, 0, D, rope, np.ascontiguousarray(idx[:, :split]))
    want_b = oracle.dequantize_and_gather_k_cache(hb, 5, 0, D, rope, np.ascontiguousarray(idx[:, split:]))
    _assert_same(got[:, 1:1 + split], want_a, "pair gather, cache A columns")
    _assert_same(got[:, 1 + split:Cc + 1], want_b, "pair gather, cache B columns")
    three = np.uint16(torch.tensor(3.0, dtype=torch.bfloat16).view(torch.int16).item())
    assert np.all(got[:, 0] == three) and np.all(got[:, Cc + 1] == three)


# ---- fused gathers (slots computed in the gather) ---------------------------------------

@pytest.mark.parametrize("seed", range(12))
def test_fused_gathers_match_two_step_oracle(cuda_device, seed):
    """gather_topk == compute_global_topk + gather and gather_window == the
    window columns of combine + gather, on random metadata (padding tokens,
    requests out of range, base offsets, replay_start, -1 table entries and
    top-k entries, odd page sizes) for the three records."""
    rng = np.random.default_rng(7000 + seed)
    d = cuda_device
    bs = int(rng.choice([1, 4, 5, 16, 64]))
    R = int(rng.integers(1, 5))
    qlen = rng.integers(0, 6, size=R)
    seq = (qlen + rng.integers(0, 40 * bs // 4 + 8, size=R)).astype(np.int32)
    qsl = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    T = int(qsl[-1])
    if T == 0:
        return
    t2r = np.repeat(np.arange(R), qlen).astype(np.int32)
    t2r[rng.random(T) < 0.1] = R
    valid = None if rng.random() < 0.5 else (rng.random(T) < 0.85)
    replay = None if rng.random() < 0.5 else rng.integers(0, 6, size=R).astype(np.int32)
    width, pages = 12, 30
    table = rng.integers(-1, pages, size=(R, width)).astype(np.int32)
    base = None if rng.random() < 0.5 else rng.integers(0, 2, size=R).astype(np.int32)
    K, W = int(rng.choice([4, 16, 20])), int(rng.choice([4, 8, 12]))
    topk = rng.integers(-1, width * bs + 3, size=(T, K)).astype(np.int32)
    for rec, D, rope in ((0, 512, 64), (0, 128, 0), (1, 128, 0), (2, 64, 0)):
        rb = oracle.fp8_record_bytes(D, rope, True) if rec == 0 else (
            D // 2 + D // 32 if rec == 1 else D + 4)
        geom = synthetic.CacheGeom(pages, bs, (bs * rb + 15) // 16 * 16)
        host = synthetic.random_cache_bytes(17 + rec, geom)
        if rec == 2:  # finite binary32 scales
            for s_ in range(pages * bs):
                pg, off = divmod(s_, bs)
                host[pg, bs * D + off * 4: bs * D + off * 4 + 4] = np.frombuffer(
                    np.float32(2.0 ** int(rng.integers(-20, 20))).tobytes(), np.uint8)
        dev_cache = torch.from_numpy(host).to(d)
        gt, _ = oracle.compute_global_topk_indices_and_lens(topk, t2r, table, bs, base_offsets=base,
                                                            is_valid_token=valid)
        want = oracle.dequantize_and_gather_k_cache(host, bs, rec, D, rope, gt)
        out = torch.full((T, K + 1, D), 5, dtype=torch.bfloat16, device=d)
        ops.dequantize_and_gather_k_cache_topk(
            out[:, 1:], dev_cache, _dev_i32(topk, d), _dev_i32(t2r, d), _dev_i32(table, d), bs,
            record=rec, rope_dim=rope, num_reqs=R, base_offsets=_dev_i32(base, d),
            is_valid_token=None if valid is None else torch.from_numpy(valid.astype(np.uint8)).to(d))
        _assert_same(_u16(out[:, 1:]), want, f"fused topk gather rec={rec} D={D}")
        if rec != 0:
            continue
        si, _ = oracle.combine_topk_swa_indices(qsl, seq, t2r, replay, table, bs, table, bs, W, 4,
                                                np.zeros((T, 0), np.int32), swa_base_offsets=base,
                                                is_valid_token=valid)
        want = oracle.dequantize_and_gather_k_cache(host, bs, 0, D, rope, np.ascontiguousarray(si[:, :W]))
        outw = torch.empty((T, W, D), dtype=torch.bfloat16, device=d)
        ops.dequantize_and_gather_k_cache_window(
            outw, dev_cache, _dev_i32(qsl, d), _dev_i32(seq, d), _dev_i32(t2r, d),
            _dev_i32(replay, d), _dev_i32(table, d), bs, W, rope_dim=rope,
            base_offsets=_dev_i32(base, d),
            is_valid_token=None if valid is None else torch.from_numpy(valid.astype(np.uint8)).to(d))
        _assert_same(_u16(outw), want, f"fused window gather D={D}")


@pytest.mark.parametrize("name,mode", [("decode", "graph"), ("tiny", "serial"),
                                       ("mixed", "concurrent"), ("mxfp4", "graph")])
def test_fused_step_matches_index_step(cuda_device, name, mode):
    """The fused step's outputs equal the index step's (itself pinned against
    the oracle): same caches, indices, lens and gathered rows."""
    from paged_sparse_kv_gb300.pipeline import Pipeline
    w = synthetic.make(name)
    outs = []
    for path in ("index", "fused"):
        p = Pipeline(w, cuda_device)
        for cname, geom in (("swa_cache", w.swa_cache), ("comp_cache", w.comp_cache),
                            ("index_cache", w.index_cache)):
            if geom is not None:
                getattr(p, cname).copy_(torch.from_numpy(synthetic.random_cache_bytes(91, geom)))
        if mode == "graph":
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(cuda_device)
            side.wait_stream(torch.cuda.current_stream(cuda_device))
            with torch.cuda.graph(g, stream=side):
                p.step(concurrent=True, path=path)
            g.replay()
        else:
            p.step(concurrent=(mode == "concurrent"), path=path)
        torch.cuda.synchronize(cuda_device)
        outs.append([t.cpu() for t in (p.sparse_indices, p.lens, p.gathered, p.global_topk,
                                       p.global_lens, p.gathered_index, p.swa_cache,
                                       p.index_cache) if t is not None])
        del p
        torch.cuda.empty_cache()
    for a, b in zip(*outs):
        assert torch.equal(a, b)
