"""Pins for the oracle's inserts and gather (record layouts and codecs).

* Hand-worked golden records (tests/golden/*_record_golden.json) fix every
  byte offset, the nibble order, the scale bytes and the skip rules.
* Round trips are checked against the quantisation error bound that the
  block-scaled formats guarantee (half a step of the code grid, times the
  block scale), with scale invariants checked in exact arithmetic.
* The gather's decode is checked against torch's own float8_e4m3fn decode
  and bfloat16 rounding on arbitrary record bytes.
"""
import json
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def _bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def _row_from_runs(runs, head_dim, rope_dim=0, rope_rule=None):
    vals = []
    for count, v in runs:
        if isinstance(v, list):
            vals.extend(v * count)
        else:
            vals.extend([v] * count)
    row = np.array(vals, dtype=np.float32)
    if rope_rule is not None:
        row = np.concatenate([row, 1.0 + np.arange(rope_dim, dtype=np.float32) / 128.0])
    assert row.size == head_dim, (row.size, head_dim)
    bits = _bf16_bits(row)
    # keep -0.0 exactly
    bits[np.signbit(row) & (row == 0)] = 0x8000
    return bits


def _check_expected(cache_flat, fill, expected):
    want = np.full_like(cache_flat, fill)
    for e in expected:
        b = bytes.fromhex(e["hex"]) * e.get("repeat", 1)
        want[e["at"]:e["at"] + len(b)] = np.frombuffer(b, dtype=np.uint8)
    diff = np.nonzero(cache_flat != want)[0]
    assert diff.size == 0, [(int(i), hex(cache_flat[i]), hex(want[i])) for i in diff[:10]]


def test_fp8_record_golden(oracle_mod):
    spec = json.load(open(os.path.join(GOLDEN, "fp8_record_golden.json")))
    for case in spec["cases"]:
        D, rope = case["head_dim"], case["rope_dim"]
        rows = [_row_from_runs(r["runs"], D, rope, r.get("rope")) for r in case["rows"]]
        k = np.stack(rows)
        slots = np.array([r["slot"] for r in case["rows"]], dtype=np.int64)
        cache = np.full((case["num_pages"], case["page_stride"]), case["fill"], np.uint8)
        err = oracle_mod.quantize_and_insert_k_cache(
            k, slots, cache, case["block_size"], D, rope, case["is_ue8m0"])
        assert err == case["expected_errors"], case["name"]
        _check_expected(cache.reshape(-1), case["fill"], case["expected"])


def _golden_row_bits(spec_runs, rope_bits):
    """bf16 bit patterns of an expected gathered row: runs of hex bf16 words,
    with "rope" standing for the row's verbatim RoPE tail."""
    out = []
    for count, v in spec_runs:
        if v == "rope":
            out.extend(rope_bits.tolist())
        elif isinstance(v, list):
            out.extend([int(x, 16) for x in v] * count)
        else:
            out.extend([int(v, 16)] * count)
    return np.array(out, dtype=np.uint16)


def test_fp8_record_golden_gather(oracle_mod):
    """Cases with a hand-worked gather: the inserted record read back through
    dequantize_and_gather_k_cache, every bf16 word as worked out by hand."""
    spec = json.load(open(os.path.join(GOLDEN, "fp8_record_golden.json")))
    cases = [c for c in spec["cases"] if "gather" in c]
    assert cases, "no hand-worked gather"
    for case in cases:
        D, rope = case["head_dim"], case["rope_dim"]
        rows = [_row_from_runs(r["runs"], D, rope, r.get("rope")) for r in case["rows"]]
        k = np.stack(rows)
        slots = np.array([r["slot"] for r in case["rows"]], dtype=np.int64)
        cache = np.full((case["num_pages"], case["page_stride"]), case["fill"], np.uint8)
        oracle_mod.quantize_and_insert_k_cache(k, slots, cache, case["block_size"], D, rope,
                                               case["is_ue8m0"])
        g = case["gather"]
        idx = np.array([g["indices"]], dtype=np.int32)
        out = oracle_mod.dequantize_and_gather_k_cache(cache, case["block_size"], 0, D, rope, idx,
                                                       is_ue8m0=case["is_ue8m0"])
        for j, want_runs in enumerate(g["rows"]):
            s = g["indices"][j]
            rope_bits = k[list(slots).index(s), D - rope:] if s >= 0 else None
            want = _golden_row_bits(want_runs, rope_bits)
            assert np.array_equal(out[0, j], want), (case["name"], j)


def test_mxfp4_record_golden(oracle_mod):
    spec = json.load(open(os.path.join(GOLDEN, "mxfp4_record_golden.json")))
    for case in spec["cases"]:
        D = case["head_dim"]
        k = np.stack([_row_from_runs(r["runs"], D) for r in case["rows"]])
        slots = np.array([r["slot"] for r in case["rows"]], dtype=np.int64)
        cache = np.full((case["num_pages"], case["page_stride"]), case["fill"], np.uint8)
        err = oracle_mod.write_indexer_mxfp4_cache(k, slots, cache, case["block_size"], D)
        assert err == case["expected_errors"]
        _check_expected(cache.reshape(-1), case["fill"], case["expected"])


def _e4m3_half_step(v):
    """Half the E4M3 grid spacing around |v| (2^-9 below 2^-6)."""
    a = np.abs(v.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return 0.5 * np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))


def _e2m1_half_step(v):
    a = np.abs(v.astype(np.float64))
    return 0.5 * np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))


@pytest.mark.parametrize("head_dim,rope_dim", [(512, 64), (128, 0), (256, 128)])
@pytest.mark.parametrize("outliers", [False, True])
def test_fp8_roundtrip_bound_and_scale_invariant(oracle_mod, head_dim, rope_dim, outliers):
    rng = np.random.default_rng(head_dim + rope_dim + outliers)
    N, bs = 300, 16
    x = rng.standard_normal((N, head_dim)).astype(np.float32)
    if outliers:
        x = np.where(rng.random(x.shape) < 0.01, x * 20, x)
    x[0, :64] = 0.0                     # an all-zero block (amax floor)
    x[1, :64] = 1e-6                    # a block below the floor
    x[2, :] = -x[2, :]
    k = _bf16_bits(x)
    xf = _bits_to_f32(k).astype(np.float64)
    num_pages = (N + bs - 1) // bs + 3
    rec = oracle_mod.fp8_record_bytes(head_dim, rope_dim)
    cache = np.zeros((num_pages, bs * rec + 16), np.uint8)
    slots = rng.permutation(num_pages * bs)[:N].astype(np.int64)
    assert oracle_mod.quantize_and_insert_k_cache(k, slots, cache, bs, head_dim, rope_dim) == 0
    out = oracle_mod.dequantize_and_gather_k_cache(cache, bs, 0, head_dim, rope_dim,
                                                   slots.astype(np.int32).reshape(-1, 1))
    deq = _bits_to_f32(out[:, 0, :]).astype(np.float64)
    nope = head_dim - rope_dim
    # rope dims are verbatim
    assert np.array_equal(out[:, 0, nope:], k[:, nope:])
    # per block: 2^(e-1) < max(amax,1e-4)/448 <= 2^e, and |x - deq| <= half step * 2^e
    ts = oracle_mod.fp8_token_stride(head_dim, rope_dim)
    for i in range(N):
        page, off = divmod(int(slots[i]), bs)
        scl = cache[page, bs * ts + off * (head_dim // 64):bs * ts + (off + 1) * (head_dim // 64)]
        for b in range(nope // 64):
            blk = xf[i, b * 64:(b + 1) * 64]
            amax = max(np.abs(blk).max(), float(np.float32(1e-4)))
            q = float(np.float32(np.float32(amax) / np.float32(448.0)))
            e = int(scl[b]) - 127
            assert 2.0 ** (e - 1) < q <= 2.0 ** e
            v = blk * 2.0 ** -e
            err = np.abs(blk - deq[i, b * 64:(b + 1) * 64])
            assert np.all(err <= _e4m3_half_step(v) * 2.0 ** e), (i, b)
        assert np.all(scl[nope // 64:] == 0)


def test_mxfp4_roundtrip_bound(oracle_mod):
    rng = np.random.default_rng(5)
    N, bs, D = 500, 64, 128
    x = rng.standard_normal((N, D)).astype(np.float32)
    x[0, :32] = 0.0
    k = _bf16_bits(x)
    xf = _bits_to_f32(k).astype(np.float64)
    num_pages = 10
    cache = np.zeros((num_pages, bs * 68), np.uint8)
    slots = rng.permutation(num_pages * bs)[:N].astype(np.int64)
    assert oracle_mod.write_indexer_mxfp4_cache(k, slots, cache, bs, D) == 0
    out = oracle_mod.dequantize_and_gather_k_cache(cache, bs, 1, D, 0,
                                                   slots.astype(np.int32).reshape(-1, 1))
    deq = _bits_to_f32(out[:, 0, :]).astype(np.float64)
    for i in range(N):
        page, off = divmod(int(slots[i]), bs)
        scl = cache[page, bs * 64 + off * 4: bs * 64 + off * 4 + 4]
        for b in range(4):
            blk = xf[i, b * 32:(b + 1) * 32]
            e = int(scl[b]) - 127
            q = float(np.float32(np.float32(max(np.abs(blk).max(), float(np.float32(1e-4))))
                                 / np.float32(6.0)))
            assert 2.0 ** (e - 1) < q <= 2.0 ** e
            v = blk * 2.0 ** -e
            assert np.all(np.abs(v) <= 6.0)
            err = np.abs(blk - deq[i, b * 32:(b + 1) * 32])
            assert np.all(err <= _e2m1_half_step(v) * 2.0 ** e), (i, b)


def test_fp8_gather_decode_vs_torch_on_random_bytes(oracle_mod):
    """Arbitrary record bytes (no NaN codes): decode with torch's e4m3 decode,
    a power-of-two scale as binary32 and torch's bf16 rounding."""
    rng = np.random.default_rng(9)
    bs, D, rope, pages = 8, 512, 64, 4
    rec = oracle_mod.fp8_record_bytes(D, rope)
    cache = rng.integers(0, 254, size=(pages, bs * rec), dtype=np.uint8)
    cache[cache >= 0x7F] += 1
    idx = np.array([[0, 5, 31, -1, 32, 7]], dtype=np.int32)
    out = oracle_mod.dequantize_and_gather_k_cache(cache, bs, 0, D, rope, idx)
    ts = D - rope + 2 * rope
    for j, s in enumerate(idx[0]):
        if s < 0 or s >= pages * bs:
            assert np.all(out[0, j] == 0)
            continue
        page, off = divmod(int(s), bs)
        data = cache[page, off * ts:(off + 1) * ts]
        scl = cache[page, bs * ts + off * 8: bs * ts + off * 8 + 8]
        vals = torch.from_numpy(data[:D - rope].copy()).view(torch.float8_e4m3fn).to(torch.float32)
        pw = torch.from_numpy(np.repeat(scl[:7].astype(np.int32) - 127, 64))
        sc = torch.pow(torch.tensor(2.0, dtype=torch.float32), pw.to(torch.float32))
        ref = (vals * sc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(out[0, j, :D - rope], ref)
        assert np.array_equal(out[0, j, D - rope:], data[D - rope:].view(np.uint16))


def test_fp32_scale_gather_decode_vs_torch_on_random_bytes(oracle_mod):
    """fp32-scale records (is_ue8m0 = 0) of arbitrary bytes: every e4m3 code
    but the two NaNs and binary32 scales of random finite bit patterns
    (normals of every exponent, subnormals, zeros of both signs), so the
    products round, overflow to +-inf and underflow.  Expected: torch's e4m3
    decode, a binary32 multiply by the little-endian scale, torch's bf16
    rounding -- with slots past the nope blocks (the pad) never read."""
    rng = np.random.default_rng(19)
    bs, D, rope, pages = 8, 512, 64, 6
    nope, ts, nb = D - rope, D - rope + 2 * rope, D // 64
    rec = oracle_mod.fp8_record_bytes(D, rope, is_ue8m0=False)
    assert rec == ts + 4 * nb
    cache = rng.integers(0, 254, size=(pages, bs * rec), dtype=np.uint8)
    cache[cache >= 0x7F] += 1                       # no 0x7F / 0xFF codes
    data = cache[:, :bs * ts].reshape(pages, bs, ts)
    scl = rng.integers(0, 1 << 32, size=(pages, bs, nb), dtype=np.uint64).astype(np.uint32)
    expo = (scl >> 23) & 0xFF
    scl[expo == 0xFF] &= ~np.uint32(0x40000000)     # inf/NaN exponent -> a finite one
    scl[0, 0, :] = np.array([0, 0x80000000, 1, 0x807FFFFF, 0x7F7FFFFF, 0x00800000, 0x3F800000,
                             0x3B800000], np.uint32)
    cache[:, bs * ts:] = scl.view(np.uint8).reshape(pages, bs * 4 * nb)
    idx = np.arange(pages * bs, dtype=np.int32).reshape(pages, bs)
    idx[1, 3] = -1
    idx[2, 5] = pages * bs        # beyond the cache: a zero row
    out = oracle_mod.dequantize_and_gather_k_cache(cache, bs, 0, D, rope, idx, is_ue8m0=False)
    for r in range(pages):
        for j in range(bs):
            s = int(idx[r, j])
            if s < 0 or s >= pages * bs:
                assert np.all(out[r, j] == 0)
                continue
            page, off = divmod(s, bs)
            vals = torch.from_numpy(data[page, off, :nope].copy()).view(
                torch.float8_e4m3fn).to(torch.float32)
            sc = torch.from_numpy(np.repeat(scl[page, off, :nope // 64], 64).view(np.float32))
            ref = (vals * sc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(out[r, j, :nope], ref), (r, j)
            assert np.array_equal(out[r, j, nope:], data[page, off, nope:].view(np.uint16))
    flat = out[:, :, :nope].reshape(-1)
    assert np.any(flat == 0x7F80) or np.any(flat == 0xFF80), "no product overflowed"
    assert np.any(((flat & 0x7F80) == 0) & ((flat & 0x7FFF) != 0)), "no subnormal result"


def test_mxfp4_gather_decode_vs_torch_on_random_bytes(oracle_mod):
    rng = np.random.default_rng(10)
    bs, D, pages = 4, 128, 3
    cache = rng.integers(0, 256, size=(pages, bs * 68), dtype=np.uint8)
    idx = np.array([[0, 11, -1, 12, 3]], dtype=np.int32)
    out = oracle_mod.dequantize_and_gather_k_cache(cache, bs, 1, D, 0, idx)
    mag = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    for j, s in enumerate(idx[0]):
        if s < 0 or s >= pages * bs:
            assert np.all(out[0, j] == 0)
            continue
        page, off = divmod(int(s), bs)
        packed = torch.from_numpy(cache[page, off * 64:(off + 1) * 64].astype(np.int64))
        nib = torch.stack([packed & 0xF, packed >> 4], dim=1).reshape(-1)
        val = mag[nib & 7] * torch.where((nib & 8) != 0, -1.0, 1.0)
        scl = cache[page, bs * 64 + off * 4: bs * 64 + off * 4 + 4].astype(np.int32) - 127
        sc = torch.pow(torch.tensor(2.0), torch.from_numpy(np.repeat(scl, 32)).float())
        ref = (val * sc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(out[0, j], ref)


def test_insert_skips_negative_and_counts_out_of_range(oracle_mod):
    rng = np.random.default_rng(1)
    bs, D, rope, pages = 4, 128, 0, 2
    k = _bf16_bits(rng.standard_normal((5, D)))
    cache = np.full((pages, bs * 130 + 8), 0xA5, np.uint8)
    before = cache.copy()
    slots = np.array([-1, 8, 9, -7, 1 << 40], dtype=np.int64)
    assert oracle_mod.quantize_and_insert_k_cache(k, slots, cache, bs, D, rope) == 3
    assert np.array_equal(cache, before)
    cache4 = np.full((pages, bs * 68), 0xA5, np.uint8)
    b4 = cache4.copy()
    assert oracle_mod.write_indexer_mxfp4_cache(k, slots, cache4, bs, D) == 3
    assert np.array_equal(cache4, b4)


def test_fp32_scale_record_division_identity(oracle_mod):
    """fp32-scale record (also pinned by a hand-worked golden record and by
    the decode against torch above): the stored
    scale is binary32 max(amax, 1e-12) / 448 and every code is the e4m3 of the
    binary32 quotient x / scale, clamped."""
    rng = np.random.default_rng(2)
    D, rope, bs = 512, 64, 4
    x = rng.standard_normal((6, D)).astype(np.float32)
    x[1, :64] = 0
    k = _bf16_bits(x)
    xf = _bits_to_f32(k)
    rec = oracle_mod.fp8_record_bytes(D, rope, is_ue8m0=False)
    assert rec == 448 + 128 + 32
    cache = np.zeros((2, bs * rec), np.uint8)
    slots = np.arange(6, dtype=np.int64)
    oracle_mod.quantize_and_insert_k_cache(k, slots, cache, bs, D, rope, is_ue8m0=False)
    ts = 576
    for i in range(6):
        page, off = divmod(i, bs)
        scl = cache[page, bs * ts + off * 32: bs * ts + off * 32 + 32].view(np.float32)
        for b in range(7):
            blk = xf[i, b * 64:(b + 1) * 64]
            want = np.float32(max(np.abs(blk).max(), np.float32(1e-12))) / np.float32(448.0)
            assert scl[b] == want
            q = np.clip(blk / scl[b], np.float32(-448), np.float32(448)).astype(np.float32)
            codes = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            data = cache[page, off * ts + b * 64: off * ts + (b + 1) * 64]
            assert np.array_equal(data, codes)
        assert scl[7] == 0.0


# ---- non-finite inputs (closed forms) ----------------------------------------------------

_NAN, _NNAN, _INF, _NINF = 0x7FC0, 0xFFC0, 0x7F80, 0xFF80


def test_codec_specials():
    """E4M3: NaN -> S.1111.111 (0x7F), +-inf and anything >= 448 saturate to
    +-448 (0x7E / 0xFE).  E2M1 has no NaN or inf: +-inf saturate to +-6, NaN -> +6."""
    import oracle
    v = np.array([np.nan, -np.nan, np.inf, -np.inf, 448.0, 1e30, -500.0], np.float32)
    assert oracle.e4m3_encode(v).tolist() == [0x7F, 0x7F, 0x7E, 0xFE, 0x7E, 0x7E, 0xFE]
    assert oracle.e2m1_encode(v).tolist() == [0x7, 0x7, 0x7, 0xF, 0x7, 0x7, 0xF]


def _fp8_insert_one(row_bits):
    import oracle
    D, rope, bs = 128, 0, 1
    cache = np.zeros((1, oracle.fp8_record_bytes(D, rope)), np.uint8)
    oracle.quantize_and_insert_k_cache(row_bits[None, :], np.zeros(1, np.int64), cache, bs, D, rope)
    return cache[0, :D], cache[0, D:D + 2]


def test_fp8_insert_block_amax_passes_over_nan():
    """Block 0 = [NaN, 3, -1, 0...]: amax 3 (NaN skipped), e = ceil(log2(3/448)) = -7,
    byte 120, codes 3 * 2^7 = 384 -> 0x7C, -128 -> 0xF0, NaN -> 0x7F.  Block 1 all NaN:
    amax 0 -> the 1e-4 floor, e = ceil(log2(1e-4/448)) = -22, byte 105, codes NaN."""
    row = np.zeros(128, np.uint16)
    row[0], row[1], row[2] = _NAN, _bf16_bits([3.0])[0], _bf16_bits([-1.0])[0]
    row[64:128] = _NNAN
    codes, scales = _fp8_insert_one(row)
    assert scales.tolist() == [120, 105]
    assert codes[:3].tolist() == [0x7F, 0x7C, 0xF0] and not codes[3:64].any()
    assert np.all(codes[64:] == 0x7F)


def test_fp8_insert_block_with_inf():
    """Block 0 = [inf, -inf, 1, 0...]: amax inf, e = 128, byte clamped to 255;
    codes +-inf * 2^-128 = +-inf -> +-448 (0x7E / 0xFE), 1 * 2^-128 -> 0."""
    row = np.zeros(128, np.uint16)
    row[0], row[1], row[2] = _INF, _NINF, _bf16_bits([1.0])[0]
    codes, scales = _fp8_insert_one(row)
    assert scales[0] == 255
    assert codes[:3].tolist() == [0x7E, 0xFE, 0x00]


def test_mxfp4_insert_block_amax_passes_over_nan():
    """Block 0 = [NaN, 3, 0...]: amax 3, e = ceil(log2(3/6)) = -1, byte 126; codes
    NaN -> 0x7 (low nibble), 3 * 2 = 6 -> 0x7 (high nibble).  Block 1 = [inf, 0...]:
    e = 128, byte clamped to 254, inf -> 0x7."""
    import oracle
    D = 128
    row = np.zeros(D, np.uint16)
    row[0], row[1] = _NAN, _bf16_bits([3.0])[0]
    row[32] = _INF
    cache = np.zeros((1, oracle.mxfp4_record_bytes(D)), np.uint8)
    oracle.write_indexer_mxfp4_cache(row[None, :], np.zeros(1, np.int64), cache, 1, D)
    vals, scales = cache[0, :D // 2], cache[0, D // 2:]
    assert vals[0] == 0x77 and not vals[1:16].any()
    assert scales[0] == 126 and scales[1] == 254
    assert vals[16] == 0x07 and not vals[17:32].any()
