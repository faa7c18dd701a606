"""Pins for the oracle's indexer-key variants: the FP8 indexer record (writer
and reader) and indexer_k_norm_rope_store.

* Hand-worked FP8 indexer records (tests/golden/indexer_fp8_golden.json).
* The writer against torch's own float8_e4m3fn cast of x / scale, with the
  scale found by an exact search over powers of two (not a log2).
* The reader against torch's float8_e4m3fn decode times the stored scale.
* indexer_k_norm_rope_store against closed forms: a constant row normalises to
  exactly 1 (sum of squares 128 c^2, rsqrt exact), a 90-degree RoPE row maps
  (e, o) to (-o, e), and the quantised bytes of those values are worked by
  hand; the emission rule (slot >= 0 and a group boundary) and the RoPE row
  (the group's first position) are checked by which rows change.
* The RMSNorm reading (binary32 square root, then a binary32 division) against
  a correctly rounded reciprocal square root, on a row whose factor differs in
  the last bit between the two and a weight that turns that bit into a code.
"""
import json
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN

REC_MXFP4, REC_FP8_INDEXER = 1, 2


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def test_fp8_indexer_golden(oracle_mod):
    with open(os.path.join(GOLDEN, "indexer_fp8_golden.json")) as f:
        g = json.load(f)
    D, bs = g["head_dim"], g["block_size"]
    rows = np.zeros((len(g["rows"]), D), np.float32)
    slots = []
    for i, r in enumerate(g["rows"]):
        for k, v in r["values"].items():
            rows[i, int(k)] = v
        slots.append(r["slot"])
    cache = np.full((2, bs * (D + 4)), 0xAB, np.uint8)
    assert oracle_mod.write_indexer_fp8_cache(_bf16(rows), np.array(slots, np.int64), cache,
                                              bs, D) == 0
    flat = cache.reshape(-1)
    for r in g["rows"]:
        page, off = divmod(r["slot"], bs)
        base = page * cache.shape[1]
        codes = np.zeros(D, np.uint8)
        for k, v in r["codes"].items():
            codes[int(k)] = v
        assert flat[base + off * D: base + off * D + D].tolist() == codes.tolist()
        sc = flat[base + bs * D + off * 4: base + bs * D + off * 4 + 4]
        assert sc.tolist() == r["scale_bytes"]


def _pow2_scale(q):
    """Smallest power of two >= q (binary32 q > 0), by exact search."""
    e = -160
    while np.ldexp(1.0, e) < float(q):
        e += 1
    return np.float32(np.ldexp(1.0, e))


@pytest.mark.parametrize("D", [32, 128, 512])
def test_fp8_indexer_writer_vs_torch(oracle_mod, D):
    rng = np.random.default_rng(D)
    n, bs = 40, 4
    x = (rng.standard_normal((n, D)) * np.exp(rng.uniform(-12, 12, size=(n, 1)))).astype(np.float32)
    x[3] = 0.0
    k = _bf16(x)
    xf = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).float().numpy()
    cache = np.zeros((n // bs + 1, bs * (D + 4)), np.uint8)
    slots = np.arange(n, dtype=np.int64)
    oracle_mod.write_indexer_fp8_cache(k, slots, cache, bs, D)
    for t in range(n):
        page, off = divmod(t, bs)
        q = np.float32(np.abs(xf[t]).max()) / np.float32(448.0)
        q = max(q, np.float32(1e-10))
        scale = _pow2_scale(q)
        want = torch.from_numpy(np.clip(xf[t] / scale, -448, 448)).to(torch.float8_e4m3fn)
        got = cache[page, off * D: off * D + D]
        assert got.tolist() == want.view(torch.uint8).numpy().tolist()
        sc = cache[page, bs * D + off * 4: bs * D + off * 4 + 4].view(np.float32)[0]
        assert sc == scale


def test_fp8_indexer_reader_vs_torch(oracle_mod):
    rng = np.random.default_rng(7)
    D, bs, pages = 64, 8, 5
    cache = rng.integers(0, 256, size=(pages, bs * (D + 4)), dtype=np.uint8)
    cache[cache == 0x7F] = 0x7E
    cache[cache == 0xFF] = 0xFE
    exps = rng.integers(-40, 40, size=pages * bs)
    for s, e in enumerate(exps):  # power-of-two and arbitrary binary32 scales
        page, off = divmod(s, bs)
        v = np.float32(np.ldexp(1.0, int(e))) * (np.float32(1.37) if s % 3 == 0 else 1)
        cache[page, bs * D + off * 4: bs * D + off * 4 + 4] = np.frombuffer(
            np.float32(v).tobytes(), np.uint8)
    idx = rng.integers(-1, pages * bs, size=(6, 9)).astype(np.int32)
    out = oracle_mod.dequantize_and_gather_k_cache(cache, bs, REC_FP8_INDEXER, D, 0, idx)
    for t in range(idx.shape[0]):
        for j in range(idx.shape[1]):
            s = int(idx[t, j])
            if s < 0:
                assert np.all(out[t, j] == 0)
                continue
            page, off = divmod(s, bs)
            codes = torch.from_numpy(cache[page, off * D: off * D + D].copy()).view(
                torch.float8_e4m3fn).float()
            sc = torch.from_numpy(cache[page, bs * D + off * 4: bs * D + off * 4 + 4].copy()).view(
                torch.float32)
            want = (codes * sc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            assert out[t, j].tolist() == want.tolist()


def _cos_sin(max_pos, special=None):
    """cos = 1, sin = 0 on every row, except `special` rows: a 90-degree turn."""
    cs = np.zeros((max_pos, 64), np.float32)
    cs[:, :32] = 1.0
    for p in special or ():
        cs[p, :32] = 0.0
        cs[p, 32:] = 1.0
    return cs


def _read_mxfp4(cache, slot, bs):
    page, off = divmod(slot, bs)
    return (cache[page, off * 64: off * 64 + 64].tolist(),
            cache[page, bs * 64 + off * 4: bs * 64 + off * 4 + 4].tolist())


def _read_fp8(cache, slot, bs):
    page, off = divmod(slot, bs)
    return (cache[page, off * 128: off * 128 + 128].tolist(),
            cache[page, bs * 128 + off * 4: bs * 128 + off * 4 + 4].tolist())


def test_norm_rope_store_closed_form(oracle_mod):
    """x = 2.0 everywhere, weight 1, eps 0: sum of squares 512, variance 4,
    r = 0.5 exactly, y = 1.  Row 0 of cos_sin is a 90-degree turn: (1, 1) ->
    (-1, 1) on the RoPE half.  MXFP4: amax 1 -> e = ceil(log2(1/6)) = -2
    (scale byte 125), codes of 4 and -4 are 0x6 and 0xE: nope bytes 0x66,
    RoPE bytes 0x6E (even element low).  FP8: 1/448 in (2^-9, 2^-8] -> scale
    2^-8 (0x3B800000), codes of 256 and -256 are 0x78 and 0xF8."""
    bs = 4
    k = _bf16(np.full((1, 128), 2.0))
    pos = np.array([0], np.int64)
    cs = _cos_sin(8, special=[0])
    w = np.ones(128, np.float32)
    cache = np.zeros((2, bs * 68), np.uint8)
    assert oracle_mod.indexer_k_norm_rope_store(k, pos, cs, w, 0.0, np.array([5], np.int64), 1,
                                                REC_MXFP4, cache, bs) == 0
    vals, scl = _read_mxfp4(cache, 5, bs)
    assert vals == [0x66] * 32 + [0x6E] * 32 and scl == [125] * 4
    cache = np.zeros((2, bs * 132), np.uint8)
    oracle_mod.indexer_k_norm_rope_store(k, pos, cs, w, 0.0, np.array([6], np.int64), 1,
                                         REC_FP8_INDEXER, cache, bs)
    vals, scl = _read_fp8(cache, 6, bs)
    assert vals == [0x78] * 64 + [0xF8, 0x78] * 32
    assert scl == [0x00, 0x00, 0x80, 0x3B]


def test_norm_rope_store_weight_and_eps(oracle_mod):
    """x = 2, eps = 12: variance + eps = 16, r = 0.25 exactly; weight 4 on every
    dim gives y = 2 -> FP8 scale 2^-7, code of 256 = 0x78 (identity RoPE)."""
    bs = 2
    k = _bf16(np.full((1, 128), 2.0))
    cache = np.zeros((1, bs * 132), np.uint8)
    oracle_mod.indexer_k_norm_rope_store(k, np.array([3], np.int64), _cos_sin(8),
                                         np.full(128, 4.0, np.float32), 12.0,
                                         np.array([1], np.int64), 1, REC_FP8_INDEXER, cache, bs)
    vals, scl = _read_fp8(cache, 1, bs)
    assert vals == [0x78] * 128 and scl == [0, 0, 0, 0x3C]


def _f32(bits):
    return np.array([bits], np.uint32).view(np.float32)[0]


def test_norm_rope_store_rsqrt_reading(oracle_mod):
    """The RMSNorm factor is a binary32 square root followed by a binary32
    division, r = RN(1 / RN(sqrt(v + eps))), and not a correctly rounded
    reciprocal square root.  x = (3, 1, ..., 1), eps = 2^-7: the sum of squares
    is 136, v = 1.0625 and v + eps = 137/128, all exact.  RN(sqrt(137/128)) =
    1.03455913066864..., and 1 over it is 0.96659530649..., which rounds down
    to 0x3F7772CA (0.96659529209...); 1 / sqrt(137/128) = 0.96659534932... lies
    above the midpoint 0.96659532189... of the two and rounds up to 0x3F7772CB.
    Weight 0x3F80490B on dim 1 makes y_1 = RN(r * w_1) one binary32 step below
    31/32 under the first reading and exactly 31/32 under the second.  The row's
    amax is RN(3 r) = 2.89978..., so the FP8 scale is 2^-7 and 31/32 is 124
    scale units, the midpoint of the codes 120 (0x6F) and 128 (0x70): the first
    reading stores 0x6F and the second, its tie going to the even code, 0x70.
    Dim 0 stores 384 (0x7C, 371.17 units), every other dim 120 (0x6F, 123.70)."""
    rA, rB = _f32(0x3F7772CA), _f32(0x3F7772CB)
    s = np.float32(137.0 / 128.0)
    assert np.float32(1.0) / np.sqrt(s) == rA  # the binary32 reading (numpy: IEEE ops)
    assert np.float32(1.0 / np.sqrt(np.float64(s))) == rB  # rounded once
    w1 = _f32(0x3F80490B)
    assert np.float32(rA * w1) < np.float32(31 / 32) == np.float32(rB * w1)
    bs = 2
    x = np.ones((1, 128), np.float32)
    x[0, 0] = 3.0
    w = np.ones(128, np.float32)
    w[1] = w1
    cache = np.zeros((1, bs * 132), np.uint8)
    n = oracle_mod.indexer_k_norm_rope_store(_bf16(x), np.array([0], np.int64), _cos_sin(4), w,
                                             2.0 ** -7, np.array([1], np.int64), 1,
                                             REC_FP8_INDEXER, cache, bs)
    assert n == 0
    vals, scl = _read_fp8(cache, 1, bs)
    assert vals == [0x7C] + [0x6F] * 127  # a correctly rounded rsqrt stores 0x70 at dim 1
    assert scl == [0, 0, 0, 0x3C]


def test_norm_rope_store_emission_and_rope_row(oracle_mod):
    """Ratio 2: only tokens with (pos + 1) % 2 == 0 and a slot write; their RoPE
    row is the group's first position pos - 1.  Row 4 is the only rotating
    row, so exactly the token at position 5 (group 4..5) comes out rotated."""
    bs = 8
    k = _bf16(np.full((6, 128), 2.0))
    pos = np.array([2, 3, 4, 5, 6, 7], np.int64)
    slots = np.array([0, 1, 2, 3, -1, 5], np.int64)
    cache = np.full((1, bs * 132), 0xAB, np.uint8)
    n_err = oracle_mod.indexer_k_norm_rope_store(k, pos, _cos_sin(8, special=[4]),
                                                 np.ones(128, np.float32), 0.0, slots, 2,
                                                 REC_FP8_INDEXER, cache, bs)
    assert n_err == 0
    ident = [0x78] * 128
    rot = [0x78] * 64 + [0xF8, 0x78] * 32
    assert _read_fp8(cache, 1, bs)[0] == ident  # pos 3: group 2..3, identity row 2
    assert _read_fp8(cache, 3, bs)[0] == rot    # pos 5: group 4..5, row 4 rotates
    assert _read_fp8(cache, 5, bs)[0] == ident  # pos 7: row 6
    for untouched in (0, 2, 4):                  # pos 2, 4 not boundaries; slot -1
        assert _read_fp8(cache, untouched, bs)[0] == [0xAB] * 128


def test_norm_rope_store_out_of_range_counted(oracle_mod):
    bs = 4
    k = _bf16(np.ones((3, 128)))
    cache = np.zeros((1, bs * 68), np.uint8)
    n = oracle_mod.indexer_k_norm_rope_store(k, np.array([0, 9, 1], np.int64), _cos_sin(8),
                                             np.ones(128, np.float32), 1e-6,
                                             np.array([4, 1, 2], np.int64), 1, REC_MXFP4,
                                             cache, bs)
    assert n == 2  # slot 4 beyond the 4-slot cache; RoPE row 9 beyond max_pos 8
    assert np.all(cache[0, 64:128] == 0)  # slot 1 (row 9) not written


@pytest.mark.parametrize("seed", range(6))
def test_norm_rope_store_error_bound(oracle_mod, seed):
    """Random rows and a GPT-J table cos(p * theta_i), sin(p * theta_i): the
    stored key dequantises to the rotated, normalised row within half a code
    step times the scale (plus binary32 rounding of the inputs)."""
    rng = np.random.default_rng(seed)
    n, bs, max_pos = 32, 8, 64
    x = (rng.standard_normal((n, 128)) * rng.uniform(0.01, 50, size=(n, 1))).astype(np.float32)
    k = _bf16(x)
    xf = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).double().numpy()
    pos = rng.integers(0, max_pos, size=n).astype(np.int64)
    theta = 10000.0 ** (-np.arange(32) / 32.0)
    ang = np.arange(max_pos)[:, None] * theta[None, :]
    cs = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    w = rng.uniform(0.5, 2.0, size=128).astype(np.float32)
    eps = 1e-6
    for rec in (REC_MXFP4, REC_FP8_INDEXER):
        rb = 68 if rec == REC_MXFP4 else 132
        cache = np.zeros((n // bs, bs * rb), np.uint8)
        slots = np.arange(n, dtype=np.int64)
        oracle_mod.indexer_k_norm_rope_store(k, pos, cs, w, eps, slots, 1, rec, cache, bs)
        got = oracle_mod.dequantize_and_gather_k_cache(cache, bs, rec, 128, 0,
                                                       slots.astype(np.int32)[None, :])[0]
        got = torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).double().numpy()
        for t in range(n):
            y = xf[t] / np.sqrt(np.mean(xf[t] ** 2) + eps) * w
            c, s = cs[pos[t], :32].astype(np.float64), cs[pos[t], 32:].astype(np.float64)
            e, o = y[64::2].copy(), y[65::2].copy()
            y[64::2], y[65::2] = e * c - o * s, e * s + o * c
            if rec == REC_FP8_INDEXER:
                scale = 2.0 ** np.ceil(np.log2(max(np.abs(y).max() / 448, 1e-10)))
                bound = 16 * scale  # half of the widest e4m3 step (32) below 448
            else:
                amax = np.abs(y.reshape(4, 32)).max(axis=1)
                scale = 2.0 ** np.ceil(np.log2(np.maximum(amax, 1e-4) / 6))
                bound = np.repeat(scale, 32) * 1.0  # half of the widest e2m1 step (2)
            err = np.abs(got[t] - y)
            assert np.all(err <= bound * (1 + 1e-5) + 1e-6 * np.abs(y).max()), (rec, t)
