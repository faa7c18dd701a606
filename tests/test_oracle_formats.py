"""Pins for the oracle's scalar formats (E4M3, E2M1, UE8M0 exponent, bf16).

Each check compares the oracle against something other than itself: values
worked by hand from the OCP format definitions (tests/golden), the library
casts of torch (float8_e4m3fn, bfloat16), or a brute-force nearest-value
search written here from the E2M1 element table.
"""
import math
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append(parts)
    return rows


def _all_finite_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    return f[np.isfinite(f)]


def test_e4m3_golden(oracle_mod):
    rows = _golden_rows("e4m3_codes.txt")
    assert len(rows) >= 15
    vals = np.array([float(r[0]) for r in rows], dtype=np.float32)
    # -0.0 must survive float parsing
    for i, r in enumerate(rows):
        if r[0].startswith("-0.0") and float(r[0]) == 0.0:
            vals[i] = np.float32(-0.0)
    got = oracle_mod.e4m3_encode(vals)
    want = np.array([int(r[1], 16) for r in rows], dtype=np.uint8)
    bad = [(rows[i][0], hex(got[i]), rows[i][1]) for i in np.nonzero(got != want)[0]]
    assert not bad, bad


def test_e4m3_decode_matches_torch_for_every_code(oracle_mod):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([oracle_mod.e4m3_decode(c) for c in range(256)], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert nan.sum() == 2  # 0x7f and 0xff


def test_e4m3_encode_exhaustive_scaled_bf16_vs_torch(oracle_mod):
    """Every value the UE8M0 insert can hand the encoder: each finite bf16 x
    scaled by 2^-e for every exponent a bf16 block can produce (e in
    [-22, 120]) and clamped to +-448, encoded by the oracle and by torch's
    float8_e4m3fn cast (RNE)."""
    x = _all_finite_bf16().astype(np.float32)
    mism = 0
    total = 0
    for e in range(-22, 121):
        with np.errstate(over="ignore"):
            v = (x * np.float32(2.0 ** -e)).astype(np.float32)
        v = np.clip(v, np.float32(-448.0), np.float32(448.0))
        got = oracle_mod.e4m3_encode(v)
        ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        mism += int((got != ref).sum())
        total += v.size
    assert total > 9_000_000
    assert mism == 0


def test_e4m3_encode_random_binary32_vs_torch(oracle_mod):
    """Arbitrary binary32 inputs within +-448 (the fp32-scale record divides
    by an arbitrary scale, so any binary32 can reach the encoder)."""
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 32, size=4_000_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    v = np.clip(v, np.float32(-448.0), np.float32(448.0))
    # add values near every rounding boundary: midpoints between codes
    codes = np.arange(0, 0x7F, dtype=np.int32).astype(np.uint8)
    grid = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(1000))])
    v = np.concatenate([v, near, -near]).astype(np.float32)
    got = oracle_mod.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_bruteforce(v: np.ndarray) -> np.ndarray:
    """Nearest of the 8 magnitudes, ties to the even code, saturating at 6,
    sign bit from the input's sign (an independent restatement of the MX
    element table)."""
    a = np.abs(v.astype(np.float64))
    d = np.abs(a[:, None] - E2M1_MAG[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among tied candidates prefer the even code index
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    pick_even = even.any(axis=1)
    code = np.where(pick_even, np.argmax(even, axis=1), np.argmax(cand, axis=1))
    code = np.where(a >= 6.0, 7, code)
    sign = np.signbit(v).astype(np.int64) << 3
    return (code | sign).astype(np.uint8)


def test_e2m1_golden(oracle_mod):
    rows = _golden_rows("e2m1_codes.txt")
    vals = np.array([float(r[0]) for r in rows], dtype=np.float32)
    for i, r in enumerate(rows):
        if r[0] == "-0.0":
            vals[i] = np.float32(-0.0)
    got = oracle_mod.e2m1_encode(vals)
    want = np.array([int(r[1], 16) for r in rows], dtype=np.uint8)
    assert np.array_equal(got, want), list(zip(vals, got, want))


def test_e2m1_encode_exhaustive_scaled_bf16_vs_bruteforce(oracle_mod):
    """Every value the MXFP4 insert can hand the encoder: finite bf16 times
    2^-e for every reachable exponent (e in [-15, 126])."""
    x = _all_finite_bf16().astype(np.float32)
    for e in range(-15, 127, 3):
        with np.errstate(over="ignore"):
            v = (x * np.float32(2.0 ** -e)).astype(np.float32)
        got = oracle_mod.e2m1_encode(v)
        ref = _e2m1_bruteforce(v)
        assert np.array_equal(got, ref), e


def test_e2m1_decode_table(oracle_mod):
    for code in range(16):
        mag = E2M1_MAG[code & 7]
        want = np.float32(-mag if code & 8 else mag)
        got = np.float32(oracle_mod.e2m1_decode(code))
        assert got.view(np.uint32) == want.view(np.uint32), code


def test_ceil_log2_definition(oracle_mod):
    """Smallest e with 2^e >= q, checked with exact double arithmetic on
    powers of two, their float neighbours and random positive floats."""
    rng = np.random.default_rng(3)
    pw = np.array([2.0 ** k for k in range(-149, 128)], dtype=np.float32)
    qs = np.concatenate([
        pw, np.nextafter(pw, np.float32(np.inf)), np.nextafter(pw, np.float32(0)),
        rng.integers(1, 0x7F800000, size=200_000, dtype=np.int64).astype(np.uint32).view(np.float32),
    ])
    qs = qs[(qs > 0) & np.isfinite(qs)]
    e = oracle_mod.ceil_log2(qs)
    q64 = qs.astype(np.float64)
    upper = np.ldexp(1.0, e)
    lower = np.ldexp(1.0, e - 1)
    assert np.all(upper >= q64)
    assert np.all(lower < q64)


def test_ue8m0_scale_golden(oracle_mod):
    """Scale bytes of a 64-block with a given amax, through the full insert."""
    rows = _golden_rows("ue8m0_scales.txt")
    for r in rows:
        amax, want_byte, want_code = float(r[0]), int(r[1]), int(r[2], 16)
        blk = np.zeros(64, dtype=np.float32)
        blk[5] = amax
        bits = torch.from_numpy(blk).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        k = bits.reshape(1, 64)
        cache = np.zeros((1, 80), dtype=np.uint8)  # bs 1: 64 data bytes + 1 scale
        err = oracle_mod.quantize_and_insert_k_cache(k, np.array([0], np.int64), cache,
                                                     block_size=1, head_dim=64, rope_dim=0)
        assert err == 0
        assert cache[0, 64] == want_byte, (amax, cache[0, 64], want_byte)
        assert cache[0, 5] == want_code, (amax, hex(cache[0, 5]), hex(want_code))


def test_bf16_rounding_vs_torch(oracle_mod):
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 1 << 32, size=300_000, dtype=np.uint64).astype(np.uint32)
    # ties: low 16 bits exactly 0x8000, with even and odd kept parts
    ties = (rng.integers(0, 1 << 16, size=20_000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    v = np.concatenate([bits, ties]).view(np.float32)
    v = v[np.isfinite(v)]
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    lib = oracle_mod._load()
    got = np.array([lib.oracle_bf16_from_f32(float(x)) for x in v[:20000]], dtype=np.uint16)
    assert np.array_equal(got, ref[:20000])
    got_t = np.array([lib.oracle_bf16_from_f32(float(x)) for x in v[-20000:]], dtype=np.uint16)
    assert np.array_equal(got_t, ref[-20000:])
