"""Pins for the oracle's compressed-KV producer: its binary32 exp, the
compressor-state writer and the window-pooling insert.

* exp: against the C library's exp (binary64, rounded to binary32) within 2 ulp
  over a dense sweep of [-104, 88], with exp(0) = 1 and exp(x) = 0 below the
  subnormal range.
* save_compressor_state: the row it writes is [kv, score + ape[pos % ratio]].
* compress_kv_cache_insert against closed forms: equal scores pool to the mean
  (weights exactly 1 / window for the power-of-two windows), a constant row
  normalises to exactly 1, the overlap window takes the first kv slice from the
  older positions and the second from the newer ones, a dominant score selects
  its row, absent pages drop out, and the emission rule / counted skips.
* The RMSNorm reading (binary32 square root, then a binary32 division) on a
  pooled row whose factor differs in the last bit from a correctly rounded
  reciprocal square root, with a weight that turns that bit into a bf16 code.
  Expected records are built through the FP8 insert of a hand-written bf16
  row (the insert is pinned on its own).
"""
import numpy as np
import pytest
import torch

D, R64 = 512, 64


def _ulp_err(got, want):
    gi = got.view(np.int32).astype(np.int64)
    wi = want.view(np.int32).astype(np.int64)
    return np.abs(gi - wi)


def test_exp_against_libm(oracle_mod):
    x = np.concatenate([np.linspace(-104, 88.7, 2_000_003, dtype=np.float32),
                        -np.abs(np.random.default_rng(0).standard_normal(200000)).astype(np.float32) * 30,
                        np.float32([0.0, -0.0, -1e-30, -1e-7, -0.3465, 0.3466])])
    got = oracle_mod.exp_cw(x)
    want = np.exp(x.astype(np.float64)).astype(np.float32)
    fin = np.isfinite(want) & (want > 0)
    assert _ulp_err(got[fin], want[fin]).max() <= 2
    assert oracle_mod.exp_cw(np.float32([0.0]))[0] == 1.0
    assert np.all(oracle_mod.exp_cw(np.float32([-104.5, -1e30, -np.inf])) == 0.0)
    assert np.isnan(oracle_mod.exp_cw(np.float32([np.nan]))[0])


def test_save_compressor_state(oracle_mod):
    rng = np.random.default_rng(1)
    sw, bs, ratio = 16, 4, 4
    kv = rng.standard_normal((6, sw)).astype(np.float32)
    score = rng.standard_normal((6, sw)).astype(np.float32)
    ape = rng.standard_normal((ratio, sw)).astype(np.float32)
    pos = np.array([0, 5, 6, 7, -3, 9], np.int64)
    slots = np.array([3, 0, -1, 7, 5, 99], np.int64)
    st = np.full((2, bs, 2 * sw), 7.0, np.float32)
    n = oracle_mod.save_compressor_state(kv, score, ape, slots, pos, ratio, st, bs)
    assert n == 1  # slot 99 beyond the 8-slot cache
    flat = st.reshape(-1, 2 * sw)
    for t, s in enumerate(slots):
        if s < 0 or s >= 8:
            continue
        a = int(pos[t]) % ratio
        assert np.array_equal(flat[s, :sw], kv[t])
        assert np.array_equal(flat[s, sw:], score[t] + ape[a])
    assert np.all(flat[[1, 2, 4, 6]] == 7.0)  # untouched rows


def _record(oracle_mod, row_f32, rope_rot):
    """Expected fp8_ds_mla record of one key: bf16 of the nope values and of the
    rotated rope tail, through the (separately pinned) FP8 insert."""
    row = np.concatenate([row_f32[:D - R64], rope_rot]).astype(np.float32)
    bf = torch.from_numpy(row).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    cache = np.zeros((1, 584), np.uint8)
    oracle_mod.quantize_and_insert_k_cache(bf[None, :], np.array([0], np.int64), cache, 1, D, R64)
    return cache[0]


def _cos_sin(max_pos, turn_rows=()):
    cs = np.zeros((max_pos, 64), np.float32)
    cs[:, :32] = 1.0
    for p in turn_rows:
        cs[p, :32], cs[p, 32:] = 0.0, 1.0
    return cs


def _setup(ratio, overlap, pos, sw, fill):
    """One request whose state rows for positions 0..pos sit at state slot
    p (identity table, page 8); fill(p) gives the [kv | score] row."""
    bs = 8
    npages = (pos + bs) // bs + 1
    st = np.zeros((npages, bs, 2 * sw), np.float32)
    for p in range(pos + 1):
        st[p // bs, p % bs] = fill(p)
    table = np.arange(npages, dtype=np.int32)[None, :]
    return st, table, bs


@pytest.mark.parametrize("ratio,overlap", [(4, True), (128, False)])
def test_compress_constant_rows(oracle_mod, ratio, overlap):
    """kv = 2 everywhere, equal scores: weights 1 / window (exact), the pooled
    row is 2, RMSNorm makes it 1 (weight 1, eps 0); RoPE at a 90-degree row
    turns each tail pair (1, 1) into (-1, 1)."""
    sw = (2 if overlap else 1) * D
    pos = 2 * ratio - 1 if overlap else ratio - 1
    st, table, bs = _setup(ratio, overlap, pos, sw,
                           lambda p: np.concatenate([np.full(sw, 2.0), np.zeros(sw)]))
    prow = (pos // ratio) * ratio
    kv_cache = np.zeros((1, 584), np.uint8)
    n = oracle_mod.compress_kv_cache_insert(
        st, np.array([0], np.int32), np.array([pos], np.int64), np.array([pos], np.int64), table,
        bs, np.ones(D, np.float32), 0.0, _cos_sin(pos + 1, [prow]), kv_cache,
        np.array([0], np.int64), 1, ratio, overlap)
    assert n == 0
    want = _record(oracle_mod, np.ones(D, np.float32), np.tile([-1.0, 1.0], 32))
    assert kv_cache[0].tolist() == want.tolist()


def test_compress_overlap_slices(oracle_mod):
    """CSA window of 8: the older four positions contribute their first kv
    slice (value 1), the newer four their second (value 3); equal scores
    give (4 * 1 + 4 * 3) / 8 = 2 per column, which normalises to 1."""
    sw = 2 * D
    pos = 11  # window 4..11
    st, table, bs = _setup(4, True, pos, sw, lambda p: np.concatenate(
        [np.full(D, 1.0), np.full(D, 3.0), np.zeros(sw)]))
    kv_cache = np.zeros((1, 584), np.uint8)
    oracle_mod.compress_kv_cache_insert(
        st, np.array([0], np.int32), np.array([pos], np.int64), np.array([pos], np.int64), table,
        bs, np.full(D, 0.5, np.float32), 0.0, _cos_sin(16), kv_cache, np.array([0], np.int64),
        1, 4, True)
    # weight 0.5 on every column: the pooled row 2 -> 1 -> 0.5; identity RoPE
    want = _record(oracle_mod, np.full(D, 0.5, np.float32), np.full(R64, 0.5, np.float32))
    assert kv_cache[0].tolist() == want.tolist()


def test_compress_dominant_score_and_absent_pages(oracle_mod):
    """HCA window 0..127 at pos 127: page 1 of the table is absent (positions
    8..15 drop out); position 40 has score 120 and kv row v; every other
    present position has score 0 and kv 9.  exp(-120) underflows to 0, so the
    pooled row is exactly v."""
    sw = D
    pos = 127
    rng = np.random.default_rng(5)
    v = np.where(rng.random(D) < 0.5, 1.0, -2.0).astype(np.float32)

    def fill(p):
        if p == 40:
            return np.concatenate([v, np.full(sw, 120.0)])
        return np.concatenate([np.full(sw, 9.0), np.zeros(sw)])
    st, table, bs = _setup(128, False, pos, sw, fill)
    table = table.copy()
    table[0, 1] = -1
    kv_cache = np.zeros((1, 584), np.uint8)
    oracle_mod.compress_kv_cache_insert(
        st, np.array([0], np.int32), np.array([pos], np.int64), np.array([pos], np.int64), table,
        bs, np.ones(D, np.float32), 0.0, _cos_sin(128), kv_cache, np.array([0], np.int64), 1, 128,
        False)
    # squares are 1 or 4, so every summation order gives the same exact sum
    r = np.float32(1.0) / np.sqrt(np.float32(np.float32((v * v).sum()) / np.float32(D)))
    y = (v * r).astype(np.float32)
    want = _record(oracle_mod, y, y[D - R64:])
    assert kv_cache[0].tolist() == want.tolist()


def test_compress_rsqrt_reading(oracle_mod):
    """The pooled row's RMSNorm factor is RN(1 / RN(sqrt(v + eps))), not a
    correctly rounded reciprocal square root.  HCA window 0..127, equal scores
    (weights 1/128, exact), every row c = (3, 3, 3, 3, 1, ..., 1): the pooled row
    is c exactly, its sum of squares 544, v = 1.0625, eps = 2^-7, v + eps =
    137/128.  The binary32 reading gives r = 0x3F7772CA, one rounded step gives
    0x3F7772CB.  Weight 0x3F8006D5 on the first RoPE dim (identity row) makes
    RN(r * w) = 0x3F777FFF under the first, which rounds to the bfloat16
    0x3F77, and exactly the bfloat16 midpoint 0x3F778000 under the second,
    whose tie goes to the even 0x3F78."""
    rA, rB = (np.array([b], np.uint32).view(np.float32)[0] for b in (0x3F7772CA, 0x3F7772CB))
    w_t = np.array([0x3F8006D5], np.uint32).view(np.float32)[0]
    assert np.float32(1.0) / np.sqrt(np.float32(137.0 / 128.0)) == rA
    assert np.float32(1.0 / np.sqrt(137.0 / 128.0)) == rB
    c = np.ones(D, np.float32)
    c[:4] = 3.0
    w = np.ones(D, np.float32)
    w[D - R64] = w_t
    st, table, bs = _setup(128, False, 127, D, lambda p: np.concatenate([c, np.zeros(D)]))
    kv_cache = np.zeros((1, 584), np.uint8)
    n = oracle_mod.compress_kv_cache_insert(
        st, np.array([0], np.int32), np.array([127], np.int64), np.array([127], np.int64),
        table, bs, w, 2.0 ** -7, _cos_sin(128), kv_cache, np.array([0], np.int64), 1, 128,
        False)
    assert n == 0
    rope = kv_cache[0, D - R64:D + R64].view(np.uint16)  # bf16 tail after the 448 FP8 bytes
    assert rope[0] == 0x3F77  # 0x3F78 under a correctly rounded rsqrt
    records = {}
    for tag, r in (("binary32", rA), ("rounded once", rB)):
        y = ((c * r).astype(np.float32) * w).astype(np.float32)
        records[tag] = _record(oracle_mod, y, y[D - R64:])
    assert kv_cache[0].tolist() == records["binary32"].tolist()
    assert records["binary32"].tolist() != records["rounded once"].tolist()


def test_compress_emission_and_skips(oracle_mod):
    """Ratio 4: tokens at positions 3 and 7 close groups; 5 does not; a kv slot
    of -1 skips; a kv slot beyond the cache and a RoPE row beyond max_pos are
    counted."""
    sw = 2 * D
    st, table, bs = _setup(4, True, 15, sw, lambda p: np.concatenate(
        [np.full(sw, 1.0 + p), np.zeros(sw)]))
    kv_cache = np.full((1, 4 * 584), 0xAB, np.uint8)
    pos = np.array([3, 5, 7, 11, 15, 7], np.int64)
    kv_slots = np.array([0, 1, -1, 9, 2, 3], np.int64)
    n = oracle_mod.compress_kv_cache_insert(
        st, np.zeros(6, np.int32), pos, pos, table, bs, np.ones(D, np.float32), 1e-6,
        _cos_sin(12), kv_cache, kv_slots, 4, 4, True)
    assert n == 2  # slot 9 beyond 4 slots; position 15's RoPE row 12 beyond max_pos 12
    rec = kv_cache.reshape(-1)
    data = lambda s: rec[s * 576:(s + 1) * 576]
    assert not np.all(data(0) == 0xAB) and not np.all(data(3) == 0xAB)
    assert np.all(data(1) == 0xAB) and np.all(data(2) == 0xAB)
