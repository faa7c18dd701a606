"""GPU parity on caches larger than 4 GiB: the inserts and the gathers address
records past byte offset 2^32 (the small-record gather switches to 64-bit
offsets there), byte for byte against the CPU oracle.

Each cache is ~4.6 GiB on the device; the oracle's copy is a zero-filled host
array of the same shape whose pages are touched only where records are
written or read."""
import numpy as np
import pytest
import torch

import oracle
from paged_sparse_kv_gb300 import ops
from test_parity_gpu import _assert_same, _bf16_dev

pytestmark = pytest.mark.gpu

BS = 64
TARGET_BYTES = (9 << 30) // 2  # 4.5 GiB


def _slots(rng, capacity, stride, n=2048):
    """n distinct slots: half anywhere, half on pages that start past byte 2^32,
    and the first and last slots of the cache."""
    first_high = (-(-(1 << 32) // stride) + 1) * BS
    lo = rng.choice(capacity, size=n // 2, replace=False)
    hi = first_high + rng.choice(capacity - first_high, size=n // 2, replace=False)
    s = np.unique(np.concatenate([lo, hi, [0, capacity - 1]]))
    rng.shuffle(s)
    return s.astype(np.int64)


def _compare_pages(dev_cache, host, slots, what):
    pages = np.unique(slots // BS)
    got = dev_cache[torch.from_numpy(pages).to(dev_cache.device)].cpu().numpy()
    _assert_same(got, host[pages], what)
    # a page no slot maps to stays zero on the device
    untouched = np.setdiff1d(np.arange(0, dev_cache.shape[0], 4099), pages)[:64]
    assert not dev_cache[torch.from_numpy(untouched).to(dev_cache.device)].any().item()


@pytest.mark.parametrize("kind", ["fp8_ds_mla", "mxfp4", "fp8_indexer"])
def test_cache_past_4_gib(cuda_device, kind):
    d = cuda_device
    rng = np.random.default_rng({"fp8_ds_mla": 1, "mxfp4": 2, "fp8_indexer": 3}[kind])
    if kind == "fp8_ds_mla":
        D, rope = 512, 64
        rec = oracle.fp8_record_bytes(D, rope)
    elif kind == "mxfp4":
        D, rope = 128, 0
        rec = oracle.mxfp4_record_bytes(D)
    else:
        D, rope = 128, 0
        rec = oracle.fp8_indexer_record_bytes(D)
    stride = BS * rec
    assert stride % 16 == 0
    pages = -(-TARGET_BYTES // stride)
    capacity = pages * BS
    assert capacity < 1 << 31 and pages * stride > 1 << 32
    slots = _slots(rng, capacity, stride)
    assert (slots // BS * stride > 1 << 32).sum() >= 1024
    n = slots.shape[0]
    x = (rng.standard_normal((n, D)) * np.exp(rng.uniform(-4, 4, size=(n, 1)))).astype(np.float32)
    k = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    dev_cache = torch.zeros((pages, stride), dtype=torch.uint8, device=d)
    host = np.zeros((pages, stride), np.uint8)  # lazily backed: only written pages are touched
    err = torch.zeros(1, dtype=torch.int32, device=d)
    kd, sd = _bf16_dev(k, d), torch.from_numpy(slots).to(d)
    if kind == "fp8_ds_mla":
        ops.quantize_and_insert_k_cache(kd, dev_cache, sd, BS, rope_dim=rope, err_count=err)
        n_err = oracle.quantize_and_insert_k_cache(k, slots, host, BS, D, rope)
        record = ops.PSK_REC_FP8_DS_MLA
    elif kind == "mxfp4":
        ops.write_indexer_mxfp4_cache(kd, dev_cache, sd, BS, err_count=err)
        n_err = oracle.write_indexer_mxfp4_cache(k, slots, host, BS, D)
        record = ops.PSK_REC_MXFP4
    else:
        ops.write_indexer_fp8_cache(kd, dev_cache, sd, BS, err_count=err)
        n_err = oracle.write_indexer_fp8_cache(k, slots, host, BS, D)
        record = ops.PSK_REC_FP8_INDEXER
    assert int(err.item()) == n_err == 0
    _compare_pages(dev_cache, host, slots, f"{kind} insert past 4 GiB")

    # gather every inserted slot plus -1 entries and slots nothing was written to
    idx = np.concatenate([slots, -np.ones(40, np.int64), rng.integers(0, capacity, size=88)])
    rng.shuffle(idx)
    idx = idx[: idx.shape[0] // 64 * 64].astype(np.int32).reshape(-1, 64)
    out = torch.empty((idx.shape[0], 64, D), dtype=torch.bfloat16, device=d)
    ops.dequantize_and_gather_k_cache(out, dev_cache, torch.from_numpy(idx).to(d), BS,
                                      record=record, rope_dim=rope)
    want = oracle.dequantize_and_gather_k_cache(host, BS, int(record), D, rope, idx)
    _assert_same(out.view(torch.int16).cpu().numpy().view(np.uint16), want,
                 f"{kind} gather past 4 GiB")

    # the fused top-k form: local indices through block tables whose pages are
    # the written pages (most of them past byte 2^32) and a few missing pages
    R, width, K = 8, 64, 256
    written = np.unique(slots // BS)
    table = rng.choice(written, size=(R, width)).astype(np.int32)
    table[rng.random(table.shape) < 0.03] = -1
    t2r = np.repeat(np.arange(R, dtype=np.int32), 2)
    topk = rng.integers(-1, width * BS, size=(t2r.shape[0], K)).astype(np.int32)
    out = torch.empty((t2r.shape[0], K, D), dtype=torch.bfloat16, device=d)
    ops.dequantize_and_gather_k_cache_topk(out, dev_cache, torch.from_numpy(topk).to(d),
                                           torch.from_numpy(t2r).to(d),
                                           torch.from_numpy(table).to(d), BS, record=record,
                                           rope_dim=rope, num_reqs=R)
    gslots, _ = oracle.compute_global_topk_indices_and_lens(topk, t2r, table, BS)
    assert (gslots.astype(np.int64) // BS * stride > 1 << 32).sum() > K
    want = oracle.dequantize_and_gather_k_cache(host, BS, int(record), D, rope, gslots)
    _assert_same(out.view(torch.int16).cpu().numpy().view(np.uint16), want,
                 f"{kind} fused top-k gather past 4 GiB")
