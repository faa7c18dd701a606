"""Every gathered row of a large batch against the oracle.

The mixed batch (256 decode tokens and two 2048-token prefill requests,
window 128, top-k 1024) runs its whole step the way the benchmark launches it
-- a CUDA graph of the concurrent step -- and every one of its 4352 x 1152
gathered fp8_ds_mla rows (the window columns from the SWA cache, the top-k
columns from the compressed cache) and 4352 x 1024 gathered MXFP4 rows is
compared bit for bit with the oracle's rows for the same indices: TokenSpeed
deepseek_v4_ops.py, dequantize_deepseek_v4_fp8_ds_mla_cache and
read_deepseek_v4_indexer_mxfp4_cache; vLLM deepseek_v41 ops,
dequantize_and_gather_k_cache.  The device rows are copied to the host one
chunk of tokens at a time and the oracle gathers the same chunk from the
oracle's own index matrices, several chunks in parallel (the oracle's C calls
release the interpreter lock).  About 20 s on a 16-core host.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from oracle.pipeline import run_step
from paged_sparse_kv_gb300 import synthetic
from paged_sparse_kv_gb300.pipeline import Pipeline

pytestmark = pytest.mark.gpu

CHUNK = 128  # tokens per host chunk (151 MB of fp8_ds_mla rows)


def _u16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _first_mismatch(got: np.ndarray, want: np.ndarray):
    bad = np.nonzero(got.reshape(-1) != want.reshape(-1))[0]
    return None if bad.size == 0 else (int(bad.size), int(bad[0]))


def test_mixed_step_every_gathered_row(cuda_device):
    w = synthetic.make("mixed")
    host = {}
    for i, cname in enumerate(("swa_cache", "comp_cache", "index_cache")):
        g = getattr(w, cname)
        host[cname] = None if g is None else synthetic.random_cache_bytes(60 + i, g)
    p = Pipeline(w, cuda_device)
    for cname, arr in host.items():
        getattr(p, cname).copy_(torch.from_numpy(arr))
    side = torch.cuda.Stream(cuda_device)
    side.wait_stream(torch.cuda.current_stream(cuda_device))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        p.step(concurrent=True, path="index")
    graph.replay()
    torch.cuda.synchronize()

    # the oracle's step: inserts, index matrices and lens in full (its gathers
    # on one token only; the full gathers follow chunk by chunk)
    ref = run_step(w, host["swa_cache"], host["comp_cache"], host["index_cache"], [0])
    for cname, arr in host.items():
        assert np.array_equal(getattr(p, cname).cpu().numpy(), arr), cname
    si, gt = ref["sparse_indices"], ref["global_topk"]
    assert np.array_equal(p.sparse_indices.cpu().numpy(), si)
    assert np.array_equal(p.lens.cpu().numpy(), ref["lens"])
    assert np.array_equal(p.global_topk.cpu().numpy(), gt)
    assert np.array_equal(p.global_lens.cpu().numpy(), ref["global_lens"])
    assert int(p.err.item()) == ref["err"] == 0

    W, D, Di = w.window, w.head_dim, w.index_head_dim
    T = w.num_tokens
    assert si.shape == (4352, W + w.padded_topk) == (4352, 1152)

    def check(t0: int):
        t1 = min(t0 + CHUNK, T)
        got = _u16(p.gathered[t0:t1])
        rows = si[t0:t1]
        want = oracle.dequantize_and_gather_k_cache(host["swa_cache"], w.swa_cache.block_size,
                                                    oracle.REC_FP8_DS_MLA, D, w.rope_dim,
                                                    np.ascontiguousarray(rows[:, :W]))
        bad = _first_mismatch(got[:, :W], want)
        if bad:
            return ("window", t0, bad)
        want = oracle.dequantize_and_gather_k_cache(host["comp_cache"], w.comp_cache.block_size,
                                                    oracle.REC_FP8_DS_MLA, D, w.rope_dim,
                                                    np.ascontiguousarray(rows[:, W:]))
        bad = _first_mismatch(got[:, W:], want)
        if bad:
            return ("top-k", t0, bad)
        got = _u16(p.gathered_index[t0:t1])
        want = oracle.dequantize_and_gather_k_cache(host["index_cache"],
                                                    w.index_cache.block_size, oracle.REC_MXFP4,
                                                    Di, 0, np.ascontiguousarray(gt[t0:t1]))
        bad = _first_mismatch(got, want)
        if bad:
            return ("mxfp4", t0, bad)
        return None

    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(check, range(0, T, CHUNK)))
    failures = [r for r in results if r is not None]
    assert not failures, failures[:5]
    # every chunk covered, and the batch holds both zero rows and real rows
    assert len(results) == (T + CHUNK - 1) // CHUNK
    assert np.any(si[:, :W] < 0) and np.any(si[:, W:] >= 0)
    del p
    torch.cuda.empty_cache()
