"""Inputs written by the kernel just before a libpsk call on the same stream.

Every libpsk kernel is launched with programmatic dependent launch and may
start while its predecessor on the stream is finishing.  The library's
contract is that no kernel reads global memory before the predecessor's grid
has completed, so an input written by an ordinary (non-PDL) torch kernel right
before the call is always seen.  This test alternates two versions of every
metadata input (top-k rows, block tables, sequence lengths, positions), each
written by a torch elementwise kernel immediately before the entry point that
reads it, eagerly and inside a CUDA graph, and requires every output to equal
the one computed with a full synchronisation in between.
"""
import pytest
import torch

from paged_sparse_kv_gb300 import ops, synthetic
from paged_sparse_kv_gb300.pipeline import Pipeline

pytestmark = pytest.mark.gpu


def _write(dst: torch.Tensor, src: torch.Tensor) -> None:
    """dst <- src by an elementwise torch kernel (not a copy-engine transfer)."""
    torch.add(src, 0, out=dst)


class _Case:
    """The decode batch with two versions of its metadata on the device."""

    def __init__(self, dev):
        w = synthetic.make("decode")
        p = Pipeline(w, dev)
        p.fill_caches_with_quantized_rows(seed=5)
        self.w, self.p = w, p
        W, K = w.window, w.topk
        T = w.num_tokens
        # version 1: rows and tables rolled by one request, contexts 3 shorter
        v0 = {"topk": p.topk.clone(), "swa_bt": p.swa_bt.clone(), "comp_bt": p.comp_bt.clone(),
              "seq_lens": p.seq_lens.clone()}
        v1 = {"topk": torch.roll(p.topk, 1, 0), "swa_bt": torch.roll(p.swa_bt, 1, 0),
              "comp_bt": torch.roll(p.comp_bt, 1, 0), "seq_lens": p.seq_lens - 3}
        for v in (v0, v1):
            v["positions"] = (v["seq_lens"] - 1).to(torch.int64)
        self.versions = (v0, v1)
        # live inputs (overwritten before every call) and outputs
        self.inp = {k: t.clone() for k, t in v0.items()}
        self.dense_w = 64
        self.out = {
            "gt": torch.empty((T, K), dtype=torch.int32, device=dev),
            "gt_lens": torch.empty((T,), dtype=torch.int32, device=dev),
            "si": torch.empty((T, W + w.padded_topk), dtype=torch.int32, device=dev),
            "si_lens": torch.empty((T,), dtype=torch.int32, device=dev),
            "swa": torch.empty((T, W), dtype=torch.int32, device=dev),
            "swa_lens": torch.empty((T,), dtype=torch.int32, device=dev),
            "g_topk": torch.empty((T, K, w.head_dim), dtype=torch.bfloat16, device=dev),
            "g_mx": torch.empty((T, K, w.index_head_dim), dtype=torch.bfloat16, device=dev),
            "g_win": torch.empty((T, W, w.head_dim), dtype=torch.bfloat16, device=dev),
            "g_dense": torch.empty((T, self.dense_w, w.head_dim), dtype=torch.bfloat16,
                                   device=dev),
            "g_rng": torch.zeros((w.num_reqs, W, w.head_dim), dtype=torch.bfloat16, device=dev),
        }

    def calls(self):
        """(input names written first, launch) for every entry point that reads metadata."""
        w, p, i, o = self.w, self.p, self.inp, self.out
        bs = w.swa_cache.block_size
        cbs = w.comp_cache.block_size
        W = w.window
        return [
            (("topk", "comp_bt"), lambda: ops.compute_global_topk_indices_and_lens(
                i["topk"], p.t2r, i["comp_bt"], w.index_cache.block_size, out=o["gt"],
                lens=o["gt_lens"])),
            (("topk", "swa_bt", "comp_bt", "seq_lens"), lambda: ops.combine_topk_swa_indices(
                p.qsl, i["seq_lens"], p.t2r, p.replay, i["swa_bt"], bs, i["comp_bt"], cbs, W,
                w.compress_ratio, i["topk"], out=o["si"], lens=o["si_lens"])),
            (("swa_bt", "seq_lens"), lambda: ops.decode_swa_indices_and_lens(
                p.qsl, i["seq_lens"], p.t2r, i["swa_bt"], bs, W, out=o["swa"],
                lens=o["swa_lens"])),
            (("topk", "comp_bt"), lambda: ops.dequantize_and_gather_k_cache_topk(
                o["g_topk"], p.comp_cache, i["topk"], p.t2r, i["comp_bt"], cbs,
                rope_dim=w.rope_dim, num_reqs=w.num_reqs)),
            (("topk", "comp_bt"), lambda: ops.dequantize_and_gather_k_cache_topk(
                o["g_mx"], p.index_cache, i["topk"], p.t2r, i["comp_bt"],
                w.index_cache.block_size, record=ops.PSK_REC_MXFP4, num_reqs=w.num_reqs)),
            (("swa_bt", "seq_lens"), lambda: ops.dequantize_and_gather_k_cache_window(
                o["g_win"], p.swa_cache, p.qsl, i["seq_lens"], p.t2r, p.replay, i["swa_bt"], bs,
                W, rope_dim=w.rope_dim)),
            (("positions", "comp_bt"), lambda: ops.dequantize_and_gather_k_cache_dense(
                o["g_dense"], p.comp_cache, i["positions"], p.t2r, i["comp_bt"], cbs,
                w.compress_ratio, rope_dim=w.rope_dim, num_reqs=w.num_reqs)),
            (("seq_lens", "swa_bt"), lambda: ops.dequantize_and_gather_k_cache_ranges(
                o["g_rng"], p.swa_cache, i["seq_lens"], None, i["swa_bt"], bs, 0,
                rope_dim=w.rope_dim)),
        ]

    def run(self, version: int, counters: torch.Tensor, expected=None, sync=False):
        """Every call with its inputs written just before it; with ``expected``,
        count mismatching elements of each output into ``counters``."""
        src = self.versions[version]
        outs = list(self.out.values())
        for names, launch in self.calls():
            for n in names:
                _write(self.inp[n], src[n])
            if sync:
                torch.cuda.synchronize()
            launch()
            if sync:
                torch.cuda.synchronize()
        if expected is not None:
            for k, (o, e) in enumerate(zip(outs, expected[version])):
                counters[k] += (o.view(torch.int16) if o.dtype == torch.bfloat16 else o).ne(
                    e.view(torch.int16) if e.dtype == torch.bfloat16 else e).sum()


@pytest.mark.parametrize("graph", [False, True])
def test_metadata_written_just_before_each_call(cuda_device, graph):
    case = _Case(cuda_device)
    nout = len(case.out)
    counters = torch.zeros(nout, dtype=torch.int64, device=cuda_device)
    expected = []
    for v in (0, 1):
        for o in case.out.values():
            o.zero_()
        case.run(v, counters, sync=True)
        expected.append([o.clone() for o in case.out.values()])
    # the two versions differ in every index matrix and gathered output, so a
    # stale read would show (lens may coincide)
    for k, name in enumerate(case.out):
        if not name.endswith("_lens"):
            assert not torch.equal(expected[0][k], expected[1][k]), name
    if not graph:
        for it in range(40):
            case.run(it % 2, counters, expected)
    else:
        s = torch.cuda.Stream(cuda_device)
        s.wait_stream(torch.cuda.current_stream(cuda_device))
        with torch.cuda.stream(s):
            case.run(0, counters, expected)
        torch.cuda.current_stream(cuda_device).wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for it in range(6):
                case.run(it % 2, counters, expected)
        for _ in range(8):
            g.replay()
    torch.cuda.synchronize()
    bad = counters.cpu().tolist()
    assert all(b == 0 for b in bad), dict(zip(case.out, bad))
