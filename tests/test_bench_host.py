"""Host-side logic of the benchmark that the roofline figures rest on, with no
GPU: the compulsory-byte accounting, the source hashing that decides whether a
recorded DRAM traffic figure still belongs to the current kernels, and the
reference arm's JSON line (the oracle on the same workload and config)."""
import json
import os
import shutil
from types import SimpleNamespace

import numpy as np

import bench
from oracle.pipeline import run_step
from paged_sparse_kv_gb300 import synthetic


def test_code_only_drops_comments_and_whitespace_only():
    src = "int a = 1; // note\n/* block\n comment */  int  b =\n 2;"
    assert bench._code_only(src) == "int a = 1; int b = 2;"
    assert bench._code_only(src) != bench._code_only(src.replace("2;", "3;"))


def test_recorded_traffic_follows_code_not_comments(tmp_path, monkeypatch):
    csrc = tmp_path / "paged_sparse_kv_gb300" / "csrc"
    shutil.copytree(os.path.join(bench.ROOT, "paged_sparse_kv_gb300", "csrc"), csrc)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    kernel = "dequantize_and_gather_k_cache_topk[topk]"
    h = bench.kernel_source_hash(kernel)
    (tmp_path / "profiles" / "traffic.txt").write_text(f"# header\ndecode {kernel} 12345 {h}\n")
    assert bench.recorded_traffic("decode", kernel) == 12345
    assert bench.recorded_traffic("prefill", kernel) is None
    g = csrc / "gather.cu"
    g.write_text(g.read_text() + "\n// a comment added later\n")
    assert bench.recorded_traffic("decode", kernel) == 12345
    g.write_text(g.read_text() + "\nstatic int psk_unused_symbol_for_the_test = 0;\n")
    assert bench.recorded_traffic("decode", kernel) is None
    assert bench.recorded_traffic("decode", "no_such_kernel") is None


def test_algorithmic_bytes_of_the_tiny_step():
    """Each launch's compulsory bytes, counted entry by entry from the oracle's
    outputs: the inserts (valid rows in and records out, every slot id read),
    the gathers (each distinct valid slot's record once, every index, every
    output row)."""
    w = synthetic.make("tiny")
    caches = {n: synthetic.random_cache_bytes(5 + i, getattr(w, n))
              for i, n in enumerate(("swa_cache", "comp_cache", "index_cache"))}
    out = run_step(w, caches["swa_cache"], caches["comp_cache"], caches["index_cache"])
    got = bench.algorithmic_bytes(SimpleNamespace(w=w),
                                  {"sparse_indices": out["sparse_indices"],
                                   "global_topk": out["global_topk"]})
    D, rope = w.head_dim, w.rope_dim
    fp8_rec = (D - rope) + 2 * rope + D // 64
    valid_rows = sum(1 for s in w.insert_slots.tolist() if s >= 0)
    assert got["quantize_and_insert_k_cache"] == (valid_rows * (2 * D + fp8_rec) +
                                                  8 * len(w.insert_slots))
    W = w.window
    for part, lo, hi in (("swa", 0, W), ("topk", W, out["sparse_indices"].shape[1])):
        entries = [int(v) for row in out["sparse_indices"][:, lo:hi] for v in row]
        distinct = {v for v in entries if v >= 0}
        assert got[f"dequantize_and_gather_k_cache[{part}]"] == (
            len(distinct) * fp8_rec + 4 * len(entries) + 2 * D * len(entries))
    Dx = w.index_head_dim
    entries = [int(v) for row in out["global_topk"] for v in row]
    distinct = {v for v in entries if v >= 0}
    assert got["dequantize_and_gather_k_cache[mxfp4]"] == (
        len(distinct) * (Dx // 2 + Dx // 32) + 4 * len(entries) + 2 * Dx * len(entries))
    # the gathers read at most every index entry's record once
    assert all(v >= 0 for v in got.values())
    assert len(distinct) <= len(entries)


def test_reference_arm_prints_the_same_config(capsys):
    """bench.py --impl reference times the oracle on the same workload and
    prints the same `config` object as the GPU arm builds for it."""
    from paged_sparse_kv_gb300.pipeline import Pipeline
    args = SimpleNamespace(config="tiny", path="auto", steps=1, warmup=1, eager=False)
    bench.run_reference(args, 0, 1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    w = synthetic.make("tiny")
    path = Pipeline.default_path_for(w)
    layout = bench.step_layout(SimpleNamespace(w=w, gather_as_pair=Pipeline.small_batch(w)),
                               path, True)
    assert line["config"] == bench.line_config(bench.workload_description(w), path, w.seed, 1,
                                               layout)
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
