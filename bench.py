"""Benchmark of the paged K-cache pipeline on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config prefill]
                    [--configs tiny,decode,mixed,mxfp4] [--path auto]
                    [--impl mine|reference] [--no-cpu-baseline]

A step is one pass of every hot-path row over one synthetic batch (see
paged_sparse_kv_gb300/pipeline.py): FP8 insert, MXFP4 insert, fused window +
top-k index build, the dequantize-and-gather of the window and top-k columns,
the global top-k mapping and the MXFP4 gather.  The headline workload is the
prefill chunk, the largest single-GPU configuration: 4 requests x 4096 new
tokens, head_dim 512 = 448 fp8 + 64 bf16 rope, page 64, window 128, top-k 512
-> sparse_indices [16384, 640] and a [16384, 640, 512] bf16 gather.  It runs
the index path (build, then gathers keyed by the index matrix) on three
streams.  The tiny, decode, mixed and MXFP4 workloads are measured after it
in the same run and reported under `configs`, each with its own per-kernel
table and dominant-kernel roofline (decode-sized batches take the fused path).

Timing: W untimed warm-up steps, then K steps, each preceded by an L2 flush
(a 512 MiB memset, then a 256 MiB read so no dirty line of the memset is left
to write back; outside the timed events) and bracketed by CUDA events on the
launching stream around an un-instrumented graph replay of the step.  `value`
is query tokens per second over all ranks (weak scaling: every rank runs its
own full batch).  `roofline` is for the kernel with the largest share of the
serialised step: algorithmic bytes per launch / its mean launch duration from
events around it in a serialised replay after each timed step, against the
measured HBM copy bandwidth; `roofline.in_step` is the same kernel timed inside
the concurrent step, where it shares the GPU with the other chains.  `e2e`
repeats the headline step through the public API with the step's inputs copied
from pinned host memory and every output copied back, all inside the timed
region.  `cpu_baseline` times the CPU oracle (test infrastructure,
single-threaded C) on a bounded sample of the same workload on this host.

--impl reference times the CPU oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time
from types import SimpleNamespace

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "K-cache tokens/s and achieved HBM GB/s (% of GB300 peak) per kernel, 1 GPU"
UNIT = "tokens/s"
NOMINAL_HBM_GBS = 8000.0
# the headline workload (the largest single-GPU configuration) and the ones
# measured after it
DEFAULT_CONFIG = "prefill"
SIDE_CONFIGS = ("tiny", "decode", "mixed", "mxfp4")


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---- algorithmic bytes per launch ----------------------------------------------------

def algorithmic_bytes(p, outputs) -> dict:
    """Compulsory bytes of each launch of a step: every distinct input byte read
    once, every output byte written once."""
    w = p.w
    res = {}
    if w.has_fp8:
        ins = w.insert_slots
        nv = int((ins >= 0).sum())
        rec = w.head_dim - w.rope_dim + 2 * w.rope_dim + w.head_dim // 64
        res["quantize_and_insert_k_cache"] = nv * (2 * w.head_dim + rec) + ins.size * 8
    if w.index_k is not None:
        ins = w.index_insert_slots
        nv = int((ins >= 0).sum())
        res["write_indexer_mxfp4_cache"] = nv * (2 * w.index_head_dim + w.index_head_dim // 2 +
                                                 w.index_head_dim // 32) + ins.size * 8
    T, K, R = w.num_tokens, w.topk, w.num_reqs
    comp_tab = w.comp_block_table if w.comp_block_table is not None else w.swa_block_table
    if w.has_fp8:
        W, P = w.window, w.padded_topk
        res["combine_topk_swa_indices"] = (T * (4 * K + 4 * (W + P) + 4 + 4) + R * 12 +
                                           R * comp_tab.shape[1] * 4)
        si = outputs["sparse_indices"]
        rec = w.head_dim - w.rope_dim + 2 * w.rope_dim + w.head_dim // 64
        for part, cols in (("swa", si[:, :W]), ("topk", si[:, W:])):
            valid = cols[cols >= 0]
            distinct = np.unique(valid).size
            res[f"dequantize_and_gather_k_cache[{part}]"] = (distinct * rec + cols.size * 4 +
                                                             cols.size * 2 * w.head_dim)
    res["compute_global_topk_indices_and_lens"] = T * (8 * K + 8) + R * comp_tab.shape[1] * 4
    gt = outputs["global_topk"]
    distinct = np.unique(gt[gt >= 0]).size
    D = w.index_head_dim
    res["dequantize_and_gather_k_cache[mxfp4]"] = (distinct * (D // 2 + D // 32) + gt.size * 4 +
                                                   gt.size * 2 * D)
    return res


def dense_algorithmic_bytes(p, outputs) -> dict:
    """Compulsory bytes of the dense (no top-k) decode step's launches."""
    w = p.w
    T, R, W, Wd = w.num_tokens, w.num_reqs, w.window, w.dense_width
    rec = w.head_dim - w.rope_dim + 2 * w.rope_dim + w.head_dim // 64
    ins = w.insert_slots
    res = {"quantize_and_insert_k_cache": int((ins >= 0).sum()) * (2 * w.head_dim + rec) +
           ins.size * 8}
    # token -> request + lens; per request qsl pair and seq_len, and the table row
    res["decode_swa_indices_and_lens"] = (T * (4 * W + 4 + 4) + R * 12 +
                                          R * w.swa_block_table.shape[1] * 4)
    # position (8) + token -> request + lens per token, and the table row
    res["compute_dense_compressed_indices_and_lens"] = (T * (4 * Wd + 8 + 4 + 4) +
                                                        R * w.comp_block_table.shape[1] * 4)
    for part, cols in (("swa", outputs["swa_indices"]), ("compressed", outputs["dense_indices"])):
        distinct = np.unique(cols[cols >= 0]).size
        res[f"dequantize_and_gather_k_cache[{part}]"] = (distinct * rec + cols.size * 4 +
                                                         cols.size * 2 * w.head_dim)
    return res


def indexer_algorithmic_bytes(p, variant: str, outputs) -> dict:
    """Compulsory bytes of the indexer_fp8 / indexer_store steps."""
    w = p.w
    T, K, R, D = w.num_tokens, w.topk, w.num_reqs, w.index_head_dim
    ins = w.index_insert_slots
    nv = int((ins >= 0).sum())
    comp_tab = w.comp_block_table if w.comp_block_table is not None else w.swa_block_table
    res = {"compute_global_topk_indices_and_lens": T * (8 * K + 8) + R * comp_tab.shape[1] * 4}
    gt = outputs["global_topk"]
    distinct = np.unique(gt[gt >= 0]).size
    if variant == "fp8":
        res["write_indexer_fp8_cache"] = nv * (2 * D + D + 4) + ins.size * 8
        res["dequantize_and_gather_k_cache[fp8_indexer]"] = (distinct * (D + 4) + gt.size * 4 +
                                                             gt.size * 2 * D)
    else:
        n = ins.size
        rows = min(n, p.INDEXER_MAX_POS)  # distinct RoPE rows read
        res["indexer_k_norm_rope_store"] = (nv * (2 * D + D // 2 + D // 32) + n * 16 +
                                            rows * 64 * 4 + D * 4)
        res["dequantize_and_gather_k_cache[mxfp4]"] = (distinct * (D // 2 + D // 32) +
                                                       gt.size * 4 + gt.size * 2 * D)
    return res


def compressor_algorithmic_bytes(p) -> dict:
    """Compulsory bytes of the compressor step: per layer the state write (kv
    and score read, the state row written, plus slot and position), and the
    compressed insert (every distinct window position's state slices once,
    the record written, per-token metadata)."""
    w = p.w
    res = {}
    for c in p.comp_layers:
        h = c["host"]
        r, sw, ov = h["ratio"], h["state_width"], h["overlap"]
        T = w.num_tokens
        nv = int((h["state_slots"] >= 0).sum())
        res[f"save_compressor_state[{r}]"] = nv * (2 * sw * 4 * 2) + T * 16 + r * sw * 4
        pos, t2r = h["positions"], w.token_to_req
        emit = (h["state_slots"] >= 0) & (h["kv_slots"] >= 0) & ((pos + 1) % r == 0)
        window = (2 if ov else 1) * r
        seen = set()
        for t in np.nonzero(emit)[0]:
            for q in range(int(pos[t]) - window + 1, int(pos[t]) + 1):
                if q >= 0:
                    seen.add((int(t2r[t]), q))
        # each present position's kv and score slices: all of a 2*sw row
        res[f"compress_kv_cache_insert[{r}]"] = (len(seen) * 2 * sw * 4 + int(emit.sum()) * 584 +
                                                 T * 24)
    return res


def workspace_algorithmic_bytes(p) -> dict:
    """Compulsory bytes of the prefill workspace step's launches."""
    from paged_sparse_kv_gb300.pipeline import workspace_geometry
    w = p.w
    g = workspace_geometry(w)
    D = w.head_dim
    rec = D - w.rope_dim + 2 * w.rope_dim + D // 64
    T, K, R = w.num_tokens, w.topk, w.num_reqs
    res = {}
    ins = w.insert_slots
    res["quantize_and_insert_k_cache"] = int((ins >= 0).sum()) * (2 * D + rec) + ins.size * 8
    ins = w.index_insert_slots
    Di = w.index_head_dim
    res["write_indexer_mxfp4_cache"] = int((ins >= 0).sum()) * (2 * Di + Di // 2 + Di // 32) + \
        ins.size * 8
    cb = g["compressed_base"]
    rows_c = int(np.minimum(g["compressed_lens"], cb).sum())
    rows_w = int(np.minimum(g["gather_lens"], g["workspace_width"] - cb).sum())
    res["dequantize_and_gather_k_cache_ranges[compressed]"] = rows_c * (rec + 2 * D) + R * 8
    res["dequantize_and_gather_k_cache_ranges[swa]"] = rows_w * (rec + 2 * D) + R * 12
    P = w.padded_topk
    res["combine_topk_swa_workspace_indices"] = T * (4 * K + 4 * (w.window + P) + 8) + R * 16
    n_raw = int(g["cu_compressed"][-1])
    res["indexer_mxfp4_paged_gather"] = n_raw * 2 * (Di // 2 + Di // 32) + (R + 1) * 4
    return res


# ---- clocks sampled during the timed region --------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---- CPU oracle (baseline / reference arm) -----------------------------------------

def _oracle_state(w):
    from paged_sparse_kv_gb300 import synthetic
    caches = {}
    for i, name in enumerate(("swa_cache", "comp_cache", "index_cache")):
        g = getattr(w, name)
        caches[name] = None if g is None else synthetic.random_cache_bytes(50 + i, g)
    return caches


def _oracle_sample_tokens(w, max_rows: int):
    """A bounded sample of the batch's tokens for the oracle's gathers."""
    cols = (w.window + w.padded_topk if w.has_fp8 else 0) + w.topk
    n = max(1, min(w.num_tokens, max_rows // max(cols, 1)))
    if n >= w.num_tokens:
        return None, w.num_tokens
    return np.linspace(0, w.num_tokens - 1, n).astype(np.int64), n


def host_description() -> dict:
    """The host the oracle is timed on: its processor and logical core count."""
    cpu = ""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model", "Hardware"):
            for line in info.splitlines():
                if line.split(":")[0].strip() == key and ":" in line:
                    cpu = line.split(":", 1)[1].strip()
                    break
            if cpu:
                break
        if not cpu:  # Arm: the implementer and part numbers
            impl = part = ""
            for line in info.splitlines():
                k = line.split(":")[0].strip()
                if k == "CPU implementer" and not impl:
                    impl = line.split(":", 1)[1].strip()
                if k == "CPU part" and not part:
                    part = line.split(":", 1)[1].strip()
            names = {("0x41", "0xd4f"): "Arm Neoverse V2", ("0x41", "0xd40"): "Arm Neoverse V1",
                     ("0x41", "0xd0c"): "Arm Neoverse N1"}
            if impl or part:
                cpu = names.get((impl, part), f"implementer {impl} part {part}")
    except OSError:
        pass
    import platform
    return {"cpu": cpu or platform.processor() or platform.machine(),
            "arch": platform.machine(), "nproc": os.cpu_count()}


def time_oracle(w, budget_s: float, path: str = "index"):
    """Run oracle steps until budget_s of CPU work; returns (tokens/s, desc)."""
    step, n, desc = _oracle_step(w, path, _oracle_state(w))
    steps, spent = 0, 0.0
    while spent < budget_s or steps == 0:
        t0 = time.perf_counter()
        step()
        spent += time.perf_counter() - t0
        steps += 1
    return n * steps / spent, f"{steps} x [{desc}] in {spent:.1f} s"


def _graph_events_supported(torch) -> bool:
    import inspect
    try:
        return "external" in inspect.signature(torch.cuda.Event.__new__).parameters
    except (TypeError, ValueError):
        return False


# CUDA sources of each timed entry point: its kernel file and that family's
# header (plus the shared headers).
_FAMILY = {"insert": ("insert.cu", "insert.h"), "index": ("index_build.cu", "index_build.h"),
           "gather": ("gather.cu", "gather.h"), "compressor": ("compressor.cu", "compressor.h")}
KERNEL_SOURCES = {
    "quantize_and_insert_k_cache": _FAMILY["insert"],
    "write_indexer_mxfp4_cache": _FAMILY["insert"],
    "write_indexer_fp8_cache": _FAMILY["insert"],
    "indexer_k_norm_rope_store": _FAMILY["insert"],
    "save_compressor_state": _FAMILY["compressor"],
    "compress_kv_cache_insert": _FAMILY["compressor"],
    "combine_topk_swa_indices": _FAMILY["index"],
    "compute_global_topk_indices_and_lens": _FAMILY["index"],
    "combine_topk_swa_workspace_indices": _FAMILY["index"],
    "decode_swa_indices_and_lens": _FAMILY["index"],
    "compute_dense_compressed_indices_and_lens": _FAMILY["index"],
    "build_dense_prefill_local_compressed_indices": _FAMILY["index"],
    "combine_dense_swa_indices": _FAMILY["index"],
    "dequantize_and_gather_k_cache": _FAMILY["gather"],
    "dequantize_and_gather_k_cache_ranges": _FAMILY["gather"],
    "dequantize_and_gather_k_cache_topk": _FAMILY["gather"],
    "dequantize_and_gather_k_cache_window": _FAMILY["gather"],
    "dequantize_and_gather_k_cache_pair": _FAMILY["gather"],
    "dequantize_and_gather_k_cache_dense": _FAMILY["gather"],
    "indexer_mxfp4_paged_gather": _FAMILY["gather"],
}
SHARED_SOURCES = ("psk_common.cuh", "launch.h")


def _code_only(text: str) -> str:
    """Source text without comments and with whitespace runs collapsed, so
    that editing a comment does not mark a kernel as changed."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel: str) -> str:
    """sha1 over the code (comments and whitespace dropped) of the CUDA
    sources a timed kernel is built from: its .cu file, its family's header
    and the shared headers.  Identifies the build a recorded ncu capture
    belongs to."""
    import hashlib
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "paged_sparse_kv_gb300", "csrc")
    base = kernel.split("[")[0]
    for f in sorted(KERNEL_SOURCES[base] + SHARED_SOURCES):
        h.update(f.encode())
        h.update(_code_only(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()


def recorded_traffic(config: str, kernel: str):
    """DRAM bytes (read + write) per launch from profiles/traffic.txt, or None
    when no capture exists for the current build of this kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    if kernel.split("[")[0] not in KERNEL_SOURCES:
        return None
    src = kernel_source_hash(kernel)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == config and \
                parts[1] == kernel and parts[3] == src:
            return int(parts[2])
    return None


def _instrumented(launches, names, evs):
    """The step serialised on the current stream, an event before each kernel;
    evs[-1] is recorded right after evs[0] with nothing between them (the gap
    two consecutive event nodes leave, subtracted from each kernel's figure)."""
    L = dict(launches)
    evs[0].record()
    evs[-1].record()
    for i, n in enumerate(names):
        L[n]()
        evs[i + 1].record()


def _capture(torch, dev, stream, fn):
    """Capture fn() into a CUDA graph (after one eager run on a side stream)."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn()
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize(dev)
    return g


# ---- main ------------------------------------------------------------------------------

def workload_description(w) -> str:
    return (f"{w.name}: {w.num_reqs} requests, {w.num_tokens} query tokens, "
            f"head_dim {w.head_dim} (rope {w.rope_dim}), window {w.window}, "
            f"top-k {w.topk}, ratio {w.compress_ratio}")


def line_config(workload: str, path: str, seed: int, world: int, launch: str) -> dict:
    """The `config` of the JSON line; both arms print the same one."""
    return {"workload": workload, "path": path,
            "storage": "bf16 rows in and out; fp8 e4m3 records with UE8M0 scales; "
                       "MXFP4 (e2m1 + E8M0) indexer keys",
            "seed": seed,
            "l2": ("flushed before every step: 512 MiB memset, then a 256 MiB read so "
                   "the lines left in L2 are clean"),
            "parallelism": f"dp{world} (independent batch per GPU)",
            "launch": launch,
            "timing": "value: events around an un-instrumented graph replay of each "
                      "step; roofline: events around the dominant kernel in a "
                      "serialised instrumented replay after each timed step "
                      "(roofline.in_step: in a concurrent instrumented replay)"}


def step_layout(p, path: str, graph: bool) -> str:
    """How the step's launches are laid out on streams (the config's `launch`)."""
    w = p.w
    if path == "fused":
        s = ("four streams: [fused top-k gather], [index build -> top-k mapping], "
             "[MXFP4 insert -> fused MXFP4 gather], [FP8 insert -> fused window gather]")
    elif path == "index" and not w.has_fp8:
        s = "a side stream: [top-k mapping -> MXFP4 insert -> MXFP4 gather]"
    elif path == "index" and p.gather_as_pair:
        s = ("two streams: [FP8 insert -> index build -> pair gather] (one PDL chain), "
             "[top-k mapping -> MXFP4 insert -> MXFP4 gather]")
    elif path == "index":
        s = ("three streams: [index build -> top-k gather], [FP8 insert -> (after the index "
             "build) window gather], [top-k mapping -> MXFP4 insert -> MXFP4 gather]")
    elif path == "workspace":
        s = ("three streams: [compressed range gather -> workspace index build], [FP8 insert "
             "-> window range gather], [MXFP4 insert -> raw MXFP4 gather]")
    elif path == "dense":
        s = ("three streams: [decode SWA indices -> (after the insert) window gather], [FP8 "
             "insert], [dense compressed indices -> compressed gather]")
    elif path == "dense_fused":
        s = ("three streams: [dense gather], [decode SWA indices -> dense compressed "
             "indices], [FP8 insert -> fused window gather]")
    elif path.startswith("indexer_"):
        s = "two streams: [key writer], [top-k mapping], then the gather of the top-k keys"
    elif path == "compressor":
        s = "two streams: one per layer, [state write -> compressed insert]"
    else:
        s = path
    return ("CUDA graph of the step on " if graph else "eager, ") + s


def step_alg_bytes(p, path: str, names) -> dict:
    """Algorithmic bytes of each launch of the step on ``path``."""
    w = p.w
    if path == "workspace":
        return workspace_algorithmic_bytes(p)
    if path.startswith("dense"):
        alg = dense_algorithmic_bytes(p, {"swa_indices": p.swa_indices.cpu().numpy(),
                                          "dense_indices": p.dense_indices.cpu().numpy()})
        if path == "dense_fused":
            # the same rows; slots from per-token metadata instead of index columns
            T = w.num_tokens
            alg["dequantize_and_gather_k_cache_window[swa]"] = (
                alg.pop("dequantize_and_gather_k_cache[swa]") - T * w.window * 4 + T * 16)
            alg["dequantize_and_gather_k_cache_dense[compressed]"] = (
                alg.pop("dequantize_and_gather_k_cache[compressed]") - T * w.dense_width * 4 +
                T * 16)
        return alg
    if path.startswith("indexer_"):
        return indexer_algorithmic_bytes(p, path.split("_")[1],
                                         {"global_topk": p.global_topk.cpu().numpy()})
    if path == "compressor":
        return compressor_algorithmic_bytes(p)
    outputs = {"global_topk": p.global_topk.cpu().numpy()}
    if w.has_fp8:
        outputs["sparse_indices"] = p.sparse_indices.cpu().numpy()
    alg = algorithmic_bytes(p, outputs)
    if path == "index" and "dequantize_and_gather_k_cache_pair" in names:
        # one launch over both column ranges: the two parts' bytes
        alg["dequantize_and_gather_k_cache_pair"] = (
            alg.pop("dequantize_and_gather_k_cache[swa]") +
            alg.pop("dequantize_and_gather_k_cache[topk]"))
    if path == "fused":
        # the fused gathers move the same rows; the top-k forms read a top-k
        # entry per item where the index form read a slot id, the window form
        # reads per-token metadata instead of its index columns
        alg["dequantize_and_gather_k_cache_topk[mxfp4]"] = alg.pop(
            "dequantize_and_gather_k_cache[mxfp4]")
        if w.has_fp8:
            alg["dequantize_and_gather_k_cache_topk[topk]"] = alg.pop(
                "dequantize_and_gather_k_cache[topk]")
            alg["dequantize_and_gather_k_cache_window[swa]"] = (
                alg.pop("dequantize_and_gather_k_cache[swa]") -
                w.num_tokens * w.window * 4 + w.num_tokens * 16)
    return alg


def _max_over_ranks(torch, dist, dev, x: float) -> float:
    if not dist:
        return x
    t = torch.tensor([x], device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_config(args, torch, dev, dist, world, rank, flush, config: str, steps: int,
               warmup: int, headline: bool) -> dict:
    """Measure one workload's step.  Returns the fields of its JSON entry;
    the headline workload also gets the end-to-end leg."""
    from paged_sparse_kv_gb300 import synthetic
    from paged_sparse_kv_gb300.pipeline import Pipeline

    w = synthetic.make(config, seed_offset=1000 * rank)
    p = Pipeline(w, dev)
    p.fill_caches_with_quantized_rows(seed=4321 + rank)
    path = args.path if headline else "auto"
    if path == "auto":  # the pipeline's size rule (fused for latency-bound batches)
        path = p.default_path
    if w.dense_width > 0 and not path.startswith("dense"):
        path = "dense"
    if path == "workspace" and not w.has_fp8:
        raise SystemExit("the workspace path needs a workload with an FP8 part")
    if path.startswith("dense") and w.dense_width <= 0:
        raise SystemExit("the dense path needs a workload with dense compressed entries")
    if path.startswith("indexer_") and (w.index_k is None or w.index_head_dim != 128):
        raise SystemExit("the indexer paths need 128-dim indexer keys")
    if path == "compressor" and not w.has_fp8:
        raise SystemExit("the compressor path needs a workload with an FP8 part")
    if path.startswith("indexer_"):
        launches = p.indexer_launches(path.split("_")[1])
    elif path == "compressor":
        launches = p.compressor_launches()
    else:
        launches = {"workspace": p.workspace_launches, "dense": p.dense_launches,
                    "dense_fused": p.dense_fused_launches,
                    "index": p.launches, "fused": p.fused_launches}[path]()
    names = [n for n, _ in launches]
    stream = torch.cuda.current_stream(dev)

    for _ in range(warmup):
        flush()
        p.step(concurrent=True, path=path)
    torch.cuda.synchronize(dev)
    alg = step_alg_bytes(p, path, names)

    visible = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x]
    local_rank = dev.index or 0
    clocks = ClockSampler(visible[local_rank] if local_rank < len(visible) else str(local_rank))
    use_graph = not args.eager and _graph_events_supported(torch)

    # (1) Per-kernel breakdown, untimed: the step serialised on one stream with
    # an event between consecutive kernels.  Each figure includes the cost of
    # the event node in front of the kernel.
    kern_ms = {n: [] for n in names}
    gap_ms = []
    n_ser = max(5, min(steps, 30))
    if use_graph:
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(names) + 2)]
        g_ser = _capture(torch, dev, stream, lambda: _instrumented(launches, names, evs))
        for _ in range(n_ser):
            flush()
            g_ser.replay()
            torch.cuda.synchronize(dev)
            gap_ms.append(evs[0].elapsed_time(evs[-1]))
            for i, n in enumerate(names):
                kern_ms[n].append((evs[-1] if i == 0 else evs[i]).elapsed_time(evs[i + 1]))
        del g_ser
    else:
        for _ in range(n_ser):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 2)]
            flush()
            _instrumented(launches, names, evs)
            torch.cuda.synchronize(dev)
            gap_ms.append(evs[0].elapsed_time(evs[-1]))
            for i, n in enumerate(names):
                kern_ms[n].append((evs[-1] if i == 0 else evs[i]).elapsed_time(evs[i + 1]))
    top = max(names, key=lambda n: statistics.mean(kern_ms[n]))

    # (2) Timed region: K steps.  Each step replays the concurrent step as a
    # CUDA graph with no event inside, timed by events on either side
    # (-> value).  After each timed step, two instrumented replays give the
    # dominant kernel's launch duration: the step serialised on one stream with
    # events only around that kernel, so it has the GPU to itself (-> roofline),
    # and the concurrent step with events around it on its own stream, where it
    # shares the GPU with the other chains (-> roofline.in_step).  Event nodes
    # inside a graph cost a few microseconds each, so they are kept out of the
    # replay that gives the step time.
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    marks = {k: torch.cuda.Event(enable_timing=True, external=use_graph)
             for k in ("iso0", "iso1", "cc0", "cc1")}
    hooks_iso = {top: (lambda: marks["iso0"].record(), lambda: marks["iso1"].record())}
    hooks_cc = {top: (lambda: marks["cc0"].record(), lambda: marks["cc1"].record())}
    g_plain = g_cc = g_iso = None
    if use_graph:
        g_plain = _capture(torch, dev, stream, lambda: p.step(concurrent=True, path=path))
        g_cc = _capture(torch, dev, stream,
                        lambda: p.step(concurrent=True, hooks=hooks_cc, path=path))
        g_iso = _capture(torch, dev, stream,
                         lambda: p.step(concurrent=False, hooks=hooks_iso, path=path))
        for _ in range(warmup):
            for g in (g_plain, g_cc, g_iso):
                flush()
                g.replay()
        torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    t_wall0 = time.perf_counter()
    step_ms, iso_ms, cc_ms = [], [], []
    for _ in range(steps):
        flush()
        t_start.record(stream)
        if g_plain is not None:
            g_plain.replay()
        else:
            p.step(concurrent=True, path=path)
        t_end.record(stream)
        flush()
        if g_cc is not None:
            g_cc.replay()
        else:
            p.step(concurrent=True, hooks=hooks_cc, path=path)
        flush()
        if g_iso is not None:
            g_iso.replay()
        else:
            p.step(concurrent=False, hooks=hooks_iso, path=path)
        marks["iso1"].synchronize()
        torch.cuda.synchronize(dev)
        step_ms.append(t_start.elapsed_time(t_end))
        iso_ms.append(marks["iso0"].elapsed_time(marks["iso1"]))
        cc_ms.append(marks["cc0"].elapsed_time(marks["cc1"]))
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    if dist:
        dist.barrier()

    # Back to back: the step graph replayed n times with no flush between (warm
    # L2), timed by one pair of events -- the latency-bound steps' throughput
    # when steps follow each other; reported beside the flushed per-step value.
    b2b = None
    if g_plain is not None:
        n_b2b = 20
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        flush()
        b0.record(stream)
        for _ in range(n_b2b):
            g_plain.replay()
        b1.record(stream)
        torch.cuda.synchronize(dev)
        b2b = {"ms_per_step": round(b0.elapsed_time(b1) / n_b2b, 5), "steps": n_b2b,
               "note": "step graph replayed back to back, no L2 flush between"}
    ms_per_step = _max_over_ranks(torch, dist, dev, statistics.mean(step_ms))
    value = w.num_tokens * world / (ms_per_step / 1e3)

    peak, peak_kind = _peaks()
    kernels = {}
    gap = statistics.median(gap_ms)
    for n in names:
        mean_ms = statistics.mean(kern_ms[n])
        gbs = alg[n] / (mean_ms / 1e3) / 1e9
        net_ms = max(mean_ms - gap, 1e-6)
        net_gbs = alg[n] / (net_ms / 1e3) / 1e9
        kernels[n] = {"us_serial_with_event_node": round(mean_ms * 1e3, 2),
                      "alg_bytes": int(alg[n]), "GBps": round(gbs, 1),
                      "frac_measured": round(gbs / peak, 3),
                      "frac_nominal_8TBps": round(gbs / NOMINAL_HBM_GBS, 3),
                      "us_net": round(net_ms * 1e3, 2),
                      "frac_measured_net": round(net_gbs / peak, 3)}
    iso_mean = _max_over_ranks(torch, dist, dev, statistics.mean(iso_ms))
    cc_mean = _max_over_ranks(torch, dist, dev, statistics.mean(cc_ms))
    achieved = alg[top] / (iso_mean / 1e3) / 1e9
    cc_gbs = alg[top] / (cc_mean / 1e3) / 1e9
    roof = {"kernel": top, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 3),
            "traffic": recorded_traffic(config, top), "us_per_launch": round(iso_mean * 1e3, 2),
            "alg_bytes_per_launch": int(alg[top]),
            "frac_nominal_8TBps": round(achieved / NOMINAL_HBM_GBS, 3),
            "timing": "events around the kernel in a serialised replay of the step after each "
                      "timed step (the kernel has the GPU to itself)",
            "us_per_launch_net": round(max(iso_mean - gap, 1e-6) * 1e3, 2),
            "frac_net": round(alg[top] / (max(iso_mean - gap, 1e-6) / 1e3) / 1e9 / peak, 3),
            "in_step": {"us_per_launch": round(cc_mean * 1e3, 2), "achieved": round(cc_gbs, 1),
                        "frac": round(cc_gbs / peak, 3),
                        "timing": "events around the kernel on its own stream in a concurrent "
                                  "replay of the step (it shares the GPU with the other chains)"}}
    step_bytes = sum(alg.values())
    res = {
        "workload": workload_description(w),
        "path": path, "seed": w.seed, "tokens_per_step": w.num_tokens,
        "launch": step_layout(p, path, g_plain is not None),
        "ms_per_step": round(ms_per_step, 5), "value": round(value, 1),
        "roofline": roof, "kernels": kernels,
        "event_gap_us": round(gap * 1e3, 2),
        "step_alg_bytes": int(step_bytes),
        "step_GBps": round(step_bytes / (ms_per_step / 1e3) / 1e9, 1),
        "step_frac_measured": round(step_bytes / (ms_per_step / 1e3) / 1e9 / peak, 3),
        "gpu_launches": 3 * len(launches) * steps,
        "clocks": clk, "wall_s_timed_region": round(t_wall, 4), "back_to_back": b2b,
    }
    del g_plain, g_cc, g_iso
    if headline:
        # every rank joins the max-over-ranks even if its own leg failed (e.g.
        # the pinned host buffers of several ranks exceed what the host allows)
        try:
            e2e = run_e2e(p, args, dev, flush, path)
            e2e_local, err = e2e["ms_per_step"], None
        except (RuntimeError, MemoryError) as ex:
            e2e, e2e_local = None, float("inf")
            err = (str(ex).splitlines() or ["error"])[0][:200]
        e2e_ms = _max_over_ranks(torch, dist, dev, e2e_local)
        if e2e is not None and e2e_ms != float("inf"):
            res["e2e"] = {"value": round(w.num_tokens * world / (e2e_ms / 1e3), 1),
                          "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"],
                          "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": round(e2e_ms, 4),
                          "launch": e2e["mode"] + " of [pinned host->device input copies, the "
                                    "step, device->host output copies], host clock around "
                                    "each replay"}
        else:
            res["e2e"] = {"value": None, "unit": UNIT, "h2d_bytes_per_step": None,
                          "d2h_bytes_per_step": None,
                          "error": err or "the end-to-end leg failed on another rank"}
        res["_w"] = w
    del p
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG,
                    choices=["tiny", "decode", "prefill", "mixed", "mxfp4", "prefill_small",
                             "decode_hca"])
    ap.add_argument("--configs", default=",".join(SIDE_CONFIGS),
                    help="comma-separated workloads measured after the headline one, each "
                         "reported under `configs` (empty: none)")
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--path", default="auto",
                    choices=["auto", "index", "fused", "workspace", "dense", "dense_fused",
                             "indexer_fp8",
                             "indexer_store", "compressor"],
                    help="auto: fused for index matrices of up to 2^20 items (latency-bound "
                         "batches), else index; "
                         "index: the index-keyed gather into [T, W+P, D]; workspace: the "
                         "prefill workspace path (range gathers + workspace indices); dense: "
                         "the no-top-k decode step of a heavily compressed layer (the "
                         "decode_hca workload always takes it); indexer_fp8 / indexer_store: "
                         "the mxfp4 workload's step with the FP8 indexer record or the fused "
                         "norm-RoPE store as the key writer; compressor: the compressed-KV "
                         "producer (ratio 4 and 128 layers) of a prefill batch.  Applies to "
                         "the headline workload; the others take auto")
    ap.add_argument("--eager", action="store_true",
                    help="launch the step eagerly instead of replaying a CUDA graph")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    from paged_sparse_kv_gb300 import build as psk_build

    psk_build.build()
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    flush = L2Flush(torch, dev)
    head = run_config(args, torch, dev, dist, world, rank, flush, args.config, args.steps,
                      args.warmup, headline=True)
    w = head.pop("_w")
    side = {}
    for name in [c for c in args.configs.split(",") if c and c != args.config]:
        r = run_config(args, torch, dev, dist, world, rank, flush, name, min(args.steps, 20),
                       args.warmup, headline=False)
        side[name] = {k: r[k] for k in ("workload", "path", "value", "ms_per_step",
                                        "step_GBps", "step_frac_measured", "roofline",
                                        "kernels", "event_gap_us", "launch", "back_to_back",
                                        "clocks", "gpu_launches")}
        side[name]["unit"] = UNIT

    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32/int32",
        "data": "synthetic",
        "config": line_config(head["workload"], head["path"], head["seed"], world,
                              head["launch"]),
        "roofline": head["roofline"],
        "kernels": head["kernels"],
        "kernels_note": ("us_serial_with_event_node: events between consecutive kernels of "
                         "the serialised step; us_net: that minus the gap two consecutive "
                         "event nodes leave (event_gap_us), i.e. the kernel with its own "
                         "launch latency"),
        "event_gap_us": head["event_gap_us"],
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "step_alg_bytes": head["step_alg_bytes"],
        "step_GBps": head["step_GBps"],
        "step_frac_measured": head["step_frac_measured"],
        "clocks": head["clocks"],
        "wall_s_timed_region": head["wall_s_timed_region"],
        "back_to_back": head["back_to_back"],
        "configs": side,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc = time_oracle(w, args.cpu_budget, path=head["path"])
        line["cpu_baseline"] = {"value": round(v, 2), "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": desc, "host": host_description()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


class L2Flush:
    """Evicts the step's data from L2 (129 MB) between timed steps: a 512 MiB
    memset, then a 256 MiB read of another buffer.  After the memset alone L2
    would hold dirty lines whose write-back the next step would pay for; the
    read replaces them with clean ones."""

    def __init__(self, torch, dev):
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.amax()


def run_e2e(p, args, dev, flush, path="index"):
    """The step through the public API with pinned host inputs and outputs."""
    import torch
    ins = [t for t in (p.k, p.insert_slots, p.index_k, p.index_insert_slots, p.qsl, p.seq_lens,
                       p.t2r, p.replay, p.topk) if t is not None]
    if path == "workspace":
        outs = [p.ws, p.ws_indices, p.ws_lens, p.raw_values, p.raw_scales]
    elif path.startswith("dense"):
        ins = [t for t in (p.k, p.insert_slots, p.qsl, p.seq_lens, p.t2r, p.positions)
               if t is not None]
        outs = [p.swa_indices, p.swa_lens, p.dense_indices, p.dense_lens, p.dense_gathered]
    elif path == "compressor":
        ins = [t for c in p.comp_layers for t in (c["kv"], c["score"], c["positions"],
                                                  c["state_slots"], c["kv_slots"])]
        outs = [c["kv_cache"] for c in p.comp_layers]
    elif path.startswith("indexer_"):
        ins = [p.index_k, p.index_insert_slots, p.topk, p.t2r]
        if path == "indexer_store":
            ins.append(p.ix_positions)
        outs = [p.global_topk, p.global_lens, p.gathered_index]
    else:
        outs = [t for t in (p.sparse_indices, p.lens, p.gathered, p.global_topk, p.global_lens,
                            p.gathered_index) if t is not None]
    h_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in ins]
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)

    def one_step():
        for d, h in zip(ins, h_in):
            d.copy_(h, non_blocking=True)
        p.step(concurrent=True, path=path)
        for h, d in zip(h_out, outs):
            h.copy_(d, non_blocking=True)

    # The whole step -- input copies from pinned host memory, the kernels, the
    # output copies back -- as one CUDA graph, replayed every step (eager if the
    # capture is refused).
    graph, mode = None, "eager"
    if not args.eager:
        try:
            graph = _capture(torch, dev, torch.cuda.current_stream(dev), one_step)
            mode = "cuda graph"
        except RuntimeError:
            graph = None
    times = []
    for s in range(args.warmup + args.steps):
        flush()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        if graph is not None:
            graph.replay()
        else:
            one_step()
        torch.cuda.synchronize(dev)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    return {"ms_per_step": statistics.mean(times) * 1e3, "h2d": h2d, "d2h": d2h, "mode": mode}


def _oracle_step(w, path: str, caches):
    """(one oracle step as a callable, tokens it covers, description) for a path."""
    from oracle.pipeline import (run_compressor_step, run_dense_step, run_indexer_step,
                                 run_step, run_workspace_step)
    if path == "compressor":
        from paged_sparse_kv_gb300 import synthetic
        layers = [synthetic.compressor_inputs(w, r, 777 + i) for i, r in enumerate((4, 128))]
        states = [np.zeros((c["state_pages"], c["state_bs"], 2 * c["state_width"]), np.float32)
                  for c in layers]
        kvc = [np.zeros((c["kv_geom"].num_pages, c["kv_geom"].page_stride), np.uint8)
               for c in layers]
        return (lambda: run_compressor_step(w, layers, states, kvc), w.num_tokens,
                f"oracle step of the {w.name} batch (compressor path) per timed step")
    if path.startswith("indexer_"):
        from paged_sparse_kv_gb300 import synthetic
        from paged_sparse_kv_gb300.pipeline import Pipeline
        variant = path.split("_")[1]
        n = w.index_k.shape[0]
        inputs = {"positions": np.arange(n, dtype=np.int64) % Pipeline.INDEXER_MAX_POS,
                  "cos_sin": synthetic.gptj_cos_sin(Pipeline.INDEXER_MAX_POS),
                  "weight": synthetic.norm_weight(w.seed), "eps": 1e-6}
        g = w.index_cache
        cache = (np.zeros((g.num_pages, g.block_size * 132), np.uint8) if variant == "fp8"
                 else caches["index_cache"])
        toks, nt = _oracle_sample_tokens(w, 80000)
        return (lambda: run_indexer_step(w, variant, cache, inputs, toks), nt,
                f"oracle step of the {w.name} batch ({path} path) per timed step; gathers over "
                f"{nt} of {w.num_tokens} tokens")
    if path.startswith("dense"):
        return (lambda: run_dense_step(w, caches["swa_cache"], caches["comp_cache"]),
                w.num_tokens, f"oracle step of the {w.name} batch (dense path) per timed step")
    if path == "workspace":
        from paged_sparse_kv_gb300.pipeline import workspace_geometry
        geom = workspace_geometry(w)
        return (lambda: run_workspace_step(w, geom, caches["swa_cache"], caches["comp_cache"],
                                           caches["index_cache"]),
                w.num_tokens,
                f"oracle step of the {w.name} batch (workspace path) per timed step")
    toks, n = _oracle_sample_tokens(w, 80000)
    return (lambda: run_step(w, caches["swa_cache"], caches["comp_cache"],
                             caches["index_cache"], toks),
            n, f"oracle step of the {w.name} batch per timed step; gathers over {n} of "
               f"{w.num_tokens} tokens")


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle, timed on this host's cores."""
    if rank != 0:
        return
    import oracle
    from paged_sparse_kv_gb300 import synthetic
    oracle.build()
    from paged_sparse_kv_gb300.pipeline import Pipeline
    w = synthetic.make(args.config)
    path = args.path
    if path == "auto":
        path = Pipeline.default_path_for(w)
    if w.dense_width > 0 and not path.startswith("dense"):
        path = "dense"
    step, n, desc = _oracle_step(w, path, _oracle_state(w))
    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    ms = statistics.mean(times) * 1e3
    value = n / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32/int32", "data": "synthetic",
        "config": line_config(workload_description(w), path, w.seed, world,
                              step_layout(SimpleNamespace(w=w, gather_as_pair=Pipeline.small_batch(w)),
                                          path, not args.eager)),
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "host": host_description(),
                         "sample": desc},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
