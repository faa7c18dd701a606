"""One step of the paged K-cache pipeline on the device, for a synthetic workload.

A step runs every hot-path row over one batch, in this order:

  1. quantize_and_insert_k_cache   new K rows -> SWA cache (FP8 fp8_ds_mla)
  2. write_indexer_mxfp4_cache     new indexer keys -> indexer cache (MXFP4)
  3. combine_topk_swa_indices      window + top-k -> sparse_indices, lens
  4. dequantize_and_gather_k_cache(_pair)  window columns from the SWA cache,
                                   top-k columns from the compressed cache,
                                   into one [T, W+P, D] output: one pair launch
                                   for index matrices of at most 2^20 items,
                                   else two launches on column ranges
  5. compute_global_topk_indices_and_lens  top-k -> indexer-cache slots
  6. dequantize_and_gather_k_cache those slots from the MXFP4 indexer cache

Workloads without an FP8 part (the MXFP4 indexer workload) run 2, 5 and 6.
All buffers are allocated once here; ``step()`` only launches kernels.

``step(concurrent=True)`` runs the independent chains of the step on two
streams (three with the two-launch gather), fork/join with events, with the
same dependencies as the serial order:

  stream M:  quantize_and_insert_k_cache -> combine_topk_swa_indices -> gather_pair
             (one PDL chain: each kernel waits for its predecessor's grid)
  (two launches: stream A runs quantize_and_insert_k_cache and then the window
  columns after the build, stream M the build and then the top-k columns)
  stream B:  compute_global_topk_indices_and_lens -> write_indexer_mxfp4_cache
             -> gather[mxfp4]

Decode-sized kernels fill only part of the GPU, so overlapping the chains
shortens the step to its critical path.  Capturing ``step(concurrent=True)``
in a CUDA graph keeps the fork/join structure.

``path="fused"`` produces the same outputs with gathers that compute their
own slots (the window rule through the SWA table, the local top-k through the
compressed / indexer table), so no gather waits for an index build; the index
builders still run for their outputs (sparse_indices, lens, the global top-k):

  stream M:  gather_topk[topk]  (issued first)
  stream A:  quantize_and_insert_k_cache -> gather_window[swa]
  stream B:  write_indexer_mxfp4_cache -> gather_topk[mxfp4]
  stream C:  combine_topk_swa_indices -> compute_global_topk_indices_and_lens

``path="workspace"`` is the prefill path of TokenSpeed's backend
(``_prefill_workspace``): the compressed rows of every request (range form,
offset 0) and its window rows (offset ``compressed_base``) are gathered into a
per-request bf16 workspace, the index build emits workspace-relative rows,
and the indexer's packed MXFP4 keys of every compressed entry are gathered
raw:

  stream M:  dequantize_and_gather_k_cache_ranges[compressed] ->
             combine_topk_swa_workspace_indices
  stream A:  quantize_and_insert_k_cache -> dequantize_and_gather_k_cache_ranges[swa]
  stream B:  write_indexer_mxfp4_cache -> indexer_mxfp4_paged_gather

``path="indexer_fp8"`` and ``path="indexer_store"`` are the indexer step of
the MXFP4 workload with the other key writers: the FP8 indexer record
(write_indexer_fp8_cache, read back as record 2) and the fused k_norm -> RoPE
-> MXFP4 store (indexer_k_norm_rope_store, ratio 1, positions cycling through
a 131072-row GPT-J table):

  stream A:  <key writer>
  stream B:  compute_global_topk_indices_and_lens
  join:      gather of the top-k keys

``path="compressor"`` is the compressed-KV producer of a prefill batch for a
ratio-4 (overlapping window) and a ratio-128 layer, one per stream:

  stream A:  save_compressor_state[4] -> compress_kv_cache_insert[4]
  stream B:  save_compressor_state[128] -> compress_kv_cache_insert[128]

``path="dense"`` is the decode step of a heavily compressed attention layer
(no top-k; TokenSpeed's decode SWA precompute and
``_decode_compressed_attention_indices_and_lens`` for a ratio other than 4):

  stream M:  decode_swa_indices_and_lens -> (wait for the insert) -> gather[swa]
  stream A:  quantize_and_insert_k_cache
  stream B:  compute_dense_compressed_indices_and_lens -> gather[compressed]

``path="dense_fused"`` produces the same outputs with gathers that compute their
own slots (the window rule; every visible compressed entry), so neither waits
for a builder:

  stream M:  gather_dense[compressed]  (issued first)
  stream B:  decode_swa_indices_and_lens -> compute_dense_compressed_indices_and_lens
  stream A:  quantize_and_insert_k_cache -> gather_window[swa]
"""
from __future__ import annotations

from typing import Callable, Optional

import numpy as np
import torch

from . import ops
from .synthetic import Workload


def _dev_i32(a: Optional[np.ndarray], dev) -> Optional[torch.Tensor]:
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def _dev_i64(a: Optional[np.ndarray], dev) -> Optional[torch.Tensor]:
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).to(dev)


def _dev_bf16(a: Optional[np.ndarray], dev) -> Optional[torch.Tensor]:
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


class Pipeline:
    """Device state for one workload: inputs, caches and outputs."""

    def __init__(self, w: Workload, device: torch.device | str = "cuda:0"):
        dev = torch.device(device)
        self.w = w
        self.dev = dev
        self.k = _dev_bf16(w.k, dev)
        self.insert_slots = _dev_i64(w.insert_slots, dev)
        self.index_k = _dev_bf16(w.index_k, dev)
        self.index_insert_slots = _dev_i64(w.index_insert_slots, dev)
        self.qsl = _dev_i32(w.query_start_loc, dev)
        self.seq_lens = _dev_i32(w.seq_lens, dev)
        self.t2r = _dev_i32(w.token_to_req, dev)
        self.replay = _dev_i32(w.replay_start, dev)
        self.valid = None if w.is_valid_token is None else torch.from_numpy(
            np.ascontiguousarray(w.is_valid_token, dtype=np.uint8)).to(dev)
        self.swa_bt = _dev_i32(w.swa_block_table, dev)
        self.comp_bt = _dev_i32(w.comp_block_table, dev)
        self.topk = _dev_i32(w.topk_local, dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

        def cache(g):
            return None if g is None else torch.zeros((g.num_pages, g.page_stride),
                                                      dtype=torch.uint8, device=dev)
        self.swa_cache = cache(w.swa_cache)
        # the compressed cache is its own buffer even when it shares the SWA table
        self.comp_cache = cache(w.comp_cache)
        self.index_cache = cache(w.index_cache)

        T, K = w.num_tokens, w.topk
        self.cols = w.window + w.padded_topk
        # Decode-sized index matrices are gathered by one launch over both
        # caches; larger ones by two column-range launches on two streams,
        # which overlap better (measured on the prefill and mixed batches).
        self.gather_as_pair = self.small_batch(w)
        self.default_path = self.default_path_for(w)
        if w.has_fp8:
            self.sparse_indices = torch.empty((T, self.cols), dtype=torch.int32, device=dev)
            self.lens = torch.empty((T,), dtype=torch.int32, device=dev)
            self.gathered = torch.empty((T, self.cols, w.head_dim), dtype=torch.bfloat16,
                                        device=dev)
            # the padding columns (sparse_indices -1) gather as zero rows; the
            # fused top-k gather writes only the K real columns
            self.gathered[:, w.window + K:].zero_()
        else:
            self.sparse_indices = self.lens = self.gathered = None
        self.global_topk = torch.empty((T, K), dtype=torch.int32, device=dev)
        self.global_lens = torch.empty((T,), dtype=torch.int32, device=dev)
        self.gathered_index = torch.empty((T, K, w.index_head_dim), dtype=torch.bfloat16,
                                          device=dev)
        self.ws = None

    def alloc_workspace(self) -> None:
        """Workspace geometry and buffers of the prefill workspace path, from
        the batch metadata on the host (as the backend sizes them)."""
        w, dev = self.w, self.dev
        g = workspace_geometry(w)
        self.ws_glen = _dev_i32(g["gather_lens"], dev)
        self.ws_lc = _dev_i32(g["compressed_lens"], dev)
        self.ws_cu = _dev_i32(g["cu_compressed"], dev)
        self.ws_cb, self.ws_width = g["compressed_base"], g["workspace_width"]
        self.ws_rows_raw = int(g["cu_compressed"][-1])
        self.ws = torch.empty((w.num_reqs, self.ws_width, w.head_dim), dtype=torch.bfloat16,
                              device=dev)
        self.ws_indices = torch.empty((w.num_tokens, self.cols), dtype=torch.int32, device=dev)
        self.ws_lens = torch.empty((w.num_tokens,), dtype=torch.int32, device=dev)
        self.raw_values = torch.empty((self.ws_rows_raw, w.index_head_dim // 2),
                                      dtype=torch.uint8, device=dev)
        self.raw_scales = torch.empty((self.ws_rows_raw, w.index_head_dim // 32),
                                      dtype=torch.uint8, device=dev)

    def workspace_launches(self) -> list[tuple[str, Callable[[], None]]]:
        """The prefill workspace step as (kernel name, launch) pairs, in order."""
        w = self.w
        if self.ws is None:
            self.alloc_workspace()
        comp_table = self.comp_bt if self.comp_bt is not None else self.swa_bt
        return [
            ("quantize_and_insert_k_cache", lambda: ops.quantize_and_insert_k_cache(
                self.k, self.swa_cache, self.insert_slots, w.swa_cache.block_size,
                rope_dim=w.rope_dim, err_count=self.err)),
            ("write_indexer_mxfp4_cache", lambda: ops.write_indexer_mxfp4_cache(
                self.index_k, self.index_cache, self.index_insert_slots,
                w.index_cache.block_size, err_count=self.err)),
            ("dequantize_and_gather_k_cache_ranges[compressed]",
             lambda: ops.dequantize_and_gather_k_cache_ranges(
                 self.ws[:, :self.ws_cb], self.comp_cache, self.ws_lc, None, comp_table,
                 w.comp_cache.block_size, 0, rope_dim=w.rope_dim)),
            ("dequantize_and_gather_k_cache_ranges[swa]",
             lambda: ops.dequantize_and_gather_k_cache_ranges(
                 self.ws, self.swa_cache, self.seq_lens, self.ws_glen, self.swa_bt,
                 w.swa_cache.block_size, self.ws_cb, rope_dim=w.rope_dim)),
            ("combine_topk_swa_workspace_indices",
             lambda: ops.combine_topk_swa_workspace_indices(
                 self.topk, self.qsl, self.seq_lens, self.ws_glen, self.t2r, w.window,
                 w.compress_ratio, self.ws_width, self.ws_cb, is_valid_token=self.valid,
                 out=self.ws_indices, lens=self.ws_lens)),
            ("indexer_mxfp4_paged_gather", lambda: ops.indexer_mxfp4_paged_gather(
                self.index_cache, comp_table, self.ws_cu, w.index_cache.block_size,
                w.index_head_dim, self.ws_rows_raw, values_out=self.raw_values,
                scales_out=self.raw_scales)),
        ]

    def alloc_dense(self) -> None:
        """Buffers of the dense (no top-k) decode step."""
        w, dev = self.w, self.dev
        T, W, Wd = w.num_tokens, w.window, w.dense_width
        self.positions = _dev_i64(w.positions, dev)
        self.swa_indices = torch.empty((T, W), dtype=torch.int32, device=dev)
        self.swa_lens = torch.empty((T,), dtype=torch.int32, device=dev)
        self.dense_indices = torch.empty((T, Wd), dtype=torch.int32, device=dev)
        self.dense_lens = torch.empty((T,), dtype=torch.int32, device=dev)
        self.dense_gathered = torch.empty((T, W + Wd, w.head_dim), dtype=torch.bfloat16,
                                          device=dev)

    def dense_launches(self) -> list[tuple[str, Callable[[], None]]]:
        """The dense decode step as (kernel name, launch) pairs, in order."""
        w = self.w
        if getattr(self, "dense_indices", None) is None:
            self.alloc_dense()
        W = w.window
        return [
            ("quantize_and_insert_k_cache", lambda: ops.quantize_and_insert_k_cache(
                self.k, self.swa_cache, self.insert_slots, w.swa_cache.block_size,
                rope_dim=w.rope_dim, err_count=self.err)),
            ("decode_swa_indices_and_lens", lambda: ops.decode_swa_indices_and_lens(
                self.qsl, self.seq_lens, self.t2r, self.swa_bt, w.swa_cache.block_size, W,
                is_valid_token=self.valid, out=self.swa_indices, lens=self.swa_lens)),
            ("compute_dense_compressed_indices_and_lens",
             lambda: ops.compute_dense_compressed_indices_and_lens(
                 self.positions, self.t2r, self.comp_bt, w.comp_cache.block_size,
                 w.compress_ratio, w.dense_width, is_valid_token=self.valid,
                 out=self.dense_indices, lens=self.dense_lens)),
            ("dequantize_and_gather_k_cache[swa]", lambda: ops.dequantize_and_gather_k_cache(
                self.dense_gathered[:, :W, :], self.swa_cache, self.swa_indices,
                w.swa_cache.block_size, rope_dim=w.rope_dim)),
            ("dequantize_and_gather_k_cache[compressed]",
             lambda: ops.dequantize_and_gather_k_cache(
                 self.dense_gathered[:, W:, :], self.comp_cache, self.dense_indices,
                 w.comp_cache.block_size, rope_dim=w.rope_dim)),
        ]

    def dense_fused_launches(self) -> list[tuple[str, Callable[[], None]]]:
        """The dense decode step with gathers that compute their own slots (the
        window rule; every visible compressed entry), as (name, launch) pairs."""
        w = self.w
        base = dict(self.dense_launches())
        W = w.window
        return [(n, base[n]) for n in ("quantize_and_insert_k_cache", "decode_swa_indices_and_lens",
                                       "compute_dense_compressed_indices_and_lens")] + [
            ("dequantize_and_gather_k_cache_window[swa]",
             lambda: ops.dequantize_and_gather_k_cache_window(
                 self.dense_gathered[:, :W, :], self.swa_cache, self.qsl, self.seq_lens,
                 self.t2r, None, self.swa_bt, w.swa_cache.block_size, W, rope_dim=w.rope_dim,
                 is_valid_token=self.valid)),
            ("dequantize_and_gather_k_cache_dense[compressed]",
             lambda: ops.dequantize_and_gather_k_cache_dense(
                 self.dense_gathered[:, W:, :], self.comp_cache, self.positions, self.t2r,
                 self.comp_bt, w.comp_cache.block_size, w.compress_ratio, rope_dim=w.rope_dim,
                 num_reqs=w.num_reqs, is_valid_token=self.valid)),
        ]

    COMPRESSOR_EPS = 1e-6

    def alloc_compressor(self, seed: int = 777) -> None:
        """Inputs and caches of the compressor step (ratio 4 and 128 layers)."""
        from . import synthetic
        w, dev = self.w, self.dev
        self.comp_layers = []
        for i, ratio in enumerate((4, 128)):
            c = synthetic.compressor_inputs(w, ratio, seed + i)
            g = c["kv_geom"]
            d = {"host": c, "ratio": ratio, "overlap": c["overlap"],
                 "kv": torch.from_numpy(c["kv"]).to(dev),
                 "score": torch.from_numpy(c["score"]).to(dev),
                 "ape": torch.from_numpy(c["ape"]).to(dev),
                 "positions": _dev_i64(c["positions"], dev),
                 "state_slots": _dev_i64(c["state_slots"], dev),
                 "state_table": _dev_i32(c["state_table"], dev),
                 "state": torch.zeros((c["state_pages"], c["state_bs"], 2 * c["state_width"]),
                                      dtype=torch.float32, device=dev),
                 "kv_slots": _dev_i64(c["kv_slots"], dev),
                 "kv_cache": (self.comp_cache if ratio == 4 else
                              torch.zeros((g.num_pages, g.page_stride), dtype=torch.uint8,
                                          device=dev)),
                 "weight": torch.from_numpy(c["weight"]).to(dev),
                 "cos_sin": torch.from_numpy(c["cos_sin"]).to(dev)}
            self.comp_layers.append(d)

    def compressor_launches(self) -> list[tuple[str, Callable[[], None]]]:
        """The compressor step as (kernel name, launch) pairs, in order."""
        w = self.w
        if getattr(self, "comp_layers", None) is None:
            self.alloc_compressor()
        L = []
        for c in self.comp_layers:
            r = c["ratio"]
            L.append((f"save_compressor_state[{r}]", lambda c=c: ops.save_compressor_state(
                c["kv"], c["score"], c["ape"], c["state"], c["state_slots"], c["positions"],
                c["state"].shape[1], c["ratio"], err_count=self.err)))
            L.append((f"compress_kv_cache_insert[{r}]", lambda c=c: ops.compress_kv_cache_insert(
                c["state"], self.t2r, c["positions"], c["state_slots"], c["state_table"],
                c["state"].shape[1], c["weight"], self.COMPRESSOR_EPS, c["cos_sin"],
                c["kv_cache"], c["kv_slots"], 64, c["ratio"], overlap=c["overlap"],
                err_count=self.err)))
        return L

    PAIR_MAX_ITEMS = 1 << 20

    @classmethod
    def small_batch(cls, w: Workload) -> bool:
        """An index matrix of at most 2^20 items: a latency-bound batch."""
        return w.num_tokens * (w.window + w.padded_topk) <= cls.PAIR_MAX_ITEMS

    @classmethod
    def default_path_for(cls, w: Workload) -> str:
        """The step a batch runs by default.  Latency-bound batches take the
        fused gathers, which wait for no index build (decode: 23.2 against
        27.1 us per step); larger, bandwidth-bound ones the index path
        (prefill, mixed: 1% faster)."""
        if w.dense_width > 0:
            return "dense_fused" if cls.small_batch(w) else "dense"
        return "fused" if (w.has_fp8 and cls.small_batch(w)) else "index"
    INDEXER_MAX_POS = 131072

    def alloc_indexer(self) -> None:
        """Buffers of the indexer_fp8 / indexer_store steps."""
        from . import synthetic
        w, dev = self.w, self.dev
        g = w.index_cache
        n = w.index_k.shape[0]
        self.fp8i_cache = torch.zeros((g.num_pages, g.block_size * 132), dtype=torch.uint8,
                                      device=dev)
        self.ix_positions = torch.arange(n, dtype=torch.int64, device=dev) % self.INDEXER_MAX_POS
        self.ix_cos_sin = torch.from_numpy(synthetic.gptj_cos_sin(self.INDEXER_MAX_POS)).to(dev)
        self.ix_weight = torch.from_numpy(synthetic.norm_weight(w.seed)).to(dev)
        self.ix_eps = 1e-6

    def indexer_launches(self, variant: str) -> list[tuple[str, Callable[[], None]]]:
        """The indexer step with the FP8 indexer record ("fp8") or the fused
        norm-RoPE-MXFP4 store ("store") as the key writer."""
        w = self.w
        if getattr(self, "fp8i_cache", None) is None:
            self.alloc_indexer()
        bs = w.index_cache.block_size
        topk = ("compute_global_topk_indices_and_lens",
                lambda: ops.compute_global_topk_indices_and_lens(
                    self.topk, self.t2r, self.index_table, bs, self.valid,
                    out=self.global_topk, lens=self.global_lens))
        if variant == "fp8":
            return [
                ("write_indexer_fp8_cache", lambda: ops.write_indexer_fp8_cache(
                    self.index_k, self.fp8i_cache, self.index_insert_slots, bs,
                    err_count=self.err)),
                topk,
                ("dequantize_and_gather_k_cache[fp8_indexer]",
                 lambda: ops.dequantize_and_gather_k_cache(
                     self.gathered_index, self.fp8i_cache, self.global_topk, bs,
                     record=ops.PSK_REC_FP8_INDEXER)),
            ]
        return [
            ("indexer_k_norm_rope_store", lambda: ops.indexer_k_norm_rope_store(
                self.index_k, self.ix_positions, self.ix_cos_sin, self.ix_weight, self.ix_eps,
                self.index_cache, self.index_insert_slots, 1, True, bs, err_count=self.err)),
            topk,
            ("dequantize_and_gather_k_cache[mxfp4]", lambda: ops.dequantize_and_gather_k_cache(
                self.gathered_index, self.index_cache, self.global_topk, bs,
                record=ops.PSK_REC_MXFP4)),
        ]

    # the indexer cache follows the compressed table
    @property
    def index_table(self) -> torch.Tensor:
        return self.comp_bt if self.comp_bt is not None else self.swa_bt

    def fill_caches_with_quantized_rows(self, seed: int = 1234, chunk: int = 1 << 18) -> None:
        """Fill every slot of every cache with quantized N(0,1) rows, through the
        library's own inserts (used by the benchmark to give the gathers real
        records to read)."""
        g = torch.Generator(device=self.dev).manual_seed(seed)
        w = self.w
        for cache, geom, fp8 in ((self.swa_cache, w.swa_cache, True),
                                 (self.comp_cache, w.comp_cache, True),
                                 (self.index_cache, w.index_cache, False)):
            if cache is None:
                continue
            cap = geom.num_pages * geom.block_size
            D = w.head_dim if fp8 else w.index_head_dim
            for s0 in range(0, cap, chunk):
                n = min(chunk, cap - s0)
                rows = torch.randn((n, D), generator=g, device=self.dev).to(torch.bfloat16)
                slots = torch.arange(s0, s0 + n, dtype=torch.int64, device=self.dev)
                if fp8:
                    ops.quantize_and_insert_k_cache(rows, cache, slots, geom.block_size,
                                                    rope_dim=w.rope_dim)
                else:
                    ops.write_indexer_mxfp4_cache(rows, cache, slots, geom.block_size)

    def launches(self) -> list[tuple[str, Callable[[], None]]]:
        """The step as a list of (kernel name, launch) pairs, in order."""
        w = self.w
        L: list[tuple[str, Callable[[], None]]] = []
        if w.has_fp8:
            L.append(("quantize_and_insert_k_cache", lambda: ops.quantize_and_insert_k_cache(
                self.k, self.swa_cache, self.insert_slots, w.swa_cache.block_size,
                rope_dim=w.rope_dim, err_count=self.err)))
        if self.index_k is not None:
            L.append(("write_indexer_mxfp4_cache", lambda: ops.write_indexer_mxfp4_cache(
                self.index_k, self.index_cache, self.index_insert_slots,
                w.index_cache.block_size, err_count=self.err)))
        if w.has_fp8:
            W = w.window
            L.append(("combine_topk_swa_indices", lambda: ops.combine_topk_swa_indices(
                self.qsl, self.seq_lens, self.t2r, self.replay, self.swa_bt,
                w.swa_cache.block_size, self.comp_bt, w.comp_cache.block_size, W,
                w.compress_ratio, self.topk, is_valid_token=self.valid,
                out=self.sparse_indices, lens=self.lens)))
            if self.gather_as_pair:
                L.append(("dequantize_and_gather_k_cache_pair", lambda: ops.dequantize_and_gather_k_cache_pair(
                    self.gathered, self.swa_cache, w.swa_cache.block_size, self.comp_cache,
                    w.comp_cache.block_size, self.sparse_indices, W, rope_dim=w.rope_dim)))
            else:
                L.append(("dequantize_and_gather_k_cache[swa]", lambda: ops.dequantize_and_gather_k_cache(
                    self.gathered[:, :W, :], self.swa_cache, self.sparse_indices[:, :W],
                    w.swa_cache.block_size, rope_dim=w.rope_dim)))
                L.append(("dequantize_and_gather_k_cache[topk]", lambda: ops.dequantize_and_gather_k_cache(
                    self.gathered[:, W:, :], self.comp_cache, self.sparse_indices[:, W:],
                    w.comp_cache.block_size, rope_dim=w.rope_dim)))
        L.append(("compute_global_topk_indices_and_lens", lambda: ops.compute_global_topk_indices_and_lens(
            self.topk, self.t2r, self.index_table, w.index_cache.block_size, self.valid,
            out=self.global_topk, lens=self.global_lens)))
        L.append(("dequantize_and_gather_k_cache[mxfp4]", lambda: ops.dequantize_and_gather_k_cache(
            self.gathered_index, self.index_cache, self.global_topk, w.index_cache.block_size,
            record=ops.PSK_REC_MXFP4)))
        return L

    def fused_launches(self) -> list[tuple[str, Callable[[], None]]]:
        """The fused step as (kernel name, launch) pairs, in serial order."""
        w = self.w
        base = dict(self.launches())
        L: list[tuple[str, Callable[[], None]]] = []
        for name in ("quantize_and_insert_k_cache", "write_indexer_mxfp4_cache",
                     "combine_topk_swa_indices", "compute_global_topk_indices_and_lens"):
            if name in base:
                L.append((name, base[name]))
        if w.has_fp8:
            W = w.window
            L.append(("dequantize_and_gather_k_cache_window[swa]",
                      lambda: ops.dequantize_and_gather_k_cache_window(
                          self.gathered[:, :W, :], self.swa_cache, self.qsl, self.seq_lens,
                          self.t2r, self.replay, self.swa_bt, w.swa_cache.block_size, W,
                          rope_dim=w.rope_dim, is_valid_token=self.valid)))
            comp_table = self.comp_bt if self.comp_bt is not None else self.swa_bt
            L.append(("dequantize_and_gather_k_cache_topk[topk]",
                      lambda: ops.dequantize_and_gather_k_cache_topk(
                          self.gathered[:, W:W + w.topk, :], self.comp_cache, self.topk, self.t2r,
                          comp_table, w.comp_cache.block_size, rope_dim=w.rope_dim,
                          num_reqs=w.num_reqs, is_valid_token=self.valid)))
        L.append(("dequantize_and_gather_k_cache_topk[mxfp4]",
                  lambda: ops.dequantize_and_gather_k_cache_topk(
                      self.gathered_index, self.index_cache, self.topk, self.t2r,
                      self.index_table, w.index_cache.block_size, record=ops.PSK_REC_MXFP4,
                      num_reqs=w.num_reqs, is_valid_token=self.valid)))
        return L

    def _fused_step(self, concurrent: bool, hooks: dict) -> None:
        L = self.fused_launches()
        fns = dict(L)

        def run(name):
            if name not in fns:
                return
            pre, post = hooks.get(name, (None, None))
            if pre:
                pre()
            fns[name]()
            if post:
                post()

        if not concurrent:
            for name, _ in L:
                run(name)
            return
        main = torch.cuda.current_stream(self.dev)
        if not hasattr(self, "_side3"):
            self._side3 = tuple(torch.cuda.Stream(self.dev) for _ in range(3))
        sa, sb, sc = self._side3
        fork = torch.cuda.Event()
        fork.record(main)
        # the longest gather is issued first so that its CTAs are resident
        # before the side chains take SMs
        run("dequantize_and_gather_k_cache_topk[topk]")
        done = []
        # chains captured in this order: the index builders, the MXFP4 chain,
        # then the insert and the window gather
        for st, names in ((sc, ("combine_topk_swa_indices",
                                "compute_global_topk_indices_and_lens")),
                          (sb, ("write_indexer_mxfp4_cache",
                                "dequantize_and_gather_k_cache_topk[mxfp4]")),
                          (sa, ("quantize_and_insert_k_cache",
                                "dequantize_and_gather_k_cache_window[swa]"))):
            st.wait_event(fork)
            with torch.cuda.stream(st):
                for n in names:
                    run(n)
                ev = torch.cuda.Event()
                ev.record(st)
                done.append(ev)
        for ev in done:
            main.wait_event(ev)

    def step(self, concurrent: bool = False, hooks: Optional[dict] = None,
             path: str = "index") -> None:
        """Launch one step.  ``hooks`` maps a kernel name to a pair of callables
        run on that kernel's stream just before and just after its launch
        (used to bracket one kernel with timing events)."""
        if path == "workspace":
            return self._workspace_step(concurrent, hooks or {})
        if path == "fused":
            return self._fused_step(concurrent, hooks or {})
        if path == "dense":
            return self._dense_step(concurrent, hooks or {})
        if path == "dense_fused":
            return self._dense_fused_step(concurrent, hooks or {})
        if path in ("indexer_fp8", "indexer_store"):
            return self._indexer_step(concurrent, hooks or {}, path.split("_")[1])
        if path == "compressor":
            return self._compressor_step(concurrent, hooks or {})
        L = dict(self.launches())
        hooks = hooks or {}

        def run(name):
            pre, post = hooks.get(name, (None, None))
            if pre:
                pre()
            L[name]()
            if post:
                post()

        if not concurrent:
            for name in L:
                run(name)
            return
        main = torch.cuda.current_stream(self.dev)
        if not hasattr(self, "_side"):
            self._side = (torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev))
        sa, sb = self._side
        fork = torch.cuda.Event()
        fork.record(main)
        sa.wait_event(fork)
        sb.wait_event(fork)
        with torch.cuda.stream(sb):
            run("compute_global_topk_indices_and_lens")
            if "write_indexer_mxfp4_cache" in L:
                run("write_indexer_mxfp4_cache")
            run("dequantize_and_gather_k_cache[mxfp4]")
            done_b = torch.cuda.Event()
            done_b.record(sb)
        if self.w.has_fp8 and self.gather_as_pair:
            # one programmatic (PDL) chain: each kernel waits for its
            # predecessor's grid before its first global access, so the gather
            # sees the insert's rows through the index build
            run("quantize_and_insert_k_cache")
            run("combine_topk_swa_indices")
            run("dequantize_and_gather_k_cache_pair")
        elif self.w.has_fp8:
            with torch.cuda.stream(sa):
                run("quantize_and_insert_k_cache")
            run("combine_topk_swa_indices")
            built = torch.cuda.Event()
            built.record(main)
            with torch.cuda.stream(sa):
                sa.wait_event(built)
                run("dequantize_and_gather_k_cache[swa]")
                done_a = torch.cuda.Event()
                done_a.record(sa)
            run("dequantize_and_gather_k_cache[topk]")
            main.wait_event(done_a)
        main.wait_event(done_b)

    def _workspace_step(self, concurrent: bool, hooks: dict) -> None:
        L = dict(self.workspace_launches())

        def run(name):
            pre, post = hooks.get(name, (None, None))
            if pre:
                pre()
            L[name]()
            if post:
                post()

        if not concurrent:
            for name in L:
                run(name)
            return
        main = torch.cuda.current_stream(self.dev)
        if not hasattr(self, "_side"):
            self._side = (torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev))
        sa, sb = self._side
        fork = torch.cuda.Event()
        fork.record(main)
        sa.wait_event(fork)
        sb.wait_event(fork)
        with torch.cuda.stream(sb):
            run("write_indexer_mxfp4_cache")
            run("indexer_mxfp4_paged_gather")
            done_b = torch.cuda.Event()
            done_b.record(sb)
        with torch.cuda.stream(sa):
            run("quantize_and_insert_k_cache")
            run("dequantize_and_gather_k_cache_ranges[swa]")
            done_a = torch.cuda.Event()
            done_a.record(sa)
        run("dequantize_and_gather_k_cache_ranges[compressed]")
        run("combine_topk_swa_workspace_indices")
        main.wait_event(done_a)
        main.wait_event(done_b)


    def _indexer_step(self, concurrent: bool, hooks: dict, variant: str) -> None:
        L = self.indexer_launches(variant)
        names = [n for n, _ in L]
        fns = dict(L)

        def run(name):
            pre, post = hooks.get(name, (None, None))
            if pre:
                pre()
            fns[name]()
            if post:
                post()

        if not concurrent:
            for name in names:
                run(name)
            return
        main = torch.cuda.current_stream(self.dev)
        if not hasattr(self, "_side"):
            self._side = (torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev))
        sa, sb = self._side
        fork = torch.cuda.Event()
        fork.record(main)
        sa.wait_event(fork)
        sb.wait_event(fork)
        with torch.cuda.stream(sb):
            run(names[1])
            done_b = torch.cuda.Event()
            done_b.record(sb)
        with torch.cuda.stream(sa):
            run(names[0])
            done_a = torch.cuda.Event()
            done_a.record(sa)
        main.wait_event(done_a)
        main.wait_event(done_b)
        run(names[2])

    def _compressor_step(self, concurrent: bool, hooks: dict) -> None:
        L = self.compressor_launches()
        fns = dict(L)

        def run(name):
            pre, post = hooks.get(name, (None, None))
            if pre:
                pre()
            fns[name]()
            if post:
                post()

        if not concurrent:
            for name, _ in L:
                run(name)
            return
        main = torch.cuda.current_stream(self.dev)
        if not hasattr(self, "_side"):
            self._side = (torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev))
        sa, _ = self._side
        fork = torch.cuda.Event()
        fork.record(main)
        sa.wait_event(fork)
        with torch.cuda.stream(sa):
            run("save_compressor_state[128]")
            run("compress_kv_cache_insert[128]")
            done = torch.cuda.Event()
            done.record(sa)
        run("save_compressor_state[4]")
        run("compress_kv_cache_insert[4]")
        main.wait_event(done)

    def _dense_step(self, concurrent: bool, hooks: dict) -> None:
        L = dict(self.dense_launches())

        def run(name):
            pre, post = hooks.get(name, (None, None))
            if pre:
                pre()
            L[name]()
            if post:
                post()

        if not concurrent:
            for name in L:
                run(name)
            return
        main = torch.cuda.current_stream(self.dev)
        if not hasattr(self, "_side"):
            self._side = (torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev))
        sa, sb = self._side
        fork = torch.cuda.Event()
        fork.record(main)
        sa.wait_event(fork)
        sb.wait_event(fork)
        with torch.cuda.stream(sb):
            run("compute_dense_compressed_indices_and_lens")
            run("dequantize_and_gather_k_cache[compressed]")
            done_b = torch.cuda.Event()
            done_b.record(sb)
        with torch.cuda.stream(sa):
            run("quantize_and_insert_k_cache")
            inserted = torch.cuda.Event()
            inserted.record(sa)
        run("decode_swa_indices_and_lens")
        main.wait_event(inserted)
        run("dequantize_and_gather_k_cache[swa]")
        main.wait_event(done_b)


    def _dense_fused_step(self, concurrent: bool, hooks: dict) -> None:
        L = self.dense_fused_launches()
        fns = dict(L)

        def run(name):
            pre, post = hooks.get(name, (None, None))
            if pre:
                pre()
            fns[name]()
            if post:
                post()

        if not concurrent:
            for name, _ in L:
                run(name)
            return
        main = torch.cuda.current_stream(self.dev)
        if not hasattr(self, "_side3"):
            self._side3 = tuple(torch.cuda.Stream(self.dev) for _ in range(3))
        sa, sb, _ = self._side3
        fork = torch.cuda.Event()
        fork.record(main)
        # the compressed entries first (they read no row this step writes), then
        # the builders' chain, then the insert and the window gather
        run("dequantize_and_gather_k_cache_dense[compressed]")
        done = []
        for st, names in ((sb, ("decode_swa_indices_and_lens",
                                "compute_dense_compressed_indices_and_lens")),
                          (sa, ("quantize_and_insert_k_cache",
                                "dequantize_and_gather_k_cache_window[swa]"))):
            st.wait_event(fork)
            with torch.cuda.stream(st):
                for n in names:
                    run(n)
                ev = torch.cuda.Event()
                ev.record(st)
                done.append(ev)
        for ev in done:
            main.wait_event(ev)


def workspace_geometry(w: Workload) -> dict:
    """Per-request gather lengths and the workspace shape of the prefill path
    (TokenSpeed backends/deepseek_v4.py, _prefill_workspace): gather_lens =
    query_lens + min(prefix, W - 1); compressed_lens = seq_lens // ratio;
    compressed_base = max compressed length; workspace_width = compressed_base +
    max gather length; cu_compressed = prefix sums of compressed_lens."""
    seq = w.seq_lens.astype(np.int64)
    qlen = np.diff(w.query_start_loc).astype(np.int64)
    glen = qlen + np.minimum(seq - qlen, max(w.window - 1, 0))
    lc = seq // w.compress_ratio
    cb = int(lc.max()) if lc.size else 0
    return {"gather_lens": glen.astype(np.int32), "compressed_lens": lc.astype(np.int32),
            "compressed_base": cb,
            "workspace_width": max(1, cb + (int(glen.max()) if glen.size else 0)),
            "cu_compressed": np.concatenate([[0], np.cumsum(lc)]).astype(np.int32)}
