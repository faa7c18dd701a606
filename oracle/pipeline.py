"""One pipeline step computed by the CPU oracle (test infrastructure only).

Mirrors the step order of the device pipeline on host numpy arrays, calling
only the oracle: FP8 insert, MXFP4 insert, fused index build, the two-part FP8
gather, the global top-k mapping and the MXFP4 gather.  For large workloads the
gathers can be restricted to a sample of tokens (every other output is still
computed in full).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from . import (REC_FP8_DS_MLA, REC_MXFP4, combine_topk_swa_indices,
               combine_topk_swa_workspace_indices, compute_dense_compressed_indices_and_lens,
               compute_global_topk_indices_and_lens, decode_swa_indices_and_lens,
               dequantize_and_gather_k_cache, dequantize_and_gather_k_cache_ranges,
               compress_kv_cache_insert, indexer_k_norm_rope_store, indexer_mxfp4_paged_gather,
               save_compressor_state,
               quantize_and_insert_k_cache, write_indexer_fp8_cache, write_indexer_mxfp4_cache)

REC_FP8_INDEXER = 2


def run_step(w, swa_cache: Optional[np.ndarray], comp_cache: Optional[np.ndarray],
             index_cache: Optional[np.ndarray],
             sample_tokens: Optional[Sequence[int]] = None) -> dict:
    """Run one step; caches are updated in place.  Returns the outputs."""
    res: dict = {"err": 0}
    if w.has_fp8:
        res["err"] += quantize_and_insert_k_cache(
            w.k, w.insert_slots, swa_cache, w.swa_cache.block_size, w.head_dim, w.rope_dim)
    if w.index_k is not None:
        res["err"] += write_indexer_mxfp4_cache(
            w.index_k, w.index_insert_slots, index_cache, w.index_cache.block_size,
            w.index_head_dim)
    toks = None if sample_tokens is None else np.asarray(sample_tokens, dtype=np.int64)
    if w.has_fp8:
        W = w.window
        si, lens = combine_topk_swa_indices(
            w.query_start_loc, w.seq_lens, w.token_to_req, w.replay_start, w.swa_block_table,
            w.swa_cache.block_size, w.comp_block_table, w.comp_cache.block_size, W,
            w.compress_ratio, w.topk_local, is_valid_token=w.is_valid_token)
        res["sparse_indices"], res["lens"] = si, lens
        rows = si if toks is None else si[toks]
        g_swa = dequantize_and_gather_k_cache(swa_cache, w.swa_cache.block_size, REC_FP8_DS_MLA,
                                              w.head_dim, w.rope_dim, np.ascontiguousarray(rows[:, :W]))
        g_top = dequantize_and_gather_k_cache(comp_cache, w.comp_cache.block_size, REC_FP8_DS_MLA,
                                              w.head_dim, w.rope_dim, np.ascontiguousarray(rows[:, W:]))
        res["gathered"] = np.concatenate([g_swa, g_top], axis=1)
    table = w.comp_block_table if w.comp_block_table is not None else w.swa_block_table
    gt, gl = compute_global_topk_indices_and_lens(
        w.topk_local, w.token_to_req, table, w.index_cache.block_size,
        is_valid_token=w.is_valid_token)
    res["global_topk"], res["global_lens"] = gt, gl
    rows = gt if toks is None else gt[toks]
    res["gathered_index"] = dequantize_and_gather_k_cache(
        index_cache, w.index_cache.block_size, REC_MXFP4, w.index_head_dim, 0,
        np.ascontiguousarray(rows))
    return res


def run_workspace_step(w, geom: dict, swa_cache, comp_cache, index_cache) -> dict:
    """The prefill workspace step (``geom`` = the workspace geometry of the
    batch: gather_lens, compressed_lens, compressed_base, workspace_width,
    cu_compressed).  Caches are updated in place."""
    res: dict = {"err": 0}
    res["err"] += quantize_and_insert_k_cache(
        w.k, w.insert_slots, swa_cache, w.swa_cache.block_size, w.head_dim, w.rope_dim)
    res["err"] += write_indexer_mxfp4_cache(
        w.index_k, w.index_insert_slots, index_cache, w.index_cache.block_size,
        w.index_head_dim)
    cb, ww = geom["compressed_base"], geom["workspace_width"]
    table = w.comp_block_table if w.comp_block_table is not None else w.swa_block_table
    comp_part = np.zeros((w.num_reqs, cb, w.head_dim), np.uint16)
    dequantize_and_gather_k_cache_ranges(comp_part, comp_cache, w.comp_cache.block_size,
                                         REC_FP8_DS_MLA, w.head_dim, w.rope_dim,
                                         geom["compressed_lens"], None, table, 0)
    ws = np.zeros((w.num_reqs, ww, w.head_dim), np.uint16)
    dequantize_and_gather_k_cache_ranges(ws, swa_cache, w.swa_cache.block_size, REC_FP8_DS_MLA,
                                         w.head_dim, w.rope_dim, w.seq_lens,
                                         geom["gather_lens"], w.swa_block_table, cb)
    res["workspace_compressed"] = comp_part
    res["workspace_window"] = ws[:, cb:]
    res["ws_indices"], res["ws_lens"] = combine_topk_swa_workspace_indices(
        w.query_start_loc, w.seq_lens, geom["gather_lens"], w.token_to_req, w.window,
        w.compress_ratio, w.topk_local, ww, cb, is_valid_token=w.is_valid_token)
    res["raw_values"], res["raw_scales"] = indexer_mxfp4_paged_gather(
        index_cache, w.index_cache.block_size, w.index_head_dim, table, geom["cu_compressed"])
    return res


def run_dense_step(w, swa_cache, comp_cache) -> dict:
    """The dense (no top-k) decode step: FP8 insert, window-only slot indices,
    every visible compressed entry's slot, and the two-part gather into
    [T, W + dense_width, D].  Caches are updated in place."""
    res: dict = {"err": 0}
    res["err"] += quantize_and_insert_k_cache(
        w.k, w.insert_slots, swa_cache, w.swa_cache.block_size, w.head_dim, w.rope_dim)
    res["swa_indices"], res["swa_lens"] = decode_swa_indices_and_lens(
        w.query_start_loc, w.seq_lens, w.token_to_req, w.swa_block_table,
        w.swa_cache.block_size, w.window, is_valid_token=w.is_valid_token)
    res["dense_indices"], res["dense_lens"] = compute_dense_compressed_indices_and_lens(
        w.positions, w.token_to_req, w.comp_block_table, w.comp_cache.block_size,
        w.compress_ratio, w.dense_width, num_reqs=w.num_reqs, is_valid_token=w.is_valid_token)
    g_swa = dequantize_and_gather_k_cache(swa_cache, w.swa_cache.block_size, REC_FP8_DS_MLA,
                                          w.head_dim, w.rope_dim, res["swa_indices"])
    g_cmp = dequantize_and_gather_k_cache(comp_cache, w.comp_cache.block_size, REC_FP8_DS_MLA,
                                          w.head_dim, w.rope_dim, res["dense_indices"])
    res["gathered"] = np.concatenate([g_swa, g_cmp], axis=1)
    return res


def run_indexer_step(w, variant: str, cache, inputs: dict, sample_tokens=None) -> dict:
    """The indexer step with the FP8 indexer record ("fp8") or the fused
    norm-RoPE-MXFP4 store ("store") as the key writer; ``cache`` is that
    writer's cache (updated in place); ``inputs`` holds positions, cos_sin,
    weight and eps for "store"."""
    res: dict = {}
    bs = w.index_cache.block_size
    if variant == "fp8":
        res["err"] = write_indexer_fp8_cache(w.index_k, w.index_insert_slots, cache, bs,
                                             w.index_head_dim)
        rec = REC_FP8_INDEXER
    else:
        res["err"] = indexer_k_norm_rope_store(
            w.index_k, inputs["positions"], inputs["cos_sin"], inputs["weight"], inputs["eps"],
            w.index_insert_slots, 1, REC_MXFP4, cache, bs)
        rec = REC_MXFP4
    table = w.comp_block_table if w.comp_block_table is not None else w.swa_block_table
    gt, gl = compute_global_topk_indices_and_lens(w.topk_local, w.token_to_req, table, bs,
                                                  is_valid_token=w.is_valid_token)
    res["global_topk"], res["global_lens"] = gt, gl
    toks = None if sample_tokens is None else np.asarray(sample_tokens, dtype=np.int64)
    rows = gt if toks is None else gt[toks]
    res["gathered_index"] = dequantize_and_gather_k_cache(cache, bs, rec, w.index_head_dim, 0,
                                                          np.ascontiguousarray(rows))
    return res


def run_compressor_step(w, layers, states, kv_caches, eps: float = 1e-6) -> dict:
    """The compressor step: for each layer (compressor_inputs of a ratio), save
    the state of every token, then insert the compressed rows of the tokens
    that close a group.  ``states`` and ``kv_caches`` are updated in place."""
    res: dict = {"err": 0}
    for c, st, kvc in zip(layers, states, kv_caches):
        res["err"] += save_compressor_state(c["kv"], c["score"], c["ape"], c["state_slots"],
                                            c["positions"], c["ratio"], st, c["state_bs"])
        res["err"] += compress_kv_cache_insert(
            st, w.token_to_req, c["positions"], c["state_slots"], c["state_table"], c["state_bs"],
            c["weight"], eps, c["cos_sin"], kvc, c["kv_slots"], c["kv_geom"].block_size,
            c["ratio"], c["overlap"])
    return res
