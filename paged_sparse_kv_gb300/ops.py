"""PyTorch-facing wrappers of the libpsk C ABI (same names as include/psk.h).

Argument marshalling only: every step runs in the CUDA kernels of libpsk.
Tensors must live on a CUDA device; each call launches on the current torch
stream of that device and returns without synchronising.  Errors from the
library raise :class:`PskError`.

Cache tensors are uint8 with pages along dim 0: ``num_pages = cache.shape[0]``
and ``page_stride = cache.stride(0)`` bytes (a 2-D ``[pages, bytes]`` tensor or
a 3-D ``[pages, block_size, record_bytes]`` view both work).
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _abi
from ._abi import PSK_REC_FP8_DS_MLA, PSK_REC_FP8_INDEXER, PSK_REC_MXFP4, PskError  # noqa: F401


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(dev: torch.device) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def _call(dev: torch.device, name: str, *args) -> None:
    """Call a libpsk entry point on ``dev``'s current stream with ``dev`` as
    the current CUDA device (the library launches, sizes grids and sets kernel
    attributes on the current device)."""
    if torch.cuda.current_device() != dev.index:
        with torch.cuda.device(dev):
            _abi.call(name, *args, _stream(dev))
    else:
        _abi.call(name, *args, _stream(dev))


def _need_cuda(*ts):
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("libpsk operates on CUDA tensors only (no CPU fallback)")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"all tensors of one call must be on one device ({dev} and "
                             f"{t.device})")


def _need(t: torch.Tensor, dtype: torch.dtype, name: str):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _pages(cache: torch.Tensor):
    _need(cache, torch.uint8, "cache")
    if cache.dim() < 2 or cache.shape[0] == 0 or not cache[0].is_contiguous():
        raise ValueError("cache must be [num_pages >= 1, ...] uint8 with contiguous pages")
    if cache.shape[0] == 1:  # a size-1 dim may carry any stride (0 from broadcasting)
        return 1, max(cache.stride(0), cache[0].numel())
    return cache.shape[0], cache.stride(0)


def _rows(t: torch.Tensor, name: str):
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.numel() == 0:
        return t.shape[1]
    if t.stride(1) != 1 and t.shape[1] > 1:
        raise ValueError(f"{name} must have unit inner stride")
    if t.shape[0] == 1:  # a size-1 dim may carry any stride (0 from broadcasting)
        return max(t.stride(0), t.shape[1])
    return t.stride(0)


def quantize_and_insert_k_cache(k: torch.Tensor, k_cache: torch.Tensor,
                                slot_mapping: torch.Tensor, block_size: int = 64, *,
                                rope_dim: int = 64, is_ue8m0: bool = True,
                                head_dim: Optional[int] = None,
                                err_count: Optional[torch.Tensor] = None) -> None:
    """FP8 (fp8_ds_mla) quantize + paged insert of ``k`` [N', D] bf16 at
    ``slot_mapping`` [N] int64 (N <= N'; -1 skips)."""
    _need_cuda(k, k_cache, slot_mapping, err_count)
    _need(k, torch.bfloat16, "k")
    _need(slot_mapping, torch.int64, "slot_mapping")
    if err_count is not None:
        _need(err_count, torch.int32, "err_count")
    if slot_mapping.dim() != 1 or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be 1-D contiguous")
    D = k.shape[1] if head_dim is None else head_dim
    num_pages, page_stride = _pages(k_cache)
    _call(k.device, "quantize_and_insert_k_cache", _ptr(k), _rows(k, "k"), _ptr(slot_mapping),
          slot_mapping.shape[0], _ptr(k_cache), num_pages, page_stride, block_size, D,
          rope_dim, int(bool(is_ue8m0)), _ptr(err_count))


def write_indexer_mxfp4_cache(index_k: torch.Tensor, cache: torch.Tensor,
                              slot_mapping: torch.Tensor, block_size: int = 64, *,
                              err_count: Optional[torch.Tensor] = None) -> None:
    """MXFP4 quantize + paged insert of indexer keys ``index_k`` [N', D] bf16."""
    _need_cuda(index_k, cache, slot_mapping, err_count)
    _need(index_k, torch.bfloat16, "index_k")
    _need(slot_mapping, torch.int64, "slot_mapping")
    if slot_mapping.dim() != 1 or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be 1-D contiguous")
    num_pages, page_stride = _pages(cache)
    _call(index_k.device, "write_indexer_mxfp4_cache", _ptr(index_k), _rows(index_k, "index_k"),
          _ptr(slot_mapping), slot_mapping.shape[0], _ptr(cache), num_pages, page_stride,
          block_size, index_k.shape[1], _ptr(err_count))


def compute_global_topk_indices_and_lens(topk_indices: torch.Tensor,
                                         token_to_req_indices: torch.Tensor,
                                         block_table: torch.Tensor, block_size: int,
                                         is_valid_token: Optional[torch.Tensor] = None, *,
                                         base_offsets: Optional[torch.Tensor] = None,
                                         out: Optional[torch.Tensor] = None,
                                         lens: Optional[torch.Tensor] = None):
    """Map local top-k [T, K] to global slots; returns (indices [T, K], lens [T])."""
    _need_cuda(topk_indices, token_to_req_indices, block_table, is_valid_token, base_offsets)
    for t, n in ((topk_indices, "topk_indices"), (token_to_req_indices, "token_to_req"),
                 (block_table, "block_table")):
        _need(t, torch.int32, n)
    T, K = topk_indices.shape
    if out is None:
        out = torch.empty((T, K), dtype=torch.int32, device=topk_indices.device)
    if lens is None:
        lens = torch.empty((T,), dtype=torch.int32, device=topk_indices.device)
    valid = None if is_valid_token is None else is_valid_token.to(torch.uint8)
    _call(topk_indices.device, "compute_global_topk_indices_and_lens", _ptr(topk_indices),
          _rows(topk_indices, "topk_indices"), T, K, _ptr(token_to_req_indices),
          _ptr(block_table), _rows(block_table, "block_table"), block_table.shape[1],
          block_table.shape[0], block_size, _ptr(base_offsets), _ptr(valid), _ptr(out),
          _rows(out, "out"), _ptr(lens))
    return out, lens


def combine_topk_swa_indices(query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
                             token_to_req_indices: torch.Tensor,
                             replay_start: Optional[torch.Tensor],
                             swa_block_table: torch.Tensor, swa_block_size: int,
                             compressed_block_table: Optional[torch.Tensor],
                             compressed_block_size: int, window_size: int,
                             compress_ratio: int, topk_indices: torch.Tensor, *,
                             swa_base_offsets: Optional[torch.Tensor] = None,
                             compressed_base_offsets: Optional[torch.Tensor] = None,
                             is_valid_token: Optional[torch.Tensor] = None,
                             num_tokens: Optional[int] = None,
                             out: Optional[torch.Tensor] = None,
                             lens: Optional[torch.Tensor] = None):
    """Fused sparse-index build; returns (sparse_indices [T, W + roundup4(K)], lens [T])."""
    _need_cuda(query_start_loc, seq_lens, token_to_req_indices, replay_start, swa_block_table,
               compressed_block_table, topk_indices, is_valid_token)
    dev = topk_indices.device
    T = topk_indices.shape[0] if num_tokens is None else num_tokens
    K = topk_indices.shape[1]
    width = window_size + (K + 3) // 4 * 4
    if out is None:
        out = torch.empty((T, width), dtype=torch.int32, device=dev)
    if lens is None:
        lens = torch.empty((T,), dtype=torch.int32, device=dev)
    cbt = compressed_block_table
    valid = None if is_valid_token is None else is_valid_token.to(torch.uint8)
    _call(dev, "combine_topk_swa_indices", _ptr(query_start_loc), _ptr(seq_lens),
          _ptr(token_to_req_indices), _ptr(replay_start), seq_lens.shape[0], T,
          _ptr(swa_block_table), _rows(swa_block_table, "swa_block_table"),
          swa_block_table.shape[1], _ptr(swa_base_offsets), swa_block_size,
          _ptr(cbt), _rows(cbt, "compressed_block_table") if cbt is not None else 0,
          cbt.shape[1] if cbt is not None else 0, _ptr(compressed_base_offsets),
          compressed_block_size, window_size, compress_ratio, _ptr(topk_indices),
          _rows(topk_indices, "topk_indices"), K, _ptr(valid), _ptr(out), _rows(out, "out"),
          _ptr(lens))
    return out, lens


def dequantize_and_gather_k_cache(out: torch.Tensor, cache: torch.Tensor,
                                  indices: torch.Tensor, block_size: int, *,
                                  record: int = PSK_REC_FP8_DS_MLA, rope_dim: int = 64,
                                  is_ue8m0: bool = True) -> torch.Tensor:
    """Gather + dequantize rows ``indices`` [T, C] into ``out`` [T, C, D] bf16
    (``out`` may be a strided view, e.g. a column range of a wider output)."""
    _need_cuda(out, cache, indices)
    _need(out, torch.bfloat16, "out")
    _need(indices, torch.int32, "indices")
    if out.dim() != 3 or out.stride(2) != 1:
        raise ValueError("out must be [T, C, D] with unit inner stride")
    T, C = indices.shape
    if out.shape[0] != T or out.shape[1] != C:
        raise ValueError(f"out {tuple(out.shape)} does not match indices {tuple(indices.shape)}")
    num_pages, page_stride = _pages(cache)
    _call(out.device, "dequantize_and_gather_k_cache", _ptr(out), out.stride(0), out.stride(1),
          _ptr(cache), num_pages, page_stride, block_size, record, out.shape[2],
          rope_dim if record == PSK_REC_FP8_DS_MLA else 0, int(bool(is_ue8m0)),
          _ptr(indices), _rows(indices, "indices"), T, C)
    return out


# ---- prefill workspace path ------------------------------------------------------------

def dequantize_and_gather_k_cache_ranges(out: torch.Tensor, cache: torch.Tensor,
                                         seq_lens: torch.Tensor,
                                         gather_lens: Optional[torch.Tensor],
                                         block_table: torch.Tensor, block_size: int,
                                         offset: int, *, rope_dim: int = 64,
                                         is_ue8m0: bool = True,
                                         base_offsets: Optional[torch.Tensor] = None
                                         ) -> torch.Tensor:
    """Range-form gather into ``out`` [R, rows, D] bf16 (a workspace); see psk.h."""
    _need_cuda(out, cache, seq_lens, gather_lens, block_table, base_offsets)
    _need(out, torch.bfloat16, "out")
    if out.dim() != 3 or out.stride(2) != 1:
        raise ValueError("out must be [R, rows, D] with unit inner stride")
    for t, n in ((seq_lens, "seq_lens"), (block_table, "block_table")):
        _need(t, torch.int32, n)
    num_pages, page_stride = _pages(cache)
    _call(out.device, "dequantize_and_gather_k_cache_ranges",
          _ptr(out), out.stride(0), out.stride(1),
          out.shape[1], _ptr(cache), num_pages, page_stride, block_size,
          PSK_REC_FP8_DS_MLA, out.shape[2], rope_dim, int(bool(is_ue8m0)), _ptr(seq_lens),
          _ptr(gather_lens), _ptr(block_table), _rows(block_table, "block_table"),
          block_table.shape[1], _ptr(base_offsets), seq_lens.shape[0], offset)
    return out


def combine_topk_swa_workspace_indices(topk_indices: torch.Tensor,
                                       query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
                                       gather_lens: torch.Tensor, token_to_req: torch.Tensor,
                                       window_size: int, compress_ratio: int,
                                       workspace_width: int, compressed_base: int, *,
                                       is_valid_token: Optional[torch.Tensor] = None,
                                       out: Optional[torch.Tensor] = None,
                                       lens: Optional[torch.Tensor] = None):
    """Workspace-relative index build; returns (indices [T, W + roundup4(K)], lens [T])."""
    _need_cuda(topk_indices, query_start_loc, seq_lens, gather_lens, token_to_req,
               is_valid_token)
    dev = topk_indices.device
    T, K = topk_indices.shape
    width = window_size + (K + 3) // 4 * 4
    if out is None:
        out = torch.empty((T, width), dtype=torch.int32, device=dev)
    if lens is None:
        lens = torch.empty((T,), dtype=torch.int32, device=dev)
    valid = None if is_valid_token is None else is_valid_token.to(torch.uint8)
    _call(dev, "combine_topk_swa_workspace_indices", _ptr(query_start_loc), _ptr(seq_lens),
          _ptr(gather_lens), _ptr(token_to_req), seq_lens.shape[0], T, window_size,
          compress_ratio, _ptr(topk_indices), _rows(topk_indices, "topk_indices"), K,
          workspace_width, compressed_base, _ptr(valid), _ptr(out), _rows(out, "out"),
          _ptr(lens))
    return out, lens


def indexer_mxfp4_paged_gather(cache: torch.Tensor, block_table: torch.Tensor,
                               cu_seq_lens: torch.Tensor, block_size: int, head_dim: int,
                               total_rows: int, values_out: Optional[torch.Tensor] = None,
                               scales_out: Optional[torch.Tensor] = None):
    """Raw MXFP4 rows over request ranges; returns (values [N, D/2], scales [N, D/32]) uint8."""
    _need_cuda(cache, block_table, cu_seq_lens)
    dev = cache.device
    if values_out is None:
        values_out = torch.empty((total_rows, head_dim // 2), dtype=torch.uint8, device=dev)
    if scales_out is None:
        scales_out = torch.empty((total_rows, head_dim // 32), dtype=torch.uint8, device=dev)
    num_pages, page_stride = _pages(cache)
    _call(dev, "indexer_mxfp4_paged_gather", _ptr(values_out), _ptr(scales_out), _ptr(cache),
          num_pages, page_stride, block_size, head_dim, _ptr(block_table),
          _rows(block_table, "block_table"), block_table.shape[1], _ptr(cu_seq_lens),
          cu_seq_lens.shape[0] - 1, total_rows)
    return values_out, scales_out


# ---- dense builders ---------------------------------------------------------------------

def decode_swa_indices_and_lens(query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
                                token_to_req: torch.Tensor, block_table: torch.Tensor,
                                block_size: int, window_size: int, *,
                                base_offsets: Optional[torch.Tensor] = None,
                                is_valid_token: Optional[torch.Tensor] = None,
                                out: Optional[torch.Tensor] = None,
                                lens: Optional[torch.Tensor] = None):
    """Window-only slot indices of decode tokens; returns (indices [T, W], lens [T])."""
    _need_cuda(query_start_loc, seq_lens, token_to_req, block_table, base_offsets,
               is_valid_token)
    dev = token_to_req.device
    T = token_to_req.shape[0]
    if out is None:
        out = torch.empty((T, window_size), dtype=torch.int32, device=dev)
    if lens is None:
        lens = torch.empty((T,), dtype=torch.int32, device=dev)
    valid = None if is_valid_token is None else is_valid_token.to(torch.uint8)
    _call(dev, "decode_swa_indices_and_lens", _ptr(query_start_loc), _ptr(seq_lens),
          _ptr(token_to_req), seq_lens.shape[0], T, _ptr(block_table),
          _rows(block_table, "block_table"), block_table.shape[1], _ptr(base_offsets),
          block_size, window_size, _ptr(valid), _ptr(out), _rows(out, "out"), _ptr(lens))
    return out, lens


def compute_dense_compressed_indices_and_lens(positions: torch.Tensor,
                                              token_to_req: torch.Tensor,
                                              block_table: torch.Tensor, block_size: int,
                                              compress_ratio: int, width: int, *,
                                              num_reqs: Optional[int] = None,
                                              base_offsets: Optional[torch.Tensor] = None,
                                              is_valid_token: Optional[torch.Tensor] = None,
                                              out: Optional[torch.Tensor] = None,
                                              lens: Optional[torch.Tensor] = None):
    """Slots of every visible compressed entry; returns (indices [T, width], lens [T])."""
    _need_cuda(positions, token_to_req, block_table, base_offsets, is_valid_token)
    _need(positions, torch.int64, "positions")
    dev = positions.device
    T = positions.shape[0]
    if out is None:
        out = torch.empty((T, width), dtype=torch.int32, device=dev)
    if lens is None:
        lens = torch.empty((T,), dtype=torch.int32, device=dev)
    valid = None if is_valid_token is None else is_valid_token.to(torch.uint8)
    R = block_table.shape[0] if num_reqs is None else num_reqs
    _call(dev, "compute_dense_compressed_indices_and_lens", _ptr(positions), T,
          _ptr(token_to_req), R, _ptr(block_table), _rows(block_table, "block_table"),
          block_table.shape[1], _ptr(base_offsets), block_size, compress_ratio, width,
          _ptr(valid), _ptr(out), _rows(out, "out"), _ptr(lens))
    return out, lens


def build_dense_prefill_local_compressed_indices(positions: torch.Tensor, compress_ratio: int,
                                                 width: int, *,
                                                 out: Optional[torch.Tensor] = None):
    """Request-local dense compressed indices [T, width] (j, or -1 past the visible count)."""
    _need_cuda(positions)
    _need(positions, torch.int64, "positions")
    dev = positions.device
    T = positions.shape[0]
    if out is None:
        out = torch.empty((T, width), dtype=torch.int32, device=dev)
    _call(dev, "build_dense_prefill_local_compressed_indices", _ptr(positions), T,
          compress_ratio, width, _ptr(out), _rows(out, "out"))
    return out


def combine_dense_swa_indices(positions: torch.Tensor, token_to_req: torch.Tensor,
                              seq_lens: torch.Tensor, gather_lens: torch.Tensor,
                              window_size: int, workspace_width: int, compressed_base: int = 0,
                              *, out: Optional[torch.Tensor] = None,
                              lens: Optional[torch.Tensor] = None):
    """Workspace-relative window indices of layers without a compressed cache;
    returns (indices [T, W], lens [T])."""
    _need_cuda(positions, token_to_req, seq_lens, gather_lens)
    _need(positions, torch.int64, "positions")
    dev = positions.device
    T = positions.shape[0]
    if out is None:
        out = torch.empty((T, window_size), dtype=torch.int32, device=dev)
    if lens is None:
        lens = torch.empty((T,), dtype=torch.int32, device=dev)
    _call(dev, "combine_dense_swa_indices", _ptr(positions), _ptr(token_to_req), _ptr(seq_lens),
          _ptr(gather_lens), seq_lens.shape[0], T, window_size, workspace_width,
          compressed_base, _ptr(out), _rows(out, "out"), _ptr(lens))
    return out, lens


# ---- indexer-key variants -------------------------------------------------------------

def write_indexer_fp8_cache(index_k: torch.Tensor, cache: torch.Tensor, slot_mapping: torch.Tensor,
                            block_size: int, *, err_count: Optional[torch.Tensor] = None) -> None:
    """FP8 indexer keys ([values | binary32 power-of-two scale] pages)."""
    _need_cuda(index_k, cache, slot_mapping, err_count)
    _need(index_k, torch.bfloat16, "index_k")
    _need(slot_mapping, torch.int64, "slot_mapping")
    num_pages, page_stride = _pages(cache)
    _call(index_k.device, "write_indexer_fp8_cache", _ptr(index_k), _rows(index_k, "index_k"),
          _ptr(slot_mapping), slot_mapping.shape[0], _ptr(cache), num_pages, page_stride,
          block_size, index_k.shape[1], _ptr(err_count))


def indexer_k_norm_rope_store(k_pre: torch.Tensor, positions: torch.Tensor,
                              cos_sin_cache: torch.Tensor, rms_norm_weight: torch.Tensor,
                              rms_norm_eps: float, k_cache: torch.Tensor,
                              kv_slot_mapping: torch.Tensor, compress_ratio: int,
                              use_fp4_cache: bool, block_size: int, *,
                              err_count: Optional[torch.Tensor] = None) -> None:
    """k_norm -> GPT-J RoPE -> MXFP4 / FP8 indexer record -> paged store of
    128-dim indexer keys (the vLLM op's argument names)."""
    _need_cuda(k_pre, positions, cos_sin_cache, rms_norm_weight, k_cache, kv_slot_mapping,
               err_count)
    _need(k_pre, torch.bfloat16, "k_pre")
    _need(positions, torch.int64, "positions")
    _need(cos_sin_cache, torch.float32, "cos_sin_cache")
    _need(rms_norm_weight, torch.float32, "rms_norm_weight")
    _need(kv_slot_mapping, torch.int64, "kv_slot_mapping")
    if k_pre.dim() != 2 or k_pre.shape[1] != 128:
        raise ValueError("k_pre must be [num_tokens, 128]")
    num_pages, page_stride = _pages(k_cache)
    record = PSK_REC_MXFP4 if use_fp4_cache else PSK_REC_FP8_INDEXER
    _call(k_pre.device, "indexer_k_norm_rope_store",
          _ptr(k_pre), _rows(k_pre, "k_pre"), _ptr(positions),
          _ptr(cos_sin_cache), _rows(cos_sin_cache, "cos_sin_cache"), cos_sin_cache.shape[0],
          _ptr(rms_norm_weight.contiguous()), float(rms_norm_eps), _ptr(kv_slot_mapping),
          kv_slot_mapping.shape[0], compress_ratio, record, _ptr(k_cache), num_pages,
          page_stride, block_size, _ptr(err_count))


# ---- compressed-KV producer -------------------------------------------------------------

def save_compressor_state(kv: torch.Tensor, score: torch.Tensor, ape: torch.Tensor,
                          state_cache: torch.Tensor, slot_mapping: torch.Tensor,
                          positions: torch.Tensor, block_size: int, compress_ratio: int, *,
                          err_count: Optional[torch.Tensor] = None) -> None:
    """state[slot] = [kv, score + ape[pos % ratio]] into the binary32 state cache
    [pages, block_size, 2 * state_width]."""
    _need_cuda(kv, score, ape, state_cache, slot_mapping, positions, err_count)
    for t, n in ((kv, "kv"), (score, "score"), (ape, "ape"), (state_cache, "state_cache")):
        _need(t, torch.float32, n)
    _need(slot_mapping, torch.int64, "slot_mapping")
    _need(positions, torch.int64, "positions")
    if kv.stride() != score.stride():
        raise ValueError("kv and score must share a layout")
    sw = kv.shape[1]
    if state_cache.dim() != 3 or state_cache.shape[1] != block_size or \
            state_cache.shape[2] != 2 * sw or not state_cache.is_contiguous():
        raise ValueError("state_cache must be contiguous [pages, block_size, 2 * state_width]")
    _call(kv.device, "save_compressor_state", _ptr(kv), _ptr(score), _rows(kv, "kv"),
          _ptr(ape.contiguous()), sw, _ptr(slot_mapping), _ptr(positions),
          slot_mapping.shape[0], compress_ratio, _ptr(state_cache), state_cache.shape[0],
          block_size, _ptr(err_count))


def compress_kv_cache_insert(state_cache: torch.Tensor, token_to_req_indices: torch.Tensor,
                             positions: torch.Tensor, compressor_slot_mapping: torch.Tensor,
                             block_table: torch.Tensor, compressor_block_size: int,
                             rms_norm_weight: torch.Tensor, rms_norm_eps: float,
                             cos_sin_cache: torch.Tensor, kv_cache_2d: torch.Tensor,
                             kv_slot_mapping: torch.Tensor, kv_cache_block_size: int,
                             compress_ratio: int, *, overlap: Optional[bool] = None,
                             block_table_base_offsets: Optional[torch.Tensor] = None,
                             err_count: Optional[torch.Tensor] = None) -> None:
    """Window-pooled, normalised, rotated fp8_ds_mla rows of the compressed KV
    cache (ratio 4 with overlap = the CSA insert, ratio 128 = the HCA insert)."""
    _need_cuda(state_cache, token_to_req_indices, positions, compressor_slot_mapping,
               block_table, rms_norm_weight, cos_sin_cache, kv_cache_2d, kv_slot_mapping,
               block_table_base_offsets, err_count)
    _need(state_cache, torch.float32, "state_cache")
    _need(positions, torch.int64, "positions")
    _need(rms_norm_weight, torch.float32, "rms_norm_weight")
    _need(cos_sin_cache, torch.float32, "cos_sin_cache")
    if overlap is None:
        overlap = compress_ratio == 4
    if state_cache.dim() != 3 or not state_cache.is_contiguous():
        raise ValueError("state_cache must be contiguous [pages, block_size, 2 * state_width]")
    num_pages, page_stride = _pages(kv_cache_2d)
    _call(state_cache.device, "compress_kv_cache_insert", _ptr(state_cache), state_cache.shape[0],
          compressor_block_size, state_cache.shape[2] // 2, _ptr(token_to_req_indices),
          _ptr(positions), _ptr(compressor_slot_mapping), _ptr(block_table),
          _rows(block_table, "block_table"), block_table.shape[1],
          _ptr(block_table_base_offsets), block_table.shape[0], positions.shape[0],
          compress_ratio, int(bool(overlap)), _ptr(rms_norm_weight.contiguous()),
          float(rms_norm_eps), _ptr(cos_sin_cache), _rows(cos_sin_cache, "cos_sin_cache"),
          cos_sin_cache.shape[0], _ptr(kv_cache_2d), num_pages, page_stride,
          kv_cache_block_size, _ptr(kv_slot_mapping), _ptr(err_count))


# ---- fused gathers ------------------------------------------------------------------------

def dequantize_and_gather_k_cache_topk(out: torch.Tensor, cache: torch.Tensor,
                                       topk_indices: torch.Tensor,
                                       token_to_req_indices: torch.Tensor,
                                       block_table: torch.Tensor, block_size: int, *,
                                       record: int = PSK_REC_FP8_DS_MLA, rope_dim: int = 64,
                                       num_reqs: Optional[int] = None,
                                       base_offsets: Optional[torch.Tensor] = None,
                                       is_valid_token: Optional[torch.Tensor] = None) -> torch.Tensor:
    """out[t, j] = the row of topk_indices[t, j] mapped through the request's table
    (= compute_global_topk_indices_and_lens + dequantize_and_gather_k_cache)."""
    _need_cuda(out, cache, topk_indices, token_to_req_indices, block_table, base_offsets,
               is_valid_token)
    _need(out, torch.bfloat16, "out")
    T, K = topk_indices.shape
    if out.dim() != 3 or out.shape[0] != T or out.shape[1] != K or out.stride(2) != 1:
        raise ValueError("out must be [T, K, D] with unit inner stride")
    num_pages, page_stride = _pages(cache)
    valid = None if is_valid_token is None else is_valid_token.to(torch.uint8)
    R = block_table.shape[0] if num_reqs is None else num_reqs
    _call(out.device, "dequantize_and_gather_k_cache_topk", _ptr(out), out.stride(0), out.stride(1),
          _ptr(cache), num_pages, page_stride, block_size, record, out.shape[2],
          rope_dim if record == PSK_REC_FP8_DS_MLA else 0, _ptr(topk_indices),
          _rows(topk_indices, "topk_indices"), T, K, _ptr(token_to_req_indices),
          _ptr(block_table), _rows(block_table, "block_table"), block_table.shape[1], R,
          _ptr(base_offsets), _ptr(valid))
    return out


def dequantize_and_gather_k_cache_window(out: torch.Tensor, cache: torch.Tensor,
                                         query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
                                         token_to_req: torch.Tensor,
                                         replay_start: Optional[torch.Tensor],
                                         block_table: torch.Tensor, block_size: int,
                                         window_size: int, *, rope_dim: int = 64,
                                         base_offsets: Optional[torch.Tensor] = None,
                                         is_valid_token: Optional[torch.Tensor] = None) -> torch.Tensor:
    """out[t, c] = the row of window column c of token t (= the window columns of
    combine_topk_swa_indices + dequantize_and_gather_k_cache)."""
    _need_cuda(out, cache, query_start_loc, seq_lens, token_to_req, replay_start, block_table,
               base_offsets, is_valid_token)
    _need(out, torch.bfloat16, "out")
    T = token_to_req.shape[0]
    if out.dim() != 3 or out.shape[0] != T or out.shape[1] != window_size or out.stride(2) != 1:
        raise ValueError("out must be [T, window, D] with unit inner stride")
    num_pages, page_stride = _pages(cache)
    valid = None if is_valid_token is None else is_valid_token.to(torch.uint8)
    _call(out.device, "dequantize_and_gather_k_cache_window",
          _ptr(out), out.stride(0), out.stride(1),
          _ptr(cache), num_pages, page_stride, block_size, out.shape[2], rope_dim,
          _ptr(query_start_loc), _ptr(seq_lens), _ptr(token_to_req), _ptr(replay_start),
          seq_lens.shape[0], T, _ptr(block_table), _rows(block_table, "block_table"),
          block_table.shape[1], _ptr(base_offsets), window_size, _ptr(valid))
    return out


def device_wait_timeouts() -> int:
    """Expired in-kernel bounded waits on the current device (0 in normal operation)."""
    return _abi.device_wait_timeouts()


def device_wait_selftest(limit_ns: int, device: torch.device) -> None:
    """Launch one bounded wait that nothing completes (counted when it expires)."""
    _call(device, "psk_device_wait_selftest", int(limit_ns))


def dequantize_and_gather_k_cache_pair(out: torch.Tensor, cache_a: torch.Tensor, block_size_a: int,
                                       cache_b: torch.Tensor, block_size_b: int,
                                       indices: torch.Tensor, split: int, *,
                                       rope_dim: int = 64) -> torch.Tensor:
    """out[t, j] = row indices[t, j] of cache_a for j < split, of cache_b for
    j >= split (fp8_ds_mla, UE8M0)."""
    _need_cuda(out, cache_a, cache_b, indices)
    _need(out, torch.bfloat16, "out")
    R, C = indices.shape
    if out.dim() != 3 or out.shape[0] != R or out.shape[1] != C or out.stride(2) != 1:
        raise ValueError("out must be [rows, cols, D] with unit inner stride")
    np_a, ps_a = _pages(cache_a)
    np_b, ps_b = _pages(cache_b)
    _call(out.device, "dequantize_and_gather_k_cache_pair", _ptr(out), out.stride(0), out.stride(1),
          _ptr(cache_a), np_a, ps_a, block_size_a, _ptr(cache_b), np_b, ps_b, block_size_b,
          out.shape[2], rope_dim, _ptr(indices), _rows(indices, "indices"), R, C, split)
    return out


def dequantize_and_gather_k_cache_dense(out: torch.Tensor, cache: torch.Tensor,
                                        positions: torch.Tensor, token_to_req: torch.Tensor,
                                        block_table: torch.Tensor, block_size: int,
                                        compress_ratio: int, *, rope_dim: int = 64,
                                        num_reqs: Optional[int] = None,
                                        base_offsets: Optional[torch.Tensor] = None,
                                        is_valid_token: Optional[torch.Tensor] = None) -> torch.Tensor:
    """out[t, c] = compressed entry c of token t when visible (= the dense
    compressed indices followed by the gather)."""
    _need_cuda(out, cache, positions, token_to_req, block_table, base_offsets, is_valid_token)
    _need(out, torch.bfloat16, "out")
    T = positions.shape[0]
    if out.dim() != 3 or out.shape[0] != T or out.stride(2) != 1:
        raise ValueError("out must be [T, width, D] with unit inner stride")
    num_pages, page_stride = _pages(cache)
    valid = None if is_valid_token is None else is_valid_token.to(torch.uint8)
    R = block_table.shape[0] if num_reqs is None else num_reqs
    _call(out.device, "dequantize_and_gather_k_cache_dense",
          _ptr(out), out.stride(0), out.stride(1),
          _ptr(cache), num_pages, page_stride, block_size, out.shape[2], rope_dim,
          _ptr(positions), T, _ptr(token_to_req), R, _ptr(block_table),
          _rows(block_table, "block_table"), block_table.shape[1], _ptr(base_offsets),
          compress_ratio, out.shape[1], _ptr(valid))
    return out
