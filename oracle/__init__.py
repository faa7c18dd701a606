"""CPU oracle for the paged sparse K-cache pipeline (ctypes over numpy).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
product library never imports it, and it imports nothing from the product.

The arithmetic lives in ``psk_oracle.c`` (plain single-threaded C, built
without fast-math or FMA contraction).  This module only marshals numpy arrays
into it.  Arrays must be C-contiguous; bf16 tensors travel as ``uint16`` bit
patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "psk_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
             "-fno-fast-math", "-Wall", "-Wextra"]

REC_FP8_DS_MLA = 0
REC_MXFP4 = 1
REC_FP8_INDEXER = 2


def build(force: bool = False) -> str:
    """Compile the oracle into ``liboracle.so`` beside its source."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    cmd = ["gcc", *GCC_FLAGS, _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    sig = {
        "oracle_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
        "oracle_e4m3_decode": (ctypes.c_float, [ctypes.c_uint8]),
        "oracle_e2m1_encode": (ctypes.c_uint8, [ctypes.c_float]),
        "oracle_e2m1_decode": (ctypes.c_float, [ctypes.c_uint8]),
        "oracle_ceil_log2": (_I32, [ctypes.c_float]),
        "oracle_bf16_from_f32": (ctypes.c_uint16, [ctypes.c_float]),
        "oracle_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
        "oracle_e4m3_encode_array": (None, [_P, _P, _I64]),
        "oracle_e2m1_encode_array": (None, [_P, _P, _I64]),
        "oracle_ceil_log2_array": (None, [_P, _P, _I64]),
        "oracle_fp8_token_stride": (_I64, [_I32, _I32]),
        "oracle_fp8_scale_bytes": (_I64, [_I32, _I32]),
        "oracle_quantize_and_insert_k_cache": (
            _I64, [_P, _I64, _P, _I64, _P, _I64, _I64, _I32, _I32, _I32, _I32]),
        "oracle_write_indexer_mxfp4_cache": (
            _I64, [_P, _I64, _P, _I64, _P, _I64, _I64, _I32, _I32]),
        "oracle_compute_global_topk_indices_and_lens": (
            None, [_P, _I64, _I64, _I32, _P, _P, _I64, _I32, _I32, _I32, _P, _P,
                   _P, _I64, _P]),
        "oracle_combine_topk_swa_indices": (
            None, [_P, _P, _P, _P, _I32, _I64,
                   _P, _I64, _I32, _P, _I32,
                   _P, _I64, _I32, _P, _I32,
                   _I32, _I32, _P, _I64, _I32, _P, _P, _I64, _P]),
        "oracle_dequantize_and_gather_k_cache": (
            None, [_P, _I64, _I64, _P, _I64, _I64, _I32, _I32, _I32, _I32, _I32,
                   _P, _I64, _I64, _I32]),
        "oracle_dequantize_and_gather_k_cache_ranges": (
            None, [_P, _I64, _I64, _I64, _P, _I64, _I64, _I32, _I32, _I32, _I32, _I32,
                   _P, _P, _P, _I64, _I32, _P, _I32, _I64]),
        "oracle_combine_topk_swa_workspace_indices": (
            None, [_P, _P, _P, _P, _I32, _I64, _I32, _I32, _P, _I64, _I32, _I64, _I64,
                   _P, _P, _I64, _P]),
        "oracle_indexer_mxfp4_paged_gather": (
            None, [_P, _P, _P, _I64, _I64, _I32, _I32, _P, _I64, _I32, _P, _I32]),
        "oracle_decode_swa_indices_and_lens": (
            None, [_P, _P, _P, _I32, _I64, _P, _I64, _I32, _P, _I32, _I32, _P, _P, _I64, _P]),
        "oracle_compute_dense_compressed_indices_and_lens": (
            None, [_P, _I64, _P, _I32, _P, _I64, _I32, _P, _I32, _I32, _I32, _P, _P, _I64,
                   _P]),
        "oracle_build_dense_prefill_local_compressed_indices": (
            None, [_P, _I64, _I32, _I32, _P, _I64]),
        "oracle_combine_dense_swa_indices": (
            None, [_P, _P, _P, _P, _I32, _I64, _I32, _I64, _I64, _P, _I64, _P]),
        "oracle_write_indexer_fp8_cache": (
            _I64, [_P, _I64, _P, _I64, _P, _I64, _I64, _I32, _I32]),
        "oracle_exp_cw": (ctypes.c_float, [ctypes.c_float]),
        "oracle_exp_cw_array": (None, [_P, _P, _I64]),
        "oracle_save_compressor_state": (
            _I64, [_P, _P, _I64, _P, _I32, _P, _P, _I64, _I32, _P, _I64, _I32]),
        "oracle_compress_kv_cache_insert": (
            _I64, [_P, _I64, _I32, _I32, _P, _P, _P, _P, _I64, _I32, _P, _I32, _I64, _I32, _I32,
                   _I32, _I32, _P, ctypes.c_float, _P, _I64, _I64, _P, _I64, _I64, _I32, _P]),
        "oracle_indexer_k_norm_rope_store": (
            _I64, [_P, _I64, _P, _P, _I64, _I64, _P, ctypes.c_float, _P, _I64, _I32, _I32, _P,
                   _I64, _I64, _I32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _as(a, dtype):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, f"expected {dtype}, got {a.dtype}"
    return a


# ---- scalar formats ---------------------------------------------------------

def e4m3_encode(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(v), _ptr(out), v.size)
    return out


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e2m1_encode_array(_ptr(v), _ptr(out), v.size)
    return out


def ceil_log2(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float32)
    out = np.empty(q.shape, dtype=np.int32)
    _load().oracle_ceil_log2_array(_ptr(q), _ptr(out), q.size)
    return out


def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(code)


def e2m1_decode(nibble: int) -> float:
    return _load().oracle_e2m1_decode(nibble)


def bf16_from_f32(f: float) -> int:
    return _load().oracle_bf16_from_f32(f)


def fp8_token_stride(head_dim: int, rope_dim: int) -> int:
    return _load().oracle_fp8_token_stride(head_dim, rope_dim)


def fp8_scale_bytes(head_dim: int, is_ue8m0: bool) -> int:
    return _load().oracle_fp8_scale_bytes(head_dim, int(bool(is_ue8m0)))


def fp8_record_bytes(head_dim: int, rope_dim: int, is_ue8m0: bool = True) -> int:
    return fp8_token_stride(head_dim, rope_dim) + fp8_scale_bytes(head_dim, is_ue8m0)


def mxfp4_record_bytes(head_dim: int) -> int:
    return head_dim // 2 + head_dim // 32


# ---- pipeline steps ---------------------------------------------------------

def quantize_and_insert_k_cache(k_bits, slot_mapping, cache, block_size, head_dim,
                                rope_dim, is_ue8m0=True) -> int:
    """Insert rows of ``k_bits`` (uint16 bf16 patterns [N, >=D]) into ``cache``
    (uint8 [num_pages, page_stride]) in place.  Returns out-of-range count."""
    k_bits = _as(k_bits, np.uint16)
    slot_mapping = _as(slot_mapping, np.int64)
    assert cache.dtype == np.uint8 and cache.ndim == 2 and cache.flags["C_CONTIGUOUS"]
    return _load().oracle_quantize_and_insert_k_cache(
        _ptr(k_bits), k_bits.shape[1], _ptr(slot_mapping), slot_mapping.shape[0],
        _ptr(cache), cache.shape[0], cache.shape[1], block_size, head_dim, rope_dim,
        int(bool(is_ue8m0)))


def write_indexer_mxfp4_cache(k_bits, slot_mapping, cache, block_size, head_dim) -> int:
    k_bits = _as(k_bits, np.uint16)
    slot_mapping = _as(slot_mapping, np.int64)
    assert cache.dtype == np.uint8 and cache.ndim == 2 and cache.flags["C_CONTIGUOUS"]
    return _load().oracle_write_indexer_mxfp4_cache(
        _ptr(k_bits), k_bits.shape[1], _ptr(slot_mapping), slot_mapping.shape[0],
        _ptr(cache), cache.shape[0], cache.shape[1], block_size, head_dim)


def compute_global_topk_indices_and_lens(topk_local, token_to_req, block_table,
                                         block_size, base_offsets=None,
                                         is_valid_token=None):
    topk_local = _as(topk_local, np.int32)
    token_to_req = _as(token_to_req, np.int32)
    block_table = _as(block_table, np.int32)
    base_offsets = _as(base_offsets, np.int32)
    if is_valid_token is not None:
        is_valid_token = np.ascontiguousarray(is_valid_token).astype(np.uint8)
    T, K = topk_local.shape
    out = np.empty((T, K), dtype=np.int32)
    lens = np.empty((T,), dtype=np.int32)
    _load().oracle_compute_global_topk_indices_and_lens(
        _ptr(topk_local), K, T, K, _ptr(token_to_req), _ptr(block_table),
        block_table.shape[1], block_table.shape[1], block_table.shape[0], block_size,
        _ptr(base_offsets), _ptr(is_valid_token), _ptr(out), K, _ptr(lens))
    return out, lens


def combine_topk_swa_indices(query_start_loc, seq_lens, token_to_req, replay_start,
                             swa_block_table, swa_block_size, comp_block_table,
                             comp_block_size, window, compress_ratio, topk_local,
                             swa_base_offsets=None, comp_base_offsets=None,
                             is_valid_token=None, num_tokens=None):
    query_start_loc = _as(query_start_loc, np.int32)
    seq_lens = _as(seq_lens, np.int32)
    token_to_req = _as(token_to_req, np.int32)
    replay_start = _as(replay_start, np.int32)
    swa_block_table = _as(swa_block_table, np.int32)
    comp_block_table = _as(comp_block_table, np.int32)
    swa_base_offsets = _as(swa_base_offsets, np.int32)
    comp_base_offsets = _as(comp_base_offsets, np.int32)
    topk_local = _as(topk_local, np.int32)
    if is_valid_token is not None:
        is_valid_token = np.ascontiguousarray(is_valid_token).astype(np.uint8)
    T = topk_local.shape[0] if num_tokens is None else num_tokens
    K = topk_local.shape[1]
    P = (K + 3) // 4 * 4
    num_reqs = seq_lens.shape[0]
    out = np.empty((T, window + P), dtype=np.int32)
    lens = np.empty((T,), dtype=np.int32)
    cbt = comp_block_table
    _load().oracle_combine_topk_swa_indices(
        _ptr(query_start_loc), _ptr(seq_lens), _ptr(token_to_req), _ptr(replay_start),
        num_reqs, T,
        _ptr(swa_block_table), swa_block_table.shape[1], swa_block_table.shape[1],
        _ptr(swa_base_offsets), swa_block_size,
        _ptr(cbt), cbt.shape[1] if cbt is not None else 0,
        cbt.shape[1] if cbt is not None else 0, _ptr(comp_base_offsets),
        comp_block_size, window, compress_ratio, _ptr(topk_local), K, K,
        _ptr(is_valid_token), _ptr(out), window + P, _ptr(lens))
    return out, lens


def dequantize_and_gather_k_cache(cache, block_size, record, head_dim, rope_dim,
                                  indices, is_ue8m0=True) -> np.ndarray:
    """Return uint16 bf16 patterns [rows, cols, head_dim] for ``indices``."""
    indices = _as(indices, np.int32)
    if indices.ndim == 1:
        indices = indices.reshape(-1, 1)
    rows, cols = indices.shape
    out = np.empty((rows, cols, head_dim), dtype=np.uint16)
    assert cache.dtype == np.uint8 and cache.ndim == 2 and cache.flags["C_CONTIGUOUS"]
    _load().oracle_dequantize_and_gather_k_cache(
        _ptr(out), cols * head_dim, head_dim, _ptr(cache), cache.shape[0],
        cache.shape[1], block_size, record, head_dim, rope_dim, int(bool(is_ue8m0)),
        _ptr(indices), cols, rows, cols)
    return out


def dequantize_and_gather_k_cache_ranges(out, cache, block_size, record, head_dim, rope_dim,
                                         seq_lens, gather_lens, block_table, offset,
                                         base_offsets=None, is_ue8m0=True) -> np.ndarray:
    """Range-form gather into ``out`` (uint16 [R, rows, head_dim], updated in place)."""
    seq_lens = _as(seq_lens, np.int32)
    gather_lens = _as(gather_lens, np.int32)
    block_table = _as(block_table, np.int32)
    base_offsets = _as(base_offsets, np.int32)
    assert out.dtype == np.uint16 and out.ndim == 3 and out.flags["C_CONTIGUOUS"]
    assert cache.dtype == np.uint8 and cache.ndim == 2 and cache.flags["C_CONTIGUOUS"]
    R, rows, D = out.shape
    assert D == head_dim and seq_lens.shape[0] == R
    _load().oracle_dequantize_and_gather_k_cache_ranges(
        _ptr(out), rows * D, D, rows, _ptr(cache), cache.shape[0], cache.shape[1], block_size,
        record, head_dim, rope_dim, int(bool(is_ue8m0)), _ptr(seq_lens), _ptr(gather_lens),
        _ptr(block_table), block_table.shape[1], block_table.shape[1], _ptr(base_offsets), R,
        offset)
    return out


def combine_topk_swa_workspace_indices(query_start_loc, seq_lens, gather_lens, token_to_req,
                                       window, compress_ratio, topk_local, workspace_width,
                                       compressed_base, is_valid_token=None):
    query_start_loc = _as(query_start_loc, np.int32)
    seq_lens = _as(seq_lens, np.int32)
    gather_lens = _as(gather_lens, np.int32)
    token_to_req = _as(token_to_req, np.int32)
    topk_local = _as(topk_local, np.int32)
    if is_valid_token is not None:
        is_valid_token = np.ascontiguousarray(is_valid_token).astype(np.uint8)
    T, K = topk_local.shape
    P = (K + 3) // 4 * 4
    out = np.empty((T, window + P), dtype=np.int32)
    lens = np.empty((T,), dtype=np.int32)
    _load().oracle_combine_topk_swa_workspace_indices(
        _ptr(query_start_loc), _ptr(seq_lens), _ptr(gather_lens), _ptr(token_to_req),
        seq_lens.shape[0], T, window, compress_ratio, _ptr(topk_local), K, K, workspace_width,
        compressed_base, _ptr(is_valid_token), _ptr(out), window + P, _ptr(lens))
    return out, lens


def indexer_mxfp4_paged_gather(cache, block_size, head_dim, block_table, cu_seq_lens):
    """Raw MXFP4 rows over per-request ranges: (values [N, D/2], scales [N, D/32])."""
    block_table = _as(block_table, np.int32)
    cu_seq_lens = _as(cu_seq_lens, np.int32)
    assert cache.dtype == np.uint8 and cache.ndim == 2 and cache.flags["C_CONTIGUOUS"]
    n = int(cu_seq_lens[-1])
    values = np.empty((n, head_dim // 2), dtype=np.uint8)
    scales = np.empty((n, head_dim // 32), dtype=np.uint8)
    _load().oracle_indexer_mxfp4_paged_gather(
        _ptr(values), _ptr(scales), _ptr(cache), cache.shape[0], cache.shape[1], block_size,
        head_dim, _ptr(block_table), block_table.shape[1], block_table.shape[1],
        _ptr(cu_seq_lens), cu_seq_lens.shape[0] - 1)
    return values, scales


# ---- dense builders -------------------------------------------------------------------

def decode_swa_indices_and_lens(query_start_loc, seq_lens, token_to_req, block_table,
                                block_size, window, base_offsets=None, is_valid_token=None):
    """Window-only indices [T, window] + lens of the decode SWA precompute."""
    query_start_loc = _as(query_start_loc, np.int32)
    seq_lens = _as(seq_lens, np.int32)
    token_to_req = _as(token_to_req, np.int32)
    block_table = _as(block_table, np.int32)
    base_offsets = _as(base_offsets, np.int32)
    if is_valid_token is not None:
        is_valid_token = np.ascontiguousarray(is_valid_token).astype(np.uint8)
    T = token_to_req.shape[0]
    out = np.empty((T, window), dtype=np.int32)
    lens = np.empty((T,), dtype=np.int32)
    _load().oracle_decode_swa_indices_and_lens(
        _ptr(query_start_loc), _ptr(seq_lens), _ptr(token_to_req), seq_lens.shape[0], T,
        _ptr(block_table), block_table.shape[1], block_table.shape[1], _ptr(base_offsets),
        block_size, window, _ptr(is_valid_token), _ptr(out), window, _ptr(lens))
    return out, lens


def compute_dense_compressed_indices_and_lens(positions, token_to_req, block_table, block_size,
                                              compress_ratio, width, num_reqs=None,
                                              base_offsets=None, is_valid_token=None):
    """Every visible compressed entry's slot [T, width] + lens (HCA decode)."""
    positions = _as(positions, np.int64)
    token_to_req = _as(token_to_req, np.int32)
    block_table = _as(block_table, np.int32)
    base_offsets = _as(base_offsets, np.int32)
    if is_valid_token is not None:
        is_valid_token = np.ascontiguousarray(is_valid_token).astype(np.uint8)
    T = positions.shape[0]
    R = block_table.shape[0] if num_reqs is None else num_reqs
    out = np.empty((T, width), dtype=np.int32)
    lens = np.empty((T,), dtype=np.int32)
    _load().oracle_compute_dense_compressed_indices_and_lens(
        _ptr(positions), T, _ptr(token_to_req), R, _ptr(block_table), block_table.shape[1],
        block_table.shape[1], _ptr(base_offsets), block_size, compress_ratio, width,
        _ptr(is_valid_token), _ptr(out), width, _ptr(lens))
    return out, lens


def build_dense_prefill_local_compressed_indices(positions, compress_ratio, width):
    """Request-local dense compressed indices [T, width]."""
    positions = _as(positions, np.int64)
    T = positions.shape[0]
    out = np.empty((T, width), dtype=np.int32)
    _load().oracle_build_dense_prefill_local_compressed_indices(
        _ptr(positions), T, compress_ratio, width, _ptr(out), width)
    return out


def combine_dense_swa_indices(positions, token_to_req, seq_lens, gather_lens, window,
                              workspace_width, compressed_base=0):
    """Window-only workspace indices [T, window] + lens (layers without a
    compressed cache)."""
    positions = _as(positions, np.int64)
    token_to_req = _as(token_to_req, np.int32)
    seq_lens = _as(seq_lens, np.int32)
    gather_lens = _as(gather_lens, np.int32)
    T = positions.shape[0]
    out = np.empty((T, window), dtype=np.int32)
    lens = np.empty((T,), dtype=np.int32)
    _load().oracle_combine_dense_swa_indices(
        _ptr(positions), _ptr(token_to_req), _ptr(seq_lens), _ptr(gather_lens),
        seq_lens.shape[0], T, window, workspace_width, compressed_base, _ptr(out), window,
        _ptr(lens))
    return out, lens


# ---- indexer-key variants -------------------------------------------------------------

def fp8_indexer_record_bytes(head_dim: int) -> int:
    """head_dim e4m3 bytes + one binary32 scale."""
    return head_dim + 4


def write_indexer_fp8_cache(k, slots, cache, block_size, head_dim) -> int:
    """FP8 indexer records (per-token power-of-two binary32 scale); returns the
    count of out-of-range slots."""
    k = np.ascontiguousarray(k, dtype=np.uint16)
    slots = _as(slots, np.int64)
    assert cache.dtype == np.uint8 and cache.ndim == 2 and cache.flags["C_CONTIGUOUS"]
    return _load().oracle_write_indexer_fp8_cache(
        _ptr(k), k.shape[1], _ptr(slots), slots.shape[0], _ptr(cache), cache.shape[0],
        cache.shape[1], block_size, head_dim)


def indexer_k_norm_rope_store(k_pre, positions, cos_sin_cache, rms_norm_weight, rms_norm_eps,
                              slots, compress_ratio, record, cache, block_size) -> int:
    """k_norm -> RoPE -> quant -> paged store of 128-dim indexer keys (record
    REC_MXFP4 or REC_FP8_INDEXER); returns the count of skipped-and-counted rows."""
    k_pre = np.ascontiguousarray(k_pre, dtype=np.uint16)
    positions = _as(positions, np.int64)
    cs = np.ascontiguousarray(cos_sin_cache, dtype=np.float32)
    wt = np.ascontiguousarray(rms_norm_weight, dtype=np.float32)
    slots = _as(slots, np.int64)
    assert cache.dtype == np.uint8 and cache.ndim == 2 and cache.flags["C_CONTIGUOUS"]
    return _load().oracle_indexer_k_norm_rope_store(
        _ptr(k_pre), k_pre.shape[1], _ptr(positions), _ptr(cs), cs.shape[1], cs.shape[0],
        _ptr(wt), float(rms_norm_eps), _ptr(slots), slots.shape[0], compress_ratio, record,
        _ptr(cache), cache.shape[0], cache.shape[1], block_size)


# ---- compressed-KV producer -------------------------------------------------------------

def exp_cw(x) -> np.ndarray:
    """The oracle's binary32 exp (Cody-Waite reduction + Taylor polynomial)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    _load().oracle_exp_cw_array(_ptr(x), _ptr(out), x.size)
    return out


def save_compressor_state(kv, score, ape, slots, positions, compress_ratio, state_cache,
                          block_size) -> int:
    """state[slot] = [kv, score + ape[pos % ratio]]; state_cache float32
    [pages, block_size, 2 * state_width] updated in place."""
    kv = np.ascontiguousarray(kv, dtype=np.float32)
    score = np.ascontiguousarray(score, dtype=np.float32)
    ape = np.ascontiguousarray(ape, dtype=np.float32)
    slots = _as(slots, np.int64)
    positions = _as(positions, np.int64)
    assert state_cache.dtype == np.float32 and state_cache.flags["C_CONTIGUOUS"]
    sw = kv.shape[1]
    assert state_cache.shape[1:] == (block_size, 2 * sw)
    return _load().oracle_save_compressor_state(
        _ptr(kv), _ptr(score), sw, _ptr(ape), sw, _ptr(slots), _ptr(positions),
        slots.shape[0], compress_ratio, _ptr(state_cache), state_cache.shape[0], block_size)


def compress_kv_cache_insert(state_cache, token_to_req, positions, state_slots, block_table,
                             state_block_size, rms_norm_weight, rms_norm_eps, cos_sin_cache,
                             kv_cache, kv_slots, kv_block_size, compress_ratio, overlap,
                             num_reqs=None, base_offsets=None, head_dim=512) -> int:
    """The compressed-KV producer: window softmax pooling of the state, RMSNorm,
    GPT-J RoPE of the tail, fp8_ds_mla insert.  Returns the counted skips."""
    assert state_cache.dtype == np.float32 and state_cache.flags["C_CONTIGUOUS"]
    token_to_req = _as(token_to_req, np.int32)
    positions = _as(positions, np.int64)
    state_slots = _as(state_slots, np.int64)
    block_table = _as(block_table, np.int32)
    base_offsets = _as(base_offsets, np.int32)
    wt = np.ascontiguousarray(rms_norm_weight, dtype=np.float32)
    cs = np.ascontiguousarray(cos_sin_cache, dtype=np.float32)
    kv_slots = _as(kv_slots, np.int64)
    assert kv_cache.dtype == np.uint8 and kv_cache.ndim == 2 and kv_cache.flags["C_CONTIGUOUS"]
    sw = state_cache.shape[2] // 2
    R = block_table.shape[0] if num_reqs is None else num_reqs
    return _load().oracle_compress_kv_cache_insert(
        _ptr(state_cache), state_cache.shape[0], state_block_size, sw, _ptr(token_to_req),
        _ptr(positions), _ptr(state_slots), _ptr(block_table), block_table.shape[1],
        block_table.shape[1], _ptr(base_offsets), R, positions.shape[0], compress_ratio,
        int(bool(overlap)), head_dim, cs.shape[1], _ptr(wt), float(rms_norm_eps), _ptr(cs),
        cs.shape[1], cs.shape[0], _ptr(kv_cache), kv_cache.shape[0], kv_cache.shape[1],
        kv_block_size, _ptr(kv_slots))
