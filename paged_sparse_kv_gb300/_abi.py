"""ctypes binding of libpsk.so (include/psk.h).  Argument marshalling only.

The library must have been built (``paged_sparse_kv_gb300.build.build()`` or
``__graft_entry__.build()``); there is no fallback implementation, so a
missing library is an ImportError-style RuntimeError at first use.
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpsk.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "psk.h")

PSK_OK = 0
PSK_ERR_INVALID_ARGUMENT = 1
PSK_ERR_UNSUPPORTED = 2
PSK_ERR_CUDA = 3
PSK_REC_FP8_DS_MLA = 0
PSK_REC_MXFP4 = 1
PSK_REC_FP8_INDEXER = 2

STATUS_NAMES = {0: "PSK_OK", 1: "PSK_ERR_INVALID_ARGUMENT", 2: "PSK_ERR_UNSUPPORTED",
                3: "PSK_ERR_CUDA"}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32

SIGNATURES = {
    "psk_last_error": (ctypes.c_char_p, []),
    "psk_abi_version": (_I32, []),
    "psk_device_wait_timeouts": (_I32, [_P]),
    "psk_device_wait_selftest": (_I32, [ctypes.c_uint64, _P]),
    "quantize_and_insert_k_cache": (
        _I32, [_P, _I64, _P, _I64, _P, _I64, _I64, _I32, _I32, _I32, _I32, _P, _P]),
    "write_indexer_mxfp4_cache": (
        _I32, [_P, _I64, _P, _I64, _P, _I64, _I64, _I32, _I32, _P, _P]),
    "compute_global_topk_indices_and_lens": (
        _I32, [_P, _I64, _I64, _I32, _P, _P, _I64, _I32, _I32, _I32, _P, _P, _P, _I64, _P, _P]),
    "combine_topk_swa_indices": (
        _I32, [_P, _P, _P, _P, _I32, _I64,
               _P, _I64, _I32, _P, _I32,
               _P, _I64, _I32, _P, _I32,
               _I32, _I32, _P, _I64, _I32, _P, _P, _I64, _P, _P]),
    "dequantize_and_gather_k_cache": (
        _I32, [_P, _I64, _I64, _P, _I64, _I64, _I32, _I32, _I32, _I32, _I32, _P, _I64, _I64,
               _I32, _P]),
    "dequantize_and_gather_k_cache_ranges": (
        _I32, [_P, _I64, _I64, _I64, _P, _I64, _I64, _I32, _I32, _I32, _I32, _I32, _P, _P, _P,
               _I64, _I32, _P, _I32, _I64, _P]),
    "combine_topk_swa_workspace_indices": (
        _I32, [_P, _P, _P, _P, _I32, _I64, _I32, _I32, _P, _I64, _I32, _I64, _I64, _P, _P, _I64,
               _P, _P]),
    "indexer_mxfp4_paged_gather": (
        _I32, [_P, _P, _P, _I64, _I64, _I32, _I32, _P, _I64, _I32, _P, _I32, _I64, _P]),
    "decode_swa_indices_and_lens": (
        _I32, [_P, _P, _P, _I32, _I64, _P, _I64, _I32, _P, _I32, _I32, _P, _P, _I64, _P, _P]),
    "compute_dense_compressed_indices_and_lens": (
        _I32, [_P, _I64, _P, _I32, _P, _I64, _I32, _P, _I32, _I32, _I32, _P, _P, _I64, _P, _P]),
    "build_dense_prefill_local_compressed_indices": (
        _I32, [_P, _I64, _I32, _I32, _P, _I64, _P]),
    "combine_dense_swa_indices": (
        _I32, [_P, _P, _P, _P, _I32, _I64, _I32, _I64, _I64, _P, _I64, _P, _P]),
    "write_indexer_fp8_cache": (
        _I32, [_P, _I64, _P, _I64, _P, _I64, _I64, _I32, _I32, _P, _P]),
    "dequantize_and_gather_k_cache_topk": (
        _I32, [_P, _I64, _I64, _P, _I64, _I64, _I32, _I32, _I32, _I32, _P, _I64, _I64, _I32, _P, _P,
               _I64, _I32, _I32, _P, _P, _P]),
    "dequantize_and_gather_k_cache_dense": (
        _I32, [_P, _I64, _I64, _P, _I64, _I64, _I32, _I32, _I32, _P, _I64, _P, _I32, _P, _I64,
               _I32, _P, _I32, _I32, _P, _P]),
    "dequantize_and_gather_k_cache_pair": (
        _I32, [_P, _I64, _I64, _P, _I64, _I64, _I32, _P, _I64, _I64, _I32, _I32, _I32, _P, _I64,
               _I64, _I32, _I32, _P]),
    "dequantize_and_gather_k_cache_window": (
        _I32, [_P, _I64, _I64, _P, _I64, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _I32, _I64, _P,
               _I64, _I32, _P, _I32, _P, _P]),
    "save_compressor_state": (
        _I32, [_P, _P, _I64, _P, _I32, _P, _P, _I64, _I32, _P, _I64, _I32, _P, _P]),
    "compress_kv_cache_insert": (
        _I32, [_P, _I64, _I32, _I32, _P, _P, _P, _P, _I64, _I32, _P, _I32, _I64, _I32, _I32, _P,
               ctypes.c_float, _P, _I64, _I64, _P, _I64, _I64, _I32, _P, _P, _P]),
    "indexer_k_norm_rope_store": (
        _I32, [_P, _I64, _P, _P, _I64, _I64, _P, ctypes.c_float, _P, _I64, _I32, _I32, _P, _I64,
               _I64, _I32, _P, _P]),
}

_lib = None


class PskError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        self.status = status
        super().__init__(f"{fn} failed with {STATUS_NAMES.get(status, status)}: {message}")


def lib() -> ctypes.CDLL:
    """Load libpsk.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"libpsk.so is missing at {LIB_PATH}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` "
            "(there is no CPU fallback)")
    l = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(l, name)
        fn.restype = res
        fn.argtypes = args
    _lib = l
    return l


def header_functions() -> list[str]:
    """Names of the functions include/psk.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(\w+)\s*\(", text, flags=re.M)


def call(name: str, *args) -> None:
    """Call an entry point and raise PskError unless it returns PSK_OK."""
    l = lib()
    st = getattr(l, name)(*args)
    if st != PSK_OK:
        msg = l.psk_last_error().decode(errors="replace")
        raise PskError(name, st, msg)


def status(name: str, *args) -> int:
    """Call an entry point and return its raw status code."""
    return getattr(lib(), name)(*args)


def device_wait_timeouts() -> int:
    """Expired in-kernel waits on the current device (0 in normal operation)."""
    v = ctypes.c_uint32(0)
    call("psk_device_wait_timeouts", ctypes.addressof(v))
    return int(v.value)


def last_error() -> str:
    return lib().psk_last_error().decode(errors="replace")
