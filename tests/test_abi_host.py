"""Host-side checks of the C ABI that need no GPU.

* libpsk.so loads and exports every function include/psk.h declares.
* Argument validation: every bad-argument call returns
  PSK_ERR_INVALID_ARGUMENT with a message, before any CUDA call, so these run
  on a machine without a GPU.
* Zero-work calls return PSK_OK without launching anything.
"""
import ctypes

import pytest

from paged_sparse_kv_gb300 import _abi

INV = _abi.PSK_ERR_INVALID_ARGUMENT
OK = _abi.PSK_OK

# Fake but well-aligned device addresses: validation never dereferences them.
A = 0x10000000
B = 0x20000000
C = 0x30000000


def test_library_exports_every_declared_symbol(psk_lib):
    declared = _abi.header_functions()
    assert set(declared) >= {"quantize_and_insert_k_cache", "write_indexer_mxfp4_cache",
                             "compute_global_topk_indices_and_lens",
                             "combine_topk_swa_indices", "dequantize_and_gather_k_cache",
                             "psk_last_error", "psk_abi_version"}
    for name in declared:
        assert hasattr(psk_lib, name), name
        assert ctypes.cast(getattr(psk_lib, name), ctypes.c_void_p).value
    assert psk_lib.psk_abi_version() >= 1


def _insert(**kw):
    a = dict(k=A, k_row_stride=512, slots=B, n=4, cache=C, num_pages=8, page_stride=64 * 584,
             bs=64, D=512, rope=64, ue=1, err=None)
    a.update(kw)
    return _abi.status("quantize_and_insert_k_cache", a["k"], a["k_row_stride"], a["slots"],
                       a["n"], a["cache"], a["num_pages"], a["page_stride"], a["bs"], a["D"],
                       a["rope"], a["ue"], a["err"], None)


@pytest.mark.parametrize("kw", [
    dict(k=None), dict(slots=None), dict(cache=None), dict(n=-1), dict(ue=2),
    dict(D=96), dict(D=500), dict(rope=32), dict(rope=512), dict(rope=-64),
    dict(bs=0), dict(num_pages=0), dict(page_stride=64 * 584 - 16),
    dict(page_stride=64 * 584 + 8), dict(cache=C + 8), dict(k=A + 2),
    dict(k_row_stride=500), dict(k_row_stride=256), dict(slots=B + 4), dict(err=B + 2),
    dict(ue=0, page_stride=64 * 584),  # fp32 scales need 32 scale bytes per token
])
def test_insert_rejects_bad_arguments(psk_lib, kw):
    assert _insert(**kw) == INV
    assert _abi.last_error()


def test_insert_zero_tokens_is_ok_without_launch(psk_lib):
    assert _insert(n=0, k=None, slots=None) == OK
    assert _abi.last_error() == ""


def _mx(**kw):
    a = dict(k=A, ks=128, slots=B, n=4, cache=C, num_pages=8, page_stride=64 * 68, bs=64,
             D=128, err=None)
    a.update(kw)
    return _abi.status("write_indexer_mxfp4_cache", a["k"], a["ks"], a["slots"], a["n"],
                       a["cache"], a["num_pages"], a["page_stride"], a["bs"], a["D"], a["err"],
                       None)


@pytest.mark.parametrize("kw", [dict(D=48), dict(D=100), dict(page_stride=64 * 68 - 16),
                                dict(cache=C + 4), dict(k=None), dict(ks=120), dict(n=-5)])
def test_mxfp4_insert_rejects_bad_arguments(psk_lib, kw):
    assert _mx(**kw) == INV


def _topk(**kw):
    a = dict(topk=A, ts=8, n=3, K=8, t2r=B, bt=C, bts=4, btw=4, R=2, bs=16, base=None,
             valid=None, out=A + 4096, os=8, lens=B + 4096)
    a.update(kw)
    return _abi.status("compute_global_topk_indices_and_lens", a["topk"], a["ts"], a["n"],
                       a["K"], a["t2r"], a["bt"], a["bts"], a["btw"], a["R"], a["bs"],
                       a["base"], a["valid"], a["out"], a["os"], a["lens"], None)


@pytest.mark.parametrize("kw", [dict(K=-1), dict(ts=4), dict(os=4), dict(bs=0), dict(R=0),
                                dict(btw=5), dict(t2r=None), dict(lens=None),
                                dict(topk=None), dict(out=A + 2), dict(n=-1)])
def test_global_topk_rejects_bad_arguments(psk_lib, kw):
    assert _topk(**kw) == INV


def test_global_topk_zero_tokens_ok(psk_lib):
    assert _topk(n=0, topk=None, t2r=None, out=None, lens=None) == OK


def _combine(**kw):
    a = dict(qsl=A, seq=A + 256, t2r=A + 512, rs=None, R=2, n=3, swa=B, swas=4, swaw=4,
             swab=None, swabs=16, comp=None, comps=0, compw=0, compb=None, compbs=16, W=8,
             ratio=4, topk=C, ts=8, K=8, valid=None, out=C + 4096, os=16, lens=C + 8192)
    a.update(kw)
    return _abi.status("combine_topk_swa_indices", a["qsl"], a["seq"], a["t2r"], a["rs"],
                       a["R"], a["n"], a["swa"], a["swas"], a["swaw"], a["swab"], a["swabs"],
                       a["comp"], a["comps"], a["compw"], a["compb"], a["compbs"], a["W"],
                       a["ratio"], a["topk"], a["ts"], a["K"], a["valid"], a["out"], a["os"],
                       a["lens"], None)


@pytest.mark.parametrize("kw", [dict(W=-1), dict(K=-2), dict(ratio=0), dict(swabs=0),
                                dict(compbs=0), dict(os=15), dict(ts=7), dict(R=0),
                                dict(qsl=None), dict(seq=None), dict(out=None),
                                dict(swa=None), dict(comp=B + 1024, comps=2, compw=3),
                                dict(K=5, os=12), dict(swaw=5), dict(lens=C + 2)])
def test_combine_rejects_bad_arguments(psk_lib, kw):
    assert _combine(**kw) == INV


def test_combine_padded_width_rule(psk_lib):
    # K=5 pads to 8: a row of W + 8 = 16 columns is enough, 15 is not.
    assert _combine(K=5, ts=5, os=16, n=0) == OK
    assert _combine(K=5, ts=5, os=15, n=0) == INV


def _gather(**kw):
    a = dict(out=A, ost=640 * 512, osj=512, cache=B, num_pages=8, page_stride=64 * 584, bs=64,
             rec=0, D=512, rope=64, ue=1, idx=C, ids=640, rows=4, cols=640)
    a.update(kw)
    return _abi.status("dequantize_and_gather_k_cache", a["out"], a["ost"], a["osj"],
                       a["cache"], a["num_pages"], a["page_stride"], a["bs"], a["rec"], a["D"],
                       a["rope"], a["ue"], a["idx"], a["ids"], a["rows"], a["cols"], None)


@pytest.mark.parametrize("kw", [dict(rec=2), dict(D=100), dict(rope=16), dict(out=A + 8),
                                dict(osj=4), dict(ost=-8), dict(ids=100), dict(idx=None),
                                dict(out=None), dict(rows=-1), dict(page_stride=1000),
                                dict(rec=1, D=128, rope=64), dict(rec=1, D=48, rope=0),
                                dict(ue=5), dict(cache=None)])
def test_gather_rejects_bad_arguments(psk_lib, kw):
    assert _gather(**kw) == INV


def test_gather_zero_rows_ok(psk_lib):
    assert _gather(rows=0, out=None, idx=None) == OK
    assert _gather(cols=0, ids=0, out=None, idx=None) == OK


def test_error_message_is_thread_local(psk_lib):
    import threading
    assert _insert(ue=7) == INV
    seen = {}

    def other():
        seen["msg"] = _abi.last_error()
    th = threading.Thread(target=other)
    th.start()
    th.join()
    assert seen["msg"] == ""
    assert "is_ue8m0" in _abi.last_error()


def _ranges(**kw):
    a = dict(out=A, osr=8 * 512, osi=512, rows=8, cache=B, num_pages=8, page_stride=64 * 584,
             bs=64, rec=0, D=512, rope=64, ue=1, seq=C, glen=None, bt=C + 4096, bts=4, btw=4,
             base=None, R=2, off=0)
    a.update(kw)
    return _abi.status("dequantize_and_gather_k_cache_ranges", a["out"], a["osr"], a["osi"],
                       a["rows"], a["cache"], a["num_pages"], a["page_stride"], a["bs"], a["rec"],
                       a["D"], a["rope"], a["ue"], a["seq"], a["glen"], a["bt"], a["bts"],
                       a["btw"], a["base"], a["R"], a["off"], None)


@pytest.mark.parametrize("kw", [dict(off=9), dict(off=-1), dict(out=None), dict(seq=None),
                                dict(osi=4), dict(out=A + 2), dict(btw=5), dict(D=100),
                                dict(page_stride=100), dict(R=-1)])
def test_range_gather_rejects_bad_arguments(psk_lib, kw):
    assert _ranges(**kw) == INV


def test_range_gather_rejects_mxfp4_record(psk_lib):
    assert _ranges(rec=1) == _abi.PSK_ERR_UNSUPPORTED


def test_range_gather_zero_work_ok(psk_lib):
    assert _ranges(R=0, out=None, seq=None) == OK
    assert _ranges(off=8, out=None) == OK


def _wsidx(**kw):
    a = dict(qsl=A, seq=A + 256, glen=A + 512, t2r=A + 768, R=2, n=3, W=8, ratio=4, topk=B,
             ts=8, K=8, ww=100, cb=10, valid=None, out=C, os=16, lens=C + 4096)
    a.update(kw)
    return _abi.status("combine_topk_swa_workspace_indices", a["qsl"], a["seq"], a["glen"],
                       a["t2r"], a["R"], a["n"], a["W"], a["ratio"], a["topk"], a["ts"], a["K"],
                       a["ww"], a["cb"], a["valid"], a["out"], a["os"], a["lens"], None)


@pytest.mark.parametrize("kw", [dict(os=15), dict(ratio=0), dict(glen=None), dict(W=-1),
                                dict(ww=-1), dict(R=0), dict(lens=None), dict(ts=4)])
def test_workspace_indices_reject_bad_arguments(psk_lib, kw):
    assert _wsidx(**kw) == INV


def _raw(**kw):
    a = dict(v=A, s=A + 4096, cache=B, num_pages=4, page_stride=64 * 68, bs=64, D=128, bt=C,
             bts=2, btw=2, cu=C + 256, R=2, n=100)
    a.update(kw)
    return _abi.status("indexer_mxfp4_paged_gather", a["v"], a["s"], a["cache"], a["num_pages"],
                       a["page_stride"], a["bs"], a["D"], a["bt"], a["bts"], a["btw"], a["cu"],
                       a["R"], a["n"], None)


@pytest.mark.parametrize("kw", [dict(D=96), dict(v=None), dict(cu=None), dict(R=0),
                                dict(s=A + 4098), dict(n=-1), dict(page_stride=64 * 68 - 16)])
def test_mxfp4_raw_gather_rejects_bad_arguments(psk_lib, kw):
    assert _raw(**kw) == INV


def _dswa(**kw):
    a = dict(qsl=A, seq=A + 256, t2r=A + 512, R=2, n=3, bt=B, bts=4, btw=4, base=None, bs=16,
             W=8, valid=None, out=C, os=8, lens=C + 4096)
    a.update(kw)
    return _abi.status("decode_swa_indices_and_lens", a["qsl"], a["seq"], a["t2r"], a["R"], a["n"],
                       a["bt"], a["bts"], a["btw"], a["base"], a["bs"], a["W"], a["valid"],
                       a["out"], a["os"], a["lens"], None)


@pytest.mark.parametrize("kw", [dict(W=-1), dict(bs=0), dict(btw=5), dict(os=7), dict(R=0),
                                dict(qsl=None), dict(out=None), dict(lens=None), dict(bt=None),
                                dict(out=C + 2), dict(n=-1)])
def test_decode_swa_rejects_bad_arguments(psk_lib, kw):
    assert _dswa(**kw) == INV


def test_decode_swa_zero_tokens_ok(psk_lib):
    assert _dswa(n=0, qsl=None, out=None, lens=None) == OK


def _dense(**kw):
    a = dict(pos=A, n=3, t2r=A + 256, R=2, bt=B, bts=4, btw=4, base=None, bs=16, ratio=128,
             width=64, valid=None, out=C, os=64, lens=C + 8192)
    a.update(kw)
    return _abi.status("compute_dense_compressed_indices_and_lens", a["pos"], a["n"], a["t2r"],
                       a["R"], a["bt"], a["bts"], a["btw"], a["base"], a["bs"], a["ratio"],
                       a["width"], a["valid"], a["out"], a["os"], a["lens"], None)


@pytest.mark.parametrize("kw", [dict(width=-1), dict(ratio=0), dict(bs=0), dict(os=63),
                                dict(btw=5), dict(R=0), dict(pos=None), dict(pos=A + 4),
                                dict(out=None), dict(lens=None), dict(t2r=None), dict(n=-2)])
def test_dense_compressed_rejects_bad_arguments(psk_lib, kw):
    assert _dense(**kw) == INV


def test_dense_compressed_zero_tokens_ok(psk_lib):
    assert _dense(n=0, pos=None, out=None, lens=None) == OK


def _local(**kw):
    a = dict(pos=A, n=3, ratio=128, width=64, out=C, os=64)
    a.update(kw)
    return _abi.status("build_dense_prefill_local_compressed_indices", a["pos"], a["n"],
                       a["ratio"], a["width"], a["out"], a["os"], None)


@pytest.mark.parametrize("kw", [dict(width=-1), dict(ratio=0), dict(os=63), dict(pos=None),
                                dict(out=None), dict(pos=A + 4), dict(out=C + 2), dict(n=-1)])
def test_dense_local_rejects_bad_arguments(psk_lib, kw):
    assert _local(**kw) == INV


def test_dense_local_zero_work_ok(psk_lib):
    assert _local(n=0, pos=None, out=None) == OK
    assert _local(width=0, os=0, pos=None, out=None) == OK


def _dswa_ws(**kw):
    a = dict(pos=A, t2r=A + 256, seq=A + 512, glen=A + 768, R=2, n=3, W=8, ww=100, cb=10, out=C,
             os=8, lens=C + 4096)
    a.update(kw)
    return _abi.status("combine_dense_swa_indices", a["pos"], a["t2r"], a["seq"], a["glen"],
                       a["R"], a["n"], a["W"], a["ww"], a["cb"], a["out"], a["os"], a["lens"], None)


@pytest.mark.parametrize("kw", [dict(W=-1), dict(ww=-1), dict(cb=-1), dict(os=7), dict(R=0),
                                dict(pos=None), dict(glen=None), dict(out=None), dict(lens=None),
                                dict(pos=A + 4), dict(seq=A + 514)])
def test_dense_swa_rejects_bad_arguments(psk_lib, kw):
    assert _dswa_ws(**kw) == INV


def test_dense_swa_zero_tokens_ok(psk_lib):
    assert _dswa_ws(n=0, pos=None, out=None, lens=None) == OK


def _fp8i(**kw):
    a = dict(k=A, ks=128, slots=B, n=4, cache=C, num_pages=8, page_stride=64 * 132, bs=64,
             D=128, err=None)
    a.update(kw)
    return _abi.status("write_indexer_fp8_cache", a["k"], a["ks"], a["slots"], a["n"], a["cache"],
                       a["num_pages"], a["page_stride"], a["bs"], a["D"], a["err"], None)


@pytest.mark.parametrize("kw", [dict(D=48), dict(D=16), dict(page_stride=64 * 132 - 16),
                                dict(cache=C + 4), dict(k=None), dict(k=A + 8), dict(ks=120),
                                dict(n=-5), dict(slots=B + 4), dict(err=B + 2)])
def test_fp8_indexer_insert_rejects_bad_arguments(psk_lib, kw):
    assert _fp8i(**kw) == INV


def test_fp8_indexer_insert_zero_tokens_ok(psk_lib):
    assert _fp8i(n=0, k=None, slots=None) == OK


def test_fp8_indexer_gather_record_checks(psk_lib):
    assert _gather(rec=2, D=128, rope=0, page_stride=64 * 132, rows=0, out=None, idx=None) == OK
    assert _gather(rec=2, D=128, rope=64, page_stride=64 * 132) == INV
    assert _gather(rec=2, D=128, rope=0, page_stride=64 * 132 - 16) == INV
    assert _gather(rec=3, D=128, rope=0) == INV


def _nrs(**kw):
    a = dict(k=A, ks=128, pos=B, cs=C, css=64, maxp=4096, w=A + 4096, eps=1e-6, slots=B + 4096,
             n=4, ratio=4, rec=1, cache=C + 65536, num_pages=8, page_stride=64 * 68, bs=64,
             err=None)
    a.update(kw)
    return _abi.status("indexer_k_norm_rope_store", a["k"], a["ks"], a["pos"], a["cs"], a["css"],
                       a["maxp"], a["w"], a["eps"], a["slots"], a["n"], a["ratio"], a["rec"],
                       a["cache"], a["num_pages"], a["page_stride"], a["bs"], a["err"], None)


@pytest.mark.parametrize("kw", [dict(rec=0), dict(rec=3), dict(ratio=0), dict(css=32),
                                dict(maxp=-1), dict(ks=126), dict(ks=132), dict(k=A + 8),
                                dict(pos=B + 4), dict(w=A + 4100), dict(cs=C + 2),
                                dict(page_stride=64 * 68 - 16), dict(rec=2, page_stride=64 * 68),
                                dict(k=None), dict(slots=None), dict(n=-1), dict(err=B + 1)])
def test_norm_rope_store_rejects_bad_arguments(psk_lib, kw):
    assert _nrs(**kw) == INV


def test_norm_rope_store_zero_tokens_ok(psk_lib):
    assert _nrs(n=0, k=None, pos=None) == OK


def _save(**kw):
    a = dict(kv=A, sc=A + 65536, ins=1024, ape=B, sw=1024, slots=B + 65536, pos=C, n=4, ratio=4,
             st=C + 65536, pages=4, bs=16, err=None)
    a.update(kw)
    return _abi.status("save_compressor_state", a["kv"], a["sc"], a["ins"], a["ape"], a["sw"],
                       a["slots"], a["pos"], a["n"], a["ratio"], a["st"], a["pages"], a["bs"],
                       a["err"], None)


@pytest.mark.parametrize("kw", [dict(sw=0), dict(sw=1022), dict(ratio=0), dict(pages=0),
                                dict(st=None), dict(st=C + 65544), dict(kv=None), dict(ins=1020),
                                dict(ins=1026), dict(kv=A + 4), dict(slots=B + 65540), dict(n=-1)])
def test_save_state_rejects_bad_arguments(psk_lib, kw):
    assert _save(**kw) == INV


def _cmp(**kw):
    a = dict(st=A, spages=8, sbs=16, sw=1024, t2r=B, pos=B + 4096, ss=B + 8192, bt=C, bts=4,
             btw=4, base=None, R=2, n=4, ratio=4, ov=1, w=C + 4096, eps=1e-6, cs=C + 8192,
             css=64, maxp=4096, kv=A + 1048576, kpages=8, kps=64 * 584, kbs=64, ks=B + 12288,
             err=None)
    a.update(kw)
    return _abi.status("compress_kv_cache_insert", a["st"], a["spages"], a["sbs"], a["sw"],
                       a["t2r"], a["pos"], a["ss"], a["bt"], a["bts"], a["btw"], a["base"],
                       a["R"], a["n"], a["ratio"], a["ov"], a["w"], a["eps"], a["cs"], a["css"],
                       a["maxp"], a["kv"], a["kpages"], a["kps"], a["kbs"], a["ks"], a["err"], None)


@pytest.mark.parametrize("kw", [dict(ov=2), dict(ratio=0), dict(ratio=129, ov=1),
                                dict(ratio=300, ov=0, sw=512), dict(sw=512), dict(ov=0),
                                dict(spages=0), dict(btw=5), dict(css=32), dict(maxp=-1),
                                dict(kps=64 * 584 - 16), dict(R=0), dict(st=None), dict(st=A + 4),
                                dict(w=C + 4100), dict(pos=B + 4100), dict(n=-1)])
def test_compress_rejects_bad_arguments(psk_lib, kw):
    assert _cmp(**kw) == INV


def test_compress_zero_tokens_ok(psk_lib):
    assert _cmp(n=0, st=None, t2r=None) == OK


def _gather_topk(**kw):
    a = dict(out=A, ost=512 * 512, osj=512, cache=B, num_pages=8, page_stride=64 * 584, bs=64,
             rec=0, D=512, rope=64, tk=C, tks=512, T=4, K=512, t2r=C + 4096, bt=C + 8192,
             bts=16, btw=16, R=2, base=None, valid=None)
    a.update(kw)
    return _abi.status("dequantize_and_gather_k_cache_topk", a["out"], a["ost"], a["osj"],
                       a["cache"], a["num_pages"], a["page_stride"], a["bs"], a["rec"], a["D"],
                       a["rope"], a["tk"], a["tks"], a["T"], a["K"], a["t2r"], a["bt"],
                       a["bts"], a["btw"], a["R"], a["base"], a["valid"], None)


@pytest.mark.parametrize("kw", [dict(rec=3), dict(D=100), dict(rope=16), dict(out=A + 8),
                                dict(osj=4), dict(ost=-8), dict(tks=100), dict(tk=None),
                                dict(t2r=None), dict(bt=None), dict(out=None), dict(T=-1),
                                dict(K=-1), dict(R=0), dict(bts=8), dict(btw=-1),
                                dict(page_stride=1000), dict(rec=1, D=128, rope=64),
                                dict(rec=1, D=48, rope=0), dict(rec=2, D=64, rope=0,
                                                                page_stride=100),
                                dict(tk=C + 2), dict(base=C + 1), dict(cache=None)])
def test_gather_topk_rejects_bad_arguments(psk_lib, kw):
    assert _gather_topk(**kw) == INV


def test_gather_topk_zero_work_ok(psk_lib):
    assert _gather_topk(T=0, out=None, tk=None, t2r=None) == OK
    assert _gather_topk(K=0, tks=0, out=None, tk=None, t2r=None) == OK
    # an empty table needs no pointer: every slot resolves to -1
    assert _gather_topk(T=0, btw=0, bt=None) == OK


def _gather_window(**kw):
    a = dict(out=A, ost=128 * 512, osj=512, cache=B, num_pages=8, page_stride=64 * 584, bs=64,
             D=512, rope=64, qsl=C, seq=C + 64, t2r=C + 128, replay=None, R=2, T=4,
             bt=C + 8192, bts=16, btw=16, base=None, W=128, valid=None)
    a.update(kw)
    return _abi.status("dequantize_and_gather_k_cache_window", a["out"], a["ost"], a["osj"],
                       a["cache"], a["num_pages"], a["page_stride"], a["bs"], a["D"], a["rope"],
                       a["qsl"], a["seq"], a["t2r"], a["replay"], a["R"], a["T"], a["bt"],
                       a["bts"], a["btw"], a["base"], a["W"], a["valid"], None)


@pytest.mark.parametrize("kw", [dict(D=100), dict(rope=16), dict(D=128, rope=128),
                                dict(out=A + 8), dict(osj=4), dict(ost=-8), dict(qsl=None),
                                dict(seq=None), dict(t2r=None), dict(bt=None), dict(out=None),
                                dict(T=-1), dict(W=-1), dict(R=0), dict(bts=8),
                                dict(page_stride=1000), dict(replay=C + 2), dict(seq=C + 1),
                                dict(cache=None)])
def test_gather_window_rejects_bad_arguments(psk_lib, kw):
    assert _gather_window(**kw) == INV


def test_gather_window_zero_work_ok(psk_lib):
    assert _gather_window(T=0, out=None, qsl=None, seq=None, t2r=None) == OK
    assert _gather_window(W=0, out=None, qsl=None, seq=None, t2r=None) == OK


@pytest.mark.parametrize("limit", [0, 999, 10**9 + 1, 2**63])
def test_wait_selftest_rejects_bad_limit(psk_lib, limit):
    assert _abi.status("psk_device_wait_selftest", limit, None) == INV


def _gather_pair(**kw):
    a = dict(out=A, ost=640 * 512, osj=512, ca=B, npa=8, psa=64 * 584, bsa=64, cb=B + 4096,
             npb=4, psb=16 * 592, bsb=16, D=512, rope=64, idx=C, ids=640, rows=4, cols=640,
             split=128)
    a.update(kw)
    return _abi.status("dequantize_and_gather_k_cache_pair", a["out"], a["ost"], a["osj"], a["ca"],
                       a["npa"], a["psa"], a["bsa"], a["cb"], a["npb"], a["psb"], a["bsb"], a["D"],
                       a["rope"], a["idx"], a["ids"], a["rows"], a["cols"], a["split"], None)


@pytest.mark.parametrize("kw", [dict(D=100), dict(rope=16), dict(out=A + 8), dict(osj=4),
                                dict(ost=-8), dict(ids=100), dict(idx=None), dict(out=None),
                                dict(rows=-1), dict(split=-1), dict(split=641),
                                dict(psa=1000), dict(psb=16 * 500), dict(ca=None), dict(cb=None),
                                dict(cb=B + 8), dict(npb=0), dict(bsb=0)])
def test_gather_pair_rejects_bad_arguments(psk_lib, kw):
    assert _gather_pair(**kw) == INV


def test_gather_pair_zero_work_ok(psk_lib):
    assert _gather_pair(rows=0, out=None, idx=None) == OK
    assert _gather_pair(cols=0, ids=0, split=0, out=None, idx=None) == OK


def _gather_dense(**kw):
    a = dict(out=A, ost=40 * 512, osj=512, cache=B, num_pages=8, page_stride=64 * 584, bs=64,
             D=512, rope=64, pos=C, T=4, t2r=C + 4096, R=2, bt=C + 8192, bts=16, btw=16,
             base=None, ratio=128, width=40, valid=None)
    a.update(kw)
    return _abi.status("dequantize_and_gather_k_cache_dense", a["out"], a["ost"], a["osj"],
                       a["cache"], a["num_pages"], a["page_stride"], a["bs"], a["D"], a["rope"],
                       a["pos"], a["T"], a["t2r"], a["R"], a["bt"], a["bts"], a["btw"], a["base"],
                       a["ratio"], a["width"], a["valid"], None)


@pytest.mark.parametrize("kw", [dict(D=100), dict(rope=16), dict(out=A + 8), dict(osj=4),
                                dict(ost=-8), dict(pos=None), dict(t2r=None), dict(bt=None),
                                dict(out=None), dict(T=-1), dict(width=-1), dict(R=0),
                                dict(ratio=0), dict(bts=8), dict(page_stride=1000),
                                dict(pos=C + 4), dict(t2r=C + 4098), dict(cache=None)])
def test_gather_dense_rejects_bad_arguments(psk_lib, kw):
    assert _gather_dense(**kw) == INV


def test_gather_dense_zero_work_ok(psk_lib):
    assert _gather_dense(T=0, out=None, pos=None, t2r=None) == OK
    assert _gather_dense(width=0, out=None, pos=None, t2r=None) == OK
