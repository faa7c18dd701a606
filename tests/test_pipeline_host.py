"""Host-side pipeline choices that need no GPU: which step a batch runs by
default, and which gather form its index matrix takes."""
import pytest

from paged_sparse_kv_gb300 import synthetic
from paged_sparse_kv_gb300.pipeline import Pipeline


@pytest.mark.parametrize("name,small,path", [("tiny", True, "fused"), ("decode", True, "fused"),
                                             ("prefill", False, "index"),
                                             ("mixed", False, "index"),
                                             ("mxfp4", True, "index"),
                                             ("decode_hca", True, "dense_fused")])
def test_default_path_follows_the_batch_size_rule(name, small, path):
    w = synthetic.make(name)
    items = w.num_tokens * (w.window + w.padded_topk)
    assert Pipeline.small_batch(w) == small == (items <= Pipeline.PAIR_MAX_ITEMS)
    # without an FP8 part (the MXFP4 indexer batch) there is no fused step; the
    # heavily compressed decode batch takes the dense step, fused when small
    assert Pipeline.default_path_for(w) == path


def test_rule_boundary():
    """The rule reads the token count, the window and the padded top-k width:
    one token past 2^20 index items flips both choices."""
    from types import SimpleNamespace
    w = synthetic.make("decode")
    cols = w.window + w.padded_topk
    at = SimpleNamespace(num_tokens=Pipeline.PAIR_MAX_ITEMS // cols, window=w.window,
                         padded_topk=w.padded_topk, has_fp8=True, dense_width=0)
    past = SimpleNamespace(**{**vars(at), "num_tokens": at.num_tokens + 1})
    assert Pipeline.small_batch(at) and Pipeline.default_path_for(at) == "fused"
    assert not Pipeline.small_batch(past) and Pipeline.default_path_for(past) == "index"


def test_size_one_leading_dims_ignore_their_stride():
    """A one-row table or one-page cache may carry any stride on its size-1
    dim (numpy broadcasting gives 0); the binding passes the row's extent
    instead, and keeps the stride of every other shape."""
    import numpy as np
    import torch
    from paged_sparse_kv_gb300 import ops
    table = torch.from_numpy(np.arange(6, dtype=np.int32)[None, :])
    assert table.stride(0) == 0 and ops._rows(table, "table") == 6
    wide = torch.zeros(1, 8, dtype=torch.int32)[:, :5]
    assert ops._rows(wide, "table") == 8
    assert ops._rows(torch.zeros(3, 8, dtype=torch.int32)[:, :5], "table") == 8
    cache = torch.from_numpy(np.zeros(592, np.uint8)[None, :])
    assert cache.stride(0) == 0 and ops._pages(cache) == (1, 592)
    assert ops._pages(torch.zeros(4, 600, dtype=torch.uint8)[:, :592]) == (4, 600)
    with pytest.raises(ValueError):
        ops._pages(torch.zeros(0, 592, dtype=torch.uint8))
