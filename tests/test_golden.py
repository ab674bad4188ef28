"""The buffer sizes the pages print (tests/golden/page_size_figures.json), recomputed
from their shapes, and what the plan needs instead for the same shapes."""
import json
import os

import numpy as np
import pytest

from sparse_attention_prefill_tcgen05_gb300 import _lib as K

HERE = os.path.dirname(os.path.abspath(__file__))
FIG = json.load(open(os.path.join(HERE, "golden", "page_size_figures.json")))["figures"]


@pytest.mark.parametrize("fig", FIG, ids=[f["name"] for f in FIG])
def test_printed_sizes_follow_from_their_shapes(fig):
    b = fig["rows"] * fig["keys"] * fig["bytes_per_pair"]
    if "printed_gib" in fig:
        assert round(b / 2**30, 2 if fig["printed_gib"] < 10 else 1) == fig["printed_gib"]
    else:
        assert round(b / 1e9, 1) == fig["printed_gb"]


def _plan(rows, keys, topk, **kw):
    cl = np.arange(keys - rows + 1, keys + 1, dtype=np.int32)
    return K.indexer_plan(np.array([0, rows], np.int32), np.array([0, keys], np.int32), cl,
                          32, 128, topk, **kw)


def test_fused_transient_of_the_long_chunk_is_below_every_printed_buffer():
    logits = next(f for f in FIG if f["name"].startswith("materialised fp32 logits"))
    plan = _plan(logits["rows"], logits["keys"], 512)
    assert plan.workspace_bytes <= 2 << 30
    assert plan.workspace_bytes < logits["rows"] * logits["keys"] * 4 / 25


def test_block_mask_is_an_eighth_of_the_key_level_mask():
    """The candidate mask here is one byte per 8-key block: the key-level mask the
    pages publish (16 GiB for a 16K chunk at 1M context) becomes 2 GiB."""
    fig = next(f for f in FIG if f["name"].startswith("key-level published mask"))
    block_bytes = fig["rows"] * ((fig["keys"] + 7) // 8)
    assert block_bytes * 8 == fig["rows"] * fig["keys"]
    assert block_bytes / 2**30 == pytest.approx(2.0)
