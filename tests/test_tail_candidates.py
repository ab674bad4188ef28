"""Tail-only candidate publish and the consumer's mask-row map: the packed masks of
a subset of rows are byte-identical to the full call's rows, and a consumer reading
masks through a row map equals one reading the gathered masks (GPU)."""
import dataclasses

import numpy as np
import pytest
import torch

from sparse_attention_prefill_tcgen05_gb300 import _lib as K
from sparse_attention_prefill_tcgen05_gb300 import workloads as W
from tests import helpers as Hp

pytestmark = pytest.mark.gpu


def _problem():
    # the third request is long enough for the sampled candidate path
    spec = dataclasses.replace(W.CONFIGS["ragged_cand"], topk=48, cand_topk=30, requests=(
        W.RequestSpec(90, 0, 1), W.RequestSpec(60, 3000, 2), W.RequestSpec(50, 16000, 1)),
        seed=21)
    p = W.make_problem(spec)
    return p, Hp.make_plan(p)


def _tail_masks(p, plan, d, tails):
    b = p.spec.cand_block
    ldm = (Hp.max_keys(p) + b - 1) // b
    packed = torch.full((max(sum(tails), 1), ldm), 7, dtype=torch.uint8, device="cuda")
    ws = Hp.workspace(plan)
    K.indexer_candidate_blocks_tail(plan, d["q"], d["s_q"], d["w"], d["k"], d["k_scale"],
                                    d["compress_len"], tails, packed, ws)
    assert K.indexer_status(plan, ws) == K.IDX_OK
    return packed[:sum(tails)]


@pytest.mark.parametrize("tails", [[7, 0, 50], [90, 60, 1], [0, 0, 0]])
def test_tail_publish_equals_the_full_rows(tails):
    p, plan = _problem()
    d = Hp.device_inputs(p)
    full = Hp.gpu_candidates(p, plan, d).cpu().numpy()
    got = _tail_masks(p, plan, d, tails).cpu().numpy()
    cu = p.cu_seqlens_q.numpy()
    want = np.concatenate([full[cu[r + 1] - n:cu[r + 1]] for r, n in enumerate(tails)])
    assert got.shape == want.shape
    assert np.array_equal(got, want)


def test_mapped_consumer_equals_gathered_masks():
    p, plan = _problem()
    d = Hp.device_inputs(p)
    tails = [30, 20, 50]
    packed = _tail_masks(p, plan, d, tails)
    T = int(p.cu_seqlens_q[-1])
    rng = np.random.default_rng(5)
    rows = torch.from_numpy(rng.integers(0, packed.shape[0], size=T).astype(np.int32)).cuda()
    d2 = Hp.device_inputs(p, layer=2)
    want_i, want_v = Hp.gpu_fused(p, plan, d2, mask=packed[rows.long()].contiguous())
    idx = torch.empty_like(want_i)
    val = torch.empty_like(want_v)
    ws = Hp.workspace(plan)
    K.indexer_fused_topk_mapped(plan, d2["q"], d2["s_q"], d2["w"], d2["k"], d2["k_scale"],
                                d2["compress_len"], packed, rows, idx, val, ws)
    assert K.indexer_status(plan, ws) == K.IDX_OK
    assert torch.equal(idx, want_i)
    assert torch.equal(val, want_v)
    # a map entry outside the mask is reported
    rows[3] = packed.shape[0]
    K.indexer_fused_topk_mapped(plan, d2["q"], d2["s_q"], d2["w"], d2["k"], d2["k_scale"],
                                d2["compress_len"], packed, rows, idx, val, ws)
    assert K.indexer_status(plan, ws) == K.IDX_ERR_DEVICE_CHECK


def test_tail_counts_out_of_range_are_rejected():
    p, plan = _problem()
    d = Hp.device_inputs(p)
    with pytest.raises(K.IndexerError) as e:
        _tail_masks(p, plan, d, [91, 0, 0])
    assert e.value.code == K.IDX_ERR_INVALID_ARG
