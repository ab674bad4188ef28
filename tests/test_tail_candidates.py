"""Tail-only candidate publish and the consumer's mask-row map ("[SGLang PR 39187]",
Modifications: publish only each request's tail rows).  Against the CPU oracle: the
packed tail masks by the near-tie rule against the fp64 oracle and bit for bit against
the oracle's block selector on the GPU's own logits; the row-mapped consumer by the
near-tie rule under the gathered masks and bit for bit against the oracle's masked
selector on the GPU's own logits.  Against the GPU's own full-row calls: the packed
masks are byte-identical to the full call's rows, and the mapped consumer equals one
given the gathered masks."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import oracle as O
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


def test_tail_publish_with_fp4_queries_equals_the_full_rows():
    """The same for e2m1 queries and keys on the fp4 MMA kind (the full call's masks are
    checked against the oracle with the other fp4-query parity cases)."""
    spec = dataclasses.replace(W.CONFIGS["ragged_cand"], topk=48, cand_topk=30, requests=(
        W.RequestSpec(90, 0, 1), W.RequestSpec(60, 3000, 2), W.RequestSpec(50, 16000, 1)),
        seed=23, kdtype="fp4", qdtype="fp4")
    p = W.make_problem(spec)
    plan = Hp.make_plan(p)
    d = Hp.device_inputs(p)
    tails = [7, 60, 30]
    full = Hp.gpu_candidates(p, plan, d).cpu().numpy()
    got = _tail_masks(p, plan, d, tails).cpu().numpy()
    cu = p.cu_seqlens_q.numpy()
    want = np.concatenate([full[cu[r + 1] - n:cu[r + 1]] for r, n in enumerate(tails)])
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


def _tail_rows(p, tails):
    cu = p.cu_seqlens_q.numpy()
    return np.concatenate([np.arange(cu[r + 1] - n, cu[r + 1]) for r, n in enumerate(tails)]
                          ).astype(np.int64)


@pytest.mark.parametrize("tails", [[7, 0, 50], [90, 60, 1]])
def test_tail_publish_matches_the_oracle(tails):
    p, plan = _problem()
    d = Hp.device_inputs(p)
    got = _tail_masks(p, plan, d, tails).cpu().numpy()
    rows = _tail_rows(p, tails)
    cl = p.compress_len.numpy()[rows]
    b, ct = p.spec.cand_block, p.spec.cand_topk
    ref = O.problem_logits(p, rows)
    for i in range(len(rows)):
        Hp.check_mask_row(got[i], ref[i], int(cl[i]), b, ct)
    g = Hp.gpu_logits(p, plan, d).cpu().numpy()[rows].astype(np.float64)
    assert np.array_equal(O.candidates_rows(g, cl, b, ct, got.shape[1]), got)


def test_mapped_consumer_matches_the_oracle():
    p, plan = _problem()
    d = Hp.device_inputs(p)
    tails = [30, 20, 50]
    packed = _tail_masks(p, plan, d, tails)
    T = int(p.cu_seqlens_q[-1])
    rng = np.random.default_rng(9)
    rows = rng.integers(0, packed.shape[0], size=T).astype(np.int32)
    d2 = Hp.device_inputs(p, layer=2)
    idx = torch.empty((T, p.topk), dtype=torch.int32, device="cuda")
    val = torch.empty((T, p.topk), dtype=torch.float32, device="cuda")
    ws = Hp.workspace(plan)
    K.indexer_fused_topk_mapped(plan, d2["q"], d2["s_q"], d2["w"], d2["k"], d2["k_scale"],
                                d2["compress_len"], packed, torch.from_numpy(rows).cuda(), idx,
                                val, ws)
    assert K.indexer_status(plan, ws) == K.IDX_OK
    fi = idx.cpu().numpy()
    gathered = packed.cpu().numpy()[rows]
    cl = p.compress_len.numpy()
    b = p.spec.cand_block
    ref2 = O.problem_logits(p, np.arange(T), layer=2)
    for t in range(T):
        Hp.check_topk_row(fi[t], ref2[t], int(cl[t]), p.topk, mask_row=gathered[t], block=b)
    g2 = Hp.gpu_logits(p, plan, d2).cpu().numpy().astype(np.float64)
    want = O.topk_rows(g2, cl, p.topk, mask=gathered, mask_block=b)
    for t in range(T):
        assert np.array_equal(np.sort(fi[t][fi[t] >= 0]), np.sort(want[t][want[t] >= 0])), t
    m = fi >= 0
    assert np.array_equal(val.cpu().numpy()[m].astype(np.float64),
                          g2[np.nonzero(m)[0], fi[m]])
