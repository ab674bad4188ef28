"""Page-index transform of the selected raw key indices: the oracle against a
worked example, the identity table and brute force (CPU), then the kernel
against the oracle, element for element (GPU)."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_attention_prefill_tcgen05_gb300 import _lib as K
from sparse_attention_prefill_tcgen05_gb300 import workloads as W
from tests import helpers as Hp


def test_oracle_worked_example():
    """Page size 4, one request of 16 keys, pages mapped 0->7, 1->2, 2 unmapped, 3->5."""
    raw = np.array([[0, 3, 4, 9, 13, -1, 16, 15]], dtype=np.int32)
    got = O.page_indices_rows(raw, [0], [16], np.array([[7, 2, -1, 5]]), 4)
    assert got.tolist() == [[28, 31, 8, -1, 21, -1, -1, 23]]


def test_oracle_identity_table_and_brute_force():
    rng = np.random.default_rng(1)
    L, P = 1000, 48
    pages = -(-L // P)
    raw = rng.integers(-1, L + 3, size=(6, 40)).astype(np.int32)
    ident = np.arange(pages)[None, :]
    got = O.page_indices_rows(raw, [0] * 6, [L], ident, P)
    want = np.where((raw >= 0) & (raw < L), raw, -1)
    assert np.array_equal(got, want)
    table = rng.permutation(4 * pages)[:pages][None, :].copy()
    table[0, 3] = -1
    got = O.page_indices_rows(raw, [0] * 6, [L], table, P)
    for t in range(6):
        for i in range(40):
            j = int(raw[t, i])
            q, rem = divmod(j, P) if 0 <= j < L else (None, None)
            want = -1 if q is None or table[0, q] < 0 else int(table[0, q]) * P + rem
            assert got[t, i] == want


def test_oracle_slot_past_int32_is_unmapped():
    got = O.page_indices_rows(np.array([[1]], np.int32), [0], [8], np.array([[2**30, 0]]), 4)
    assert got.tolist() == [[-1]]


def _plan_problem(topk):
    spec = dataclasses.replace(W.CONFIGS["ragged_cand"], topk=topk, cand_topk=0, requests=(
        W.RequestSpec(40, 0, 1), W.RequestSpec(30, 5000, 2), W.RequestSpec(25, 9000, 1)))
    p = W.make_problem(spec)
    return p, Hp.make_plan(p)


@pytest.mark.gpu
@pytest.mark.parametrize("topk,page", [(100, 64), (128, 48), (128, 256)])
def test_page_indices_match_the_oracle(topk, page):
    p, plan = _plan_problem(topk)
    rng = np.random.default_rng(topk + page)
    cu_q, cu_k = p.cu_seqlens_q.numpy(), p.cu_seqlens_k.numpy()
    T, R = int(cu_q[-1]), len(cu_q) - 1
    Ls = np.diff(cu_k)
    row_req = np.repeat(np.arange(R), np.diff(cu_q))
    raw = np.stack([rng.integers(-1, Ls[row_req[t]] + 4, size=topk) for t in range(T)])
    raw = raw.astype(np.int32)
    ld = -(-int(Ls.max()) // page) + 3
    table = rng.permutation(R * ld * 2)[:R * ld].reshape(R, ld).astype(np.int32)
    table[rng.random(table.shape) < 0.1] = -1
    want = O.page_indices_rows(raw, row_req, Ls, table, page)
    raw_d, table_d = torch.from_numpy(raw).cuda(), torch.from_numpy(table).cuda()
    got = K.indexer_page_indices(plan, raw_d, table_d, page).cpu().numpy()
    assert np.array_equal(got, want)
    # in place
    K.indexer_page_indices(plan, raw_d, table_d, page, page_idx=raw_d)
    assert np.array_equal(raw_d.cpu().numpy(), want)


@pytest.mark.gpu
def test_page_indices_of_a_fused_topk():
    """The transform applied to the fused top-k's own output."""
    p, plan = _plan_problem(64)
    d = Hp.device_inputs(p)
    fi, _ = Hp.gpu_fused(p, plan, d)
    cu_q, cu_k = p.cu_seqlens_q.numpy(), p.cu_seqlens_k.numpy()
    R = len(cu_q) - 1
    Ls = np.diff(cu_k)
    row_req = np.repeat(np.arange(R), np.diff(cu_q))
    page = 64
    ld = -(-int(Ls.max()) // page)
    table = np.arange(R * ld, dtype=np.int32).reshape(R, ld)[:, ::-1].copy()
    got = K.indexer_page_indices(plan, fi.contiguous(), torch.from_numpy(table).cuda(), page)
    want = O.page_indices_rows(fi.cpu().numpy(), row_req, Ls, table, page)
    assert np.array_equal(got.cpu().numpy(), want)


@pytest.mark.gpu
def test_page_table_too_short_is_rejected():
    p, plan = _plan_problem(32)
    raw = torch.zeros((int(p.cu_seqlens_q[-1]), 32), dtype=torch.int32, device="cuda")
    table = torch.zeros((3, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(K.IndexerError) as e:
        K.indexer_page_indices(plan, raw, table, 64)
    assert e.value.code == K.IDX_ERR_INVALID_ARG
