"""The allocation-free fused top-k (indexer_fused_topk_noalloc).

Some callers cannot allocate device memory: a plugin whose host application
owns all device memory through its own pool, or a serving loop where a
cudaMalloc would stall the device.  For them the library runs the fused
top-k out of a fixed 64 MiB device array it holds itself.  This checks,
through the C ABI, that two calls in a row (on different problems, so the
second one starts from the first one's leftovers) give what the regular
entry point gives with a caller-allocated workspace, and that a plan too
big for the array is refused.  Kept in its own file, collected last.
"""
import dataclasses

import numpy as np
import pytest
import torch

from sparse_attention_prefill_tcgen05_gb300 import _lib as K
from sparse_attention_prefill_tcgen05_gb300 import workloads as W

from . import helpers as Hp

pytestmark = pytest.mark.gpu


def _problem(name, rows_div, keys_div, topk, seed):
    spec = dataclasses.replace(W.scaled(W.CONFIGS[name], rows_div, keys_div), topk=topk,
                               seed=seed)
    return W.make_problem(spec)


def _regular(p, plan, d):
    return Hp.gpu_fused(p, plan, d)


def _noalloc(p, plan, d):
    T = int(p.cu_seqlens_q[-1])
    idx = torch.full((T, plan.problem.topk), -7, dtype=torch.int32, device="cuda")
    val = torch.full((T, plan.problem.topk), 7.0, dtype=torch.float32, device="cuda")
    K.indexer_fused_topk_noalloc(plan, d["q"], d["s_q"], d["w"], d["k"], d["k_scale"],
                                 d["compress_len"], None, idx, val)
    torch.cuda.synchronize()
    return idx, val


def _same(a_idx, a_val, b_idx, b_val):
    ai, bi = a_idx.cpu().numpy(), b_idx.cpu().numpy()
    av, bv = a_val.cpu().numpy().astype(np.float64), b_val.cpu().numpy().astype(np.float64)
    for t in range(ai.shape[0]):
        assert set(ai[t].tolist()) == set(bi[t].tolist()), t
        m = ai[t] >= 0
        order_a = np.argsort(ai[t][m])
        order_b = np.argsort(bi[t][bi[t] >= 0])
        va = av[t][m][order_a]
        vb = bv[t][bi[t] >= 0][order_b]
        assert np.all(np.abs(va - vb) <= Hp.LOGIT_RTOL * (1 + np.abs(vb))), t


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    budget = K.IDX_NOALLOC_SCRATCH_BYTES
    problems = [_problem("cold64k", 8, 8, 300, seed=21),
                _problem("long488k", 64, 64, 128, seed=22)]
    for p in problems:
        plan = Hp.make_plan(p, budget=budget)
        assert plan.workspace_bytes <= budget
        d = Hp.device_inputs(p)
        ri, rv = _regular(p, plan, d)
        ni, nv = _noalloc(p, plan, d)
        _same(ni, nv, ri, rv)


def test_noalloc_refuses_a_plan_larger_than_its_array():
    """The full cold chunk planned with the default 2 GiB budget needs ~0.5 GiB: refused on
    the host before anything is launched."""
    spec = W.CONFIGS["cold64k"]
    T, L = spec.total_rows, spec.total_keys
    cl = torch.tensor([r + 1 for r in range(L - T, L)], dtype=torch.int32)
    plan = K.indexer_plan(torch.tensor([0, T], dtype=torch.int32),
                          torch.tensor([0, L], dtype=torch.int32), cl, spec.H, spec.D, spec.topk)
    assert plan.workspace_bytes > K.IDX_NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(K.IndexerError) as e:
        K.indexer_fused_topk_noalloc(plan, dummy, dummy, dummy, dummy, dummy, dummy, None, dummy,
                                     None)
    assert e.value.code == K.IDX_ERR_WORKSPACE
