"""The allocation-free fused top-k (indexer_fused_topk_noalloc).

Some callers cannot allocate device memory: a plugin whose host application
owns all device memory through its own pool, or a serving loop where a
cudaMalloc would stall the device.  For them the library runs the fused
top-k out of a fixed 64 MiB device array it holds itself.  This checks,
through the C ABI, that two calls in a row (on different problems, so the
second one starts from the first one's leftovers) give, bit for bit, what
the regular entry point gives with a caller-allocated workspace: for fp8
keys, for e2m1 keys (block-scaled MMA), for e2m1 queries and keys (fp4 MMA kind)
and for a consumer reading a candidate mask.  A call whose e2m1 keys the conversion refuses reports it through
indexer_noalloc_status, and a plan too big for the array is refused.  Kept in
its own file, collected last.
"""
import dataclasses

import pytest
import torch

from sparse_attention_prefill_tcgen05_gb300 import _lib as K
from sparse_attention_prefill_tcgen05_gb300 import workloads as W

from . import helpers as Hp

pytestmark = pytest.mark.gpu

BUDGET = K.IDX_NOALLOC_SCRATCH_BYTES


def _problem(name, rows_div, keys_div, topk, seed, **over):
    spec = dataclasses.replace(W.scaled(W.CONFIGS[name], rows_div, keys_div), topk=topk,
                               seed=seed, **over)
    return W.make_problem(spec)


def _noalloc(p, plan, d, mask=None):
    T = int(p.cu_seqlens_q[-1])
    idx = torch.full((T, plan.problem.topk), -7, dtype=torch.int32, device="cuda")
    val = torch.full((T, plan.problem.topk), 7.0, dtype=torch.float32, device="cuda")
    K.indexer_fused_topk_noalloc(plan, d["q"], d["s_q"], d["w"], d["k"], d["k_scale"],
                                 d["compress_len"], mask, idx, val)
    assert K.indexer_noalloc_status() == K.IDX_OK
    return idx, val


def _check_pair(p, mask=None, layer=1):
    plan = Hp.make_plan(p, budget=BUDGET)
    assert plan.workspace_bytes <= BUDGET
    d = Hp.device_inputs(p, layer=layer)
    ri, rv = Hp.gpu_fused(p, plan, d, mask=mask)
    ni, nv = _noalloc(p, plan, d, mask=mask)
    # the same kernels on the same plan: identical bits, indices and values
    assert torch.equal(ni, ri)
    assert torch.equal(nv, rv)


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    problems = [_problem("cold64k", 8, 8, 300, seed=21),
                _problem("long488k", 64, 64, 128, seed=22)]
    for p in problems:
        _check_pair(p)


def test_noalloc_fp4_keys_and_masked_consumer():
    """e2m1 keys scored by the block-scaled MMA; a consumer reads a block mask."""
    _check_pair(_problem("v4ratio2", 16, 32, 64, seed=31))
    spec = dataclasses.replace(W.CONFIGS["ragged_cand"], topk=40, cand_topk=30, seed=32,
                               requests=(W.RequestSpec(90, 0, 1), W.RequestSpec(50, 2000, 1)))
    p = W.make_problem(spec)
    plan = Hp.make_plan(p)
    mask = Hp.gpu_candidates(p, plan, Hp.device_inputs(p))
    _check_pair(p, mask=mask, layer=2)


def test_noalloc_fp4_queries_and_keys():
    """e2m1 queries and keys on the fp4 MMA kind through the allocation-free entry point."""
    _check_pair(_problem("v4fp4qk", 16, 32, 64, seed=34))


def test_noalloc_reports_a_refused_fp4_key():
    """With 16 heads e2m1 keys are converted to e4m3 inside the array; a key whose block
    scales span 2^10 with a 0.5 code in the small block has no exact e4m3 form.  The
    status word in the array reports it, and the next good call clears it."""
    spec = W.ProblemSpec("H=16 fp4", (W.RequestSpec(24, 400, 1),), H=16, D=128, topk=16,
                         kdtype="fp4", seed=33)
    p = W.make_problem(spec)
    k, ks = p.k.clone(), p.k_scale.clone()
    ks[0, 0] = 127 + 10
    ks[0, 1] = 127
    k[0, 16] = 0x11
    bad = dataclasses.replace(p, k=k, k_scale=ks)
    plan = Hp.make_plan(bad, budget=BUDGET)
    d = Hp.device_inputs(bad)
    T = int(bad.cu_seqlens_q[-1])
    idx = torch.empty((T, bad.topk), dtype=torch.int32, device="cuda")
    K.indexer_fused_topk_noalloc(plan, d["q"], d["s_q"], d["w"], d["k"], d["k_scale"],
                                 d["compress_len"], None, idx, None)
    assert K.indexer_noalloc_status() == K.IDX_ERR_DEVICE_CHECK
    _noalloc(p, Hp.make_plan(p, budget=BUDGET), Hp.device_inputs(p))


def test_noalloc_refuses_a_plan_larger_than_its_array():
    """The full cold chunk planned with the default 2 GiB budget needs more than the array
    holds: refused on the host before anything is launched."""
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
