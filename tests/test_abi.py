"""The C ABI on the host (CPU only): the library loads, exports every entry
point the header declares, and the plan validates and sizes problems
without a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from sparse_attention_prefill_tcgen05_gb300 import _lib as K
from sparse_attention_prefill_tcgen05_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "indexer.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(indexer_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = K.lib()
    syms = declared_symbols()
    assert len(syms) >= 12
    for s in syms:
        assert hasattr(lib, s), s
    assert set(syms) == set(K.EXPORTED)
    assert K.indexer_version() >= 1
    assert K.error_string(K.IDX_ERR_WORKSPACE).startswith("workspace")


def lens(spec):
    cu_q = np.concatenate([[0], np.cumsum([r.rows for r in spec.requests])]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum([r.keys for r in spec.requests])]).astype(np.int32)
    cl = np.concatenate([(np.arange(r.pos0, r.pos0 + r.rows) + 1) // r.ratio
                         for r in spec.requests]).astype(np.int32)
    return cu_q, cu_k, cl


@pytest.mark.parametrize("name", ["tiny", "cold64k", "long488k", "ragged_cand"])
def test_plans_fit_the_transient_budget(name):
    spec = W.CONFIGS[name]
    cu_q, cu_k, cl = lens(spec)
    plan = K.indexer_plan(cu_q, cu_k, cl, spec.H, spec.D, spec.topk,
                          cand_topk=spec.cand_topk, key_block=spec.key_block)
    assert plan.workspace_bytes <= 2 << 30
    info = plan.info()
    assert info["key_block"] % 128 == 0 and info["row_chunk"] >= 1


def test_long_context_transient_is_far_below_materialised_logits():
    """The pages print 16384 x 487936 x 4 B = 29.8 GiB for the [T, L] fp32 logits of this
    shape ("[DeepSeek-V4.1] Bound the dense prefill indexer transient", Motivation)."""
    spec = W.CONFIGS["long488k"]
    cu_q, cu_k, cl = lens(spec)
    materialised = 16384 * 487936 * 4
    assert round(materialised / 2**30, 1) == 29.8
    plan = K.indexer_plan(cu_q, cu_k, cl, spec.H, spec.D, spec.topk)
    assert plan.workspace_bytes <= 2 << 30 < materialised
    small = K.indexer_plan(cu_q, cu_k, cl, spec.H, spec.D, spec.topk,
                           transient_budget_bytes=512 << 20)
    assert small.workspace_bytes <= 512 << 20
    assert small.info()["key_block"] <= plan.info()["key_block"]


def expect(code, fn, *a, **kw):
    with pytest.raises(K.IndexerError) as e:
        fn(*a, **kw)
    assert e.value.code == code


def test_plan_rejects_bad_problems():
    cu_q = np.array([0, 4], np.int32)
    cu_k = np.array([0, 10], np.int32)
    cl = np.array([1, 2, 3, 4], np.int32)
    K.indexer_plan(cu_q, cu_k, cl, 32, 128, 8)
    expect(K.IDX_ERR_INVALID_ARG, K.indexer_plan, cu_q, cu_k, cl, 32, 128, 0)
    expect(K.IDX_ERR_INVALID_ARG, K.indexer_plan, cu_q, cu_k, cl, 32, 128, 4096)
    expect(K.IDX_ERR_INVALID_ARG, K.indexer_plan, cu_q, cu_k, np.array([1, 2, 3, 11], np.int32),
           32, 128, 8)                                    # compress_len > keys of the request
    expect(K.IDX_ERR_INVALID_ARG, K.indexer_plan, cu_q, cu_k, np.array([1, -1, 3, 4], np.int32),
           32, 128, 8)
    expect(K.IDX_ERR_INVALID_ARG, K.indexer_plan, np.array([0, 5, 4], np.int32),
           np.array([0, 5, 10], np.int32), np.zeros(4, np.int32), 32, 128, 8)  # decreasing
    expect(K.IDX_ERR_UNSUPPORTED, K.indexer_plan, cu_q, cu_k, cl, 24, 128, 8)
    expect(K.IDX_ERR_UNSUPPORTED, K.indexer_plan, cu_q, cu_k, cl, 32, 96, 8)
    # e2m1 keys: 32 heads are scored by the block-scaled MMA (no converted copy of the
    # keys in the workspace); 16 heads go through the exact e4m3 conversion
    fp4 = K.indexer_plan(cu_q, cu_k, cl, 16, 128, 8, kdtype=K.IDX_K_FP4_E2M1_UE8M0)
    fp8 = K.indexer_plan(cu_q, cu_k, cl, 16, 128, 8)
    assert fp4.workspace_bytes >= fp8.workspace_bytes + 10 * (128 + 4)   # converted keys
    fp4 = K.indexer_plan(cu_q, cu_k, cl, 32, 128, 8, kdtype=K.IDX_K_FP4_E2M1_UE8M0)
    fp8 = K.indexer_plan(cu_q, cu_k, cl, 32, 128, 8)
    assert fp4.workspace_bytes <= fp8.workspace_bytes + 256
    expect(K.IDX_ERR_INVALID_ARG, K.indexer_plan, cu_q, cu_k, cl, 32, 128, 8, key_block=100)
    expect(K.IDX_ERR_WORKSPACE, K.indexer_plan, cu_q, cu_k, cl, 32, 128, 8,
           transient_budget_bytes=512)


def test_plan_with_empty_rows_and_requests():
    cu_q = np.array([0, 0, 3, 3], np.int32)
    cu_k = np.array([0, 7, 7, 20], np.int32)
    cl = np.array([0, 0, 0], np.int32)
    plan = K.indexer_plan(cu_q, cu_k, cl, 32, 128, 4)
    assert plan.workspace_bytes >= 256


def test_calls_validate_arguments_before_touching_the_gpu():
    """Null/unaligned pointers are rejected on the host (no GPU is needed to see that)."""
    cu_q = np.array([0, 4], np.int32)
    cu_k = np.array([0, 10], np.int32)
    cl = np.array([1, 2, 3, 4], np.int32)
    plan = K.indexer_plan(cu_q, cu_k, cl, 32, 128, 8)
    lib = K.lib()
    rc = lib.indexer_fused_topk(plan.handle, None, None, None, None, None, None, None, 0, None,
                                None, ctypes.c_void_p(256), plan.workspace_bytes, None)
    assert rc == K.IDX_ERR_INVALID_ARG
    rc = lib.indexer_logits(plan.handle, ctypes.c_void_p(4096), ctypes.c_void_p(4096),
                            ctypes.c_void_p(4096), ctypes.c_void_p(4096), ctypes.c_void_p(4096),
                            ctypes.c_void_p(4096), ctypes.c_void_p(4096), 10,
                            ctypes.c_void_p(4096), 1, None)
    assert rc == K.IDX_ERR_WORKSPACE
    rc = lib.indexer_logits(plan.handle, ctypes.c_void_p(4097), ctypes.c_void_p(4096),
                            ctypes.c_void_p(4096), ctypes.c_void_p(4096), ctypes.c_void_p(4096),
                            ctypes.c_void_p(4096), ctypes.c_void_p(4096), 10,
                            ctypes.c_void_p(4096), plan.workspace_bytes, None)
    assert rc == K.IDX_ERR_INVALID_ARG
    assert lib.indexer_selftest_timeout(None, 10, None) == K.IDX_ERR_INVALID_ARG
