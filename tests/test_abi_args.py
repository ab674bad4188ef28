"""Argument checks of the C ABI on the host (CPU only): every entry point rejects bad
arguments with IDX_ERR_INVALID_ARG (or IDX_ERR_WORKSPACE) before it touches a device.
Pointers are dummy, well-aligned addresses: none of these calls dereferences them."""
import ctypes

import numpy as np
import pytest

from sparse_attention_prefill_tcgen05_gb300 import _lib as K

A = ctypes.c_void_p(0x100000)          # a 1 MiB-aligned dummy address, never dereferenced
NULL = ctypes.c_void_p(0)


def _plan(topk=16, requests=((40, 300), (20, 900))):
    cu_q = np.concatenate([[0], np.cumsum([r for r, _ in requests])]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum([l for _, l in requests])]).astype(np.int32)
    cl = np.concatenate([np.full(r, l) for r, l in requests]).astype(np.int32)
    return K.indexer_plan(cu_q, cu_k, cl, 32, 128, topk, cand_block=8, cand_topk=8)


def test_page_indices_arguments():
    L = K.lib()
    plan = _plan()
    h = plan.handle
    assert L.indexer_page_indices(h, A, A, 1000, 0, A, NULL) == K.IDX_ERR_INVALID_ARG    # page 0
    assert L.indexer_page_indices(h, A, A, 14, 64, A, NULL) == K.IDX_ERR_INVALID_ARG     # 900/64 -> 15
    assert L.indexer_page_indices(h, NULL, A, 15, 64, A, NULL) == K.IDX_ERR_INVALID_ARG
    assert L.indexer_page_indices(None, A, A, 15, 64, A, NULL) == K.IDX_ERR_INVALID_ARG


def test_convert_fp4_arguments():
    L = K.lib()
    def call(codes=A, sf=A, rows=10, D=128, out=A, scale=A, ws=A, ws_bytes=256):
        return L.indexer_convert_fp4(codes, sf, rows, D, out, scale, ws, ws_bytes, NULL)
    assert call(D=48) == K.IDX_ERR_INVALID_ARG                       # not a multiple of 32
    assert call(ws_bytes=128) == K.IDX_ERR_INVALID_ARG               # no room for the status
    assert call(ws=ctypes.c_void_p(0x100010)) == K.IDX_ERR_INVALID_ARG   # not 256-aligned
    assert call(codes=ctypes.c_void_p(0x100002)) == K.IDX_ERR_INVALID_ARG
    assert call(rows=-1) == K.IDX_ERR_INVALID_ARG
    assert call(out=NULL) == K.IDX_ERR_INVALID_ARG


def test_tail_and_mapped_arguments():
    L = K.lib()
    plan = _plan()
    h = plan.handle
    ws_bytes = plan.workspace_bytes
    ldm = (900 + 7) // 8
    for bad in ([41, 0], [-1, 0], [0, 21]):
        tails = np.array(bad, dtype=np.int32)
        rc = L.indexer_candidate_blocks_tail(h, A, A, A, A, A, A,
                                             tails.ctypes.data_as(ctypes.c_void_p), A, ldm, A,
                                             ws_bytes, NULL)
        assert rc == K.IDX_ERR_INVALID_ARG, bad
    rc = L.indexer_candidate_blocks_tail(h, A, A, A, A, A, A, NULL, A, ldm, A, ws_bytes, NULL)
    assert rc == K.IDX_ERR_INVALID_ARG
    # a workspace below the plan's size is a workspace error, not an argument error
    tails = np.array([1, 1], dtype=np.int32)
    rc = L.indexer_candidate_blocks_tail(h, A, A, A, A, A, A,
                                         tails.ctypes.data_as(ctypes.c_void_p), A, ldm, A,
                                         ws_bytes - 1, NULL)
    assert rc == K.IDX_ERR_WORKSPACE
    # the mapped consumer needs a mask and a row map with at least one row
    rc = L.indexer_fused_topk_mapped(h, A, A, A, A, A, A, A, ldm, NULL, 4, A, NULL, A,
                                     ws_bytes, NULL)
    assert rc == K.IDX_ERR_INVALID_ARG
    rc = L.indexer_fused_topk_mapped(h, A, A, A, A, A, A, A, ldm, A, 0, A, NULL, A, ws_bytes,
                                     NULL)
    assert rc == K.IDX_ERR_INVALID_ARG
    rc = L.indexer_fused_topk_mapped(h, A, A, A, A, A, A, NULL, ldm, A, 4, A, NULL, A,
                                     ws_bytes, NULL)
    assert rc == K.IDX_ERR_INVALID_ARG


def test_fallback_rows_arguments():
    L = K.lib()
    plan = _plan()
    assert L.indexer_fallback_rows(None, A, NULL) == K.IDX_ERR_INVALID_ARG
    assert L.indexer_fallback_rows(plan.handle, NULL, NULL) == K.IDX_ERR_INVALID_ARG
