"""Thin ctypes binding of ``libindexer.so`` (argument marshalling only).

Every function here has the name of the C entry point it calls (see
``include/indexer.h``) and does nothing but turn torch tensors into raw
pointers and the current CUDA stream into a ``cudaStream_t``.  All compute
runs in the library's CUDA kernels.  If the library has not been built,
loading it raises: there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libindexer.so")

IDX_OK = 0
IDX_ERR_INVALID_ARG = -1
IDX_ERR_UNSUPPORTED = -2
IDX_ERR_WORKSPACE = -3
IDX_ERR_CUDA = -4
IDX_ERR_TIMEOUT = -5
IDX_ERR_DEVICE_CHECK = -6
IDX_K_FP8_E4M3 = 0
IDX_K_FP4_E2M1_UE8M0 = 1
IDX_Q_FP8_E4M3 = 0
IDX_Q_FP4_E2M1_UE8M0 = 1
IDX_SELECT_AUTO = 0
IDX_SELECT_STREAM = 1

EXPORTED = ("indexer_plan", "indexer_plan_destroy", "indexer_plan_info", "indexer_logits",
            "indexer_topk", "indexer_fused_topk", "indexer_candidate_blocks",
            "indexer_expand_mask", "indexer_status", "indexer_selftest_timeout",
            "indexer_set_wait_budget", "indexer_launch_count", "indexer_error_string",
            "indexer_version", "indexer_fused_topk_noalloc", "indexer_profile_main_kernel",
            "indexer_chunk_rows", "indexer_page_indices", "indexer_candidate_blocks_tail",
            "indexer_fused_topk_mapped", "indexer_convert_fp4", "indexer_fallback_rows",
            "indexer_noalloc_status")
IDX_NOALLOC_SCRATCH_BYTES = 64 << 20


class IndexerError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {code} ({error_string(code)})")


class _Problem(ctypes.Structure):
    _fields_ = [
        ("num_requests", ctypes.c_int32), ("total_rows", ctypes.c_int32),
        ("total_keys", ctypes.c_int32), ("H", ctypes.c_int32), ("D", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.POINTER(ctypes.c_int32)),
        ("cu_seqlens_k", ctypes.POINTER(ctypes.c_int32)),
        ("compress_len", ctypes.POINTER(ctypes.c_int32)),
        ("kdtype", ctypes.c_int32), ("cand_block", ctypes.c_int32),
        ("cand_topk", ctypes.c_int32), ("key_block", ctypes.c_int32),
        ("transient_budget_bytes", ctypes.c_uint64),
        ("select_mode", ctypes.c_int32), ("qdtype", ctypes.c_int32),
    ]


_lib = None


def lib():
    """Load the library (raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run "
                               "python -m sparse_attention_prefill_tcgen05_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        L.indexer_plan.argtypes = [ctypes.POINTER(_Problem), ctypes.POINTER(P),
                                   ctypes.POINTER(sz)]
        L.indexer_plan_destroy.argtypes = [P]
        L.indexer_plan_destroy.restype = None
        L.indexer_plan_info.argtypes = [P, ctypes.POINTER(ctypes.c_int32),
                                        ctypes.POINTER(ctypes.c_int32),
                                        ctypes.POINTER(ctypes.c_int32),
                                        ctypes.POINTER(ctypes.c_int32)]
        L.indexer_logits.argtypes = [P, P, P, P, P, P, P, P, i64, P, sz, P]
        L.indexer_topk.argtypes = [P, P, i64, P, P, P, P, sz, P]
        L.indexer_fused_topk.argtypes = [P, P, P, P, P, P, P, P, i64, P, P, P, sz, P]
        L.indexer_candidate_blocks.argtypes = [P, P, P, P, P, P, P, P, i64, P, sz, P]
        L.indexer_expand_mask.argtypes = [P, P, i64, P, P, i64, P]
        L.indexer_status.argtypes = [P, P, P]
        L.indexer_selftest_timeout.argtypes = [P, ctypes.c_longlong, P]
        L.indexer_set_wait_budget.argtypes = [P, ctypes.c_longlong]
        L.indexer_launch_count.argtypes = []
        L.indexer_profile_main_kernel.argtypes = [P, P]
        L.indexer_profile_main_kernel.restype = None
        L.indexer_fused_topk_noalloc.argtypes = [P, P, P, P, P, P, P, P, i64, P, P, P]
        L.indexer_noalloc_status.argtypes = [P]
        L.indexer_chunk_rows.argtypes = [i64, ctypes.c_double, i32, i32, i32, i32]
        L.indexer_page_indices.argtypes = [P, P, P, i64, i32, P, P]
        L.indexer_convert_fp4.argtypes = [P, P, i64, i32, P, P, P, sz, P]
        L.indexer_candidate_blocks_tail.argtypes = [P, P, P, P, P, P, P, P, P, i64, P, sz, P]
        L.indexer_fused_topk_mapped.argtypes = [P, P, P, P, P, P, P, P, i64, P, i64, P, P, P,
                                                sz, P]
        L.indexer_error_string.argtypes = [i32]
        L.indexer_error_string.restype = ctypes.c_char_p
        for name in EXPORTED:
            if name not in ("indexer_plan_destroy", "indexer_error_string"):
                getattr(L, name).restype = ctypes.c_int
        L.indexer_launch_count.restype = ctypes.c_longlong
        L.indexer_fallback_rows.argtypes = [P, P, P]
        L.indexer_fallback_rows.restype = ctypes.c_longlong
        _lib = L
    return _lib


def error_string(code: int) -> str:
    try:
        return lib().indexer_error_string(int(code)).decode()
    except Exception:  # library missing: still format the code
        return str(code)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, rc: int):
    if rc != IDX_OK:
        raise IndexerError(fn, rc)


class Plan:
    """Owns an ``indexer_plan_t``; destroyed with the object."""

    def __init__(self, handle, workspace_bytes: int, problem: _Problem, keepalive):
        self.handle = handle
        self.workspace_bytes = workspace_bytes
        self.problem = problem
        self._keep = keepalive

    def info(self):
        kb, rc, ns, st = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check("indexer_plan_info", lib().indexer_plan_info(
            self.handle, ctypes.byref(kb), ctypes.byref(rc), ctypes.byref(ns), ctypes.byref(st)))
        return {"key_block": kb.value, "row_chunk": rc.value, "max_splits": ns.value,
                "sample_stride": st.value}

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h is not None and _lib is not None:
            _lib.indexer_plan_destroy(h)


def indexer_plan(cu_seqlens_q, cu_seqlens_k, compress_len, H: int, D: int, topk: int,
                 kdtype: int = IDX_K_FP8_E4M3, cand_block: int = 0, cand_topk: int = 0,
                 key_block: int = 0, transient_budget_bytes: int = 0,
                 select_mode: int = 0, qdtype: int = IDX_Q_FP8_E4M3) -> Plan:
    """Host-only planning: lengths are host (CPU) int32 arrays/tensors.  With
    ``qdtype=IDX_Q_FP4_E2M1_UE8M0`` the calls take q as packed e2m1 [T, H, D/2] and its
    ue8m0 block scales [T, H, D/32] (uint8) in the ``s_q`` argument."""
    def host_i32(x):
        t = torch.as_tensor(x).to(device="cpu", dtype=torch.int32).contiguous()
        return t, t.numpy().ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

    cq, pq = host_i32(cu_seqlens_q)
    ck, pk = host_i32(cu_seqlens_k)
    cl, pl = host_i32(compress_len)
    prob = _Problem(num_requests=cq.numel() - 1, total_rows=int(cq[-1]), total_keys=int(ck[-1]),
                    H=H, D=D, topk=topk, cu_seqlens_q=pq, cu_seqlens_k=pk, compress_len=pl,
                    kdtype=kdtype, cand_block=cand_block, cand_topk=cand_topk,
                    key_block=key_block, transient_budget_bytes=transient_budget_bytes,
                    select_mode=select_mode, qdtype=qdtype)
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    _check("indexer_plan", lib().indexer_plan(ctypes.byref(prob), ctypes.byref(handle),
                                              ctypes.byref(ws)))
    return Plan(handle, ws.value, prob, (cq, ck, cl))


def indexer_logits(plan: Plan, q, s_q, w, k, k_scale, compress_len, logits, ws, stream=None):
    _check("indexer_logits", lib().indexer_logits(
        plan.handle, _ptr(q), _ptr(s_q), _ptr(w), _ptr(k), _ptr(k_scale), _ptr(compress_len),
        _ptr(logits), logits.stride(0), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def indexer_topk(plan: Plan, logits, compress_len, out_idx, out_val, ws, stream=None):
    _check("indexer_topk", lib().indexer_topk(
        plan.handle, _ptr(logits), logits.stride(0), _ptr(compress_len), _ptr(out_idx),
        _ptr(out_val), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def indexer_fused_topk(plan: Plan, q, s_q, w, k, k_scale, compress_len, cand_mask, out_idx,
                       out_val, ws, stream=None):
    ldm = cand_mask.stride(0) if cand_mask is not None else 0
    _check("indexer_fused_topk", lib().indexer_fused_topk(
        plan.handle, _ptr(q), _ptr(s_q), _ptr(w), _ptr(k), _ptr(k_scale), _ptr(compress_len),
        _ptr(cand_mask), ldm, _ptr(out_idx), _ptr(out_val), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def indexer_candidate_blocks(plan: Plan, q, s_q, w, k, k_scale, compress_len, cand_mask, ws,
                             stream=None):
    _check("indexer_candidate_blocks", lib().indexer_candidate_blocks(
        plan.handle, _ptr(q), _ptr(s_q), _ptr(w), _ptr(k), _ptr(k_scale), _ptr(compress_len),
        _ptr(cand_mask), cand_mask.stride(0), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def indexer_candidate_blocks_tail(plan: Plan, q, s_q, w, k, k_scale, compress_len,
                                  publish_rows, cand_mask, ws, stream=None):
    """Candidate blocks of each request's last ``publish_rows[r]`` rows only, packed into
    ``cand_mask`` [sum(publish_rows), ld_mask] (``publish_rows``: a host sequence)."""
    pr = np.ascontiguousarray(np.asarray(publish_rows, dtype=np.int32))
    _check("indexer_candidate_blocks_tail", lib().indexer_candidate_blocks_tail(
        plan.handle, _ptr(q), _ptr(s_q), _ptr(w), _ptr(k), _ptr(k_scale), _ptr(compress_len),
        pr.ctypes.data_as(ctypes.c_void_p), _ptr(cand_mask), cand_mask.stride(0), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def indexer_fused_topk_mapped(plan: Plan, q, s_q, w, k, k_scale, compress_len, cand_mask,
                              mask_rows, out_idx, out_val, ws, stream=None):
    """indexer_fused_topk where row t reads candidate-mask row ``mask_rows[t]`` (device int32)."""
    _check("indexer_fused_topk_mapped", lib().indexer_fused_topk_mapped(
        plan.handle, _ptr(q), _ptr(s_q), _ptr(w), _ptr(k), _ptr(k_scale), _ptr(compress_len),
        _ptr(cand_mask), cand_mask.stride(0), _ptr(mask_rows), cand_mask.shape[0],
        _ptr(out_idx), _ptr(out_val), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def indexer_expand_mask(plan: Plan, cand_mask, compress_len, key_mask, stream=None):
    _check("indexer_expand_mask", lib().indexer_expand_mask(
        plan.handle, _ptr(cand_mask), cand_mask.stride(0), _ptr(compress_len), _ptr(key_mask),
        key_mask.stride(0), _stream(stream)))


def indexer_status(plan: Optional[Plan], ws, stream=None) -> int:
    return int(lib().indexer_status(plan.handle if plan is not None else None, _ptr(ws),
                                    _stream(stream)))


def indexer_selftest_timeout(ws, cycles: int, stream=None):
    _check("indexer_selftest_timeout",
           lib().indexer_selftest_timeout(_ptr(ws), int(cycles), _stream(stream)))


def indexer_set_wait_budget(plan: Plan, cycles: int):
    _check("indexer_set_wait_budget", lib().indexer_set_wait_budget(plan.handle, int(cycles)))


def indexer_fused_topk_noalloc(plan: Plan, q, s_q, w, k, k_scale, compress_len, cand_mask,
                               out_idx, out_val, stream=None):
    """indexer_fused_topk with the library's fixed device scratch as the workspace."""
    ldm = cand_mask.stride(0) if cand_mask is not None else 0
    _check("indexer_fused_topk_noalloc", lib().indexer_fused_topk_noalloc(
        plan.handle, _ptr(q), _ptr(s_q), _ptr(w), _ptr(k), _ptr(k_scale), _ptr(compress_len),
        _ptr(cand_mask), ldm, _ptr(out_idx), _ptr(out_val), _stream(stream)))


def indexer_noalloc_status(stream=None) -> int:
    """Status word of the last indexer_fused_topk_noalloc call on this device (syncs)."""
    return int(lib().indexer_noalloc_status(_stream(stream)))


def indexer_launch_count() -> int:
    return int(lib().indexer_launch_count())


def indexer_profile_main_kernel(start_event=None, stop_event=None):
    """Record two torch.cuda.Event (already created, timing enabled) around the main
    logits launch of the following top-k calls; no arguments turns it off."""
    h = lambda e: ctypes.c_void_p(e.cuda_event) if e is not None else None
    lib().indexer_profile_main_kernel(h(start_event), h(stop_event))


def indexer_fallback_rows(plan: Plan, ws, stream=None) -> int:
    """Rows the last top-k / candidate call on ``ws`` sent to the exact path (syncs)."""
    n = int(lib().indexer_fallback_rows(plan.handle, _ptr(ws), _stream(stream)))
    if n < 0:
        raise IndexerError("indexer_fallback_rows", n)
    return n


def indexer_version() -> int:
    return int(lib().indexer_version())


def indexer_convert_fp4(codes, block_scales, out_e4m3, out_scale, ws, stream=None):
    """e2m1 + ue8m0/32 rows -> e4m3 rows + fp32 row scales, exactly (see the header);
    ``codes`` [rows, D/2] and ``block_scales`` [rows, D/32] uint8 on the device."""
    rows, half = codes.shape[0], codes.shape[-1]
    _check("indexer_convert_fp4", lib().indexer_convert_fp4(
        _ptr(codes), _ptr(block_scales), rows, 2 * half, _ptr(out_e4m3), _ptr(out_scale),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def indexer_page_indices(plan: Plan, raw_idx, page_table, page_size: int, page_idx=None,
                         stream=None):
    """KV-slot indices of selected raw key indices: page_table[r, j // page_size] *
    page_size + j % page_size, -1 for -1 / out-of-range keys / unmapped pages.  ``raw_idx``
    int32 [rows, topk] and ``page_table`` int32 [requests, ld] on the device; writes into
    ``page_idx`` (default: a new tensor; may be ``raw_idx``) and returns it."""
    if page_idx is None:
        page_idx = torch.empty_like(raw_idx)
    for name, t in (("raw_idx", raw_idx), ("page_table", page_table), ("page_idx", page_idx)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name}: contiguous int32 CUDA tensor expected")
    _check("indexer_page_indices", lib().indexer_page_indices(
        plan.handle, _ptr(raw_idx), _ptr(page_table), page_table.stride(0), int(page_size),
        _ptr(page_idx), _stream(stream)))
    return page_idx


def indexer_chunk_rows(prefix_len: int, budget_token2: float = 2.0e8, chunk_min: int = 256,
                       chunk_max: int = 2048, page: int = 256, pow2: bool = False) -> int:
    """Prefill chunk size for a prefix of ``prefix_len`` compressed keys under a T x L budget
    (the library's host-only planner helper; raises on invalid arguments)."""
    r = int(lib().indexer_chunk_rows(int(prefix_len), float(budget_token2), int(chunk_min),
                                     int(chunk_max), int(page), 1 if pow2 else 0))
    if r < 0:
        raise IndexerError("indexer_chunk_rows", r)
    return r
