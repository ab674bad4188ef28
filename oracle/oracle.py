"""Python front end of the CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  It loads ``liboracle.so`` (built from
``oracle.c`` by :func:`build`) and works on numpy / CPU torch arrays.  It
imports nothing from the CUDA package: inputs come from the shared seeded
generator as plain arrays.

The arithmetic lives in ``oracle.c`` (see its header for the definition and
the passages it follows); this file only marshals arguments and walks the
ragged batch one request at a time, except for two small definitions written
out here in plain Python: the adaptive chunk size (:func:`chunk_rows`) and the
page-index transform (:func:`page_indices_rows`).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (OpenMP when the compiler has it)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:5] + ["-fopenmp"] + base[5:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int
        L.oracle_logits.argtypes = [i32, i32, i32, i64, P, P, P, i64, P, P, P, P, i32]
        L.oracle_logits.restype = i32
        L.oracle_topk.argtypes = [i64, P, i64, P, P, i64, i32, i32, P, P, i32]
        L.oracle_topk.restype = i32
        L.oracle_candidates.argtypes = [i64, P, i64, P, i32, i32, P, i64, P, i32]
        L.oracle_candidates.restype = i32
        L.oracle_select_pairs.argtypes = [i64, P, P, i32, P, P]
        L.oracle_select_pairs.restype = i32
        L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_value.restype = ctypes.c_double
        L.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        L.oracle_e2m1_value.restype = ctypes.c_double
        L.oracle_ue8m0_value.argtypes = [ctypes.c_uint8]
        L.oracle_ue8m0_value.restype = ctypes.c_double
        L.oracle_max_threads.restype = i32
        _lib = L
    return _lib


def _np(x, dtype):
    if hasattr(x, "numpy"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x), dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def e4m3_value(b: int) -> float:
    return float(lib().oracle_e4m3_value(b))


def e2m1_value(nib: int) -> float:
    return float(lib().oracle_e2m1_value(nib))


def ue8m0_value(e: int) -> float:
    return float(lib().oracle_ue8m0_value(e))


def logits_request(H, D, kdtype, q, s_q, w, k, k_scale, compress_len, nthreads=0):
    """fp64 logits of some rows of one request against that request's keys.

    q [n, H, D] e4m3 bytes, s_q/w [n, H], k [L, D] (fp8) or [L, D/2] (fp4),
    k_scale [L] float (fp8) or [L, D/32] ue8m0 bytes (fp4), compress_len [n].
    Returns [n, L] float64 with -inf past compress_len.
    """
    kd = {"fp8": 0, "fp4": 1}[kdtype] if isinstance(kdtype, str) else int(kdtype)
    q = _np(q, np.uint8)
    n = q.shape[0]
    s_q = _np(s_q, np.float32)
    w = _np(w, np.float32)
    k = _np(k, np.uint8)
    L = k.shape[0]
    ks = _np(k_scale, np.float32 if kd == 0 else np.uint8)
    cl = _np(compress_len, np.int32)
    out = np.empty((n, L), dtype=np.float64)
    rc = lib().oracle_logits(H, D, kd, n, _ptr(q), _ptr(s_q), _ptr(w), L, _ptr(k), _ptr(ks),
                             _ptr(cl), _ptr(out), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_logits failed: {rc}")
    return out


def topk_rows(vals, compress_len, k, mask=None, mask_block=8, nthreads=0, with_values=False):
    """Per-row top-k (ties to the lower index) over dense rows ``vals`` [n, ld]."""
    v = _np(vals, np.float64)
    n, ld = v.shape
    cl = _np(compress_len, np.int32)
    out = np.empty((n, k), dtype=np.int32)
    outv = np.empty((n, k), dtype=np.float64) if with_values else None
    if mask is not None:
        m = _np(mask, np.uint8)
        mp, ldm = _ptr(m), m.shape[1]
    else:
        mp, ldm = None, 0
    rc = lib().oracle_topk(n, _ptr(v), ld, _ptr(cl), mp, ldm, int(mask_block), int(k), _ptr(out),
                           _ptr(outv) if outv is not None else None, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_topk failed: {rc}")
    return (out, outv) if with_values else out


def candidates_rows(vals, compress_len, block, cand_topk, ld_mask, nthreads=0,
                    with_pooled=False):
    """Per-row candidate-block mask [n, ld_mask] (uint8 0/1) over dense rows ``vals``."""
    v = _np(vals, np.float64)
    n, ld = v.shape
    cl = _np(compress_len, np.int32)
    out = np.empty((n, ld_mask), dtype=np.uint8)
    pooled = np.empty((n, ld_mask), dtype=np.float64) if with_pooled else None
    rc = lib().oracle_candidates(n, _ptr(v), ld, _ptr(cl), int(block), int(cand_topk), _ptr(out),
                                 ld_mask, _ptr(pooled) if pooled is not None else None,
                                 int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_candidates failed: {rc}")
    return (out, pooled) if with_pooled else out


def select_pairs(vals, idx, k):
    """Top-k of explicit (value, index) pairs; returns (indices, values) padded with -1/-inf."""
    v = _np(vals, np.float64)
    i = _np(idx, np.int64)
    out = np.empty(k, dtype=np.int64)
    outv = np.empty(k, dtype=np.float64)
    rc = lib().oracle_select_pairs(v.shape[0], _ptr(v), _ptr(i), int(k), _ptr(out), _ptr(outv))
    if rc != 0:
        raise RuntimeError(f"oracle_select_pairs failed: {rc}")
    return out, outv


# ----------------------------------------------------------------- batches

def _request_arrays(p, rows, layer):
    """Group the requested rows by request; yield (r, local rows, global rows)."""
    cu_q = _np(p.cu_seqlens_q, np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    req = np.searchsorted(cu_q, rows, side="right") - 1
    for r in np.unique(req):
        sel = rows[req == r]
        yield int(r), sel


def _layer(p, layer):
    if layer == 2:
        return p.q2, p.s_q2, p.w2
    return p.q, p.s_q, p.w


def problem_logits(p, rows=None, layer=1, nthreads=0, ld=None):
    """fp64 logits of ``rows`` (global row ids) of problem ``p``.

    Returns [len(rows), ld] with ld = the largest L in the batch by default;
    entries past a row's compress_len (and past its request's L) are -inf.
    """
    T = int(p.cu_seqlens_q[-1])
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    cu_k = _np(p.cu_seqlens_k, np.int64)
    Lmax = int(np.max(np.diff(cu_k)))
    ld = Lmax if ld is None else ld
    q, s_q, w = _layer(p, layer)
    q, s_q, w = _np(q, np.uint8), _np(s_q, np.float32), _np(w, np.float32)
    k, ks = _np(p.k, np.uint8), p.k_scale
    ks = _np(ks, np.float32 if p.spec.kdtype == "fp8" else np.uint8)
    cl = _np(p.compress_len, np.int32)
    out = np.full((len(rows), ld), -np.inf, dtype=np.float64)
    pos_of = {int(g): i for i, g in enumerate(rows)}
    for r, sel in _request_arrays(p, rows, layer):
        k0, k1 = int(cu_k[r]), int(cu_k[r + 1])
        res = logits_request(p.H, p.D, p.spec.kdtype, q[sel], s_q[sel], w[sel], k[k0:k1],
                             ks[k0:k1], cl[sel], nthreads)
        idx = [pos_of[int(g)] for g in sel]
        out[idx, : k1 - k0] = res
    return out


def problem_topk(p, rows=None, layer=1, mask=None, nthreads=0, logits=None, k=None):
    """Oracle top-k indices [len(rows), k] (request-local key ids, -1 padded)."""
    T = int(p.cu_seqlens_q[-1])
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    vals = problem_logits(p, rows, layer, nthreads) if logits is None else logits
    cl = _np(p.compress_len, np.int32)[rows]
    return topk_rows(vals, cl, p.topk if k is None else k, mask=mask,
                     mask_block=p.spec.cand_block, nthreads=nthreads)


def problem_candidates(p, rows=None, nthreads=0, logits=None, ld_mask=None):
    """Oracle candidate-block masks [len(rows), ld_mask] of the source layer."""
    T = int(p.cu_seqlens_q[-1])
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    vals = problem_logits(p, rows, 1, nthreads) if logits is None else logits
    cl = _np(p.compress_len, np.int32)[rows]
    b = p.spec.cand_block
    if ld_mask is None:
        ld_mask = (vals.shape[1] + b - 1) // b
    return candidates_rows(vals, cl, b, p.spec.cand_topk, ld_mask, nthreads)


def chunk_rows(prefix_len, budget_token2=2.0e8, chunk_min=256, chunk_max=2048, page=256,
               pow2=False):
    """Adaptive prefill chunk ("chunked-prefill-memory.md", section 2.1):
    clamp(round_down(BUDGET / L), CHUNK_MIN, CHUNK_MAX), round_down to a multiple of the
    page (the section's formula) or, with ``pow2``, to a power of two (the rounding its
    printed schedule follows).  Exact rational arithmetic; prefix_len <= 0 -> chunk_max."""
    from fractions import Fraction
    import math
    if prefix_len <= 0:
        return chunk_max
    x = math.floor(Fraction(budget_token2) / prefix_len)
    if pow2:
        c = 0
        while x >= 1 and (c * 2 if c else 1) <= x:
            c = c * 2 if c else 1
    else:
        c = x // page * page
    return min(chunk_max, max(chunk_min, c))


def page_indices_rows(raw_idx, row_request, key_count, page_table, page_size):
    """KV-cache slot of each selected key ("[SGLang PR 39187]", Accuracy / equivalence:
    the indexer emits page_indices beside raw_indices; the usual paged addressing):
    slot = page_table[r, j // page_size] * page_size + j % page_size for 0 <= j < L_r,
    -1 for j = -1, keys outside [0, L_r), negative (unmapped) table entries and slots past
    the int32 range.  Plain loops over numpy arrays."""
    raw = np.asarray(raw_idx, dtype=np.int64)
    table = np.asarray(page_table, dtype=np.int64)
    out = np.full(raw.shape, -1, dtype=np.int64)
    for t in range(raw.shape[0]):
        r = int(row_request[t])
        for i in range(raw.shape[1]):
            j = int(raw[t, i])
            if j < 0 or j >= int(key_count[r]):
                continue
            page = int(table[r, j // page_size])
            if page < 0:
                continue
            slot = page * page_size + j % page_size
            if slot <= 2**31 - 1:
                out[t, i] = slot
    return out.astype(np.int32)


# ------------------------------------------------------------ fp4 x fp4

def decode_fp4(codes, block_exp):
    """e2m1 codes [..., D/2] (element 2i in the low nibble) with one ue8m0 exponent per 32
    elements [..., D/32] -> fp64 values [..., D] = e2m1(code) * 2^(e - 127), exactly (the
    OCP MX fp4 format the pages' "fp8_fp4" kernel reads for keys)."""
    tab = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
    c = np.asarray(codes, dtype=np.uint8)
    v = np.empty(c.shape[:-1] + (2 * c.shape[-1],), dtype=np.float64)
    v[..., 0::2] = tab[c & 15]
    v[..., 1::2] = tab[c >> 4]
    e = np.asarray(block_exp, dtype=np.int64)
    return v * np.repeat(np.ldexp(1.0, e - 127), 32, axis=-1)


def _key_values(p, k0, k1):
    """fp64 key values [L, D] of keys k0..k1 (scale included)."""
    if p.spec.kdtype == "fp4":
        return decode_fp4(_np(p.k, np.uint8)[k0:k1], _np(p.k_scale, np.uint8)[k0:k1])
    tab = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)
    return tab[_np(p.k, np.uint8)[k0:k1]] * _np(p.k_scale, np.float32)[k0:k1, None].astype(
        np.float64)


def problem_logits_fp4q(p, rows=None, ld=None, batch=8):
    """fp64 logits when the queries too are e2m1 + ue8m0/32 (fp4 x fp4, ``p.q4`` /
    ``p.q_sf``): the definition's step 3 with decoded values (the scales live in the
    values, so s_q = 1): x = <q_h, k_j> by an fp64 matmul (every product and partial sum
    of these short dyadic values is exact), logit = sum over h in order of w * max(x, 0)
    in fp64, -inf past compress_len.  Same layout as problem_logits."""
    T = int(p.cu_seqlens_q[-1])
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    cu_k = _np(p.cu_seqlens_k, np.int64)
    ld = int(np.max(np.diff(cu_k))) if ld is None else ld
    w = _np(p.w, np.float32).astype(np.float64)
    cl = _np(p.compress_len, np.int64)
    out = np.full((len(rows), ld), -np.inf, dtype=np.float64)
    pos_of = {int(g): i for i, g in enumerate(rows)}
    for r, sel in _request_arrays(p, rows, 1):
        k0, k1 = int(cu_k[r]), int(cu_k[r + 1])
        kv = _key_values(p, k0, k1)                                   # [L, D]
        for a in range(0, len(sel), batch):
            part = sel[a:a + batch]
            qv = decode_fp4(_np(p.q4, np.uint8)[part], _np(p.q_sf, np.uint8)[part])
            s = np.einsum("nhd,ld->nhl", qv, kv)                      # [n, H, L]
            acc = np.zeros((len(part), k1 - k0), dtype=np.float64)
            for h in range(p.H):
                acc += w[part, h][:, None] * np.maximum(s[:, h, :], 0.0)
            j = np.arange(k1 - k0)[None, :]
            acc[j >= np.minimum(cl[part], k1 - k0)[:, None]] = -np.inf
            out[[pos_of[int(g)] for g in part], : k1 - k0] = acc
    return out
