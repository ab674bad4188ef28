"""Shared test helpers: run the CUDA path through the C ABI and compare with the oracle.

Acceptance rules (1e-3 relative logits tolerance and exact index sets, made precise):
  * logits: |gpu - oracle| <= 1e-3 * (1 + |oracle|) on eligible keys; -inf on
    exactly the ineligible ones.
  * top-k: with v_k, v_k1 the oracle's k-th and (k+1)-th eligible scores and
    tau = 1e-3 * (1 + |v_k|), a row is a near-tie row when v_k - v_k1 < tau.
    Other rows must return exactly the oracle's index set.  Near-tie rows
    must still be a valid answer: no duplicates, the right count, every key
    scoring above v_k + tau present, every returned key scoring >= v_k - tau.
  * candidate masks: the same rule at block level over pooled scores.
"""
from __future__ import annotations

import numpy as np
import torch

from sparse_attention_prefill_tcgen05_gb300 import _lib as K

LOGIT_RTOL = 1e-3


def device_inputs(p, layer=1, dev="cuda"):
    """The call's inputs on the device.  e2m1 queries (qdtype "fp4", first layer) go in as
    their packed codes, with their ue8m0 block scales in the s_q slot."""
    q, s_q, w = (p.q, p.s_q, p.w) if layer == 1 else (p.q2, p.s_q2, p.w2)
    if layer == 1 and p.spec.qdtype == "fp4":
        q, s_q = p.q4, p.q_sf
    return dict(q=q.to(dev), s_q=s_q.to(dev), w=w.to(dev), k=p.k.to(dev),
                k_scale=p.k_scale.to(dev), compress_len=p.compress_len.to(dev))


def make_plan(p, key_block=0, budget=0, topk=None, select_mode=K.IDX_SELECT_AUTO,
              qdtype=None):
    kd = K.IDX_K_FP8_E4M3 if p.spec.kdtype == "fp8" else K.IDX_K_FP4_E2M1_UE8M0
    if qdtype is None:
        qdtype = K.IDX_Q_FP4_E2M1_UE8M0 if p.spec.qdtype == "fp4" else K.IDX_Q_FP8_E4M3
    return K.indexer_plan(p.cu_seqlens_q, p.cu_seqlens_k, p.compress_len, p.H, p.D,
                          topk or p.topk, kdtype=kd, cand_block=p.spec.cand_block,
                          cand_topk=p.spec.cand_topk, key_block=key_block,
                          transient_budget_bytes=budget, select_mode=select_mode,
                          qdtype=qdtype)


def workspace(plan, dev="cuda"):
    n = max(plan.workspace_bytes, 256)
    return torch.empty(n, dtype=torch.uint8, device=dev)


def max_keys(p):
    return int(torch.diff(p.cu_seqlens_k).max())


def gpu_logits(p, plan, d, ld=None):
    ld = ld or max_keys(p)
    out = torch.empty((int(p.cu_seqlens_q[-1]), ld), dtype=torch.float32, device="cuda")
    ws = workspace(plan)
    K.indexer_logits(plan, d["q"], d["s_q"], d["w"], d["k"], d["k_scale"], d["compress_len"],
                     out, ws)
    st = K.indexer_status(plan, ws)
    assert st == K.IDX_OK, K.error_string(st)
    return out


def gpu_fused(p, plan, d, mask=None, with_values=True):
    T = int(p.cu_seqlens_q[-1])
    k = plan.problem.topk
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    val = torch.empty((T, k), dtype=torch.float32, device="cuda") if with_values else None
    ws = workspace(plan)
    K.indexer_fused_topk(plan, d["q"], d["s_q"], d["w"], d["k"], d["k_scale"],
                         d["compress_len"], mask, idx, val, ws)
    st = K.indexer_status(plan, ws)
    assert st == K.IDX_OK, K.error_string(st)
    return idx, val


def gpu_topk(p, plan, logits, d):
    T = int(p.cu_seqlens_q[-1])
    k = plan.problem.topk
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    val = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = workspace(plan)
    K.indexer_topk(plan, logits, d["compress_len"], idx, val, ws)
    st = K.indexer_status(plan, ws)
    assert st == K.IDX_OK, K.error_string(st)
    return idx, val


def gpu_candidates(p, plan, d, ld_mask=None):
    T = int(p.cu_seqlens_q[-1])
    b = p.spec.cand_block
    ld_mask = ld_mask or (max_keys(p) + b - 1) // b
    mask = torch.full((T, ld_mask), 7, dtype=torch.uint8, device="cuda")
    ws = workspace(plan)
    K.indexer_candidate_blocks(plan, d["q"], d["s_q"], d["w"], d["k"], d["k_scale"],
                               d["compress_len"], mask, ws)
    st = K.indexer_status(plan, ws)
    assert st == K.IDX_OK, K.error_string(st)
    return mask


def check_logits(gpu_rows: np.ndarray, ref_rows: np.ndarray):
    """Element-wise logits rule; returns the max normalised error."""
    g = gpu_rows.astype(np.float64)
    elig = np.isfinite(ref_rows)
    assert np.array_equal(np.isneginf(g), ~elig), "ineligible pattern differs"
    err = np.abs(g[elig] - ref_rows[elig]) / (1.0 + np.abs(ref_rows[elig]))
    worst = float(err.max()) if err.size else 0.0
    assert worst <= LOGIT_RTOL, f"logit error {worst}"
    return worst


def eligible_scores(ref_row, clen, mask_row=None, block=8):
    j = np.arange(min(clen, ref_row.shape[0]))
    if mask_row is not None:
        j = j[mask_row[j // block] != 0]
    return j, ref_row[j]


def check_topk_row(gpu_idx_row: np.ndarray, ref_row: np.ndarray, clen: int, k: int,
                   mask_row=None, block=8):
    """Returns True when the row was an exact match, False when it was a near-tie row that
    passed the validity check; raises on failure."""
    j, v = eligible_scores(ref_row, clen, mask_row, block)
    n = len(j)
    got = gpu_idx_row[gpu_idx_row >= 0]
    assert np.all(gpu_idx_row[len(got):] == -1), "padding must trail"
    assert len(got) == min(k, n), f"count {len(got)} != {min(k, n)}"
    assert len(np.unique(got)) == len(got), "duplicate indices"
    if n <= k:
        assert set(got.tolist()) == set(j.tolist())
        return True
    order = np.lexsort((j, -v))
    want = j[order[:k]]
    vk, vk1 = v[order[k - 1]], v[order[k]]
    tau = LOGIT_RTOL * (1.0 + abs(vk))
    if set(got.tolist()) == set(want.tolist()):
        return True
    assert vk - vk1 < tau, f"not a near-tie row (gap {vk - vk1}) but sets differ"
    score = dict(zip(j.tolist(), v.tolist()))
    assert all(x in score for x in got.tolist()), "ineligible index returned"
    assert set(j[v > vk + tau].tolist()) <= set(got.tolist()), "a clear winner is missing"
    assert min(score[x] for x in got.tolist()) >= vk - tau, "a clear loser was returned"
    return False


def pooled_scores(ref_row, clen, block):
    n = min(clen, ref_row.shape[0])
    nb = (n + block - 1) // block
    pooled = np.full(nb, -np.inf)
    for b in range(nb):
        pooled[b] = ref_row[b * block:min(n, (b + 1) * block)].max()
    return pooled


def check_mask_row(gpu_mask_row: np.ndarray, ref_row: np.ndarray, clen: int, block: int,
                   cand_topk: int):
    pooled = pooled_scores(ref_row, clen, block)
    nb = len(pooled)
    assert np.all(gpu_mask_row[nb:] == 0), "mask set past the row's blocks"
    got = np.nonzero(gpu_mask_row[:nb])[0]
    assert np.all(np.isin(gpu_mask_row, (0, 1)))
    return check_topk_row(np.concatenate([got, -np.ones(max(0, cand_topk - len(got)), np.int64)])
                          .astype(np.int64), pooled, nb, cand_topk)
