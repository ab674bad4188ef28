"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Small cases are checked element by element; the full-size workloads are
checked on sampled rows (the oracle computes rows independently, so a
sampled row is checked exactly).  Also: the selector is bit-exact against
the oracle's selector applied to the GPU's own fp32 logits, exact-arithmetic
inputs give bitwise-equal logits and tie-exact selections, results do not
depend on key-block size or run, and bounded waits report instead of hang.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_attention_prefill_tcgen05_gb300 import _lib as K
from sparse_attention_prefill_tcgen05_gb300 import workloads as W

from . import helpers as Hp

pytestmark = pytest.mark.gpu


def small(name, rows_div, keys_div, topk=None, **over):
    spec = W.scaled(W.CONFIGS[name], rows_div, keys_div, **over)
    if topk:
        spec = dataclasses.replace(spec, topk=topk)
    return W.make_problem(spec)


def oracle_rows(p, rows, layer=1):
    if layer == 1 and p.spec.qdtype == "fp4":
        return O.problem_logits_fp4q(p, rows)
    return O.problem_logits(p, rows, layer=layer)


# ----------------------------------------------------------------- logits

def check_all(p, key_block=0):
    plan = Hp.make_plan(p, key_block=key_block)
    d = Hp.device_inputs(p)
    T = int(p.cu_seqlens_q[-1])
    rows = np.arange(T)
    ref = oracle_rows(p, rows)
    g = Hp.gpu_logits(p, plan, d).cpu().numpy()
    Hp.check_logits(g, ref)
    cl = p.compress_len.numpy()
    # selector isolation: oracle selector on the GPU's own logits == GPU top-k, ties included
    sel_ref = O.topk_rows(g.astype(np.float64), cl, p.topk)
    ti, tv = Hp.gpu_topk(p, plan, torch.from_numpy(g).cuda(), d)
    fi, fv = Hp.gpu_fused(p, plan, d)
    # both selection strategies give the same result, bit for bit
    si, sv = Hp.gpu_fused(p, Hp.make_plan(p, key_block=key_block,
                                          select_mode=K.IDX_SELECT_STREAM), d)
    assert torch.equal(si, fi) and torch.equal(sv, fv)
    ti, fi = ti.cpu().numpy(), fi.cpu().numpy()
    for t in range(T):
        want = sorted(x for x in sel_ref[t].tolist() if x >= 0)
        assert sorted(x for x in ti[t].tolist() if x >= 0) == want, t
        assert np.array_equal(ti[t], fi[t]), t
    assert torch.equal(tv.cpu(), fv.cpu())
    # values are the GPU's own logits at the indices
    gv = fv.cpu().numpy()
    for t in range(T):
        m = fi[t] >= 0
        assert np.array_equal(gv[t][m], g[t][fi[t][m]])
        assert np.all(np.isneginf(gv[t][~m]))
    # against the fp64 oracle
    exact = 0
    for t in range(T):
        exact += Hp.check_topk_row(fi[t], ref[t], int(cl[t]), p.topk)
    return exact


def test_tiny_full_parity():
    p = W.make_problem(W.CONFIGS["tiny"])
    exact = check_all(p)
    assert exact >= 60


@pytest.mark.parametrize("key_block", [0, 512])
def test_cold_chunk_scaled_parity(key_block):
    # 128 rows ending a 4096-key prefix, H=32, D=128, top-256: several tiles, ragged tail
    p = small("cold64k", 16, 16, topk=256)
    check_all(p, key_block=key_block)


def test_long_context_scaled_parity_with_ties():
    p = small("long488k", 128, 96, topk=96)
    check_all(p, key_block=1024)


@pytest.mark.parametrize("H", [16, 64])
def test_other_head_counts_parity(H):
    """The other built head counts (16 rows x 16 heads and 4 rows x 64 heads per MMA tile),
    several tiles and a ragged tail, sampled thresholds on."""
    spec = W.ProblemSpec(f"H={H}", (W.RequestSpec(72, 4100, 1),), H=H, D=128, topk=100,
                         seed=40 + H)
    p = W.make_problem(spec)
    check_all(p)


def test_ragged_requests_parity():
    spec = dataclasses.replace(W.CONFIGS["ragged_cand"], topk=64, cand_topk=48, requests=(
        W.RequestSpec(100, 0, 1), W.RequestSpec(37, 0, 2), W.RequestSpec(0, 0, 1),
        W.RequestSpec(129, 300, 1), W.RequestSpec(70, 5000, 1)))
    p = W.make_problem(spec)
    check_all(p, key_block=1024)


def test_fp4_keys_scaled_parity():
    """fp8 queries x e2m1 keys with one ue8m0 scale per 32 elements (converted exactly to
    e4m3 keys with a per-key power-of-two scale, then the fp8 MMA)."""
    p = small("v4ratio2", 16, 32, topk=64)
    check_all(p, key_block=1024)


def test_fp4_exact_arithmetic_inputs_are_bit_exact():
    spec = dataclasses.replace(W.scaled(W.CONFIGS["v4ratio2"], 32, 64), topk=50, exact=True)
    p = W.make_problem(spec)
    plan = Hp.make_plan(p, key_block=512)
    d = Hp.device_inputs(p)
    T = int(p.cu_seqlens_q[-1])
    ref = oracle_rows(p, np.arange(T))
    g = Hp.gpu_logits(p, plan, d).cpu().numpy().astype(np.float64)
    assert np.array_equal(g, ref)


def _wide_scale_key(p):
    """Key 0 gets block scales 2^10 apart with a 0.5 code in the small block: an e2m1 key
    with no exact e4m3 form under one per-key scale."""
    k, ks = p.k.clone(), p.k_scale.clone()
    ks[0, 0] = 127 + 10
    ks[0, 1] = 127
    k[0, 16] = 0x11                       # elements 32, 33 (block 1): code 1 = 0.5
    return dataclasses.replace(p, k=k, k_scale=ks)


def test_fp4_keys_with_widely_spread_block_scales_match_the_oracle():
    """The block-scaled MMA applies each 32-element block's scale itself, so a key whose
    block scales are far apart is scored like any other: logits within tolerance of the
    oracle, the key's own row entries included, and the top-k sets."""
    p = _wide_scale_key(small("v4ratio2", 64, 256, topk=16))
    plan = Hp.make_plan(p)
    d = Hp.device_inputs(p)
    T = int(p.cu_seqlens_q[-1])
    ref = oracle_rows(p, np.arange(T))
    g = Hp.gpu_logits(p, plan, d).cpu().numpy()
    Hp.check_logits(g, ref)
    fi, _ = Hp.gpu_fused(p, plan, d)
    fi = fi.cpu().numpy()
    cl = p.compress_len.numpy()
    for t in range(T):
        Hp.check_topk_row(fi[t], ref[t], int(cl[t]), p.topk)


@pytest.mark.parametrize("name", ["v4ratio2", "v4fp4qk"])
def test_fp4_scores_far_above_the_fp8_range_match_the_oracle(name):
    """Block scales put a few keys' scores above 2^29, far beyond anything e4m3 x e4m3 can
    reach (D * 448^2 < 2^25); the epilogue's ReLU must still be exact on every head
    column (logits element by element, and those keys at the top of every row)."""
    p = small(name, 64, 256, topk=16)
    ks = p.k_scale.clone()
    ks[:48] = (ks[:48].to(torch.int32) + 24).clamp(max=254).to(torch.uint8)
    p = dataclasses.replace(p, k_scale=ks)
    T = int(p.cu_seqlens_q[-1])
    ref = oracle_rows(p, np.arange(T))
    # the raw scores the MMA accumulates: query codes (e4m3 values, or e2m1 with their
    # block scales) against the keys' block-scaled values
    if p.spec.qdtype == "fp4":
        qv = O.decode_fp4(p.q4.numpy(), p.q_sf.numpy())
    else:
        qv = np.array([O.e4m3_value(b) for b in range(256)])[p.q.numpy()]
    kv = O.decode_fp4(p.k.numpy(), ks.numpy())
    assert np.abs(np.einsum("thd,ld->thl", qv[:4], kv[:48])).max() > 2.0 ** 25
    plan = Hp.make_plan(p)
    d = Hp.device_inputs(p)
    g = Hp.gpu_logits(p, plan, d).cpu().numpy()
    Hp.check_logits(g, ref)
    fi, _ = Hp.gpu_fused(p, plan, d)
    fi = fi.cpu().numpy()
    cl = p.compress_len.numpy()
    for t in range(T):
        Hp.check_topk_row(fi[t], ref[t], int(cl[t]), p.topk)


def test_fp4_key_outside_the_e4m3_range_is_reported_by_the_conversion():
    """Head counts without a block-scaled kernel (16 heads here) score e2m1 keys through
    their exact e4m3 form; a key that has none is reported as IDX_ERR_DEVICE_CHECK
    through indexer_status instead of being scored wrongly."""
    spec = W.ProblemSpec("H=16 fp4", (W.RequestSpec(24, 400, 1),), H=16, D=128, topk=16,
                         kdtype="fp4", seed=51)
    p = _wide_scale_key(W.make_problem(spec))
    plan = Hp.make_plan(p)
    d = Hp.device_inputs(p)
    out = torch.empty((int(p.cu_seqlens_q[-1]), Hp.max_keys(p)), dtype=torch.float32,
                      device="cuda")
    ws = Hp.workspace(plan)
    K.indexer_logits(plan, d["q"], d["s_q"], d["w"], d["k"], d["k_scale"], d["compress_len"],
                     out, ws)
    assert K.indexer_status(plan, ws) == K.IDX_ERR_DEVICE_CHECK


def test_fp4_keys_other_head_counts_parity():
    """e2m1 keys with 16 heads (the exact conversion) against the oracle."""
    spec = W.ProblemSpec("H=16 fp4", (W.RequestSpec(40, 3000, 2),), H=16, D=128, topk=48,
                         kdtype="fp4", seed=52)
    check_all(W.make_problem(spec), key_block=1024)


def test_fp4_queries_and_keys_scaled_parity():
    """e2m1 queries x e2m1 keys, one ue8m0 scale per 32 elements on both sides, through the
    block-scaled fp4 MMA (neither operand converted) against the oracle's fp4-query mode:
    logits element by element, top-k against the oracle and against the oracle's selector on
    the GPU's own logits, both selection strategies bit-identical."""
    p = small("v4fp4qk", 16, 32, topk=64)
    check_all(p, key_block=1024)


def test_fp4_queries_exact_arithmetic_inputs_are_bit_exact():
    spec = dataclasses.replace(W.scaled(W.CONFIGS["v4fp4qk"], 32, 64), topk=50, exact=True)
    p = W.make_problem(spec)
    T = int(p.cu_seqlens_q[-1])
    # the premise: per (row, key) the sum over heads of w * sum_d |q k| stays below
    # 2^15 while every term is a multiple of 2^-9, so fp32 holds every partial sum exactly
    qv = O.decode_fp4(p.q4.numpy(), p.q_sf.numpy())
    kv = O.decode_fp4(p.k.numpy(), p.k_scale.numpy())
    bound = np.einsum("th,thl->tl", p.w.numpy().astype(np.float64),
                      np.einsum("thd,ld->thl", np.abs(qv), np.abs(kv)))
    assert bound.max() < 2.0 ** 15
    plan = Hp.make_plan(p, key_block=512)
    d = Hp.device_inputs(p)
    ref = oracle_rows(p, np.arange(T))
    g = Hp.gpu_logits(p, plan, d).cpu().numpy().astype(np.float64)
    assert np.array_equal(g, ref)
    fi, _ = Hp.gpu_fused(p, plan, d)
    want = O.topk_rows(ref, p.compress_len.numpy(), p.topk)
    fi = fi.cpu().numpy()
    for t in range(T):
        assert sorted(fi[t][fi[t] >= 0].tolist()) == sorted(want[t][want[t] >= 0].tolist())


def test_fp4_queries_and_keys_with_widely_spread_block_scales_match_the_oracle():
    """A query vector and a key whose block scales are 2^20 and 2^10 apart, with small codes
    in the small blocks (neither has an exact e4m3 form under one scale per vector): the
    fp4 MMA applies every block's scale itself, so both are scored like any other."""
    p = _wide_scale_key(small("v4fp4qk", 64, 256, topk=16))
    q4, qsf = p.q4.clone(), p.q_sf.clone()
    qsf[0, 0, 0] = 127 + 10
    qsf[0, 0, 1] = 127 - 10
    q4[0, 0, 16] = 0x11                   # elements 32, 33 (block 1): code 1 = 0.5
    p = dataclasses.replace(p, q4=q4, q_sf=qsf)
    plan = Hp.make_plan(p)
    d = Hp.device_inputs(p)
    T = int(p.cu_seqlens_q[-1])
    ref = oracle_rows(p, np.arange(T))
    g = Hp.gpu_logits(p, plan, d).cpu().numpy()
    Hp.check_logits(g, ref)
    fi, _ = Hp.gpu_fused(p, plan, d)
    fi = fi.cpu().numpy()
    cl = p.compress_len.numpy()
    for t in range(T):
        Hp.check_topk_row(fi[t], ref[t], int(cl[t]), p.topk)


@pytest.mark.parametrize("name", ["cold64k", "v4fp4qk"])
def test_mixed_sign_head_weights(name):
    """Head weights of both signs (a learned projection has no sign constraint): negative
    weighted ReLU terms, rows whose logits are mostly negative, negative sampled
    thresholds; logits, top-k and both selection strategies against the oracle."""
    p = small(name, 32, 8, topk=100)     # long enough rows to be sampled
    gen = torch.Generator().manual_seed(77)
    w = torch.randn(tuple(p.w.shape), generator=gen) / float(np.sqrt(p.H))
    w[: w.shape[0] // 4] -= 0.5          # the first rows mostly negative
    p = dataclasses.replace(p, w=w.float().contiguous())
    assert Hp.make_plan(p, key_block=1024).info()["sample_stride"] >= 2
    check_all(p, key_block=1024)


def test_exact_arithmetic_inputs_are_bit_exact():
    """Small integer codes and power-of-two scales: every fp32 step is exact, so GPU logits
    equal the oracle's bitwise and selections match including ties."""
    spec = dataclasses.replace(W.scaled(W.CONFIGS["cold64k"], 32, 32), topk=100, exact=True)
    p = W.make_problem(spec)
    plan = Hp.make_plan(p, key_block=512)
    d = Hp.device_inputs(p)
    T = int(p.cu_seqlens_q[-1])
    ref = oracle_rows(p, np.arange(T))
    g = Hp.gpu_logits(p, plan, d).cpu().numpy().astype(np.float64)
    assert np.array_equal(g, ref)
    fi, _ = Hp.gpu_fused(p, plan, d)
    want = O.topk_rows(ref, p.compress_len.numpy(), p.topk)
    fi = fi.cpu().numpy()
    for t in range(T):
        assert sorted(fi[t][fi[t] >= 0].tolist()) == sorted(want[t][want[t] >= 0].tolist())


def test_runs_and_key_blocks_are_bitwise_identical():
    p = small("cold64k", 16, 8, topk=300)
    d = Hp.device_inputs(p)
    outs = []
    for kb in (0, 1024, 2048, 0):
        i, v = Hp.gpu_fused(p, Hp.make_plan(p, key_block=kb), d)
        outs.append((i.cpu(), v.cpu()))
    for i, v in outs[1:]:
        assert torch.equal(i, outs[0][0]) and torch.equal(v, outs[0][1])


def test_row_chunking_is_bitwise_invariant():
    """Scoring rows in one call or in pieces gives the same bits (SGLang PR #39187 Accuracy)."""
    p = small("cold64k", 16, 16, topk=64)
    d = Hp.device_inputs(p)
    full = Hp.gpu_logits(p, Hp.make_plan(p), d)
    T = int(p.cu_seqlens_q[-1])
    for a, b in ((0, 8), (8, 9), (9, 77), (77, T)):
        sub = dataclasses.replace(p, q=p.q[a:b], s_q=p.s_q[a:b], w=p.w[a:b],
                                  compress_len=p.compress_len[a:b],
                                  cu_seqlens_q=torch.tensor([0, b - a], dtype=torch.int32))
        ds = Hp.device_inputs(sub)
        part = Hp.gpu_logits(sub, Hp.make_plan(sub), ds)
        assert torch.equal(part, full[a:b])


def _structured_problem(L, rows, topk, key_scale):
    """H=32, D=128 with q = 1.0 everywhere, k = 2.0 everywhere, w = 1/32, s_q = 1 and a
    chosen per-key scale, so logit[t, j] = 128 * 2 * key_scale[j] exactly."""
    spec = W.ProblemSpec("structured", (W.RequestSpec(rows, L - rows, 1),), H=32, D=128,
                         topk=topk, seed=0)
    p = W.make_problem(spec)
    T = rows
    q = torch.full((T, 32, 128), 0x38, dtype=torch.uint8)
    k = torch.full((L, 128), 0x40, dtype=torch.uint8)
    return dataclasses.replace(p, q=q, s_q=torch.ones(T, 32), w=torch.full((T, 32), 1.0 / 32),
                               k=k, k_scale=key_scale.float())


@pytest.mark.parametrize("mode", [K.IDX_SELECT_STREAM, K.IDX_SELECT_AUTO])
def test_increasing_scores_force_list_compaction(mode):
    """Scores rise with the key index, so every key passes the running threshold and the
    per-row lists must be compacted many times inside the kernel (stream); the sampled
    threshold lets only the top few hundred through (auto)."""
    L, rows, topk = 8192, 24, 64
    p = _structured_problem(L, rows, topk, 1.0 + torch.arange(L, dtype=torch.float64) / L)
    plan = Hp.make_plan(p, select_mode=mode)
    assert plan.info()["max_splits"] == 1
    d = Hp.device_inputs(p)
    fi, fv = Hp.gpu_fused(p, plan, d)
    ref = oracle_rows(p, np.arange(rows))
    cl = p.compress_len.numpy()
    fi = fi.cpu().numpy()
    for t in range(rows):
        want = list(range(int(cl[t]) - topk, int(cl[t])))
        assert fi[t].tolist() == want, t
        Hp.check_topk_row(fi[t], ref[t], int(cl[t]), topk)


@pytest.mark.parametrize("mode", [K.IDX_SELECT_STREAM, K.IDX_SELECT_AUTO])
def test_all_equal_scores_keep_the_lowest_indices(mode):
    """Every key ties: the top-k is the k lowest key indices, through compaction too."""
    L, rows, topk = 8192, 20, 100
    p = _structured_problem(L, rows, topk, torch.ones(L, dtype=torch.float64))
    plan = Hp.make_plan(p, select_mode=mode)
    d = Hp.device_inputs(p)
    fi, fv = Hp.gpu_fused(p, plan, d)
    fi = fi.cpu().numpy()
    for t in range(rows):
        assert fi[t].tolist() == list(range(topk)), t
    assert torch.all(fv == 256.0)


def _sampled_tiles_scores(L, stride, sampled_high):
    """Distinct scores rising with the key index, every key of the sampled tiles
    (0, stride, 2 stride, ...) one unit above (or below) every other key."""
    j = torch.arange(L, dtype=torch.float64)
    on = ((j // 128) % stride) == 0
    hi, lo = 2.0 + j / L, 1.0 + j / L
    return torch.where(on, hi, lo) if sampled_high else torch.where(on, lo, hi)


def _check_structured_topk(p, plan, rows, topk):
    d = Hp.device_inputs(p)
    fi, fv = Hp.gpu_fused(p, plan, d)
    ref = oracle_rows(p, np.arange(rows))
    cl = p.compress_len.numpy()
    fi = fi.cpu().numpy()
    for t in range(rows):
        want = np.sort(np.argsort(-ref[t][: int(cl[t])], kind="stable")[:topk])
        assert fi[t].tolist() == want.tolist(), t
        Hp.check_topk_row(fi[t], ref[t], int(cl[t]), topk)
    return fi


def _sampled_problem(L, rows, topk, sampled_high):
    """A structured problem whose sampled tiles (at the plan's stride) score above (or
    below) every other key."""
    probe = _structured_problem(L, rows, topk, torch.ones(L, dtype=torch.float64))
    stride = Hp.make_plan(probe).info()["sample_stride"]
    assert stride >= 2
    p = _structured_problem(L, rows, topk, _sampled_tiles_scores(L, stride, sampled_high))
    return p, Hp.make_plan(p)


def test_sampled_threshold_too_high_falls_back_to_the_stream():
    """The sampled tiles hold the highest scores, so each row's threshold (the rank-th
    sample) lets fewer than k keys through: every row is decided again by the stream."""
    L, rows, topk = 16384, 24, 1024
    p, plan = _sampled_problem(L, rows, topk, True)
    _check_structured_topk(p, plan, rows, topk)


def test_sampled_threshold_too_low_overflows_and_falls_back():
    """The sampled tiles hold the lowest scores, so most of every row passes the
    threshold and the lists overflow: the stream decides every row again."""
    L, rows, topk = 16384, 24, 64
    p, plan = _sampled_problem(L, rows, topk, False)
    _check_structured_topk(p, plan, rows, topk)


# ------------------------------------------------------------- candidates

def test_candidate_blocks_and_masked_consumer_scaled():
    spec = dataclasses.replace(W.CONFIGS["ragged_cand"], topk=40, cand_topk=30, requests=(
        W.RequestSpec(90, 0, 1), W.RequestSpec(90, 0, 2), W.RequestSpec(50, 2000, 1)))
    p = W.make_problem(spec)
    plan = Hp.make_plan(p, key_block=1024)
    d = Hp.device_inputs(p)
    T = int(p.cu_seqlens_q[-1])
    rows = np.arange(T)
    ref = oracle_rows(p, rows)
    mask = Hp.gpu_candidates(p, plan, d).cpu().numpy()
    cl = p.compress_len.numpy()
    for t in rows:
        Hp.check_mask_row(mask[t], ref[t], int(cl[t]), 8, 30)
    # selector isolation at block level on the GPU's own logits
    g = Hp.gpu_logits(p, plan, d).cpu().numpy().astype(np.float64)
    want = O.candidates_rows(g, cl, 8, 30, mask.shape[1])
    assert np.array_equal(want, mask)
    # consumer: new queries, same keys, top-k within the candidate blocks
    d2 = Hp.device_inputs(p, layer=2)
    fi, _ = Hp.gpu_fused(p, plan, d2, mask=torch.from_numpy(mask).cuda())
    fi = fi.cpu().numpy()
    ref2 = oracle_rows(p, rows, layer=2)
    for t in rows:
        Hp.check_topk_row(fi[t], ref2[t], int(cl[t]), p.topk, mask_row=mask[t])
    # key-level expansion of the block mask
    km = torch.empty((T, Hp.max_keys(p)), dtype=torch.uint8, device="cuda")
    K.indexer_expand_mask(plan, torch.from_numpy(mask).cuda(), d["compress_len"], km)
    km = km.cpu().numpy()
    j = np.arange(km.shape[1])
    for t in rows:
        assert np.array_equal(km[t], ((j < cl[t]) & (mask[t][j // 8] != 0)).astype(np.uint8))


def test_fp4_queries_candidate_blocks_and_masked_call():
    """e2m1 queries and keys on the fp4 MMA kind through the candidate path: the block
    masks against the oracle (fp4-query mode) and against the oracle's block selector on
    the GPU's own logits, then a masked fused call on the same queries against the oracle's
    top-k within those blocks (short requests, and one long enough to be sampled)."""
    spec = W.ProblemSpec("fp4 x fp4 candidates", (W.RequestSpec(90, 0, 1),
                         W.RequestSpec(90, 0, 2), W.RequestSpec(50, 12000, 1)),
                         H=32, D=128, topk=40, kdtype="fp4", qdtype="fp4", seed=61,
                         cand_block=8, cand_topk=30)
    p = W.make_problem(spec)
    plan = Hp.make_plan(p, key_block=1024)
    assert plan.info()["sample_stride"] >= 2
    d = Hp.device_inputs(p)
    T = int(p.cu_seqlens_q[-1])
    rows = np.arange(T)
    ref = oracle_rows(p, rows)
    mask = Hp.gpu_candidates(p, plan, d).cpu().numpy()
    cl = p.compress_len.numpy()
    for t in rows:
        Hp.check_mask_row(mask[t], ref[t], int(cl[t]), 8, 30)
    g = Hp.gpu_logits(p, plan, d).cpu().numpy().astype(np.float64)
    assert np.array_equal(O.candidates_rows(g, cl, 8, 30, mask.shape[1]), mask)
    fi, _ = Hp.gpu_fused(p, plan, d, mask=torch.from_numpy(mask).cuda())
    fi = fi.cpu().numpy()
    for t in rows:
        Hp.check_topk_row(fi[t], ref[t], int(cl[t]), p.topk, mask_row=mask[t])


@pytest.mark.parametrize("block,cand_topk", [(8, 64), (4, 200)])
def test_sampled_candidate_blocks_match_the_stream(block, cand_topk):
    """Requests long enough to be sampled: the block threshold from pooled samples, the
    fixed-threshold block lists and the verify merge give the same masks, bit for bit,
    as the exact stream, and the oracle's (also on the GPU's own logits)."""
    spec = dataclasses.replace(
        W.CONFIGS["ragged_cand"], topk=64, cand_block=block, cand_topk=cand_topk,
        requests=(W.RequestSpec(20, 16364, 1), W.RequestSpec(12, 9000, 2)), seed=11)
    p = W.make_problem(spec)
    plan = Hp.make_plan(p)
    assert plan.info()["sample_stride"] >= 2
    d = Hp.device_inputs(p)
    n0 = K.indexer_launch_count()
    mask = Hp.gpu_candidates(p, plan, d).cpu().numpy()
    n1 = K.indexer_launch_count()
    mask_s = Hp.gpu_candidates(p, Hp.make_plan(p, select_mode=K.IDX_SELECT_STREAM),
                               d).cpu().numpy()
    # the sampled flow (samples, thresholds, filter, verify) launches more kernels
    assert n1 - n0 > K.indexer_launch_count() - n1
    assert np.array_equal(mask, mask_s)
    T = int(p.cu_seqlens_q[-1])
    ref = oracle_rows(p, np.arange(T))
    cl = p.compress_len.numpy()
    for t in range(T):
        Hp.check_mask_row(mask[t], ref[t], int(cl[t]), block, cand_topk)
    g = Hp.gpu_logits(p, plan, d).cpu().numpy().astype(np.float64)
    assert np.array_equal(O.candidates_rows(g, cl, block, cand_topk, mask.shape[1]), mask)


@pytest.mark.parametrize("sampled_high", [True, False])
def test_sampled_candidate_threshold_fallbacks(sampled_high):
    """Sampled tiles scoring above every other key put the block threshold too high (the
    rows go to the exact stream); scoring below, nearly every block passes."""
    L, rows, cand_topk = 16384, 24, 256
    p, _ = _sampled_problem(L, rows, 64, sampled_high)
    p = dataclasses.replace(p, spec=dataclasses.replace(p.spec, cand_block=8,
                                                        cand_topk=cand_topk))
    plan = Hp.make_plan(p)
    d = Hp.device_inputs(p)
    mask = Hp.gpu_candidates(p, plan, d).cpu().numpy()
    ref = oracle_rows(p, np.arange(rows))
    cl = p.compress_len.numpy()
    for t in range(rows):
        pooled = Hp.pooled_scores(ref[t], int(cl[t]), 8)
        want = np.zeros(mask.shape[1], dtype=np.uint8)
        want[np.argsort(-pooled, kind="stable")[:cand_topk]] = 1
        assert np.array_equal(mask[t], want), t


# ----------------------------------------------------------- full size
#
# At full size the oracle scores 256 sampled rows per request (first and last rows,
# the shortest causal rows, duplicated-query rows, the rest seeded at random) against
# the request's whole prefix.  Each sampled row gets three checks:
#   * indexer_logits at full size, element by element within 1e-3 * (1 + |ref|);
#   * the fused top-k (or candidate mask) against the fp64 oracle by the near-tie rule;
#   * the same output against the oracle's selector applied to the GPU's own fp32
#     logits: bit-exact index sets for every row, ties to the lower index included, with
#     no near-tie exemption (at L = 487,936 this enforces the tie rule on the
#     duplicated keys' exact ties).

FULL_ROWS = 256


def _rows_of(t, rows):
    """Rows ``rows`` of a device tensor, on the host."""
    return t[torch.from_numpy(rows).to(t.device)].cpu().numpy()


def _same_sets(got, want):
    for i in range(got.shape[0]):
        a = np.sort(got[i][got[i] >= 0])
        b = np.sort(want[i][want[i] >= 0])
        assert np.array_equal(a, b), i


def full_size_check(name, per_request=FULL_ROWS):
    p = W.make_problem(W.CONFIGS[name])
    plan = Hp.make_plan(p, key_block=p.spec.key_block)
    assert plan.workspace_bytes <= 2 << 30
    d = Hp.device_inputs(p)
    rows = W.sample_rows(p, per_request)
    fi, fv = Hp.gpu_fused(p, plan, d)
    fi, fv = _rows_of(fi, rows), _rows_of(fv, rows)
    torch.cuda.empty_cache()
    g = Hp.gpu_logits(p, plan, d)
    g = _rows_of(g, rows).astype(np.float64)
    torch.cuda.empty_cache()
    ref = oracle_rows(p, rows)
    Hp.check_logits(g, ref)
    cl = p.compress_len.numpy()[rows]
    _same_sets(fi, O.topk_rows(g, cl, p.topk))
    for i in range(len(rows)):
        m = fi[i] >= 0
        assert np.array_equal(fv[i][m].astype(np.float64), g[i][fi[i][m]]), i
        Hp.check_topk_row(fi[i], ref[i], int(cl[i]), p.topk)
    return p, rows


def test_full_cold_chunk_t2048_l65536_top2048():
    full_size_check("cold64k")


def test_full_v4_low_ratio_fp4_t2048_l100000_top512():
    full_size_check("v4ratio2")


def test_full_v4_fp4_queries_and_keys_t2048_l100000_top512():
    full_size_check("v4fp4qk")


def test_full_long_context_t16384_l487936_top512():
    p, rows = full_size_check("long488k")
    # the sample holds the rows whose queries were copied (their logits tie exactly with
    # the source rows' in every key) besides the keys' own 1 % of exact ties
    assert set(p.dup_rows[:16]) <= set(rows.tolist())


def test_full_ragged_candidates():
    p = W.make_problem(W.CONFIGS["ragged_cand"])
    plan = Hp.make_plan(p)
    assert plan.workspace_bytes <= 2 << 30
    d = Hp.device_inputs(p)
    rows = W.sample_rows(p, FULL_ROWS)
    cl = p.compress_len.numpy()[rows]
    b, ct = p.spec.cand_block, p.spec.cand_topk
    mask = Hp.gpu_candidates(p, plan, d)
    m = _rows_of(mask, rows)
    g = _rows_of(Hp.gpu_logits(p, plan, d), rows).astype(np.float64)
    torch.cuda.empty_cache()
    ref = oracle_rows(p, rows)
    Hp.check_logits(g, ref)
    # source layer: the oracle's block selector on the GPU's own logits, bit for bit
    assert np.array_equal(O.candidates_rows(g, cl, b, ct, m.shape[1]), m)
    for i in range(len(rows)):
        Hp.check_mask_row(m[i], ref[i], int(cl[i]), b, ct)
    # consumer layer: fresh queries, top-k within the candidate blocks
    d2 = Hp.device_inputs(p, layer=2)
    fi, _ = Hp.gpu_fused(p, plan, d2, mask=mask)
    fi = _rows_of(fi, rows)
    g2 = _rows_of(Hp.gpu_logits(p, plan, d2), rows).astype(np.float64)
    torch.cuda.empty_cache()
    ref2 = oracle_rows(p, rows, layer=2)
    Hp.check_logits(g2, ref2)
    _same_sets(fi, O.topk_rows(g2, cl, p.topk, mask=m, mask_block=b))
    for i in range(len(rows)):
        Hp.check_topk_row(fi[i], ref2[i], int(cl[i]), p.topk, mask_row=m[i])


# ------------------------------------------------------------ failure paths

def test_bounded_wait_reports_timeout_instead_of_hanging():
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    K.indexer_selftest_timeout(ws, 200000)
    assert K.indexer_status(None, ws) == K.IDX_ERR_TIMEOUT
    # the context is still usable afterwards
    p = W.make_problem(W.CONFIGS["tiny"])
    plan = Hp.make_plan(p)
    Hp.gpu_logits(p, plan, Hp.device_inputs(p))


def test_workspace_too_small_is_rejected():
    p = W.make_problem(W.CONFIGS["tiny"])
    plan = Hp.make_plan(p)
    assert plan.workspace_bytes > 256
    d = Hp.device_inputs(p)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    idx = torch.empty((64, p.topk), dtype=torch.int32, device="cuda")
    with pytest.raises(K.IndexerError) as e:
        K.indexer_fused_topk(plan, d["q"], d["s_q"], d["w"], d["k"], d["k_scale"],
                             d["compress_len"], None, idx, None, ws)
    assert e.value.code == K.IDX_ERR_WORKSPACE


# ------------------------------------------------- top-k over caller logits

@pytest.mark.parametrize("structured", [None, True, False])
def test_topk_over_logits_sampled_equals_direct(structured):
    """indexer_topk with the plan's workspace (sampled thresholds, one filtering read,
    verify merge, direct kernel for undecided rows) equals the direct kernel alone (a
    status-only workspace), bit for bit, and the oracle's selector; entries past a row's
    length are ignored even when huge."""
    L, rows, topk = 16384, 24, 256
    if structured is None:
        spec = W.ProblemSpec("long rows", (W.RequestSpec(rows, L - rows, 1),
                                           W.RequestSpec(10, 3000, 1)), H=32, D=128,
                             topk=topk, seed=17)
        p = W.make_problem(spec)
        plan = Hp.make_plan(p)
    else:
        p, plan = _sampled_problem(L, rows, topk, structured)
    assert plan.info()["sample_stride"] >= 2
    d = Hp.device_inputs(p)
    g = Hp.gpu_logits(p, plan, d)
    cl = p.compress_len.cuda().long()
    j = torch.arange(g.shape[1], device="cuda")[None, :]
    g = torch.where(j >= cl[:, None], torch.full_like(g, 1e30), g)    # past the row: ignored
    T = g.shape[0]
    n0 = K.indexer_launch_count()
    ti, tv = Hp.gpu_topk(p, plan, g, d)
    n1 = K.indexer_launch_count()
    assert n1 - n0 > 1                                   # the sampled path ran
    di = torch.empty_like(ti)
    dv = torch.empty_like(tv)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    K.indexer_topk(plan, g, d["compress_len"], di, dv, small)
    assert K.indexer_status(plan, small) == K.IDX_OK
    assert torch.equal(ti, di) and torch.equal(tv, dv)
    ref = O.topk_rows(g.cpu().numpy().astype(np.float64), p.compress_len.numpy(), topk)
    for t in range(T):
        assert sorted(x for x in ti[t].tolist() if x >= 0) == sorted(
            x for x in ref[t].tolist() if x >= 0), t


def test_topk_single_read_edge_rows():
    """The single-read top-k (rows of at most 65,536 keys, aligned rows) on rows built to
    reach each of its exits: a row of equal logits (every entry passes the threshold, the
    candidate buffer overflows, the direct kernel decides it; ties go to the lower index),
    a row of -inf but a few entries (the threshold lets everything through and fewer than
    k are finite), a row whose tail is -inf, a row with a few huge values, a short request
    that is not sampled; against the oracle's selector and, bit for bit, the direct kernel
    alone."""
    L, rows, topk = 32768, 12, 512
    spec = W.ProblemSpec("edge rows", (W.RequestSpec(rows, L - rows, 1),
                                       W.RequestSpec(6, 1500, 1)), H=32, D=128, topk=topk,
                         seed=29)
    p = W.make_problem(spec)
    plan = Hp.make_plan(p)
    assert plan.info()["sample_stride"] >= 2
    d = Hp.device_inputs(p)
    g = Hp.gpu_logits(p, plan, d).clone()
    cl = p.compress_len.numpy()
    g[0, :] = 1.0                                        # ties everywhere
    g[1, :] = -float("inf")
    g[1, 100:100 + topk // 3] = torch.linspace(-5.0, 5.0, topk // 3)
    g[2, int(cl[2]) // 2:] = -float("inf")               # the second half of the row
    g[3, 7::997] = 1.0e30                                # a few huge values
    T = g.shape[0]
    ti, tv = Hp.gpu_topk(p, plan, g, d)
    di = torch.empty_like(ti)
    dv = torch.empty_like(tv)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    K.indexer_topk(plan, g, d["compress_len"], di, dv, small)
    assert K.indexer_status(plan, small) == K.IDX_OK
    assert torch.equal(ti, di) and torch.equal(tv, dv)
    # -inf entries are not eligible (the entry point's contract): the oracle's selector
    # gets that rule as its eligibility mask, one byte per key
    gh = g.cpu().numpy().astype(np.float64)
    finite = np.isfinite(gh).astype(np.uint8)
    ref = O.topk_rows(gh, cl, topk, mask=finite, mask_block=1)
    ti = ti.cpu().numpy()
    for t in range(T):                                   # (the oracle lists by score)
        assert sorted(x for x in ti[t].tolist() if x >= 0) == sorted(
            x for x in ref[t].tolist() if x >= 0), t
        assert (ti[t] < 0).sum() == (ref[t] < 0).sum(), t
    assert ti[0].tolist() == list(range(topk))           # equal logits: the lowest indices


def test_topk_single_read_uneven_candidates_use_the_spill_area():
    """Every large logit of a row in one filter warp's key slice (the 512 keys j with
    128 <= j % 2048 < 160, none of them in a sampled tile): that warp's region fills and the
    rest of its candidates go to the shared spill area; the row is still decided by the
    single read (no fallback row), and matches the oracle's selector and the direct kernel
    bit for bit."""
    L, rows, topk = 32768, 8, 512
    spec = W.ProblemSpec("clustered", (W.RequestSpec(rows, L - rows, 1),), H=32, D=128,
                         topk=topk, seed=41)
    p = W.make_problem(spec)
    plan = Hp.make_plan(p)
    assert plan.info()["sample_stride"] >= 2
    d = Hp.device_inputs(p)
    gen = torch.Generator().manual_seed(41)
    g = torch.randn((rows, L), generator=gen, dtype=torch.float32)
    j = torch.arange(L)
    g[:, ((j % 2048) >= 128) & ((j % 2048) < 160)] += 20.0
    g = g.cuda()
    T = rows
    idx = torch.empty((T, topk), dtype=torch.int32, device="cuda")
    val = torch.empty((T, topk), dtype=torch.float32, device="cuda")
    ws = Hp.workspace(plan)
    K.indexer_topk(plan, g, d["compress_len"], idx, val, ws)
    assert K.indexer_status(plan, ws) == K.IDX_OK
    assert K.indexer_fallback_rows(plan, ws) == 0
    di = torch.empty_like(idx)
    dv = torch.empty_like(val)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    K.indexer_topk(plan, g, d["compress_len"], di, dv, small)
    assert torch.equal(idx, di) and torch.equal(val, dv)
    ref = O.topk_rows(g.cpu().numpy().astype(np.float64), p.compress_len.numpy(), topk)
    ti = idx.cpu().numpy()
    for t in range(T):
        assert sorted(x for x in ti[t].tolist() if x >= 0) == sorted(
            x for x in ref[t].tolist() if x >= 0), t


def test_topk_over_rows_longer_than_the_single_read_takes():
    """Rows of more than 65,536 keys (the single-read kernel's key field is 16 bits) take
    the gather / filtering read / verify merge path: against the oracle's selector on the
    same logits and, bit for bit, the direct kernel alone."""
    L, rows, topk = 70000, 6, 300
    spec = W.ProblemSpec("rows past 65,536 keys", (W.RequestSpec(rows, L - rows, 1),), H=32,
                         D=128, topk=topk, seed=37)
    p = W.make_problem(spec)
    plan = Hp.make_plan(p)
    assert plan.info()["sample_stride"] >= 2
    d = Hp.device_inputs(p)
    g = Hp.gpu_logits(p, plan, d)
    ti, tv = Hp.gpu_topk(p, plan, g, d)
    di = torch.empty_like(ti)
    dv = torch.empty_like(tv)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    K.indexer_topk(plan, g, d["compress_len"], di, dv, small)
    assert K.indexer_status(plan, small) == K.IDX_OK
    assert torch.equal(ti, di) and torch.equal(tv, dv)
    ref = O.topk_rows(g.cpu().numpy().astype(np.float64), p.compress_len.numpy(), topk)
    ti = ti.cpu().numpy()
    for t in range(rows):
        assert sorted(x for x in ti[t].tolist() if x >= 0) == sorted(
            x for x in ref[t].tolist() if x >= 0), t


def test_topk_over_unaligned_logits_rows():
    """Rows that do not start on a 16-byte boundary (a view one column into a wider
    buffer, odd row stride) take the one-entry-per-load path of the filtering read and
    the sample gather: same result, bit for bit, as the aligned rows, and the oracle's
    selector."""
    L, rows, topk = 16384, 24, 256
    spec = W.ProblemSpec("long rows", (W.RequestSpec(rows, L - rows, 1),
                                       W.RequestSpec(10, 3000, 1)), H=32, D=128, topk=topk,
                         seed=19)
    p = W.make_problem(spec)
    plan = Hp.make_plan(p)
    assert plan.info()["sample_stride"] >= 2
    d = Hp.device_inputs(p)
    g = Hp.gpu_logits(p, plan, d)
    T = g.shape[0]
    wide = torch.full((T, L + 3), 5.0e30, dtype=torch.float32, device="cuda")
    wide[:, 1:L + 1] = g
    view = wide[:, 1:L + 1]                     # 4-byte offset, row stride L + 3
    assert view.data_ptr() % 16 != 0 and view.stride(0) % 4 != 0
    ai, av = Hp.gpu_topk(p, plan, g, d)
    ui, uv = Hp.gpu_topk(p, plan, view, d)
    assert torch.equal(ai, ui) and torch.equal(av, uv)
    ref = O.topk_rows(g.cpu().numpy().astype(np.float64), p.compress_len.numpy(), topk)
    ui = ui.cpu().numpy()
    for t in range(T):
        assert sorted(x for x in ui[t].tolist() if x >= 0) == sorted(
            x for x in ref[t].tolist() if x >= 0), t


def test_repeated_calls_on_one_workspace_decide_the_same_rows():
    """Requests with different numbers of sampled tiles share a pass (the widest sets the
    sample row length): a second call on the same workspace must not read the first
    call's leftovers as samples, so no row needs the exact path on either call."""
    spec = W.ProblemSpec("mixed sampling", (W.RequestSpec(40, 7128, 1), W.RequestSpec(30, 40000, 1),
                                            W.RequestSpec(20, 2000, 1)), H=32, D=128, topk=256,
                         seed=23)
    p = W.make_problem(spec)
    plan = Hp.make_plan(p)
    assert plan.info()["sample_stride"] >= 2
    d = Hp.device_inputs(p)
    ws = Hp.workspace(plan)
    T = int(p.cu_seqlens_q[-1])
    outs = []
    for _ in range(3):
        idx = torch.empty((T, p.topk), dtype=torch.int32, device="cuda")
        K.indexer_fused_topk(plan, d["q"], d["s_q"], d["w"], d["k"], d["k_scale"],
                             d["compress_len"], None, idx, None, ws)
        assert K.indexer_status(plan, ws) == K.IDX_OK
        assert K.indexer_fallback_rows(plan, ws) == 0
        outs.append(idx)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


def test_calls_between_torch_kernels_on_one_stream():
    """Every kernel of the library may start while the previous kernel of its stream is
    still running, and waits for it before touching memory.  A call right after a PyTorch
    kernel that rewrites an input (the head weights doubled in place: every logit doubles
    exactly) sees the new values, and a PyTorch kernel right after the call reads its
    outputs; the same for indexer_topk after a kernel that writes its logits."""
    spec = dataclasses.replace(W.scaled(W.CONFIGS["cold64k"], 8, 4), topk=256, seed=43)
    p = W.make_problem(spec)
    plan = Hp.make_plan(p)
    assert plan.info()["sample_stride"] >= 2
    d = Hp.device_inputs(p)
    ri, rv = Hp.gpu_fused(p, plan, d, with_values=True)
    T = int(p.cu_seqlens_q[-1])
    idx = torch.empty((T, p.topk), dtype=torch.int32, device="cuda")
    val = torch.empty((T, p.topk), dtype=torch.float32, device="cuda")
    ws = Hp.workspace(plan)
    d["w"].mul_(2.0)                                     # a kernel, just before the call
    K.indexer_fused_topk(plan, d["q"], d["s_q"], d["w"], d["k"], d["k_scale"],
                         d["compress_len"], None, idx, val, ws)
    half = val.mul(0.5)                                  # a kernel, just after it
    i2 = idx.clone()
    assert K.indexer_status(plan, ws) == K.IDX_OK
    assert torch.equal(i2, ri)
    assert torch.equal(half, rv)
    d["w"].mul_(0.5)
    # indexer_topk over logits a kernel has just written
    g = Hp.gpu_logits(p, plan, d)
    ti, tv = Hp.gpu_topk(p, plan, g, d)
    g2 = torch.empty_like(g)
    torch.mul(g, 2.0, out=g2)
    K.indexer_topk(plan, g2, d["compress_len"], idx, val, ws)
    half = val.mul(0.5)
    assert K.indexer_status(plan, ws) == K.IDX_OK
    assert torch.equal(idx, ti) and torch.equal(half, tv)
