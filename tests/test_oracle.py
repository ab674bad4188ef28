"""Pins of the CPU oracle against things other than itself (CPU only).

Each test names what it pins the oracle to:
  * a library routine (torch's fp8 e4m3 conversion, numpy matmul/lexsort),
  * a closed form, or the published e2m1 element grid,
  * exact brute force with rational arithmetic on tiny inputs,
  * invariants the method must satisfy (block-merge identity from
    "chunked-prefill-memory.md" section 2.3, row-chunk invariance from SGLang
    PR #39187 Accuracy, the causal-length rule).
A plausible slip in the oracle (a dropped scale, a sign, a transposed
operand, a wrong tie-break or block edge) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

from oracle import brute
from oracle import oracle as O
from sparse_attention_prefill_tcgen05_gb300 import workloads as W


def small_problem(H=2, D=32, rows=4, L=40, kdtype="fp8", seed=1, ratio=1, exact=False, topk=7):
    spec = W.ProblemSpec("pin", (W.RequestSpec(rows, L * ratio - rows, ratio),), H=H, D=D,
                         topk=topk, kdtype=kdtype, seed=seed, exact=exact)
    return W.make_problem(spec)


# ------------------------------------------------------------------ formats

def test_e4m3_decode_matches_torch_for_every_code():
    """Pin: torch's float8_e4m3fn conversion (a library routine)."""
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = O.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c], (c, v, ref[c])


def test_e4m3_range_and_grid():
    """Closed form: largest finite 448, smallest subnormal 2^-9, NaN only at 0x7F/0xFF."""
    vals = [O.e4m3_value(c) for c in range(256)]
    finite = [v for v in vals if not math.isnan(v)]
    assert max(finite) == 448.0 and min(finite) == -448.0
    assert min(abs(v) for v in finite if v != 0) == 2.0 ** -9
    assert [c for c in range(256) if math.isnan(vals[c])] == [0x7F, 0xFF]
    for v in finite:  # every value is an integer multiple of 2^-9
        assert (v * 512) == int(v * 512)


def test_e2m1_decode_is_the_published_grid():
    """Pin: the OCP MX e2m1 element grid {0, .5, 1, 1.5, 2, 3, 4, 6} with a sign bit."""
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        want = grid[c & 7] * (-1 if c & 8 else 1)
        assert O.e2m1_value(c) == want
        assert float(brute.e2m1(c)) == want


def test_ue8m0_decode():
    assert O.ue8m0_value(127) == 1.0
    assert O.ue8m0_value(130) == 8.0
    assert O.ue8m0_value(0) == 2.0 ** -127
    assert math.isnan(O.ue8m0_value(255))


def test_brute_decode_agrees_with_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert float(brute.e4m3(c)) == ref[c]


# ------------------------------------------------------------------- scores

@pytest.mark.parametrize("H,D,kdtype,seed", [(1, 32, "fp8", 1), (2, 64, "fp8", 2),
                                             (4, 32, "fp8", 3), (2, 64, "fp4", 4),
                                             (1, 32, "fp4", 5)])
def test_logits_match_exact_brute_force(H, D, kdtype, seed):
    """Pin: exact rational brute force on tiny inputs (PIN1)."""
    p = small_problem(H=H, D=D, rows=3, L=23, kdtype=kdtype, seed=seed)
    got = O.problem_logits(p)
    q, sq, w = p.q.numpy(), p.s_q.numpy(), p.w.numpy()
    k, ks = p.k.numpy(), p.k_scale.numpy()
    cl = p.compress_len.numpy()
    for r in range(3):
        exact = brute.row_scores(q[r], sq[r], w[r], k, ks, int(cl[r]), kdtype)
        for j, e in enumerate(exact):
            assert abs(got[r, j] - float(e)) <= 4e-16 * max(1.0, abs(float(e))), (r, j)
        assert np.all(np.isneginf(got[r, int(cl[r]):]))
        # selection: exact scores, full sort, ties to the lower index
        want = brute.topk(exact, 7)
        sel = O.topk_rows(got[r:r + 1], cl[r:r + 1], 7)[0].tolist()
        assert sel == want


def test_textbook_reduction_single_head_unit_scales():
    """Pin: H=1, w=1, s=1 reduces to relu(Q K^T) by numpy matmul; top-k = lexsort (PIN3)."""
    rng = np.random.default_rng(7)
    D, n, L, k = 64, 5, 300, 19
    qf = torch.tensor(rng.integers(-20, 21, (n, 1, D)), dtype=torch.float32)
    kf = torch.tensor(rng.integers(-20, 21, (L, D)), dtype=torch.float32)
    qb = qf.to(torch.float8_e4m3fn).view(torch.uint8)
    kb = kf.to(torch.float8_e4m3fn).view(torch.uint8)
    Qv = qb.view(torch.float8_e4m3fn).double().numpy()[:, 0, :]
    Kv = kb.view(torch.float8_e4m3fn).double().numpy()
    ref = np.maximum(Qv @ Kv.T, 0.0)
    ones = np.ones((n, 1), np.float32)
    clen = np.full(n, L, np.int32)
    got = O.logits_request(1, D, "fp8", qb, ones, ones, kb, np.ones(L, np.float32), clen)
    assert np.array_equal(got, ref)
    sel = O.topk_rows(got, clen, k)
    for r in range(n):
        order = np.lexsort((np.arange(L), -ref[r]))[:k]
        assert sel[r].tolist() == order.tolist()
    # pooling over aligned 8-key blocks is reshape(-1, 8).max(1) on a -inf padded row
    pad = (-L) % 8
    mask, pooled = O.candidates_rows(got, clen, 8, 10, (L + pad) // 8, with_pooled=True)
    padded = np.concatenate([ref, np.full((n, pad), -np.inf)], 1)
    assert np.array_equal(pooled, padded.reshape(n, -1, 8).max(2))
    for r in range(n):
        top = np.lexsort((np.arange(pooled.shape[1]), -pooled[r]))[:10]
        want = np.zeros(pooled.shape[1], np.uint8)
        want[top] = 1
        assert np.array_equal(mask[r], want)


def test_closed_form_constant_vectors():
    """Closed form: q, k constant codes -> <q_h, k_j> = D * a * b for every head and key."""
    H, D, L = 3, 32, 9
    a_code, b_code = 0x38, 0x40          # 1.0 and 2.0 in e4m3
    q = np.full((1, H, D), a_code, np.uint8)
    k = np.full((L, D), b_code, np.uint8)
    k[4] = 0xC0                            # -2.0: negative dot -> ReLU zero
    s_q = np.array([[0.5, 0.25, 2.0]], np.float32)
    w = np.array([[1.0, -3.0, 0.125]], np.float32)
    s_k = np.linspace(0.5, 2.0, L).astype(np.float32)
    got = O.logits_request(H, D, "fp8", q, s_q, w, k, s_k, np.array([L], np.int32))[0]
    for j in range(L):
        dot = D * 1.0 * (2.0 if j != 4 else -2.0)
        want = sum(float(w[0, h]) * max(float(s_q[0, h]) * float(s_k[j]) * dot, 0.0)
                   for h in range(H))
        assert got[j] == pytest.approx(want, rel=1e-15, abs=0)
    assert got[4] == 0.0


def test_operand_orientation_is_not_transposed():
    """A single non-zero element pairs q[h, d] with k[j, d] only (same d)."""
    H, D, L = 2, 32, 5
    q = np.zeros((1, H, D), np.uint8)
    k = np.zeros((L, D), np.uint8)
    q[0, 1, 3] = 0x38          # q[h=1, d=3] = 1
    k[2, 3] = 0x48             # k[j=2, d=3] = 4
    k[3, 1] = 0x48             # k[j=3, d=1] = 4 (would pair only if d/h were swapped)
    ones = np.ones((1, H), np.float32)
    got = O.logits_request(H, D, "fp8", q, ones, ones, k, np.ones(L, np.float32),
                           np.array([L], np.int32))[0]
    assert got.tolist() == [0.0, 0.0, 4.0, 0.0, 0.0]


def test_fp4_block_scales_apply_per_32_elements():
    """Closed form: e2m1 code 2 (=1.0) with ue8m0 exponents per 32-element block."""
    H, D, L = 1, 128, 2
    q = np.full((1, H, D), 0x38, np.uint8)             # q = 1.0
    k = np.full((L, D // 2), 0x22, np.uint8)           # both nibbles code 2 = 1.0
    ue = np.array([[127, 128, 126, 130], [127, 127, 127, 127]], np.uint8)
    ones = np.ones((1, H), np.float32)
    got = O.logits_request(H, D, "fp4", q, ones, ones, k, ue, np.array([L], np.int32))[0]
    assert got[0] == 32 * (1 + 2 + 0.5 + 8)
    assert got[1] == 128.0
    # low nibble is element 2i: make element 0 negative in key 1 only
    k2 = k.copy()
    k2[1, 0] = 0x2A                                     # low nibble 0xA = -1.0
    got2 = O.logits_request(H, D, "fp4", q, ones, ones, k2, ue, np.array([L], np.int32))[0]
    assert got2[1] == 126.0


def test_fp4_keys_with_more_than_eight_scale_blocks_are_refused():
    """One ue8m0 scale per 32 elements and at most eight of them per key (D <= 256): a
    wider fp4 key is an argument error, not a key whose last blocks are dropped."""
    H, D, L = 1, 288, 1
    q = np.full((1, H, D), 0x38, np.uint8)
    k = np.full((L, D // 2), 0x22, np.uint8)
    ue = np.full((L, D // 32), 127, np.uint8)
    ones = np.ones((1, H), np.float32)
    with pytest.raises(RuntimeError):
        O.logits_request(H, D, "fp4", q, ones, ones, k, ue, np.array([L], np.int32))
    # the widest accepted key uses all eight scales
    D = 256
    q = np.full((1, H, D), 0x38, np.uint8)
    k = np.full((L, D // 2), 0x22, np.uint8)
    ue = (127 + np.arange(8, dtype=np.uint8))[None, :]
    got = O.logits_request(H, D, "fp4", q, ones, ones, k, ue, np.array([L], np.int32))[0]
    assert got[0] == 32 * sum(2.0 ** b for b in range(8))


# ---------------------------------------------------------------- invariants

def test_block_merge_identity():
    """topk(all keys) == topk(union of per-block top-k) for many block sizes (PIN4)."""
    p = small_problem(H=2, D=32, rows=3, L=257, seed=11, topk=16)
    vals = O.problem_logits(p)
    cl = p.compress_len.numpy()
    k = 16
    full = O.topk_rows(vals, cl, k)
    for B in (1, 7, k - 1, k, 3 * k, 257):
        for r in range(3):
            cv, ci = [], []
            for b0 in range(0, int(cl[r]), B):
                b1 = min(int(cl[r]), b0 + B)
                idx, v = O.select_pairs(vals[r, b0:b1], np.arange(b0, b1), k)
                keep = idx >= 0
                cv += v[keep].tolist()
                ci += idx[keep].tolist()
            merged, _ = O.select_pairs(np.array(cv), np.array(ci), k)
            assert merged.tolist() == full[r].tolist(), (B, r)


def test_block_merge_identity_candidate_blocks():
    p = small_problem(H=2, D=32, rows=2, L=200, seed=12)
    vals = O.problem_logits(p)
    cl = p.compress_len.numpy()
    ldm = 25
    full = O.candidates_rows(vals, cl, 8, 6, ldm)
    _, pooled = O.candidates_rows(vals, cl, 8, 6, ldm, with_pooled=True)
    for r in range(2):
        nb = (int(cl[r]) + 7) // 8
        cv, ci = [], []
        for b0 in range(0, nb, 5):
            b1 = min(nb, b0 + 5)
            idx, v = O.select_pairs(pooled[r, b0:b1], np.arange(b0, b1), 6)
            cv += v[idx >= 0].tolist()
            ci += idx[idx >= 0].tolist()
        merged, _ = O.select_pairs(np.array(cv), np.array(ci), 6)
        want = np.zeros(ldm, np.uint8)
        want[merged[merged >= 0]] = 1
        assert np.array_equal(full[r], want)


def test_row_chunking_and_order_do_not_change_results():
    """Row-chunk invariance: scoring rows in any grouping gives identical bits."""
    p = small_problem(H=4, D=64, rows=9, L=120, seed=13)
    all_rows = O.problem_logits(p)
    for chunk in (1, 2, 4):
        parts = [O.problem_logits(p, rows=np.arange(a, min(9, a + chunk)))
                 for a in range(0, 9, chunk)]
        assert np.array_equal(np.concatenate(parts), all_rows)
    perm = np.array([5, 0, 8, 2])
    assert np.array_equal(O.problem_logits(p, rows=perm), all_rows[perm])


def test_keys_past_compress_len_have_no_effect_and_causal_step():
    """Causal rule: keys j >= compress_len are never read; raising it by 1 admits exactly one key."""
    p = small_problem(H=2, D=32, rows=4, L=60, seed=14)
    base = O.problem_logits(p)
    cl = p.compress_len.numpy().copy()
    k2 = p.k.clone()
    k2[int(cl.min()):] = 0x7E  # 448 everywhere past the shortest row's length
    p2 = W.Problem(**{**p.__dict__, "k": k2})
    got = O.problem_logits(p2)
    for r in range(4):
        c = int(cl[r])
        assert np.array_equal(got[r, :int(cl.min())], base[r, :int(cl.min())])
        assert np.all(np.isneginf(got[r, c:]))
    # one more admitted key
    cl3 = cl.copy()
    cl3[0] = cl[0] - 1
    p3 = W.Problem(**{**p.__dict__, "compress_len": torch.tensor(cl3)})
    v3 = O.problem_logits(p3)
    assert np.array_equal(v3[0, :cl3[0]], base[0, :cl3[0]])
    assert np.isneginf(v3[0, cl3[0]]) and np.isfinite(base[0, cl3[0]])


def test_zero_length_rows_and_short_rows_pad_with_minus_one():
    p = small_problem(H=2, D=32, rows=4, L=20, seed=15, ratio=2)
    cl = p.compress_len.numpy().copy()
    cl[0], cl[1] = 0, 3
    p = W.Problem(**{**p.__dict__, "compress_len": torch.tensor(cl)})
    sel = O.problem_topk(p, k=7)
    assert sel[0].tolist() == [-1] * 7
    assert sorted(sel[1][:3].tolist()) == [0, 1, 2] and sel[1][3:].tolist() == [-1] * 4
    m = O.problem_candidates(p, ld_mask=3) if p.spec.cand_topk else None
    assert m is None or not m[0].any()


def test_weights_scale_linearly_and_nonnegative_weights_give_nonnegative_logits():
    p = small_problem(H=4, D=32, rows=3, L=50, seed=16)
    base = O.problem_logits(p)
    fin = np.isfinite(base)
    assert np.all(base[fin] >= 0)
    p2 = W.Problem(**{**p.__dict__, "w": p.w * 2})
    assert np.array_equal(O.problem_logits(p2)[fin], 2 * base[fin])
    # negating all weights negates all logits; heads are summed, not maxed
    p3 = W.Problem(**{**p.__dict__, "w": -p.w})
    assert np.array_equal(O.problem_logits(p3)[fin], -base[fin])


def test_head_permutation_changes_only_rounding():
    p = small_problem(H=4, D=32, rows=2, L=50, seed=17)
    base = O.problem_logits(p)
    perm = torch.tensor([2, 0, 3, 1])
    p2 = W.Problem(**{**p.__dict__, "q": p.q[:, perm], "s_q": p.s_q[:, perm], "w": p.w[:, perm]})
    got = O.problem_logits(p2)
    fin = np.isfinite(base)
    assert np.allclose(got[fin], base[fin], rtol=1e-14, atol=0)


def test_exact_ties_go_to_the_lower_index():
    """Tie-break: duplicated keys score identically; the lower key index wins."""
    p = small_problem(H=2, D=32, rows=2, L=64, seed=18, topk=5)
    k = p.k.clone()
    ks = p.k_scale.clone()
    vals = O.problem_logits(p)
    top = int(np.argmax(vals[0, :int(p.compress_len[0])]))
    # copy the best key into slots before and after it: all tie with it
    dup = [j for j in range(0, int(p.compress_len[0]), 7) if j != top][:6]
    for j in dup:
        k[j] = k[top]
        ks[j] = ks[top]
    p2 = W.Problem(**{**p.__dict__, "k": k, "k_scale": ks})
    v2 = O.problem_logits(p2)
    assert all(v2[0, j] == v2[0, top] for j in dup)
    sel = O.problem_topk(p2, k=5)[0].tolist()
    assert sel == sorted([top] + dup)[:5]


def test_selected_dominate_unselected():
    p = small_problem(H=4, D=64, rows=5, L=150, seed=19, topk=20)
    vals = O.problem_logits(p)
    cl = p.compress_len.numpy()
    sel = O.topk_rows(vals, cl, 20)
    for r in range(5):
        s = set(sel[r].tolist())
        chosen = [vals[r, j] for j in s]
        rest = [vals[r, j] for j in range(int(cl[r])) if j not in s]
        assert min(chosen) >= max(rest)
        assert len(s) == 20


def test_masked_topk_equals_topk_of_minus_inf_filled_scores():
    """Consumer masking: selecting within candidate blocks == selecting over scores with the
    non-candidate keys removed (brute force)."""
    p = small_problem(H=2, D=32, rows=3, L=100, seed=20, topk=9)
    vals = O.problem_logits(p)
    cl = p.compress_len.numpy()
    rng = np.random.default_rng(0)
    mask = (rng.random((3, 13)) < 0.4).astype(np.uint8)
    got = O.topk_rows(vals, cl, 9, mask=mask, mask_block=8)
    for r in range(3):
        elig = [j < cl[r] and mask[r, j // 8] for j in range(100)]
        want = brute.topk([float(x) for x in vals[r]], 9, elig)
        assert got[r].tolist() == want


def test_candidate_partial_last_block_pools_only_eligible_keys():
    p = small_problem(H=2, D=32, rows=2, L=45, seed=21)
    vals = O.problem_logits(p)
    cl = np.array([42, 17], np.int32)
    poisoned = vals.copy()
    for r in range(2):
        poisoned[r, cl[r]:] = 1e30      # values past compress_len must never be pooled
    m1, p1 = O.candidates_rows(vals, cl, 8, 3, 6, with_pooled=True)
    m2, p2 = O.candidates_rows(poisoned, cl, 8, 3, 6, with_pooled=True)
    assert np.array_equal(m1, m2) and np.array_equal(p1, p2)
    assert np.isneginf(p1[1, 3:]).all() and np.isfinite(p1[1, :3]).all()
    # fewer existing blocks than cand_topk: all of them are kept
    m3 = O.candidates_rows(vals, cl, 8, 100, 6)
    assert m3[0].tolist() == [1] * 6 and m3[1].tolist() == [1, 1, 1, 0, 0, 0]
    # brute force on the pooled scores
    for r in range(2):
        mb, _ = brute.candidate_mask([float(x) for x in vals[r, :cl[r]]], 8, 3, 6)
        assert m1[r].tolist() == mb


def test_generator_is_seeded_and_structured():
    spec = W.scaled(W.CONFIGS["long488k"], rows_div=64, keys_div=256)
    a, b = W.make_problem(spec), W.make_problem(spec)
    assert torch.equal(a.q, b.q) and torch.equal(a.k, b.k)
    # duplicated positions give byte-identical keys
    kk = a.k.numpy()
    _, inv, counts = np.unique(kk, axis=0, return_inverse=True, return_counts=True)
    assert counts.max() >= 2
    cl = a.compress_len.numpy()
    pos = a.pos.numpy()
    assert np.array_equal(cl, pos + 1)
    spec3 = W.scaled(W.CONFIGS["v4ratio2"], rows_div=64, keys_div=256)
    c = W.make_problem(spec3)
    assert np.array_equal(c.compress_len.numpy(), (c.pos.numpy() + 1) // 2)
    assert c.k.shape[1] == 64 and c.k_scale.shape[1] == 4
