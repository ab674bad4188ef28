"""fp4 x fp4 (e2m1 + ue8m0/32 queries and keys): the oracle's fp4-query mode pinned
against the fp8 oracle on equal values and against exact rationals (CPU); plans for e2m1
queries (CPU); the exact conversion kernel and the conversion route against the oracle
(GPU).  The native route (the block-scaled fp4 MMA) is checked with the other parity
cases."""
import dataclasses
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_attention_prefill_tcgen05_gb300 import _lib as K
from sparse_attention_prefill_tcgen05_gb300 import workloads as W
from tests import helpers as Hp


def _fp4q_problem(rows_div=64, keys_div=256, topk=40):
    spec = dataclasses.replace(W.scaled(W.CONFIGS["v4fp4qk"], rows_div, keys_div), topk=topk)
    return W.make_problem(spec)


def _as_fp8_queries(p):
    """The same query values as e4m3 codes with one power-of-two scale per head vector
    (2^(largest block exponent - 127)); asserts every value survives the cast exactly."""
    v = O.decode_fp4(p.q4.numpy(), p.q_sf.numpy())                    # [T, H, D]
    s = np.ldexp(1.0, p.q_sf.numpy().astype(np.int64).max(axis=-1) - 127)
    x = torch.from_numpy(v / s[..., None])
    codes = x.to(torch.float8_e4m3fn)
    assert torch.equal(codes.to(torch.float64), x), "a value has no exact e4m3 form"
    return codes.view(torch.uint8).contiguous(), torch.from_numpy(s).float()


def test_fp4_query_oracle_equals_fp8_oracle_on_equal_values():
    p = _fp4q_problem()
    q8, s_q = _as_fp8_queries(p)
    p8 = dataclasses.replace(p, q=q8, s_q=s_q, spec=dataclasses.replace(p.spec, qdtype="fp8"))
    a = O.problem_logits_fp4q(p)
    b = O.problem_logits(p8)
    assert np.array_equal(a, b)


def test_fp4_query_oracle_exact_rationals():
    """H=2, D=32, 12 keys: every logit equal to its exact rational value."""
    spec = W.ProblemSpec("tiny fp4", (W.RequestSpec(3, 9, 1),), H=2, D=32, topk=4,
                         kdtype="fp4", qdtype="fp4", seed=3)
    p = W.make_problem(spec)
    got = O.problem_logits_fp4q(p)
    tab = [Fraction(O.e2m1_value(c)) for c in range(16)]
    q4, qsf, k4, ksf = p.q4.numpy(), p.q_sf.numpy(), p.k.numpy(), p.k_scale.numpy()
    w, cl = p.w.numpy(), p.compress_len.numpy()
    for t in range(3):
        for j in range(12):
            if j >= cl[t]:
                assert got[t, j] == -np.inf
                continue
            kv = [tab[n] * Fraction(2) ** (int(ksf[j, 0]) - 127)
                  for b in k4[j] for n in (b & 15, b >> 4)]
            want = Fraction(0)
            for h in range(2):
                qv = [tab[n] * Fraction(2) ** (int(qsf[t, h, 0]) - 127)
                      for b in q4[t, h] for n in (b & 15, b >> 4)]
                x = sum(a * b for a, b in zip(qv, kv))
                want += Fraction(float(w[t, h])) * max(x, Fraction(0))
            assert abs(Fraction(got[t, j]) - want) <= abs(want) * Fraction(1, 2**50), (t, j)


@pytest.mark.gpu
def test_convert_fp4_is_exact():
    p = _fp4q_problem()
    T, H, D = p.q.shape
    codes = p.q4.reshape(T * H, D // 2).cuda()
    sf = p.q_sf.reshape(T * H, D // 32).cuda()
    q8 = torch.empty((T * H, D), dtype=torch.uint8, device="cuda")
    s = torch.empty(T * H, dtype=torch.float32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    K.indexer_convert_fp4(codes, sf, q8, s, ws)
    assert K.indexer_status(None, ws) == K.IDX_OK
    tab = np.array([O.e4m3_value(b) for b in range(256)], dtype=np.float64)
    got = tab[q8.cpu().numpy()] * s.cpu().numpy().astype(np.float64)[:, None]
    want = O.decode_fp4(p.q4.numpy(), p.q_sf.numpy()).reshape(T * H, D)
    assert np.array_equal(got, want)
    # a row whose second block is far below its first has no exact e4m3 form
    bad_sf = sf.clone()
    bad_sf[0, 1] = max(int(bad_sf[0, 0]) - 20, 0)
    bad_codes = codes.clone()
    bad_codes[0, 16] = 0x11            # 0.5, 0.5 in the second block
    K.indexer_convert_fp4(bad_codes, bad_sf, q8, s, ws)
    assert K.indexer_status(None, ws) == K.IDX_ERR_DEVICE_CHECK


@pytest.mark.gpu
def test_fp4_queries_and_keys_end_to_end():
    """The conversion route (for head counts without the fp4 MMA kind): convert q on the
    GPU, then the fp4-key logits and fused top-k, against the oracle."""
    p = _fp4q_problem()
    T, H, D = p.q.shape
    d = Hp.device_inputs(p)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    q8 = torch.empty((T * H, D), dtype=torch.uint8, device="cuda")
    s_q = torch.empty(T * H, dtype=torch.float32, device="cuda")
    K.indexer_convert_fp4(p.q4.reshape(T * H, D // 2).cuda(), p.q_sf.reshape(T * H, D // 32).cuda(),
                          q8, s_q, ws)
    assert K.indexer_status(None, ws) == K.IDX_OK
    d["q"], d["s_q"] = q8.reshape(T, H, D), s_q.reshape(T, H)
    plan = Hp.make_plan(p, qdtype=K.IDX_Q_FP8_E4M3)
    ref = O.problem_logits_fp4q(p)
    g = Hp.gpu_logits(p, plan, d).cpu().numpy()
    Hp.check_logits(g, ref)
    fi, _ = Hp.gpu_fused(p, plan, d)
    fi = fi.cpu().numpy()
    cl = p.compress_len.numpy()
    for t in range(T):
        Hp.check_topk_row(fi[t], ref[t], int(cl[t]), p.topk)


def _tiny_plan(qdtype, kdtype=K.IDX_K_FP4_E2M1_UE8M0, H=32, D=128):
    cu_q = torch.tensor([0, 4], dtype=torch.int32)
    cu_k = torch.tensor([0, 300], dtype=torch.int32)
    clen = torch.tensor([100, 200, 300, 300], dtype=torch.int32)
    return K.indexer_plan(cu_q, cu_k, clen, H, D, 8, kdtype=kdtype, qdtype=qdtype)


def test_plans_for_fp4_queries():
    """e2m1 queries plan with e2m1 keys and 32 heads of 128; other pairings are refused."""
    assert _tiny_plan(K.IDX_Q_FP4_E2M1_UE8M0).workspace_bytes > 0
    for bad in ({"kdtype": K.IDX_K_FP8_E4M3}, {"H": 16}, {"H": 8, "D": 64}):
        with pytest.raises(K.IndexerError) as e:
            _tiny_plan(K.IDX_Q_FP4_E2M1_UE8M0, **bad)
        assert e.value.code == K.IDX_ERR_UNSUPPORTED, bad
    with pytest.raises(K.IndexerError) as e:
        _tiny_plan(7)
    assert e.value.code == K.IDX_ERR_INVALID_ARG
