"""The host-only chunk planner helper ("chunked-prefill-memory.md", section 2.1):
the library against the oracle's exact-arithmetic restatement, the schedule the
section prints, hand-computed values of the formula and its invariants (CPU only)."""
import json
import os

import pytest

from oracle import oracle as O
from sparse_attention_prefill_tcgen05_gb300 import _lib as K

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "chunk_schedule.json")))


def test_printed_schedule_is_power_of_two_rounding():
    """Every band of the printed schedule, on the library and the oracle, with the
    section's budget and limits (the page is irrelevant in power-of-two mode)."""
    args = dict(budget_token2=GOLD["budget_token2"], chunk_min=GOLD["chunk_min"],
                chunk_max=GOLD["chunk_max"], page=GOLD["page"], pow2=True)
    for band in GOLD["bands"]:
        lo, hi = band["prefix_from"], band["prefix_to"]
        for L in (int(lo * 1.02) + 1, (lo + hi) // 2, int(hi * 0.98)):
            assert O.chunk_rows(L, **args) == band["chunk"], (L, band)
            assert K.indexer_chunk_rows(L, **args) == band["chunk"], (L, band)


def test_formula_values_by_hand():
    """BUDGET / L rounded down to a multiple of 256, clamped to [256, 2048]."""
    cases = {50_000: 2048,          # 4000 -> clamped to the maximum
             100_000: 1792,         # 2000 -> 7 pages
             150_000: 1280,         # 1333.3 -> 5 pages
             400_000: 256,          # 500 -> 1 page
             1_000_000: 256,        # 200 -> 0 pages -> clamped to the minimum
             0: 2048}               # no prefix yet
    for L, want in cases.items():
        assert O.chunk_rows(L) == want, L
        assert K.indexer_chunk_rows(L) == want, L


@pytest.mark.parametrize("params", [
    dict(budget_token2=2.0e8, chunk_min=256, chunk_max=2048, page=256),
    dict(budget_token2=2.6e8, chunk_min=128, chunk_max=4096, page=64),
    dict(budget_token2=1.0e6, chunk_min=1, chunk_max=1000, page=7),
])
@pytest.mark.parametrize("pow2", [False, True])
def test_library_matches_oracle_and_keeps_the_budget(params, pow2):
    prev = None
    for e in range(0, 70):
        L = int(round(1.3 ** e))
        got = K.indexer_chunk_rows(L, pow2=pow2, **params)
        assert got == O.chunk_rows(L, pow2=pow2, **params), L
        assert params["chunk_min"] <= got <= params["chunk_max"]
        if got > params["chunk_min"]:
            assert got * L <= params["budget_token2"]      # T x L stays within the budget
        if params["chunk_min"] < got < params["chunk_max"]:       # not clamped: rounded
            assert (got & (got - 1)) == 0 if pow2 else got % params["page"] == 0
        if prev is not None:
            assert got <= prev                              # never grows with the prefix
        prev = got


@pytest.mark.parametrize("bad", [
    dict(budget_token2=0.0), dict(budget_token2=float("inf")), dict(chunk_min=0),
    dict(chunk_min=512, chunk_max=256), dict(page=0)])
def test_invalid_arguments_are_rejected(bad):
    with pytest.raises(K.IndexerError) as e:
        K.indexer_chunk_rows(100_000, **bad)
    assert e.value.code == K.IDX_ERR_INVALID_ARG
