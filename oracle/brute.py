"""Exact brute force for tiny inputs -- TEST INFRASTRUCTURE ONLY.

Pure Python with ``fractions.Fraction``: every input (fp8/fp4 codes, fp32
scales, fp32 head weights) is a dyadic rational, so the scores below are
exact, with no rounding at all.  Used to pin the C oracle on tiny problems;
it is far too slow for anything else.

The number formats are decoded here from the bit layouts directly (sign,
exponent field, mantissa field), independently of ``oracle.c``.
"""
from __future__ import annotations

from fractions import Fraction


def e4m3(b: int) -> Fraction:
    s = -1 if b & 0x80 else 1
    e = (b >> 3) & 0xF
    m = b & 7
    if e == 15 and m == 7:
        raise ValueError("e4m3 NaN code")
    if e == 0:
        return s * Fraction(m, 8) * Fraction(1, 64)
    return s * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


def e2m1(nib: int) -> Fraction:
    s = -1 if nib & 0x8 else 1
    e = (nib >> 1) & 3
    m = nib & 1
    if e == 0:
        return s * Fraction(m, 2)
    return s * (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)


def f32(x) -> Fraction:
    return Fraction(float(x))


def score(q_row, s_q_row, w_row, k_row, k_scale_row, kdtype: str) -> Fraction:
    """Exact logit of one (row, key): sum_h w_h * max(s_q,h * s_k * <q_h, k>, 0)."""
    H = len(q_row)
    D = len(q_row[0])
    if kdtype == "fp8":
        kv = [e4m3(int(b)) for b in k_row]
        sk = f32(k_scale_row)
    else:
        kv = []
        for d in range(D):
            byte = int(k_row[d // 2])
            nib = (byte >> 4) if d & 1 else (byte & 0xF)
            kv.append(e2m1(nib) * Fraction(2) ** (int(k_scale_row[d // 32]) - 127))
        sk = Fraction(1)
    total = Fraction(0)
    for h in range(H):
        dot = sum(e4m3(int(q_row[h][d])) * kv[d] for d in range(D))
        x = f32(s_q_row[h]) * sk * dot
        total += f32(w_row[h]) * (x if x > 0 else 0)
    return total


def row_scores(q_row, s_q_row, w_row, k, k_scale, clen, kdtype):
    return [score(q_row, s_q_row, w_row, k[j], k_scale[j], kdtype) for j in range(clen)]


def topk(scores, k, eligible=None):
    """Indices of the k largest scores, ties to the lower index, -1 padded."""
    idx = [j for j in range(len(scores)) if eligible is None or eligible[j]]
    idx.sort(key=lambda j: (-scores[j], j))
    out = idx[:k]
    return out + [-1] * (k - len(out))


def candidate_mask(scores, block, cand_topk, nblocks_out):
    """Pool eligible scores over aligned blocks, keep the top blocks (ties to lower block)."""
    n = len(scores)
    nb = (n + block - 1) // block
    pooled = [max(scores[b * block: min(n, (b + 1) * block)]) for b in range(nb)]
    order = sorted(range(nb), key=lambda b: (-pooled[b], b))[:cand_topk]
    mask = [0] * nblocks_out
    for b in order:
        mask[b] = 1
    return mask, pooled
