"""Seeded synthetic inputs for the dense prefill indexer.

This module only *draws and quantises inputs*; it holds none of the
indexer's arithmetic (no dot products, no ReLU/head reduction, no top-k).
Both the CUDA path and the CPU oracle consume the bytes it produces, so it
is the one piece the two sides share.

Shapes follow the workloads the source pages describe:
  * "[DeepSeek-V4.1] Bound the dense prefill indexer transient" (SGLang PR
    #39187), Motivation: a 16,384-token chunk of a 487,936-token request,
    DeepGEMM ``fp8_fp4_mqa_logits`` (fp8 q, fp4 k).
  * "chunked-prefill-memory.md", section 1: ratio-1/2 low-ratio layers, chunks
    of T rows scored against the compressed prefix L; section 2.3: key blocks
    of 32k, top-512, 8-key block pooling, top-2048 blocks.
  * SGLang fork commit log ("test/manual"), the logits-chunk-cap commit:
    GLM-5.1 shapes H=32, D=128, topk=2048, cold 64K chunk.

Quantisation (a reading, the pages never spell it out):
  * fp8 e4m3: one fp32 scale per head vector of q (``s_q[t,h]``) and per key
    (``s_k[j]``), ``s = absmax/448`` (1.0 for an all-zero vector), codes by
    round-to-nearest-even with saturation at +-448.
  * fp4 e2m1 + ue8m0: one power-of-two scale per 32 consecutive elements of
    a key, exponent ``floor(log2(absmax)) - 2`` as in the OCP MX recipe,
    elements rounded to nearest-even on the e2m1 grid and saturated at +-6;
    two elements per byte, element 2i in the low nibble.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Sequence

import numpy as np
import torch

E4M3_MAX = 448.0
E2M1_MAX = 6.0

# e2m1 magnitudes by 3-bit code (sign is bit 3): the OCP MX element grid.
_E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
_E2M1_MIDPOINTS = tuple((a + b) / 2 for a, b in zip(_E2M1_GRID[:-1], _E2M1_GRID[1:]))


@dataclass(frozen=True)
class RequestSpec:
    """One request of a prefill batch.

    ``rows`` query rows sit at absolute positions ``pos0 .. pos0+rows-1``;
    the request's compressed prefix holds ``L = floor((pos0+rows)/ratio)``
    keys and row t may look at ``compress_len(t) = floor((pos(t)+1)/ratio)``
    of them.
    """

    rows: int
    pos0: int
    ratio: int = 1

    @property
    def keys(self) -> int:
        return (self.pos0 + self.rows) // self.ratio


@dataclass(frozen=True)
class ProblemSpec:
    name: str
    requests: tuple
    H: int
    D: int
    topk: int
    kdtype: str = "fp8"          # "fp8" or "fp4" (e2m1 + ue8m0 per 32)
    seed: int = 0
    qdtype: str = "fp8"          # "fp8", or "fp4": e2m1 + ue8m0 per 32 queries (fp4 x fp4)
    heavy_keys_frac: float = 0.0  # fraction of keys multiplied before quantising
    heavy_keys_mult: float = 4.0
    dup_frac: float = 0.0         # fraction of key positions copied from earlier ones
    cand_block: int = 8           # candidate path: keys per pooled block
    cand_topk: int = 0            # candidate path: blocks kept per row (0 = no candidate path)
    key_block: int = 0            # key-block size the workload names (0 = planner's choice)
    exact: bool = False           # small-integer codes + power-of-two scales

    @property
    def total_rows(self) -> int:
        return sum(r.rows for r in self.requests)

    @property
    def total_keys(self) -> int:
        return sum(r.keys for r in self.requests)

    @property
    def dense_pairs(self) -> int:
        """Sum over requests of T_r * L_r (the dense pairs the metric counts)."""
        return sum(r.rows * r.keys for r in self.requests)


# The five workloads: a tiny oracle-sized case and four shaped like the pages'.
CONFIGS = {
    "tiny": ProblemSpec(
        "tiny: T=64 rows at pos 960..1023, L=1024, H=4, D=64, fp8, top-32",
        (RequestSpec(64, 960, 1),), H=4, D=64, topk=32, seed=0),
    "cold64k": ProblemSpec(
        "cold chunk: T=2048 rows ending a 65,536-token prefix, L=65,536, H=32, D=128, fp8, "
        "5% of keys x4, top-2048",
        (RequestSpec(2048, 63488, 1),), H=32, D=128, topk=2048, seed=2,
        heavy_keys_frac=0.05, heavy_keys_mult=4.0),
    "v4ratio2": ProblemSpec(
        "low-ratio layer: T=2048 rows at prefix 200,000, ratio 2, L=100,000, H=32, D=128, "
        "fp8 q x fp4(e2m1+ue8m0/32) k, top-512, key blocks of 32,768",
        (RequestSpec(2048, 197952, 2),), H=32, D=128, topk=512, kdtype="fp4", seed=3,
        key_block=32768),
    "long488k": ProblemSpec(
        "long-context chunk: T=16,384 rows ending a 487,936-token prefix, L=487,936, H=32, "
        "D=128, fp8, 1% of positions duplicated (exact ties), top-512",
        (RequestSpec(16384, 471552, 1),), H=32, D=128, topk=512, seed=4, dup_frac=0.01),
    "v4fp4qk": ProblemSpec(
        "low-ratio layer, fp4 x fp4: T=2048 rows at prefix 200,000, ratio 2, L=100,000, "
        "H=32, D=128, e2m1+ue8m0/32 queries and keys, top-512, key blocks of 32,768",
        (RequestSpec(2048, 197952, 2),), H=32, D=128, topk=512, kdtype="fp4", seed=6,
        key_block=32768, qdtype="fp4"),
    "ragged_cand": ProblemSpec(
        "ragged batch + candidates: 4 cold requests of 7,168 rows (ratios 1,2,1,2) and a "
        "2,048-row chunk on a 150,000-token cached prefix; 8-key block pooling, top-2048 "
        "blocks, consumer top-512",
        (RequestSpec(7168, 0, 1), RequestSpec(7168, 0, 2), RequestSpec(7168, 0, 1),
         RequestSpec(7168, 0, 2), RequestSpec(2048, 150000, 1)),
        H=32, D=128, topk=512, seed=5, cand_block=8, cand_topk=2048),
}


@dataclass
class Problem:
    """Quantised inputs of one batch, all on the CPU (torch tensors)."""

    spec: ProblemSpec
    q: torch.Tensor            # uint8 [T, H, D] fp8 e4m3 codes
    s_q: torch.Tensor          # float32 [T, H]
    w: torch.Tensor            # float32 [T, H]
    k: torch.Tensor            # uint8 [Lk, D] (fp8) or [Lk, D/2] (fp4 packed)
    k_scale: torch.Tensor      # float32 [Lk] (fp8) or uint8 [Lk, D/32] (ue8m0)
    cu_seqlens_q: torch.Tensor  # int32 [R+1]
    cu_seqlens_k: torch.Tensor  # int32 [R+1]
    compress_len: torch.Tensor  # int32 [T]
    pos: torch.Tensor           # int64 [T] absolute positions
    # second layer's queries for the candidate consumer (same k, same compress_len)
    q2: Optional[torch.Tensor] = None
    s_q2: Optional[torch.Tensor] = None
    w2: Optional[torch.Tensor] = None
    dup_rows: list = field(default_factory=list)   # rows whose q was copied from an earlier row
    # qdtype "fp4": the queries as e2m1 codes [T, H, D/2] and ue8m0 exponents [T, H, D/32]
    # (q and s_q then hold zeros / ones and are not inputs)
    q4: Optional[torch.Tensor] = None
    q_sf: Optional[torch.Tensor] = None

    @property
    def H(self):
        return self.spec.H

    @property
    def D(self):
        return self.spec.D

    @property
    def topk(self):
        return self.spec.topk

    def request_of_row(self) -> np.ndarray:
        cu = self.cu_seqlens_q.numpy()
        return np.searchsorted(cu, np.arange(int(cu[-1])), side="right") - 1


def quantize_fp8(x: torch.Tensor):
    """Absmax-scaled fp8 e4m3 codes along the last axis. Returns (uint8 codes, fp32 scales)."""
    amax = x.abs().amax(dim=-1, keepdim=True)
    s = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    y = (x / s).clamp_(-E4M3_MAX, E4M3_MAX)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, s.squeeze(-1).to(torch.float32)


def _e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    """Round v (already divided by its block scale) onto the e2m1 grid.

    Nearest grid point, ties to the even 3-bit code, saturating at +-6; a
    value that rounds to zero keeps a positive sign.
    """
    mag = v.abs()
    code = torch.zeros(mag.shape, dtype=torch.int64)
    for i, m in enumerate(_E2M1_MIDPOINTS):
        up = mag > m
        if (i + 1) % 2 == 0:
            up |= mag == m
        code += up.to(torch.int64)
    sign = (v < 0) & (code > 0)
    return (code | (sign.to(torch.int64) << 3)).to(torch.uint8)


def quantize_fp4(x: torch.Tensor, block: int = 32):
    """e2m1 codes with one ue8m0 scale per ``block`` elements along the last axis.

    Returns (uint8 packed [.., D/2] with element 2i in the low nibble,
    uint8 ue8m0 exponents [.., D/block]).
    """
    *lead, D = x.shape
    xb = x.reshape(*lead, D // block, block)
    amax = xb.abs().amax(dim=-1)
    e = torch.zeros_like(amax, dtype=torch.int64)
    nz = amax > 0
    e[nz] = torch.floor(torch.log2(amax[nz].double())).to(torch.int64) - 2
    ue = (e + 127).clamp(0, 254)
    ue[~nz] = 127
    scale = torch.pow(2.0, (ue - 127).double()).to(torch.float64)
    v = (xb.double() / scale.unsqueeze(-1)).to(torch.float32)
    codes = _e2m1_codes(v).reshape(*lead, D)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    return packed.contiguous(), ue.to(torch.uint8).contiguous()


def _exact_fp8(gen, shape):
    """fp8 codes of small integers in [-8, 8] (all exactly representable in e4m3)."""
    ints = torch.randint(-8, 9, shape, generator=gen).to(torch.float32)
    return ints.to(torch.float8_e4m3fn).view(torch.uint8)


def make_problem(spec: ProblemSpec) -> Problem:
    gen = torch.Generator().manual_seed(spec.seed)
    H, D = spec.H, spec.D
    qs, sqs, ws, ks, kss, clens, poss = [], [], [], [], [], [], []
    q2s, sq2s, w2s = [], [], []
    q4s, qsfs = [], []
    dup_rows = []
    row_base = 0
    for req in spec.requests:
        T_r, L_r = req.rows, req.keys
        pos = torch.arange(req.pos0, req.pos0 + T_r, dtype=torch.int64)
        clen = ((pos + 1) // req.ratio).to(torch.int32)
        if spec.exact:
            q = _exact_fp8(gen, (T_r, H, D))
            s_q = torch.pow(2.0, torch.randint(-4, 1, (T_r, H), generator=gen).float())
            w = torch.full((T_r, H), 0.125)
            if spec.kdtype == "fp8":
                k = _exact_fp8(gen, (L_r, D))
                s_k = torch.pow(2.0, torch.randint(-4, 1, (L_r,), generator=gen).float())
            else:
                k = torch.randint(0, 256, (L_r, D // 2), generator=gen).to(torch.uint8)
                s_k = torch.randint(124, 131, (L_r, D // 32), generator=gen).to(torch.uint8)
            if spec.qdtype == "fp4":
                # e2m1 codes of magnitude <= 1.5 (codes 0-3 and 8-11) and block exponents
                # 126..128: with the keys above, every product, block sum and head sum is
                # a short dyadic number, exact in fp32 in any order
                codes = (torch.randint(0, 4, (T_r, H, D), generator=gen) |
                         (torch.randint(0, 2, (T_r, H, D), generator=gen) << 3))
                q4s.append((codes[..., 0::2] | (codes[..., 1::2] << 4)).to(torch.uint8))
                qsfs.append(torch.randint(126, 129, (T_r, H, D // 32),
                                          generator=gen).to(torch.uint8))
                q, s_q = torch.zeros((T_r, H, D), dtype=torch.uint8), torch.ones((T_r, H))
            qs.append(q); sqs.append(s_q); ws.append(w); ks.append(k); kss.append(s_k)
        else:
            qf = torch.randn((T_r, H, D), generator=gen)
            kf = torch.randn((L_r, D), generator=gen)
            w = torch.rand((T_r, H), generator=gen) / math.sqrt(H)
            if spec.heavy_keys_frac > 0:
                n = int(spec.heavy_keys_frac * L_r)
                idx = torch.randperm(L_r, generator=gen)[:n]
                kf[idx] *= spec.heavy_keys_mult
            if spec.dup_frac > 0 and L_r > 1:
                n = int(spec.dup_frac * L_r)
                ps = torch.sort(torch.randperm(L_r - 1, generator=gen)[:n] + 1).values
                srcs = (torch.rand(n, generator=gen, dtype=torch.float64) * ps.double()).floor().long()
                for p, p_src in zip(ps.tolist(), srcs.tolist()):
                    kf[p] = kf[p_src]
                    # the query rows of those positions too, when both lie in this chunk
                    a, b = p * req.ratio - req.pos0, p_src * req.ratio - req.pos0
                    if req.ratio == 1 and 0 <= a < T_r and 0 <= b < T_r:
                        qf[a] = qf[b]
                        w[a] = w[b]
                        dup_rows.append(row_base + a)
            if spec.qdtype == "fp4":
                q4, qsf = quantize_fp4(qf)
                q4s.append(q4); qsfs.append(qsf)
                q, s_q = torch.zeros((T_r, H, D), dtype=torch.uint8), torch.ones((T_r, H))
            else:
                q, s_q = quantize_fp8(qf)
            qs.append(q); sqs.append(s_q); ws.append(w.float())
            if spec.kdtype == "fp8":
                k, s_k = quantize_fp8(kf)
            else:
                k, s_k = quantize_fp4(kf)
            ks.append(k); kss.append(s_k)
        clens.append(clen); poss.append(pos)
        row_base += T_r
    if spec.cand_topk > 0:
        # the consumer layer: fresh queries against the same keys
        for req in spec.requests:
            qf = torch.randn((req.rows, H, D), generator=gen)
            w = torch.rand((req.rows, H), generator=gen) / math.sqrt(H)
            q, s_q = quantize_fp8(qf)
            q2s.append(q); sq2s.append(s_q); w2s.append(w.float())
    cu_q = torch.zeros(len(spec.requests) + 1, dtype=torch.int32)
    cu_k = torch.zeros(len(spec.requests) + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(torch.tensor([r.rows for r in spec.requests]), 0)
    cu_k[1:] = torch.cumsum(torch.tensor([r.keys for r in spec.requests]), 0)
    p = Problem(
        spec=spec,
        q=torch.cat(qs).contiguous(), s_q=torch.cat(sqs).float().contiguous(),
        w=torch.cat(ws).float().contiguous(),
        k=torch.cat(ks).contiguous(), k_scale=torch.cat(kss).contiguous(),
        cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
        compress_len=torch.cat(clens).contiguous(), pos=torch.cat(poss),
        dup_rows=dup_rows)
    if q4s:
        p.q4 = torch.cat(q4s).contiguous()
        p.q_sf = torch.cat(qsfs).contiguous()
    if q2s:
        p.q2 = torch.cat(q2s).contiguous()
        p.s_q2 = torch.cat(sq2s).float().contiguous()
        p.w2 = torch.cat(w2s).float().contiguous()
    return p


def scaled(spec: ProblemSpec, rows_div: int = 1, keys_div: int = 1, name: str = None,
           **over) -> ProblemSpec:
    """A smaller copy of ``spec`` with the same structure (for oracle-sized parity runs).

    Each request keeps its chunk-at-the-end-of-prefix shape: ``rows/rows_div`` rows ending
    at the prefix ``(pos0+rows)/keys_div``.
    """
    reqs = []
    for r in spec.requests:
        rows = max(1, r.rows // rows_div)
        end = max(rows, (r.pos0 + r.rows) // keys_div)
        reqs.append(RequestSpec(rows, end - rows, r.ratio))
    return replace(spec, requests=tuple(reqs), name=name or spec.name + " (scaled)", **over)


def sample_rows(p: Problem, per_request: int = 256, seed: int = 0) -> np.ndarray:
    """Rows checked against the oracle for full-size problems.

    Always includes each request's first and last rows, its rows with the
    smallest compress_len, and rows whose queries were duplicated; the rest
    are drawn at random (seeded).
    """
    rng = np.random.default_rng(seed)
    cu = p.cu_seqlens_q.numpy()
    clen = p.compress_len.numpy()
    out = set()
    for r in range(len(cu) - 1):
        a, b = int(cu[r]), int(cu[r + 1])
        n = b - a
        if n <= per_request:
            out.update(range(a, b))
            continue
        chosen = {a, a + 1, b - 2, b - 1}
        order = np.argsort(clen[a:b], kind="stable")[:4]
        chosen.update(int(a + i) for i in order)
        chosen.update(x for x in p.dup_rows[:16] if a <= x < b)
        rest = rng.choice(np.arange(a, b), size=per_request, replace=False)
        for x in rest:
            if len(chosen) >= per_request:
                break
            chosen.add(int(x))
        out.update(chosen)
    return np.array(sorted(out), dtype=np.int64)
