"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no attention arithmetic: it only draws numbers.  Recipe:
a CPU ``torch.Generator`` seeded with ``seed`` draws float32 i.i.d. N(0, 1)
values in the order q, k, v; each is then cast to the requested dtype
(bf16 rounding is round-to-nearest-even).  An optional power-of-two
``q_scale`` (e.g. 8 for the near-one-hot "outlier" variant) multiplies q
before the cast, which is exact in bf16.

Layouts: q [B, Nq, Hq, d], k and v [B, Nk, Hkv, d], all row-major.
"""
from __future__ import annotations

import torch


def make_qkv(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int, seed: int,
             dtype: torch.dtype = torch.bfloat16, q_scale: float = 1.0):
    """Return CPU tensors (q, k, v) of the given shapes and dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, Nq, Hq, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, Nk, Hkv, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, Nk, Hkv, d), generator=g, dtype=torch.float32)
    if q_scale != 1.0:
        q = q * q_scale
    return q.to(dtype), k.to(dtype), v.to(dtype)


def make_partials(P: int, rows: int, d: int, seed: int, empty_frac: float = 0.0):
    """Random normalised partial outputs and log-sum-exps for merge tests.

    Returns float32 CPU tensors (o_parts [P, rows, d], lse_parts [P, rows]);
    a fraction ``empty_frac`` of the parts get lse = -inf (empty segments).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    o_parts = torch.randn((P, rows, d), generator=g, dtype=torch.float32)
    lse_parts = 4.0 * torch.randn((P, rows), generator=g, dtype=torch.float32)
    if empty_frac > 0.0:
        mask = torch.rand((P, rows), generator=g) < empty_frac
        lse_parts = lse_parts.masked_fill(mask, float("-inf"))
        o_parts = o_parts.masked_fill(mask[..., None], 0.0)
    return o_parts, lse_parts


def sample_rows(B: int, Hq: int, Nq: int, n: int, seed: int):
    """``n`` distinct (b, hq, i) rows, always including the first and last
    row of every tile boundary case (i = 0 and i = Nq - 1)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 7919)
    total = B * Hq * Nq
    n = min(n, total)
    idx = torch.randperm(total, generator=g)[:n].tolist()
    idx += [0, total - 1]
    out = []
    seen = set()
    for r in idx:
        if r in seen:
            continue
        seen.add(r)
        b = r // (Hq * Nq)
        hq = (r // Nq) % Hq
        i = r % Nq
        out.append((b, hq, i))
    return out
