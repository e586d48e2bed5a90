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


def make_paged(B: int, Hq: int, Hkv: int, d: int, page_size: int, seq_lens, seed: int,
               extra_pages: int = 3, poison: bool = True, dtype: torch.dtype = torch.bfloat16):
    """A random paged KV cache on the CPU.

    Sequence b owns ceil(seq_lens[b] / page_size) distinct pages, drawn in
    random order from a shuffled pool with ``extra_pages`` pages nobody owns.
    Table entries past a sequence's pages are -1.  With ``poison`` every pool
    slot that no sequence's first seq_lens[b] positions use is NaN.
    Returns (q [B,1,Hq,d], k_pages, v_pages [num_pages, page_size, Hkv, d],
    block_table [B, max_pages] int32, seq_lens [B] int32).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    lens = [int(x) for x in seq_lens]
    need = [(L + page_size - 1) // page_size for L in lens]
    max_pages = max(1, max(need))
    num_pages = sum(need) + extra_pages
    perm = torch.randperm(num_pages, generator=g).tolist()
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    owned = torch.zeros((num_pages, page_size), dtype=torch.bool)
    pos = 0
    for b in range(B):
        for j in range(need[b]):
            pg = perm[pos]
            pos += 1
            table[b, j] = pg
            n_used = min(page_size, lens[b] - j * page_size)
            owned[pg, :n_used] = True
    q = torch.randn((B, 1, Hq, d), generator=g, dtype=torch.float32)
    kp = torch.randn((num_pages, page_size, Hkv, d), generator=g, dtype=torch.float32)
    vp = torch.randn((num_pages, page_size, Hkv, d), generator=g, dtype=torch.float32)
    q, kp, vp = q.to(dtype), kp.to(dtype), vp.to(dtype)
    if poison:
        kp[~owned] = float("nan")
        vp[~owned] = float("nan")
    return q, kp, vp, table, torch.tensor(lens, dtype=torch.int32)
