"""Parity of attn_decode_paged against the oracle's paged decode.

Block tables are random permutations of a pool with unowned pages; every
slot no sequence owns is NaN (it must not reach the output).  Cases cover
page sizes 16, 32, 64 and 256, lengths on both sides of page and tile
boundaries, empty sequences (with one and with several segments), GQA
ratios 1, 3, 4 and 8, d = 64 and 128, and fixed and automatic segment counts;
with pages of 16 keys and 2, 4 or 8 KV heads, the kernel that takes every KV
head of a segment in one CTA."""
import math

import numpy as np
import pytest
import torch

from exact_attention_62_gb300.inputs import make_paged
from parity import compare

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    # B, Hq, Hkv, d, page_size, seq_lens, splits, max_seq_len (None = max of lens)
    (4, 8, 2, 128, 16, [1, 15, 16, 17], 0, None),
    (3, 32, 8, 128, 64, [0, 64, 1000], 0, None),
    (2, 16, 4, 64, 32, [500, 33], 3, None),
    (2, 8, 8, 128, 256, [5000, 4097], 0, None),
    (2, 8, 2, 128, 64, [0, 100], 1, None),
    (3, 8, 2, 64, 16, [63, 64, 65], 2, 400),          # segments past every sequence
    (2, 16, 2, 128, 32, [2047, 1], 7, None),
    # pages of 16 keys with 8 KV heads: one CTA takes all KV heads of a segment
    (4, 32, 8, 128, 16, [1, 15, 16, 17], 0, None),
    (3, 24, 8, 64, 16, [0, 33, 700], 3, None),         # 3 query heads per KV head, an empty sequence
    (2, 64, 8, 128, 16, [1000, 2048], 1, None),        # 8 per KV head; one segment writes O itself
    (2, 8, 8, 128, 16, [63, 65], 4, 400),              # 1 per KV head; segments past every sequence
    (1, 32, 8, 128, 16, [5000], 0, None),              # the automatic count: one wave of CTAs
    # ... with 4 and 2 KV heads: 2 or 4 pages per stage, the warps of a head merged
    (3, 16, 4, 128, 16, [1, 40, 1000], 0, None),
    (2, 32, 4, 64, 16, [0, 700], 3, None),
    (2, 16, 2, 128, 16, [2048, 33], 1, None),          # one segment: the merged warp writes O
    (2, 8, 2, 128, 16, [63, 65], 5, 400),              # stages with fewer pages than slots
]


@pytest.mark.parametrize("B,Hq,Hkv,d,ps,lens,S,maxlen", CASES)
def test_paged_decode_matches_oracle(attn, oracle_mod, B, Hq, Hkv, d, ps, lens, S, maxlen):
    q, kp, vp, table, sl = make_paged(B, Hq, Hkv, d, ps, lens, seed=sum(lens) + ps)
    scale = 1.0 / math.sqrt(d)
    max_seq_len = maxlen if maxlen is not None else max(lens)
    cols = (max_seq_len + ps - 1) // ps          # the table must cover max_seq_len
    if table.shape[1] < cols:
        table = torch.cat([table, torch.full((B, cols - table.shape[1]), -1, dtype=torch.int32)], 1)
    o, lse = attn.attn_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV),
                                    max_seq_len, scale, num_splits=S)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    ro, rl = oracle_mod.decode_paged(q, kp.float(), vp.float(), table.numpy(), sl.numpy(), scale)
    compare(o, lse, ro, rl, torch.bfloat16, "paged %s" % (lens,))
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.all(o[b] == 0) and torch.all(torch.isneginf(lse[b]))


def test_paged_long_context_and_many_sequences(attn, oracle_mod):
    """The two decode workloads' shapes on a paged cache: one 64K sequence in
    64-key pages, and 16 sequences of random length up to 8K in 16-key pages."""
    for (B, lens, ps) in [(1, [65536], 64),
                          (16, torch.randint(1, 8193, (16,), generator=torch.Generator().manual_seed(5)).tolist(), 16)]:
        q, kp, vp, table, sl = make_paged(B, 32, 8, 128, ps, lens, seed=77, poison=True)
        o, lse = attn.attn_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV),
                                        sl.to(DEV), max(lens), 128 ** -0.5)
        torch.cuda.synchronize()
        assert attn.attn_check_device_status() == 0
        ro, rl = oracle_mod.decode_paged(q, kp.float(), vp.float(), table.numpy(), sl.numpy(),
                                         128 ** -0.5)
        compare(o, lse, ro, rl, torch.bfloat16, "paged B=%d" % B)


def test_paged_equals_contiguous_decode(attn):
    """With pages laid out in order, the paged call sees the same keys as the
    dense decode of the same cache; both use the same kernels, so with the
    same segment count the results agree bit for bit."""
    B, Hq, Hkv, d, N, ps = 2, 16, 4, 128, 3000, 64
    g = torch.Generator().manual_seed(9)
    q = torch.randn((B, 1, Hq, d), generator=g).to(torch.bfloat16).to(DEV)
    kc = torch.randn((B, N, Hkv, d), generator=g).to(torch.bfloat16).to(DEV)
    vc = torch.randn((B, N, Hkv, d), generator=g).to(torch.bfloat16).to(DEV)
    npg = (N + ps - 1) // ps
    pad = npg * ps - N
    kp = torch.cat([kc, torch.zeros((B, pad, Hkv, d), dtype=kc.dtype, device=DEV)], 1)
    vp = torch.cat([vc, torch.zeros((B, pad, Hkv, d), dtype=vc.dtype, device=DEV)], 1)
    kp = kp.reshape(B * npg, ps, Hkv, d).contiguous()
    vp = vp.reshape(B * npg, ps, Hkv, d).contiguous()
    table = torch.arange(B * npg, dtype=torch.int32, device=DEV).reshape(B, npg)
    sl = torch.full((B,), N, dtype=torch.int32, device=DEV)
    for S in (1, 5):   # segment lengths are whole tiles in both when N/S is
        o1, l1 = attn.attn_decode_paged(q, kp, vp, table, sl, N, num_splits=S)
        o2, l2 = attn.attn_decode_splitkv(q, kc, vc, num_splits=S)
        torch.cuda.synchronize()
        if S == 1:
            assert torch.equal(o1, o2) and torch.equal(l1, l2)
        else:
            assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
            assert (l1 - l2).abs().max().item() <= 1e-4


@pytest.mark.parametrize("Hkv,ps", [(8, 16), (4, 16), (2, 64)])
def test_auto_count_keeps_segments_within_the_table(attn, Hkv, ps):
    """For very long sequences the automatic segment count is raised until
    one segment's pages fit the 4096-entry block-table staging area, which
    attn_decode_paged requires of every count (both kernels)."""
    for max_len in (1 << 20, 1 << 26, (1 << 27) + 5):
        S = attn.attn_decode_paged_num_splits(1, 4 * Hkv, Hkv, 128, ps, max_len)
        assert S >= 1
        seg = -(-max_len // S)
        seg = -(-seg // 64) * 64
        assert seg // ps + 2 <= 4096, (Hkv, ps, max_len, S)
