"""Sizes whose element offsets pass 2^31: the forward with Q and O of more
than 2^31 elements, and flash-decoding over a cache of more than 2^31 K (and
V) elements.  The oracle checks sampled rows: for a row i of a causal forward
it gets that row's query and the keys the row may see (j <= i + Nk - Nq, the
bottom-right rule), run without a mask, which is the same attention."""
import math

import numpy as np
import pytest
import torch

from parity import compare

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _randn(shape, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=DEV, dtype=torch.float32).to(torch.bfloat16)


def _row_oracle(oracle_mod, q_row, k_head, v_head, scale):
    """q_row [d], k_head/v_head [n, d] (CPU bf16) -> oracle (o [d], lse)."""
    d = q_row.shape[-1]
    o, lse = oracle_mod.attn_fwd(q_row.reshape(1, 1, 1, d), k_head.reshape(1, -1, 1, d),
                                 v_head.reshape(1, -1, 1, d), False, scale)
    return o.reshape(d), float(np.asarray(lse).reshape(-1)[0])


def test_forward_offsets_past_2_31(attn, oracle_mod):
    """B=1, Hq=64, Hkv=8, N=263168, d=128, causal: Q and O hold 2.16e9
    elements, so rows near the end of the last heads sit past 2^31."""
    B, Hq, Hkv, N, d = 1, 64, 8, 262144 + 1024, 128
    assert B * N * Hq * d > 2 ** 31
    q = _randn((B, N, Hq, d), 101)
    k = _randn((B, N, Hkv, d), 102)
    v = _randn((B, N, Hkv, d), 103)
    scale = 1.0 / math.sqrt(d)
    o, lse = attn.attn_fwd(q, k, v, True, scale)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    G = Hq // Hkv
    rows = [(63, N - 1), (63, N - 129), (63, N - 128), (62, N - 1000), (0, N - 1), (31, 200000),
            (63, 0), (40, 127), (7, 140000)]
    kh = {}
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for hq, i in rows:
        g = hq // G
        if g not in kh:
            kh[g] = (k[0, :, g].contiguous().cpu(), v[0, :, g].contiguous().cpu())
        kk, vv = kh[g]
        ro, rl = _row_oracle(oracle_mod, q[0, i, hq].cpu(), kk[:i + 1], vv[:i + 1], scale)
        ref_o.append(ro)
        ref_l.append(rl)
        got_o.append(o[0, i, hq].float().cpu())
        got_l.append(lse[0, hq, i].float().cpu())
    compare(torch.stack(got_o), torch.stack(got_l), np.stack(ref_o), np.array(ref_l), torch.bfloat16,
            "forward past 2^31")
    assert torch.isfinite(lse).all()


def test_decode_cache_past_2_31(attn, oracle_mod):
    """B=1, Hq=Hkv=16, Nk=2^20+37, d=128: K and V hold 2.15e9 elements each;
    automatic segment count."""
    B, Hq, Hkv, Nk, d = 1, 16, 16, (1 << 20) + 37, 128
    assert B * Nk * Hkv * d > 2 ** 31
    q = _randn((B, 1, Hq, d), 111)
    k = _randn((B, Nk, Hkv, d), 112)
    v = _randn((B, Nk, Hkv, d), 113)
    scale = 1.0 / math.sqrt(d)
    o, lse = attn.attn_decode_splitkv(q, k, v, scale)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for hq in (0, 7, 15):
        ro, rl = _row_oracle(oracle_mod, q[0, 0, hq].cpu(), k[0, :, hq].contiguous().cpu(),
                             v[0, :, hq].contiguous().cpu(), scale)
        ref_o.append(ro)
        ref_l.append(rl)
        got_o.append(o[0, 0, hq].float().cpu())
        got_l.append(lse[0, hq].float().cpu())
    compare(torch.stack(got_o), torch.stack(got_l), np.stack(ref_o), np.array(ref_l), torch.bfloat16,
            "decode past 2^31")
