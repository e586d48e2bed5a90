"""Parity of attn_decode_splitkv and attn_merge_lse against the oracle."""
import math

import numpy as np
import pytest
import torch

from exact_attention_62_gb300.inputs import make_partials, make_qkv
from parity import compare, guarded, guards_intact, to_np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def decode_case(attn, oracle_mod, B, Hq, Hkv, Nk, d, splits, seed, check_parts=True):
    q, k, v = make_qkv(B, Hq, Hkv, 1, Nk, d, seed)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    S = splits if splits > 0 else attn.attn_decode_num_splits(B, Hq, Hkv, Nk, d)
    assert S >= 1
    wbytes = attn.attn_decode_workspace_bytes(B, Hq, Hkv, Nk, d, S)
    ws, wb, wg = guarded((max(wbytes, 16),), torch.uint8, DEV, fill=0x5A)
    o, ob, og = guarded((B, 1, Hq, d), torch.bfloat16, DEV)
    lse, lb, lg = guarded((B, Hq), torch.float32, DEV)
    attn.attn_decode_splitkv(qd, kd, vd, scale, S, workspace=ws if wbytes else None, o=o, lse=lse)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    assert guards_intact(ob, og) and guards_intact(lb, lg), "write outside O/LSE"
    assert guards_intact(wb, wg, fill=0x5A), "write outside the workspace"
    o_ref, lse_ref = oracle_mod.attn_fwd(q, k, v, False, scale)
    res = compare(o.view(B, Hq, d), lse, o_ref.reshape(B, Hq, d), lse_ref.reshape(B, Hq),
                  torch.bfloat16, "decode B%d Hq%d Hkv%d Nk%d d%d S%d" % (B, Hq, Hkv, Nk, d, S))
    if check_parts and S > 1:
        # the workspace holds the per-segment partials in the documented layout
        R = B * Hq
        o_bytes = S * R * d * 4
        lse_off = (o_bytes + 255) // 256 * 256
        flat = ws.view(-1)
        o_parts = flat[:o_bytes].view(torch.float32).view(S, R, d)
        lse_parts = flat[lse_off:lse_off + S * R * 4].view(torch.float32).view(S, R)
        op_ref, lp_ref = oracle_mod.decode_split(q, k, v, scale, S)
        # partial outputs are fp32 but built from bf16 P: same bound as O
        compare(o_parts, lse_parts, op_ref, lp_ref, torch.bfloat16, "decode partials")
    return res, S


def test_flash_decoding_long_context(attn, oracle_mod):
    """Nq=1, Hq=32, Hkv=8, d=128, Nk=65536, B=1, automatic segment count."""
    (_, _), S = decode_case(attn, oracle_mod, 1, 32, 8, 65536, 128, 0, seed=5)
    assert S > 1


def test_flash_decoding_batched(attn, oracle_mod):
    """Nq=1, Hq=32, Hkv=8, d=128, Nk=8192, B=16, automatic segment count."""
    decode_case(attn, oracle_mod, 16, 32, 8, 8192, 128, 0, seed=6)


@pytest.mark.parametrize("splits", [1, 7, 64, 1000])
def test_segment_counts_agree(attn, oracle_mod, splits):
    """Lecture 11 section 6.2: 1, 7, 64 and 1000 segments give the same result."""
    decode_case(attn, oracle_mod, 2, 8, 2, 5000, 128, splits, seed=7)


@pytest.mark.parametrize("B,Hq,Hkv,Nk,d,S", [
    (1, 8, 8, 1000, 64, 3),      # G = 1
    (2, 16, 8, 333, 128, 5),     # G = 2
    (1, 16, 2, 4097, 128, 9),    # G = 8
    (1, 32, 2, 2000, 64, 4),     # G = 16: two CTAs per KV head
    (1, 12, 4, 700, 128, 2),     # G = 3
    (3, 4, 1, 1, 128, 1),        # a single key
    (1, 4, 2, 65, 64, 65),       # one key per segment
    (1, 4, 2, 10, 64, 6),        # a trailing empty segment
])
def test_decode_shapes(attn, oracle_mod, B, Hq, Hkv, Nk, d, S):
    decode_case(attn, oracle_mod, B, Hq, Hkv, Nk, d, S, seed=Nk + S)


def test_decode_outlier(attn, oracle_mod):
    q, k, v = make_qkv(2, 8, 2, 1, 3000, 128, seed=8, q_scale=8.0)
    o, lse = attn.attn_decode_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), 1 / math.sqrt(128), 6)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle_mod.attn_fwd(q, k, v, False, 1 / math.sqrt(128))
    compare(o.view(2, 8, 128), lse, o_ref.reshape(2, 8, 128), l_ref.reshape(2, 8), torch.bfloat16)


def test_decode_empty_cache(attn):
    q = torch.randn(2, 1, 4, 128, device=DEV).to(torch.bfloat16)
    k = torch.empty(2, 0, 2, 128, device=DEV, dtype=torch.bfloat16)
    o, lse = attn.attn_decode_splitkv(q, k, k.clone(), 0.1, 0)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(lse == float("-inf"))


@pytest.mark.parametrize("P,rows,d,out", [(1, 5, 64, torch.float32), (12, 300, 128, torch.float32),
                                          (7, 1000, 128, torch.bfloat16), (40, 33, 4, torch.float32),
                                          (3, 17, 512, torch.bfloat16),
                                          # more parts than one staged chunk of weights
                                          (2500, 3, 128, torch.float32), (1025, 4, 64, torch.bfloat16),
                                          # 4-column groups that do not divide the thread count
                                          (9, 6, 12, torch.float32), (33, 5, 20, torch.bfloat16),
                                          # the one-pass merge with 19 segments per thread, up to its
                                          # limit (152 parts at d = 128, 304 at d = 64), and one past it
                                          (33, 40, 128, torch.bfloat16), (128, 7, 128, torch.float32),
                                          (200, 9, 64, torch.float32), (129, 3, 128, torch.bfloat16),
                                          (152, 5, 128, torch.bfloat16), (153, 5, 128, torch.float32),
                                          (304, 3, 64, torch.bfloat16), (305, 3, 64, torch.float32)])
def test_merge_lse(attn, oracle_mod, P, rows, d, out):
    """attn_merge_lse against the oracle's log-sum-exp merge, with some empty
    parts and some rows whose parts are all empty."""
    o_parts, lse_parts = make_partials(P, rows, d, seed=P * rows, empty_frac=0.3)
    lse_parts[:, :2] = float("-inf")
    o_parts[:, :2] = 0.0
    o, lse = attn.attn_merge_lse(o_parts.to(DEV), lse_parts.to(DEV), out_dtype=out)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle_mod.merge_lse(o_parts.double().numpy(), lse_parts.double().numpy())
    tol = 1e-5 if out == torch.float32 else 2e-2
    got = to_np64(o)
    assert np.abs(got - o_ref).max() <= tol * max(1.0, np.abs(o_ref).max())
    lg = to_np64(lse)
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    assert np.abs(lg[fin] - l_ref[fin]).max() <= 1e-5 * max(1.0, np.abs(l_ref[fin]).max())
    assert np.all(got[:2] == 0.0)
