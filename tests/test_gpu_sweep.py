"""Seeded random shapes against the oracle: the forward (bf16 and fp32),
split-KV decode, paged decode, the backward and the two FP8 forwards on
combinations of batch,
GQA ratio, lengths (tile multiples or not, Nq != Nk), head dimension, mask
and segment count that the hand-picked cases do not spell out.  The shapes
are drawn once from a fixed seed, so every run checks the same list."""
import math
import random

import pytest
import torch

from exact_attention_62_gb300.inputs import make_paged, make_qkv
from parity import compare

pytestmark = pytest.mark.gpu
DEV = "cuda"

_R = random.Random(20261203)


def _fwd_shapes(n):
    out = []
    for i in range(n):
        Hkv = _R.choice([1, 2, 3])
        G = _R.choice([1, 2, 3, 4, 8])
        Nq = _R.randint(1, 640)
        Nk = Nq if _R.random() < 0.5 else _R.randint(1, 640)
        dtype = "f32" if i % 6 == 5 else "bf16"
        out.append((_R.randint(1, 3), Hkv * G, Hkv, Nq, Nk, _R.choice([64, 128]), _R.random() < 0.5, dtype))
    return out


def _decode_shapes(n):
    out = []
    for _ in range(n):
        Hkv = _R.choice([1, 2, 4])
        Nk = _R.randint(1, 6000)
        S = 0 if _R.random() < 0.4 else _R.randint(1, min(Nk, 48))
        out.append((_R.randint(1, 4), Hkv * _R.choice([1, 2, 3, 4, 8, 16]), Hkv, Nk, _R.choice([64, 128]), S))
    return out


def _paged_shapes(n):
    out = []
    for _ in range(n):
        B = _R.randint(1, 4)
        lens = [_R.randint(0, 3000) for _ in range(B)]
        lens[_R.randrange(B)] = max(1, lens[0])
        Hkv = _R.choice([1, 2, 4])
        out.append((B, Hkv * _R.choice([1, 2, 4, 8]), Hkv, _R.choice([64, 128]), _R.choice([16, 32, 64, 128]),
                    lens, 0 if _R.random() < 0.5 else _R.randint(1, 12)))
    return out


def _bwd_shapes(n):
    out = []
    for _ in range(n):
        Hkv = _R.choice([1, 2])
        Nq = _R.randint(40, 600)
        Nk = Nq if _R.random() < 0.5 else _R.randint(40, 600)
        out.append((_R.randint(1, 2), Hkv * _R.choice([1, 2, 4]), Hkv, Nq, Nk, _R.choice([64, 128]),
                    _R.random() < 0.5))
    return out


def _fp8_shapes(n):
    out = []
    for _ in range(n):
        Hkv = _R.choice([1, 2, 4])
        Nq = _R.randint(1, 700)
        Nk = Nq if _R.random() < 0.5 else _R.randint(1, 700)
        out.append((_R.randint(1, 2), Hkv * _R.choice([1, 2, 4, 8]), Hkv, Nq, Nk, _R.random() < 0.5))
    return out


FWD = _fwd_shapes(40)
DEC = _decode_shapes(20)
PAGED = _paged_shapes(16)
BWD = _bwd_shapes(16)
FP8 = _fp8_shapes(12)  # drawn last, so the lists above stay as they were


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal,dt", FWD)
def test_forward_random_shapes(attn, oracle_mod, B, Hq, Hkv, Nq, Nk, d, causal, dt):
    dtype = torch.float32 if dt == "f32" else torch.bfloat16
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nk, d, Nq * 7 + Nk, dtype=dtype)
    scale = 1.0 / math.sqrt(d)
    o, lse = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal, scale)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    ro, rl = oracle_mod.attn_fwd(q, k, v, causal, scale)
    compare(o, lse, ro, rl, dtype, "fwd B%d Hq%d Hkv%d Nq%d Nk%d d%d c%d" % (B, Hq, Hkv, Nq, Nk, d, causal))


@pytest.mark.parametrize("B,Hq,Hkv,Nk,d,S", DEC)
def test_decode_random_shapes(attn, oracle_mod, B, Hq, Hkv, Nk, d, S):
    q, k, v = make_qkv(B, Hq, Hkv, 1, Nk, d, Nk + S)
    scale = 1.0 / math.sqrt(d)
    o, lse = attn.attn_decode_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), scale, S)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    ro, rl = oracle_mod.attn_fwd(q, k, v, False, scale)
    compare(o.view(B, Hq, d), lse, ro.reshape(B, Hq, d), rl.reshape(B, Hq), torch.bfloat16,
            "decode B%d Hq%d Hkv%d Nk%d d%d S%d" % (B, Hq, Hkv, Nk, d, S))


@pytest.mark.parametrize("B,Hq,Hkv,d,ps,lens,S", PAGED)
def test_paged_random_shapes(attn, oracle_mod, B, Hq, Hkv, d, ps, lens, S):
    q, kp, vp, table, sl = make_paged(B, Hq, Hkv, d, ps, lens, seed=sum(lens) + ps + S)
    scale = 1.0 / math.sqrt(d)
    o, lse = attn.attn_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV),
                                    max(lens), scale, num_splits=S)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    ro, rl = oracle_mod.decode_paged(q, kp.float(), vp.float(), table.numpy(), sl.numpy(), scale)
    compare(o, lse, ro, rl, torch.bfloat16, "paged %s ps%d S%d" % (lens, ps, S))


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", BWD)
def test_backward_random_shapes(attn, oracle_mod, B, Hq, Hkv, Nq, Nk, d, causal):
    from test_gpu_bwd import check
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nk, d, Nq + 3 * Nk)
    dout = torch.randn((B, Nq, Hq, d), generator=torch.Generator().manual_seed(Nq)).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    qg, kg, vg, dog = q.to(DEV), k.to(DEV), v.to(DEV), dout.to(DEV)
    o, lse = attn.attn_fwd(qg, kg, vg, causal, scale)
    dq, dk, dv = attn.attn_bwd(qg, kg, vg, o, lse, dog, causal, scale)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    rq, rk, rv = oracle_mod.attn_bwd(q, k, v, dout, causal, scale)
    check("dq", dq, rq)
    check("dk", dk, rk)
    check("dv", dv, rv)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,causal", FP8)
def test_fp8_random_shapes(attn, oracle_mod, B, Hq, Hkv, Nq, Nk, causal):
    """attn_fwd_fp8 within the bf16 bar of the oracle on the dequantised Q,
    K, and attn_fwd_fp8_pv within the e4m3 P-rounding bound of the oracle on
    the dequantised Q, K, V (d = 128)."""
    import numpy as np
    from parity import check_fp8_pv
    from test_gpu_fp8 import fp8_pv_reference
    d = 128
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nk, d, 5 * Nq + Nk)
    scale = 1.0 / math.sqrt(d)
    q8, qsc = attn.attn_quantize_fp8(q.to(DEV))
    k8, ksc = attn.attn_quantize_fp8(k.to(DEV))
    vt8, vsc = attn.attn_quantize_fp8_v(v.to(DEV))
    o8, l8 = attn.attn_fwd_fp8(q8, k8, v.to(DEV), qsc, ksc, causal, scale)
    opv, lpv = attn.attn_fwd_fp8_pv(q8, k8, vt8, qsc, ksc, vsc, causal, scale)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    what = "B%d Hq%d Hkv%d Nq%d Nk%d c%d" % (B, Hq, Hkv, Nq, Nk, causal)
    ro, rl, rabs, vabs_sum, _ = fp8_pv_reference(oracle_mod, q8, qsc, k8, ksc, vt8, vsc, Nk, causal, scale,
                                                 Hq, Hkv)
    check_fp8_pv(opv, lpv, ro, rl, rabs, vabs_sum, "fp8 P V " + what)
    qd = oracle_mod.dequantize_fp8_blocks(q8.cpu().numpy(), qsc.cpu().numpy()).astype(np.float32)
    kd = oracle_mod.dequantize_fp8_blocks(k8.cpu().numpy(), ksc.cpu().numpy()).astype(np.float32)
    r8o, r8l = oracle_mod.attn_fwd(qd, kd, v, causal, scale)
    compare(o8, l8, r8o, r8l, torch.bfloat16, "fp8 " + what)
