"""FP8 (e4m3, block-quantised) Q and K for the forward.

1. attn_quantize_fp8 matches the oracle's block quantisation bit for bit
   (codes and scales): every step is IEEE-defined, including the tie rule
   of e4m3 rounding (blocks of exact midpoints between codes).  The rotated
   quantiser matches the oracle's exact (float64) rotation up to the
   rounding of a float32 evaluation of it, within the bound the oracle
   derives (tests/parity.check_rotated_codes).
2. attn_fwd_fp8 matches the oracle run on the dequantised Q and K within the
   bf16 tolerance of attn_fwd: the kernel's arithmetic on the codes is exact
   up to that.  attn_quantize_fp8_v (one block per head, transposed) is bit
   exact as in 1, and attn_fwd_fp8_pv (e4m3 P and V) matches the oracle on
   the dequantised Q, K and V within the bound that follows from rounding
   256 P to e4m3 (parity.check_fp8_pv).
3. Against the exact attention of the unquantised inputs, each row obeys the
   bound that follows from how far quantisation moves its scaled scores:
   with delta_i = max_j |S'_ij - S_ij| (from the oracle),
   |dLSE_i| <= delta_i + 1e-3 and
   |dO_i| <= (exp(2 delta_i) - 1) * max_j |v_j - O_i| + 2e-2
   (softmax weights change by at most exp(2 delta) - 1 in L1, and a change of
   weights that sums to zero moves O by at most that times max |v_j - c|)."""
import math

import numpy as np
import pytest
import torch

from exact_attention_62_gb300.inputs import make_qkv
from parity import check_fp8_pv, check_rotated_codes, compare

pytestmark = pytest.mark.gpu
DEV = "cuda"


# d = 64 and 128 take the single-pass kernel, other even d the two-pass one
@pytest.mark.parametrize("B,N,H,d,seed", [(2, 300, 3, 128, 1), (1, 1000, 2, 64, 2), (1, 128, 1, 128, 3),
                                         (1, 200, 2, 96, 4)])
def test_quantisation_is_bit_exact(attn, oracle_mod, B, N, H, d, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((B, N, H, d), generator=g) * 3).to(torch.bfloat16)
    x[0, :, 0, 5] *= 40                       # outlier column
    if N > 128:
        x[-1, 128:256, -1] = 0                # an all-zero block
    codes, scales = attn.attn_quantize_fp8(x.to(DEV))
    torch.cuda.synchronize()
    rc, rs = oracle_mod.quantize_fp8_blocks(x.float())
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), rs)


@pytest.mark.parametrize("d", [64, 128, 96])
def test_quantisation_ties_round_to_even(attn, oracle_mod, d):
    """A block with maximum 448 (scale 1) holding exact midpoints between
    e4m3 codes, and a block whose maximum times float32(448 / amax) rounds
    above 448: the kernel's codes equal the oracle's, whose tie rule is
    pinned by hand-derived codes in the oracle tests."""
    mids = [448.0, 1.0625, 1.1875, -1.0625, 17.0, 19.0, 432.0, -432.0, 2.0 ** -10, 3 * 2.0 ** -10,
            1.0703125, 2.0 ** -10 * (1 + 2.0 ** -7), 0.1875, -0.3125, 3.25, 208.0]
    x = torch.zeros((1, 256, 2, d), dtype=torch.float32)
    x[0, :len(mids), 0, : d // 2] = torch.tensor(mids)[:, None]
    x[0, :len(mids), 1, ::3] = -torch.tensor(mids)[:, None]
    x[0, 128 + 7, 0, 3] = 1.359375                    # amax * fl(448 / amax) = 448.00003
    x[0, 128 + 9, 0, 1] = -0.6796875
    x = x.to(torch.bfloat16)
    assert torch.equal(x.float()[0, :len(mids), 0, 0], torch.tensor(mids))  # exact in bf16
    codes, scales = attn.attn_quantize_fp8(x.to(DEV))
    torch.cuda.synchronize()
    rc, rs = oracle_mod.quantize_fp8_blocks(x.float())
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert int(codes[0, 128 + 7, 0, 3]) == 0x7E


CASES = [
    # B, Hq, Hkv, Nq, Nk, causal, q_scale
    (1, 2, 2, 300, 300, True, 1.0),
    (2, 4, 1, 520, 520, False, 1.0),
    (1, 2, 2, 1000, 300, True, 1.0),      # causal rows with no allowed key
    (1, 2, 2, 700, 700, True, 8.0),       # near one-hot rows
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,causal,qs", CASES)
def test_fp8_forward(attn, oracle_mod, B, Hq, Hkv, Nq, Nk, causal, qs):
    d = 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nk, d, 12, q_scale=qs)
    q8, qsc = attn.attn_quantize_fp8(q.to(DEV))
    k8, ksc = attn.attn_quantize_fp8(k.to(DEV))
    o, lse = attn.attn_fwd_fp8(q8, k8, v.to(DEV), qsc, ksc, causal, scale)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    qd = oracle_mod.dequantize_fp8_blocks(q8.cpu().numpy(), qsc.cpu().numpy())
    kd = oracle_mod.dequantize_fp8_blocks(k8.cpu().numpy(), ksc.cpu().numpy())
    # (2) the kernel's arithmetic on the quantised inputs
    ro, rl = oracle_mod.attn_fwd(qd.astype(np.float32), kd.astype(np.float32), v, causal, scale)
    compare(o, lse, ro, rl, torch.bfloat16, "fp8 vs dequantised oracle")
    # (3) the quantisation error against the exact inputs, row by row
    eo, el = oracle_mod.attn_fwd(q, k, v, causal, scale)
    delta = oracle_mod.score_perturbation(qd, kd, q.double().numpy(), k.double().numpy(), causal, scale)
    og = o.float().cpu().numpy().astype(np.float64)
    lg = lse.cpu().numpy().astype(np.float64)
    vv = v.double().numpy()
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            for i in range(Nq):
                last = Nk - 1 if not causal else min(Nk - 1, i + (Nk - Nq))
                if last < 0:
                    assert np.all(og[b, i, h] == 0.0) and lg[b, h, i] == -np.inf
                    continue
                dl = delta[b, h, i]
                assert abs(lg[b, h, i] - el[b, h, i]) <= dl + 1e-3, (b, h, i)
                spread = np.abs(vv[b, :last + 1, h // G, :] - eo[b, i, h][None, :]).max()
                bound = math.expm1(2 * dl) * spread + 2e-2
                assert np.abs(og[b, i, h] - eo[b, i, h]).max() <= bound, (b, h, i)


@pytest.mark.parametrize("B,Hq,Hkv,N", [(4, 16, 16, 4096), (1, 32, 8, 16384)],
                         ids=["training_prefill", "long_sequence"])
def test_fp8_forward_full_size_sampled(attn, oracle_mod, B, Hq, Hkv, N):
    """The FP8 workloads at full size (B=4, Hq=Hkv=16, N=4096 and B=1,
    Hq=32, Hkv=8, N=16384; d=128, causal), on sampled rows against the
    oracle run on the dequantised Q and K (bar 2 above)."""
    from exact_attention_62_gb300.inputs import sample_rows
    H, d = Hq, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_qkv(B, Hq, Hkv, N, N, d, 14)
    q8, qsc = attn.attn_quantize_fp8(q.to(DEV))
    k8, ksc = attn.attn_quantize_fp8(k.to(DEV))
    o, lse = attn.attn_fwd_fp8(q8, k8, v.to(DEV), qsc, ksc, True, scale)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    qd = oracle_mod.dequantize_fp8_blocks(q8.cpu().numpy(), qsc.cpu().numpy()).astype(np.float32)
    kd = oracle_mod.dequantize_fp8_blocks(k8.cpu().numpy(), ksc.cpu().numpy()).astype(np.float32)
    rows = sample_rows(B, H, N, 256, 15)
    rows += [(0, 0, 127), (B - 1, H // 2, 128), (B - 1, H - 1, N - 1), (0, 3, 0)]
    ro, rl = oracle_mod.attn_rows(qd, kd, v, True, scale, rows)
    o_sel = torch.stack([o[b, i, h] for b, h, i in rows])
    l_sel = torch.stack([lse[b, h, i] for b, h, i in rows])
    compare(o_sel, l_sel, ro, rl, torch.bfloat16, "fp8 full size vs dequantised oracle")


def _signs(d, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randint(0, 2, (d,), generator=g) * 2 - 1).to(torch.float32)


# incoherent processing: Hadamard rotation with random signs before quantising
@pytest.mark.parametrize("B,N,H,d,seed", [(2, 300, 3, 128, 21), (1, 1000, 2, 64, 22), (1, 128, 1, 128, 23)])
def test_rotated_quantisation_matches_the_exact_rotation(attn, oracle_mod, B, N, H, d, seed):
    """The kernel rotates in float32 (butterflies), the oracle exactly in
    float64; codes and scales agree up to the derived float32 rounding bound:
    every differing code is one step off, at a rounding boundary."""
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((B, N, H, d), generator=g) * 3).to(torch.bfloat16)
    x[0, :, 0, 5] *= 40                       # outlier column
    if N > 128:
        x[-1, 128:256, -1] = 0                # an all-zero block
    s = _signs(d, seed)
    codes, scales = attn.attn_quantize_fp8_rotated(x.to(DEV), s.to(DEV))
    torch.cuda.synchronize()
    check_rotated_codes(codes.cpu().numpy(), scales.cpu().numpy(), x.float().numpy(), s.numpy(),
                        oracle_mod)


@pytest.mark.parametrize("outlier", [1.0, 20.0])
def test_fp8_forward_rotated(attn, oracle_mod, outlier):
    """attn_fwd_fp8 on rotated Q and K (the same signs): (2) equals the
    oracle on the dequantised rotated inputs within the bf16 tolerance (their
    dot products are the scores); (3) obeys the per-row bound against the
    exact attention; and with outlier features the rotation lowers the error
    against the exact attention compared with plain block quantisation."""
    B, Hq, Hkv, N, d = 1, 4, 2, 640, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_qkv(B, Hq, Hkv, N, N, d, 24)
    if outlier != 1.0:
        q[..., 17] = (q[..., 17].float() * outlier).to(torch.bfloat16)
        k[..., 17] = (k[..., 17].float() * outlier).to(torch.bfloat16)
    s = _signs(d, 25).to(DEV)
    q8, qsc = attn.attn_quantize_fp8_rotated(q.to(DEV), s)
    k8, ksc = attn.attn_quantize_fp8_rotated(k.to(DEV), s)
    o, lse = attn.attn_fwd_fp8(q8, k8, v.to(DEV), qsc, ksc, True, scale)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    qd = oracle_mod.dequantize_fp8_blocks(q8.cpu().numpy(), qsc.cpu().numpy())
    kd = oracle_mod.dequantize_fp8_blocks(k8.cpu().numpy(), ksc.cpu().numpy())
    ro, rl = oracle_mod.attn_fwd(qd.astype(np.float32), kd.astype(np.float32), v, True, scale)
    compare(o, lse, ro, rl, torch.bfloat16, "rotated fp8 vs dequantised rotated oracle")
    eo, el = oracle_mod.attn_fwd(q, k, v, True, scale)
    delta = oracle_mod.score_perturbation(qd, kd, q.double().numpy(), k.double().numpy(), True, scale)
    og = o.float().cpu().numpy().astype(np.float64)
    lg = lse.cpu().numpy().astype(np.float64)
    vv = v.double().numpy()
    G = Hq // Hkv
    for h in range(Hq):
        for i in range(N):
            dl = delta[0, h, i]
            assert abs(lg[0, h, i] - el[0, h, i]) <= dl + 1e-3, (h, i)
            spread = np.abs(vv[0, :i + 1, h // G, :] - eo[0, i, h][None, :]).max()
            assert np.abs(og[0, i, h] - eo[0, i, h]).max() <= math.expm1(2 * dl) * spread + 2e-2, (h, i)
    if outlier != 1.0:
        p8, psc = attn.attn_quantize_fp8(q.to(DEV))
        pk8, pksc = attn.attn_quantize_fp8(k.to(DEV))
        po, plse = attn.attn_fwd_fp8(p8, pk8, v.to(DEV), psc, pksc, True, scale)
        torch.cuda.synchronize()
        err_rot = np.abs(lg - el).mean()
        err_plain = np.abs(plse.cpu().numpy().astype(np.float64) - el).mean()
        assert err_rot < err_plain, (err_rot, err_plain)


# ---------------------------------------------------------------- e4m3 V and P V
def _v_codes_bnhd(vt8, N):
    """attn_quantize_fp8_v's transposed codes [B, H, d, ld] back to [B, N, H, d]."""
    return vt8[..., :N].permute(0, 3, 1, 2).contiguous()


@pytest.mark.parametrize("B,N,H,d,seed", [(2, 300, 3, 128, 31), (1, 1000, 2, 64, 32), (1, 128, 1, 128, 33),
                                         (3, 17, 2, 128, 34), (1, 4100, 1, 64, 35)])
def test_v_quantisation_is_bit_exact(attn, oracle_mod, B, N, H, d, seed):
    """attn_quantize_fp8_v is the block quantisation with one block per
    (batch, head), the whole sequence (the oracle's quantize_fp8_blocks with
    block = N), written transposed; the padding keys up to a multiple of 16
    hold code 0 and an all-zero head gets scale 1."""
    g = torch.Generator().manual_seed(seed)
    v = (torch.randn((B, N, H, d), generator=g) * 2).to(torch.bfloat16)
    v[0, :, 0, 3] *= 40                        # outlier column
    if B > 1:
        v[1, :, -1] = 0                        # an all-zero head
    vt8, vsc = attn.attn_quantize_fp8_v(v.to(DEV))
    torch.cuda.synchronize()
    ld = (N + 15) // 16 * 16
    assert tuple(vt8.shape) == (B, H, d, ld) and tuple(vsc.shape) == (B, H)
    rc, rs = oracle_mod.quantize_fp8_blocks(v.float(), block=N)
    assert np.array_equal(_v_codes_bnhd(vt8, N).cpu().numpy(), rc)
    assert np.array_equal(vsc.cpu().numpy(), rs[:, :, 0])
    assert torch.all(vt8[..., N:] == 0)
    if B > 1:
        assert vsc[1, -1].item() == 1.0 and torch.all(vt8[1, -1] == 0)


def fp8_pv_reference(oracle_mod, q8, qsc, k8, ksc, vt8, vsc, Nk, causal, scale, Hq, Hkv):
    """The oracle on the dequantised Q, K and V of an attn_fwd_fp8_pv call,
    with the terms of its error bound: (o, lse, sum_j w_ij |v_jc| from the
    oracle on |V|, sum_j |v_jc| over the KV head's keys, as [B, 1, Hq, d])."""
    qd = oracle_mod.dequantize_fp8_blocks(q8.cpu().numpy(), qsc.cpu().numpy()).astype(np.float32)
    kd = oracle_mod.dequantize_fp8_blocks(k8.cpu().numpy(), ksc.cpu().numpy()).astype(np.float32)
    vd = oracle_mod.dequantize_fp8_blocks(_v_codes_bnhd(vt8, Nk).cpu().numpy(),
                                          vsc.cpu().numpy()[:, :, None], block=Nk).astype(np.float32)
    ro, rl = oracle_mod.attn_fwd(qd, kd, vd, causal, scale)
    rabs, _ = oracle_mod.attn_fwd(qd, kd, np.abs(vd), causal, scale)
    vsum = np.abs(vd.astype(np.float64)).sum(axis=1)                        # [B, Hkv, d]
    vabs_sum = np.repeat(vsum, Hq // Hkv, axis=1)[:, None, :, :]           # [B, 1, Hq, d]
    return ro, rl, rabs, vabs_sum, vd


PV_CASES = [
    # B, Hq, Hkv, Nq, Nk, causal, q_scale
    (1, 2, 2, 300, 300, True, 1.0),
    (2, 4, 1, 520, 520, False, 1.0),
    (1, 2, 2, 1000, 300, True, 1.0),      # causal rows with no allowed key
    (1, 2, 2, 700, 700, True, 8.0),       # near one-hot rows
    (1, 8, 2, 257, 1000, False, 1.0),     # GQA, Nk not a multiple of 16
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,causal,qs", PV_CASES)
def test_fp8_pv_forward(attn, oracle_mod, B, Hq, Hkv, Nq, Nk, causal, qs):
    d = 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nk, d, 41, q_scale=qs)
    v[:, :, 0, 7] *= 20                    # an outlier feature in V
    q8, qsc = attn.attn_quantize_fp8(q.to(DEV))
    k8, ksc = attn.attn_quantize_fp8(k.to(DEV))
    vt8, vsc = attn.attn_quantize_fp8_v(v.to(DEV))
    o, lse = attn.attn_fwd_fp8_pv(q8, k8, vt8, qsc, ksc, vsc, causal, scale)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    ro, rl, rabs, vabs_sum, vd = fp8_pv_reference(oracle_mod, q8, qsc, k8, ksc, vt8, vsc, Nk, causal, scale,
                                                  Hq, Hkv)
    err = check_fp8_pv(o, lse, ro, rl, rabs, vabs_sum, "fp8 P V vs dequantised oracle")
    # and the rounding of P is visible: the result is not the bf16-P result
    ob, _ = attn.attn_fwd_fp8(q8, k8, torch.from_numpy(vd).to(torch.bfloat16).to(DEV), qsc, ksc, causal, scale)
    torch.cuda.synchronize()
    assert not torch.equal(ob, o) and err > 0


@pytest.mark.parametrize("B,Hq,Hkv,N", [(4, 16, 16, 4096), (1, 32, 8, 16384)],
                         ids=["training_prefill", "long_sequence"])
def test_fp8_pv_forward_full_size_sampled(attn, oracle_mod, B, Hq, Hkv, N):
    """The e4m3 P V forward at the two full FP8 sizes (d = 128, causal), on
    sampled rows against the oracle run on the dequantised Q, K and V,
    within the P-rounding bound above."""
    from exact_attention_62_gb300.inputs import sample_rows
    d = 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_qkv(B, Hq, Hkv, N, N, d, 42)
    q8, qsc = attn.attn_quantize_fp8(q.to(DEV))
    k8, ksc = attn.attn_quantize_fp8(k.to(DEV))
    vt8, vsc = attn.attn_quantize_fp8_v(v.to(DEV))
    o, lse = attn.attn_fwd_fp8_pv(q8, k8, vt8, qsc, ksc, vsc, True, scale)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    qd = oracle_mod.dequantize_fp8_blocks(q8.cpu().numpy(), qsc.cpu().numpy()).astype(np.float32)
    kd = oracle_mod.dequantize_fp8_blocks(k8.cpu().numpy(), ksc.cpu().numpy()).astype(np.float32)
    vd = oracle_mod.dequantize_fp8_blocks(_v_codes_bnhd(vt8, N).cpu().numpy(),
                                          vsc.cpu().numpy()[:, :, None], block=N).astype(np.float32)
    rows = sample_rows(B, Hq, N, 192, 43)
    rows += [(0, 0, 127), (B - 1, Hq // 2, 128), (B - 1, Hq - 1, N - 1), (0, 3, 0)]
    ro, rl = oracle_mod.attn_rows(qd, kd, vd, True, scale, rows)
    rabs, _ = oracle_mod.attn_rows(qd, kd, np.abs(vd), True, scale, rows)
    G = Hq // Hkv
    vsum = np.abs(vd.astype(np.float64)).sum(axis=1)                        # [B, Hkv, d]
    vabs_sum = np.stack([vsum[b, h // G] for b, h, _ in rows])
    o_sel = torch.stack([o[b, i, h] for b, h, i in rows])
    l_sel = torch.stack([lse[b, h, i] for b, h, i in rows])
    check_fp8_pv(o_sel, l_sel, ro, rl, rabs, vabs_sum, "fp8 P V full size vs dequantised oracle")
