"""Bounded device waits: a lost signal ends in a status code, not a hung GPU.

Every mbarrier wait in the kernels gives up after a bound, sets the block's
abort flag (so every role of the block drains to its teardown and frees its
tensor memory) and records ATTN_ERR_TIMEOUT in a status word that
attn_check_device_status() reads and clears.  These tests make one wait run
out on purpose through the test-only entry points of include/attn_test.h: the
TMA producer of block 0 skips one load (no byte count posted, no copy
issued), so nothing in flight is lost and the consumer's wait can only end
by its bound, here about a millisecond.  Each test then checks that the call
returned, that the status reports the timeout once, and that the next normal
call on the same context matches the oracle.
"""
import math

import pytest
import torch

from exact_attention_62_gb300.inputs import make_qkv
from parity import compare

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUT = 4
SHORT_WAIT = 2_000_000  # SM cycles, about 1 ms


@pytest.mark.parametrize("d,N,skip", [(128, 256, 0), (64, 256, 1), (128, 700, 3), (64, 700, 2)])
def test_forward_lost_load_times_out_and_context_survives(attn, oracle_mod, d, N, skip):
    """One work unit per block (B = H = 1 and N <= 256; three blocks at
    N = 700, the injected one working on the longest unit): block 0 never
    receives the K/V tiles at ring position `skip`; its MMA warp's wait runs
    out."""
    q, k, v = make_qkv(1, 1, 1, N, N, d, seed=40 + d)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    scale = 1.0 / math.sqrt(d)
    assert attn.attn_check_device_status() == 0
    opt = attn.AttnTestOptions(wait_limit_cycles=SHORT_WAIT, skip_load=skip)
    attn.attn_fwd_test(qd, kd, vd, True, scale, opt)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == TIMEOUT
    assert attn.attn_check_device_status() == 0  # read and cleared
    o, lse = attn.attn_fwd(qd, kd, vd, True, scale)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    o_ref, l_ref = oracle_mod.attn_fwd(q, k, v, True, scale)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, "forward after a timed-out call")


def test_forward_short_bound_without_injection_is_correct(attn, oracle_mod):
    """The same short bound with nothing skipped: no wait runs out on a
    multi-block grid, and the result matches the oracle."""
    B, H, N, d = 4, 8, 1000, 64
    q, k, v = make_qkv(B, H, H, N, N, d, seed=44)
    scale = 1.0 / math.sqrt(d)
    opt = attn.AttnTestOptions(wait_limit_cycles=SHORT_WAIT)
    o, lse = attn.attn_fwd_test(q.to(DEV), k.to(DEV), v.to(DEV), True, scale, opt)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    o_ref, l_ref = oracle_mod.attn_fwd(q, k, v, True, scale)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, "forward with a short wait bound")


@pytest.mark.parametrize("S,skip", [(3, 0), (1, 5), (4, 2)])
def test_decode_lost_load_times_out_and_context_survives(attn, oracle_mod, S, skip):
    """Block (0, 0, 0) of the split kernel never receives its tile `skip`;
    the consumer group that owns it times out, the other group and the
    producer see the abort flag, and the merge still runs."""
    B, Hq, Hkv, Nk, d = 2, 8, 2, 3000, 128
    q, k, v = make_qkv(B, Hq, Hkv, 1, Nk, d, seed=45 + S)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    scale = 1.0 / math.sqrt(d)
    assert attn.attn_check_device_status() == 0
    opt = attn.AttnTestOptions(wait_limit_cycles=SHORT_WAIT, skip_load=skip)
    attn.attn_decode_test(qd, kd, vd, scale, S, opt)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == TIMEOUT
    assert attn.attn_check_device_status() == 0
    o, lse = attn.attn_decode_splitkv(qd, kd, vd, scale, S)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    o_ref, l_ref = oracle_mod.attn_fwd(q, k, v, False, scale)
    compare(o, lse.reshape(B, Hq, 1), o_ref, l_ref, torch.bfloat16, "decode after a timed-out call")


def test_decode_short_bound_without_injection_is_correct(attn, oracle_mod):
    B, Hq, Hkv, Nk, d = 3, 32, 8, 20000, 128
    q, k, v = make_qkv(B, Hq, Hkv, 1, Nk, d, seed=49)
    scale = 1.0 / math.sqrt(d)
    opt = attn.AttnTestOptions(wait_limit_cycles=SHORT_WAIT)
    o, lse = attn.attn_decode_test(q.to(DEV), k.to(DEV), v.to(DEV), scale, 0, opt)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    o_ref, l_ref = oracle_mod.attn_fwd(q, k, v, False, scale)
    compare(o, lse.reshape(B, Hq, 1), o_ref, l_ref, torch.bfloat16, "decode with a short wait bound")
