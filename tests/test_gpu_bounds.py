"""The bounds-checked debug build, libattn_bounds.so (compiled with
ATTN_BOUNDS_CHECK).  In it, every global load and store that is not a TMA
copy (forward, decode, merge, backward and FP8 kernels) is checked against
its buffer's extent.  A refused access is skipped and reported by
attn_check_device_status as ATTN_ERR_BOUNDS; nothing traps.

1. On correct calls the checks never fire and change nothing: every result
   equals the production library's bit for bit, and the status stays OK.
2. The check itself works: with the test option o_extent_slack the kernels
   take O to end `slack` elements early.  They refuse exactly the stores past
   that point, leave those elements as they were, write everything else as
   the production library does, and report ATTN_ERR_BOUNDS.  The buffers are
   whole, so no access ever leaves them."""
import math

import pytest
import torch

from exact_attention_62_gb300.inputs import make_paged, make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def bounds_lib(attn):
    from exact_attention_62_gb300 import build
    return attn.load_library(build.build(bounds_check=True))


def _with(attn, L, fn):
    """fn() with every entry point calling the library L."""
    old = attn.use_library(L)
    try:
        out = fn()
        torch.cuda.synchronize()
        return out, attn.attn_check_device_status()
    finally:
        attn.use_library(old)


def _both(attn, bounds_lib, fn):
    ref, st_ref = _with(attn, None, fn)
    got, st = _with(attn, bounds_lib, fn)
    assert st_ref == attn.ATTN_OK and st == attn.ATTN_OK, (st_ref, st)
    for a, b in zip(ref, got):
        assert torch.equal(a, b)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal,dt", [
    (2, 4, 2, 300, 300, 64, True, "bf16"),
    (1, 2, 2, 1000, 300, 128, True, "bf16"),   # rows with no key
    (2, 8, 2, 257, 700, 128, False, "bf16"),
    (1, 2, 1, 200, 333, 64, True, "f32"),
    (2, 3, 3, 97, 97, 128, False, "f32"),
])
def test_forward_unchanged(attn, bounds_lib, B, Hq, Hkv, Nq, Nk, d, causal, dt):
    dtype = torch.float32 if dt == "f32" else torch.bfloat16
    q, k, v = (x.to(DEV) for x in make_qkv(B, Hq, Hkv, Nq, Nk, d, Nq + Nk, dtype=dtype))
    _both(attn, bounds_lib, lambda: attn.attn_fwd(q, k, v, causal, 1.0 / math.sqrt(d)))


@pytest.mark.parametrize("B,Hq,Hkv,Nk,d,S", [
    (2, 8, 2, 5000, 128, 1), (2, 8, 2, 5000, 128, 7), (1, 32, 8, 9000, 128, 64),
    (3, 4, 1, 1000, 128, 40), (1, 4, 2, 10, 64, 6),     # 40 at d = 128: the two-pass merge; 6: empty segments
])
def test_decode_unchanged(attn, bounds_lib, B, Hq, Hkv, Nk, d, S):
    q, k, v = (x.to(DEV) for x in make_qkv(B, Hq, Hkv, 1, Nk, d, Nk + S))
    _both(attn, bounds_lib, lambda: attn.attn_decode_splitkv(q, k, v, 1.0 / math.sqrt(d), S))


@pytest.mark.parametrize("ps,S,Hq,Hkv", [(16, 0, 8, 2), (64, 3, 8, 2), (16, 5, 32, 8)])
def test_paged_decode_unchanged(attn, bounds_lib, ps, S, Hq, Hkv):
    lens = [700, 1, 2049]
    q, kp, vp, table, sl = (x.to(DEV) for x in make_paged(3, Hq, Hkv, 128, ps, lens, seed=ps + S))
    _both(attn, bounds_lib, lambda: attn.attn_decode_paged(q, kp, vp, table, sl, max(lens), 0.088,
                                                           num_splits=S))


def test_merge_unchanged(attn, bounds_lib):
    g = torch.Generator().manual_seed(3)
    o_parts = torch.randn((40, 33, 128), generator=g).to(DEV)
    lse_parts = torch.randn((40, 33), generator=g).to(DEV)
    lse_parts[:, 0] = float("-inf")
    _both(attn, bounds_lib, lambda: attn.attn_merge_lse(o_parts, lse_parts))


def _refused_rows(total_rows, d, slack):
    """Rows (of d elements) whose stores end past total_rows * d - slack."""
    return [r for r in range(total_rows) if (r + 1) * d > total_rows * d - slack]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,slack", [
    (2, 4, 2, 300, 128, 128),          # the last row of O
    (1, 8, 2, 257, 64, 8 * 64 + 5),    # a whole query position and part of the row before
])
def test_forward_check_refuses_past_the_extent(attn, bounds_lib, B, Hq, Hkv, N, d, slack):
    q, k, v = (x.to(DEV) for x in make_qkv(B, Hq, Hkv, N, N, d, 77))
    scale = 1.0 / math.sqrt(d)
    ref, _ = _with(attn, None, lambda: attn.attn_fwd(q, k, v, True, scale))
    o = torch.full((B, N, Hq, d), 7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, Hq, N), device=DEV)
    opt = attn.AttnTestOptions(o_extent_slack=slack)
    _, st = _with(attn, bounds_lib, lambda: attn.attn_fwd_test(q, k, v, True, scale, opt, o=o, lse=lse))
    assert st == attn.ATTN_ERR_BOUNDS
    rows = o.view(-1, d)
    refused = _refused_rows(rows.shape[0], d, slack)
    assert refused and torch.all(rows[refused] == 7.0)
    keep = torch.ones(rows.shape[0], dtype=torch.bool)
    keep[refused] = False
    assert torch.equal(rows[keep.to(DEV)], ref[0].view(-1, d)[keep.to(DEV)])
    assert torch.equal(lse, ref[1])                       # LSE's extent is whole
    _, st = _with(attn, bounds_lib, lambda: None)
    assert st == attn.ATTN_OK                             # the status was read and cleared


@pytest.mark.parametrize("S", [1, 7, 40])   # the split kernel's stores; the short merge; the two-pass merge
def test_decode_check_refuses_past_the_extent(attn, bounds_lib, S):
    B, Hq, Hkv, Nk, d = 2, 8, 2, 3000, 128
    q, k, v = (x.to(DEV) for x in make_qkv(B, Hq, Hkv, 1, Nk, d, 78 + S))
    scale = 1.0 / math.sqrt(d)
    ref, _ = _with(attn, None, lambda: attn.attn_decode_splitkv(q, k, v, scale, S))
    o = torch.full((B, 1, Hq, d), 7.0, dtype=torch.bfloat16, device=DEV)
    opt = attn.AttnTestOptions(o_extent_slack=d)
    (o_got, lse_got), st = _with(attn, bounds_lib,
                                 lambda: attn.attn_decode_test(q, k, v, scale, S, opt, o=o))
    assert st == attn.ATTN_ERR_BOUNDS
    rows, rrows = o_got.view(-1, d), ref[0].view(-1, d)
    assert torch.all(rows[-1] == 7.0)                     # the last row: refused
    assert torch.equal(rows[:-1], rrows[:-1])
    assert torch.equal(lse_got, ref[1])


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (2, 4, 2, 300, 300, 64, True),
    (1, 8, 2, 257, 400, 128, False),
])
def test_backward_unchanged(attn, bounds_lib, B, Hq, Hkv, Nq, Nk, d, causal):
    q, k, v = (x.to(DEV) for x in make_qkv(B, Hq, Hkv, Nq, Nk, d, Nq + 2 * Nk))
    dout = torch.randn((B, Nq, Hq, d), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).to(DEV)
    scale = 1.0 / math.sqrt(d)

    def run():
        o, lse = attn.attn_fwd(q, k, v, causal, scale)
        return (o, lse) + tuple(attn.attn_bwd(q, k, v, o, lse, dout, causal, scale))

    _both(attn, bounds_lib, run)


def test_fp8_unchanged(attn, bounds_lib):
    B, Hq, Hkv, N, d = 1, 4, 2, 300, 128
    q, k, v = (x.to(DEV) for x in make_qkv(B, Hq, Hkv, N, N, d, 9))
    signs = (torch.randint(0, 2, (d,), generator=torch.Generator().manual_seed(2)) * 2 - 1).float().to(DEV)

    def run():
        q8, qs = attn.attn_quantize_fp8(q)
        k8, ks = attn.attn_quantize_fp8(k)
        r8, rs = attn.attn_quantize_fp8_rotated(q, signs)
        vt8, vs = attn.attn_quantize_fp8_v(v)
        o8, l8 = attn.attn_fwd_fp8(q8, k8, v, qs, ks, True)
        opv, lpv = attn.attn_fwd_fp8_pv(q8, k8, vt8, qs, ks, vs, True)
        return q8, qs, r8, rs, vt8, vs, o8, l8, opv, lpv

    _both(attn, bounds_lib, run)
