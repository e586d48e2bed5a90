"""attn_decode_splitkv_static: flash-decoding for callers that cannot allocate.

Callers that may not call cudaMalloc (device memory owned by a host
framework's allocator, a pre-planned memory budget, or a latency-critical path
where an allocation could block or synchronise) use this entry point instead
of attn_decode_splitkv: it keeps the per-segment partials in a scratch area
built into the library.  These tests call it through the C ABI and check that
it returns what the workspace-taking entry point returns, bit for bit (the
same kernels with the same segment count; a read of stale partials would
show), on two calls in a row with different inputs (the shared scratch area
is reused), and that sizes needing more scratch than the library holds are
refused before any launch, after the usual argument checks.

This file is collected last on purpose.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from exact_attention_62_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda"
OK, INVALID, UNSUPPORTED = 0, 1, 2
BF16 = 0


def _static_call(L, q, k, v, o, lse, S, scale):
    B, _, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    return L.attn_decode_splitkv_static(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), B, Hq, Hkv, Nk, d, scale, S, BF16,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("B,Hq,Hkv,Nk,d,S", [
    (1, 32, 8, 65536, 128, 0),   # long-context decode, automatic segment count
    (2, 8, 2, 5000, 128, 7),
    (3, 16, 4, 3000, 64, 5),
    (16, 32, 8, 8192, 128, 1),   # one segment: no scratch needed
])
def test_static_scratch_matches_workspace_entry_point(attn, B, Hq, Hkv, Nk, d, S):
    L = attn.lib()
    scale = 1.0 / math.sqrt(d)
    for call, seed in enumerate((101, 202)):  # two calls in a row, different inputs
        q, k, v = (x.to(DEV) for x in make_qkv(B, Hq, Hkv, 1, Nk, d, seed))
        o_ref, l_ref = attn.attn_decode_splitkv(q, k, v, scale, S)
        o = torch.full_like(q, 7.0)
        lse = torch.full((B, Hq), 7.0, dtype=torch.float32, device=DEV)
        assert _static_call(L, q, k, v, o, lse, S, scale) == OK
        torch.cuda.synchronize()
        assert attn.attn_check_device_status() == 0
        assert torch.equal(o, o_ref), (call, (o.float() - o_ref.float()).abs().max().item())
        assert torch.equal(lse, l_ref), (call, (lse - l_ref).abs().max().item())


def test_static_scratch_refuses_oversized_requests(attn):
    L = attn.lib()
    B, Hq, Hkv, Nk, d, S = 64, 32, 8, 100000, 128, 64
    need = attn.attn_decode_workspace_bytes(B, Hq, Hkv, Nk, d, S)
    assert need > attn.DECODE_STATIC_SCRATCH_BYTES
    o = torch.full((B, 1, Hq, d), 7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, Hq), 7.0, dtype=torch.float32, device=DEV)
    fake = ctypes.c_void_p(0x7f0000000000)  # never dereferenced: refused first
    st = L.attn_decode_splitkv_static(fake, fake, fake, ctypes.c_void_p(o.data_ptr()),
                                      ctypes.c_void_p(lse.data_ptr()), B, Hq, Hkv, Nk, d,
                                      0.1, S, BF16, None)
    assert st == UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(o == 7.0) and torch.all(lse == 7.0)


def test_static_scratch_checks_arguments_first(attn):
    """An invalid call (more segments than keys) is reported as invalid, not
    as too large for the scratch area, and writes nothing."""
    L = attn.lib()
    B, Hq, Hkv, Nk, d, S = 64, 32, 8, 1000, 128, 2000
    o = torch.full((B, 1, Hq, d), 7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, Hq), 7.0, dtype=torch.float32, device=DEV)
    fake = ctypes.c_void_p(0x7f0000000000)  # never dereferenced: refused first
    st = L.attn_decode_splitkv_static(fake, fake, fake, ctypes.c_void_p(o.data_ptr()),
                                      ctypes.c_void_p(lse.data_ptr()), B, Hq, Hkv, Nk, d,
                                      0.1, S, BF16, None)
    assert st == INVALID
    torch.cuda.synchronize()
    assert torch.all(o == 7.0) and torch.all(lse == 7.0)
