"""attn_fwd_host: the forward on host buffers with the transfers overlapped.

Sequences are independent, so whatever the chunking the results equal one
device-side attn_fwd call over the whole batch bit for bit; a small case is
also checked against the oracle.  Covers page-locked and pageable host
memory, 1 to B chunks, fp32, causal and GQA shapes, an empty key set, and
that work queued earlier on the compute stream is ordered before the
copies (a buffer still being written by an earlier kernel)."""
import math

import pytest
import torch

from exact_attention_62_gb300.inputs import make_qkv
from parity import compare

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _device_reference(attn, q, k, v, causal, scale):
    o, lse = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal, scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,chunks,pinned,dtype", [
    (4, 8, 2, 700, 128, True, 0, True, torch.bfloat16),
    (4, 8, 2, 700, 128, True, 1, True, torch.bfloat16),
    (5, 4, 4, 300, 64, False, 5, True, torch.bfloat16),
    (3, 4, 1, 257, 128, True, 2, False, torch.bfloat16),
    (2, 2, 2, 200, 64, False, 2, True, torch.float32),
])
def test_fwd_host_equals_device_call(attn, B, Hq, Hkv, N, d, causal, chunks, pinned, dtype):
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_qkv(B, Hq, Hkv, N, N, d, 41 + B, dtype=dtype)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o, lse = attn.attn_fwd_host(q, k, v, causal, scale, chunks=chunks)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    ro, rl = _device_reference(attn, q, k, v, causal, scale)
    assert torch.equal(o, ro) and torch.equal(lse, rl)


@pytest.mark.parametrize("Hq,Hkv,Nq,Nk,d,causal,chunks", [
    (8, 2, 1300, 1300, 128, True, 0),   # causal, 6 units of 256 rows in 4 chunks
    (4, 4, 1300, 1300, 64, False, 3),   # no mask: every key goes with the first chunk
    (8, 4, 700, 1500, 128, True, 0),    # Nq < Nk: bottom-right causal, keys in prefixes
    (4, 2, 1024, 1024, 128, True, 16),  # more chunks asked than units: one per unit
    (4, 2, 900, 300, 128, True, 0),     # Nq > Nk causal: whole-sequence path
])
def test_fwd_host_one_sequence_in_row_chunks(attn, Hq, Hkv, Nq, Nk, d, causal, chunks):
    """One sequence is cut by query rows (with the key prefix each chunk's
    rows may see); the result equals one device call bit for bit."""
    scale = 1.0 / math.sqrt(d)
    q, k, v = (t.pin_memory() for t in make_qkv(1, Hq, Hkv, Nq, Nk, d, 46 + Nq))
    o, lse = attn.attn_fwd_host(q, k, v, causal, scale, chunks=chunks)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    ro, rl = _device_reference(attn, q, k, v, causal, scale)
    assert torch.equal(o, ro) and torch.equal(lse, rl)


def test_fwd_host_matches_oracle(attn, oracle_mod):
    B, Hq, Hkv, N, d = 3, 4, 2, 333, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_qkv(B, Hq, Hkv, N, N, d, 44)
    o, lse = attn.attn_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), True, scale, chunks=3)
    torch.cuda.synchronize()
    ro, rl = oracle_mod.attn_fwd(q, k, v, True, scale)
    compare(o, lse, ro, rl, torch.bfloat16, "attn_fwd_host vs oracle")


def test_fwd_host_empty_keys(attn):
    q = torch.randn(2, 16, 2, 64).to(torch.bfloat16).pin_memory()
    k = torch.empty(2, 0, 2, 64, dtype=torch.bfloat16).pin_memory()
    o, lse = attn.attn_fwd_host(q, k, k.clone(), False, 0.125)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_fwd_host_orders_after_queued_work(attn):
    """The device input buffer is filled by a kernel queued just before the
    call on the compute stream; the pipeline's copy into it must come after,
    so the result is that of the host inputs."""
    B, Hq, Hkv, N, d = 4, 4, 4, 512, 128
    q, k, v = (t.pin_memory() for t in make_qkv(B, Hq, Hkv, N, N, d, 45))
    bufs = (torch.empty(q.shape, dtype=q.dtype, device=DEV), torch.empty(k.shape, dtype=k.dtype, device=DEV),
            torch.empty(v.shape, dtype=v.dtype, device=DEV), torch.empty(q.shape, dtype=q.dtype, device=DEV),
            torch.empty((B, Hq, N), dtype=torch.float32, device=DEV))
    torch.cuda.synchronize()
    torch.cuda._sleep(20_000_000)          # keep the compute stream busy for a while
    bufs[0].fill_(float("nan"))            # then overwrite the q buffer on it
    o, lse = attn.attn_fwd_host(q, k, v, True, 1.0 / math.sqrt(d), device_buffers=bufs)
    torch.cuda.synchronize()
    ro, rl = _device_reference(attn, q, k, v, True, 1.0 / math.sqrt(d))
    assert torch.equal(o, ro) and torch.equal(lse, rl)


@pytest.mark.parametrize("slow", ["h2d", "d2h"])
def test_fwd_host_done_when_its_stream_is(attn, slow):
    """The results are in the host buffers once the caller's compute stream
    has completed, with nothing else synchronised: the chunks' forwards on
    the library's second compute stream and the read-back copies are all
    ordered before that stream's end.  One copy stream is held back by a
    kernel queued on it before the call, so the pipeline finishes late."""
    Hq, Hkv, N, d = 8, 2, 2048, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = (t.pin_memory() for t in make_qkv(1, Hq, Hkv, N, N, d, 46))
    st, up, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ro, rl = _device_reference(attn, q, k, v, True, scale)
    with torch.cuda.stream(up if slow == "h2d" else down):
        torch.cuda._sleep(20_000_000)
    o, lse = attn.attn_fwd_host(q, k, v, True, scale, chunks=8, stream=st, h2d_stream=up, d2h_stream=down)
    st.synchronize()
    assert torch.equal(o, ro) and torch.equal(lse, rl)
    torch.cuda.synchronize()
