"""Every entry point can be captured into a CUDA graph and replayed
(attn_fwd_host included: its copy streams and second compute stream join
the capture through its events).

A launch path that synchronises, allocates or reads back from the device
would break stream capture; one that baked input values into the launch
(rather than pointers to them) would replay stale results.  Each test
captures a call on static buffers, writes new inputs into those buffers,
replays, and requires the replay to equal an eager call on the new inputs
bit for bit (every kernel here is deterministic: each output element is
written by one CTA in a fixed order), and the forward replay to match the
oracle."""
import math

import numpy as np
import pytest
import torch

from exact_attention_62_gb300.inputs import make_paged, make_qkv
from parity import compare

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _capture(fn):
    """Warm up on a side stream (one-time setup happens outside capture),
    then capture fn into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_forward_graph(attn, oracle_mod):
    B, Hq, Hkv, N, d = 2, 4, 2, 300, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = (x.to(DEV) for x in make_qkv(B, Hq, Hkv, N, N, d, 31))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), device=DEV)
    g = _capture(lambda: attn.attn_fwd(q, k, v, True, scale, o=o, lse=lse))
    q2, k2, v2 = make_qkv(B, Hq, Hkv, N, N, d, 32)
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    eo, el = attn.attn_fwd(q, k, v, True, scale)
    torch.cuda.synchronize()
    assert torch.equal(o, eo) and torch.equal(lse, el)
    ro, rl = oracle_mod.attn_fwd(q2, k2, v2, True, scale)
    compare(o, lse, ro, rl, torch.bfloat16, "graph replay vs oracle")


def test_decode_graph(attn):
    B, Hq, Hkv, Nk, d = 2, 32, 8, 5000, 128
    q, k, v = (x.to(DEV) for x in make_qkv(B, Hq, Hkv, 1, Nk, d, 33))
    S = attn.attn_decode_num_splits(B, Hq, Hkv, Nk, d)
    assert S > 1
    ws = torch.empty(attn.attn_decode_workspace_bytes(B, Hq, Hkv, Nk, d, S), dtype=torch.uint8, device=DEV)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), device=DEV)
    g = _capture(lambda: attn.attn_decode_splitkv(q, k, v, num_splits=S, workspace=ws, o=o, lse=lse))
    o_s = torch.empty_like(q)
    lse_s = torch.empty((B, Hq), device=DEV)
    gs = _capture(lambda: attn.attn_decode_splitkv_static(q, k, v, num_splits=S, o=o_s, lse=lse_s))
    q2, k2, v2 = make_qkv(B, Hq, Hkv, 1, Nk, d, 34)
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2)
    g.replay()
    gs.replay()
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    eo, el = attn.attn_decode_splitkv(q, k, v, num_splits=S)
    torch.cuda.synchronize()
    assert torch.equal(o, eo) and torch.equal(lse, el)
    assert torch.equal(o_s, eo) and torch.equal(lse_s, el)


def test_paged_graph_with_new_table(attn):
    """The serving pattern: capture once with a maximum length, then change
    the block table and the sequence lengths in place between replays."""
    B, Hq, Hkv, d, ps = 3, 8, 2, 128, 16
    max_len = 700
    qh, kp, vp, table, lens = make_paged(B, Hq, Hkv, d, ps, [700, 333, 16], seed=35, extra_pages=6,
                                         poison=False)
    qh, kp, vp, table, lens = (x.to(DEV) for x in (qh, kp, vp, table, lens))
    S = attn.attn_decode_paged_num_splits(B, Hq, Hkv, d, ps, max_len)
    ws = torch.empty(max(16, attn.attn_decode_workspace_bytes(B, Hq, Hkv, max_len, d, S)), dtype=torch.uint8,
                     device=DEV)
    o = torch.empty_like(qh)
    lse = torch.empty((B, Hq), device=DEV)
    g = _capture(lambda: attn.attn_decode_paged(qh, kp, vp, table, lens, max_len, num_splits=S, workspace=ws,
                                                o=o, lse=lse))
    # same pools, a new assignment of pages (sequences may share pages) and new lengths
    gen = torch.Generator().manual_seed(36)
    table.copy_(torch.randint(0, kp.shape[0], tuple(table.shape), generator=gen, dtype=torch.int32))
    lens.copy_(torch.tensor([1, 699, 400], dtype=torch.int32))
    q2 = torch.randn(qh.shape, generator=gen).to(torch.bfloat16)
    qh.copy_(q2)
    g.replay()
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    eo, el = attn.attn_decode_paged(qh, kp, vp, table, lens, max_len, num_splits=S)
    torch.cuda.synchronize()
    assert torch.equal(o, eo) and torch.equal(lse, el)


def test_backward_graph(attn):
    B, Hq, Hkv, N, d = 1, 4, 2, 400, 128
    q, k, v = (x.to(DEV) for x in make_qkv(B, Hq, Hkv, N, N, d, 37))
    dout = torch.randn(q.shape, device=DEV).to(torch.bfloat16)
    o, lse = attn.attn_fwd(q, k, v, True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(max(16, attn.attn_bwd_workspace_bytes(B, Hq, N)), dtype=torch.uint8, device=DEV)

    def step():
        attn.attn_fwd(q, k, v, True, o=o, lse=lse)
        attn.attn_bwd(q, k, v, o, lse, dout, True, dq=dq, dk=dk, dv=dv, workspace=ws)

    g = _capture(step)
    q2, k2, v2 = make_qkv(B, Hq, Hkv, N, N, d, 38)
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    eo, el = attn.attn_fwd(q, k, v, True)
    edq, edk, edv = attn.attn_bwd(q, k, v, eo, el, dout, True)
    torch.cuda.synchronize()
    assert torch.equal(o, eo) and torch.equal(lse, el)
    assert torch.equal(dq, edq) and torch.equal(dk, edk) and torch.equal(dv, edv)


def test_fp8_graph(attn):
    B, Hq, Hkv, N, d = 1, 2, 2, 500, 128
    q, k, v = (x.to(DEV) for x in make_qkv(B, Hq, Hkv, N, N, d, 39))
    nb = (N + 127) // 128
    q8, k8 = torch.empty(q.shape, dtype=torch.uint8, device=DEV), torch.empty(k.shape, dtype=torch.uint8, device=DEV)
    qs, ks = torch.empty((B, Hq, nb), device=DEV), torch.empty((B, Hkv, nb), device=DEV)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), device=DEV)

    def step():
        attn.attn_quantize_fp8(q, codes=q8, scales=qs)
        attn.attn_quantize_fp8(k, codes=k8, scales=ks)
        attn.attn_fwd_fp8(q8, k8, v, qs, ks, True, o=o, lse=lse)

    g = _capture(step)
    q2, k2, v2 = make_qkv(B, Hq, Hkv, N, N, d, 40)
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    eq8, eqs = attn.attn_quantize_fp8(q)
    ek8, eks = attn.attn_quantize_fp8(k)
    eo, el = attn.attn_fwd_fp8(eq8, ek8, v, eqs, eks, True)
    torch.cuda.synchronize()
    assert torch.equal(q8, eq8) and torch.equal(qs, eqs) and torch.equal(k8, ek8) and torch.equal(ks, eks)
    assert torch.equal(o, eo) and torch.equal(lse, el)


def test_fp8_pv_graph(attn):
    """Quantise Q, K, V and run the e4m3 P V forward from one graph: the
    V quantiser's memset, amax, codes and scale passes replay too."""
    B, Hq, Hkv, N, d = 1, 4, 2, 500, 128
    q, k, v = (x.to(DEV) for x in make_qkv(B, Hq, Hkv, N, N, d, 45))
    nb = (N + 127) // 128
    ld = (N + 15) // 16 * 16
    q8, k8 = torch.empty(q.shape, dtype=torch.uint8, device=DEV), torch.empty(k.shape, dtype=torch.uint8, device=DEV)
    qs, ks = torch.empty((B, Hq, nb), device=DEV), torch.empty((B, Hkv, nb), device=DEV)
    vt8 = torch.empty((B, Hkv, d, ld), dtype=torch.uint8, device=DEV)
    vs = torch.empty((B, Hkv), device=DEV)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), device=DEV)

    def step():
        attn.attn_quantize_fp8(q, codes=q8, scales=qs)
        attn.attn_quantize_fp8(k, codes=k8, scales=ks)
        attn.attn_quantize_fp8_v(v, vt8=vt8, scales=vs)
        attn.attn_fwd_fp8_pv(q8, k8, vt8, qs, ks, vs, True, o=o, lse=lse)

    g = _capture(step)
    q2, k2, v2 = make_qkv(B, Hq, Hkv, N, N, d, 46)
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2 * 3)
    g.replay()
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    eq8, eqs = attn.attn_quantize_fp8(q)
    ek8, eks = attn.attn_quantize_fp8(k)
    evt, evs = attn.attn_quantize_fp8_v(v)
    eo, el = attn.attn_fwd_fp8_pv(eq8, ek8, evt, eqs, eks, evs, True)
    torch.cuda.synchronize()
    assert torch.equal(vt8, evt) and torch.equal(vs, evs)
    assert torch.equal(o, eo) and torch.equal(lse, el)


@pytest.mark.parametrize("B,Nq,Nk,causal,chunks", [(1, 1000, 1000, True, 4),   # chunks of query rows
                                                   (3, 300, 500, False, 3)])    # chunks of sequences
def test_host_pipeline_graph(attn, B, Nq, Nk, causal, chunks):
    """attn_fwd_host in a graph: its copies, events and second compute stream
    join the capture; a replay reads the page-locked inputs' new contents and
    writes the results into the same host outputs."""
    Hq, Hkv, d = 4, 2, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nk, d, 41)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    lh = torch.empty((B, Hq, Nq), dtype=torch.float32).pin_memory()
    bufs = (torch.empty(q.shape, dtype=q.dtype, device=DEV), torch.empty(k.shape, dtype=k.dtype, device=DEV),
            torch.empty(v.shape, dtype=v.dtype, device=DEV), torch.empty(q.shape, dtype=q.dtype, device=DEV),
            torch.empty((B, Hq, Nq), dtype=torch.float32, device=DEV))
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    g = _capture(lambda: attn.attn_fwd_host(qh, kh, vh, causal, scale, o=oh, lse=lh, device_buffers=bufs,
                                            chunks=chunks, h2d_stream=up, d2h_stream=down))
    q2, k2, v2 = make_qkv(B, Hq, Hkv, Nq, Nk, d, 42)
    qh.copy_(q2)
    kh.copy_(k2)
    vh.copy_(v2)
    oh.zero_()
    lh.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    eo, el = attn.attn_fwd(q2.to(DEV), k2.to(DEV), v2.to(DEV), causal, scale)
    torch.cuda.synchronize()
    assert torch.equal(oh, eo.cpu()) and torch.equal(lh, el.cpu())
