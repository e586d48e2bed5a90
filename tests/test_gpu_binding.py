"""The Python binding rejects caller-provided buffers of the wrong shape,
dtype or layout with ValueError before anything is launched: a kernel never
sees an output, workspace or scale array smaller than the problem it is told
to solve.  After every rejected call the device status is still clean and a
correct call on the same inputs still works."""
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bf(shape, seed=0):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=DEV, dtype=torch.float32).to(torch.bfloat16)


def _rejects(fn, *args, **kw):
    with pytest.raises(ValueError):
        fn(*args, **kw)


def test_forward_buffers(attn):
    B, N, Hq, Hkv, d = 1, 200, 4, 2, 128
    q, k, v = _bf((B, N, Hq, d), 1), _bf((B, N, Hkv, d), 2), _bf((B, N, Hkv, d), 3)
    _rejects(attn.attn_fwd, q, k, v, True, o=torch.empty((B, N - 1, Hq, d), device=DEV, dtype=torch.bfloat16))
    _rejects(attn.attn_fwd, q, k, v, True, o=torch.empty((B, N, Hq, d), device=DEV, dtype=torch.float32))
    _rejects(attn.attn_fwd, q, k, v, True, lse=torch.empty((B, Hq, N - 1), device=DEV))
    _rejects(attn.attn_fwd, q, k, v, True, lse=torch.empty((B, Hq, N), device=DEV, dtype=torch.bfloat16))
    _rejects(attn.attn_fwd, q, k.float(), v, True)                       # mixed input dtypes
    _rejects(attn.attn_fwd, q, k.transpose(1, 2).contiguous().transpose(1, 2), v, True)  # not contiguous
    _rejects(attn.attn_fwd, q, k.cpu(), v, True)                        # not on the device
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    o, lse = attn.attn_fwd(q, k, v, True)
    torch.cuda.synchronize()
    assert torch.isfinite(lse).all() and attn.attn_check_device_status() == 0


def test_decode_buffers(attn):
    B, Nk, Hq, Hkv, d = 2, 1000, 8, 2, 128
    q, k, v = _bf((B, 1, Hq, d), 4), _bf((B, Nk, Hkv, d), 5), _bf((B, Nk, Hkv, d), 6)
    S = attn.attn_decode_num_splits(B, Hq, Hkv, Nk, d)
    need = attn.attn_decode_workspace_bytes(B, Hq, Hkv, Nk, d, S)
    _rejects(attn.attn_decode_splitkv, q, k, v, num_splits=S,
             workspace=torch.empty(need, device=DEV, dtype=torch.float32))
    _rejects(attn.attn_decode_splitkv, q, k, v, o=torch.empty((B, 1, Hq, d - 8), device=DEV, dtype=torch.bfloat16))
    _rejects(attn.attn_decode_splitkv, q, k, v, lse=torch.empty((B * Hq,), device=DEV))
    _rejects(attn.attn_decode_splitkv_static, q, k, v, o=torch.empty((B, 1, Hq - 1, d), device=DEV,
                                                                      dtype=torch.bfloat16))
    _rejects(attn.attn_decode_splitkv_static, q, k, v, lse=torch.empty((B, Hq), device=DEV, dtype=torch.float64))
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    o, lse = attn.attn_decode_splitkv(q, k, v)
    torch.cuda.synchronize()
    assert torch.isfinite(lse).all() and attn.attn_check_device_status() == 0


def test_merge_buffers(attn):
    P, rows, d = 3, 50, 128
    op = torch.randn((P, rows, d), device=DEV)
    lp = torch.randn((P, rows), device=DEV)
    _rejects(attn.attn_merge_lse, op, lp, o=torch.empty((rows - 1, d), device=DEV))
    _rejects(attn.attn_merge_lse, op, lp, lse=torch.empty((rows, 1), device=DEV))
    _rejects(attn.attn_merge_lse, op.to(torch.bfloat16), lp)
    _rejects(attn.attn_merge_lse, op, lp, out_dtype=torch.bfloat16, o=torch.empty((rows, d), device=DEV))
    o, lse = attn.attn_merge_lse(op, lp)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and attn.attn_check_device_status() == 0


def test_paged_buffers(attn):
    B, Hq, Hkv, d, ps, pages_per_seq = 2, 4, 2, 128, 16, 8
    num_pages = B * pages_per_seq
    q = _bf((B, 1, Hq, d), 7)
    kp, vp = _bf((num_pages, ps, Hkv, d), 8), _bf((num_pages, ps, Hkv, d), 9)
    table = torch.arange(num_pages, device=DEV, dtype=torch.int32).reshape(B, pages_per_seq)
    lens = torch.tensor([100, 128], device=DEV, dtype=torch.int32)
    _rejects(attn.attn_decode_paged, q, kp, vp, table.long(), lens, 128)
    _rejects(attn.attn_decode_paged, q, kp, vp, table, lens[:1], 128)
    _rejects(attn.attn_decode_paged, q, kp, vp, table, lens, 128,
             o=torch.empty((B, 1, Hq, d), device=DEV, dtype=torch.float32))
    _rejects(attn.attn_decode_paged, q, kp, vp, table, lens, 128, lse=torch.empty((B, Hq + 1), device=DEV))
    _rejects(attn.attn_decode_paged, q, kp, vp, table, lens, 128, num_splits=2,
             workspace=torch.empty(64, device=DEV, dtype=torch.int32))
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    o, lse = attn.attn_decode_paged(q, kp, vp, table, lens, 128)
    torch.cuda.synchronize()
    assert torch.isfinite(lse).all() and attn.attn_check_device_status() == 0


def test_backward_buffers(attn):
    B, N, Hq, Hkv, d = 1, 256, 2, 1, 128
    q, k, v = _bf((B, N, Hq, d), 10), _bf((B, N, Hkv, d), 11), _bf((B, N, Hkv, d), 12)
    o, lse = attn.attn_fwd(q, k, v, True)
    do = _bf((B, N, Hq, d), 13)
    _rejects(attn.attn_bwd, q, k, v, o, lse[:, :, :-1].contiguous(), do, True)
    _rejects(attn.attn_bwd, q, k, v, o, lse, do.float(), True)
    _rejects(attn.attn_bwd, q, k, v, o, lse, do, True, dq=torch.empty_like(k))
    _rejects(attn.attn_bwd, q, k, v, o, lse, do, True, dk=torch.empty_like(q))
    _rejects(attn.attn_bwd, q, k, v, o, lse, do, True, dv=torch.empty_like(v, dtype=torch.float32))
    _rejects(attn.attn_bwd, q, k, v, o, lse, do, True,
             workspace=torch.empty(1 << 16, device=DEV, dtype=torch.float32))
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    dq, dk, dv = attn.attn_bwd(q, k, v, o, lse, do, True)
    torch.cuda.synchronize()
    assert torch.isfinite(dq.float()).all() and attn.attn_check_device_status() == 0


def test_fp8_buffers(attn):
    B, N, Hq, Hkv, d = 1, 300, 2, 2, 128
    q, k, v = _bf((B, N, Hq, d), 14), _bf((B, N, Hkv, d), 15), _bf((B, N, Hkv, d), 16)
    nb = (N + 127) // 128
    _rejects(attn.attn_quantize_fp8, q, codes=torch.empty((B, N - 1, Hq, d), device=DEV, dtype=torch.uint8))
    _rejects(attn.attn_quantize_fp8, q, scales=torch.empty((B, Hq, nb - 1), device=DEV))
    _rejects(attn.attn_quantize_fp8, q, codes=torch.empty((B, N, Hq, d), device=DEV, dtype=torch.int8))
    q8, qs = attn.attn_quantize_fp8(q)
    k8, ks = attn.attn_quantize_fp8(k)
    _rejects(attn.attn_fwd_fp8, q8, k8, v, qs[:, :, :-1].contiguous(), ks, True)
    _rejects(attn.attn_fwd_fp8, q8, k8, v, qs, ks.double(), True)
    _rejects(attn.attn_fwd_fp8, q8, k8, v, qs, ks, True, o=torch.empty((B, N, Hq, d), device=DEV))
    _rejects(attn.attn_fwd_fp8, q8, k8, v, qs, ks, True, lse=torch.empty((B, N, Hq), device=DEV))
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    o, lse = attn.attn_fwd_fp8(q8, k8, v, qs, ks, True)
    torch.cuda.synchronize()
    assert torch.isfinite(lse).all() and attn.attn_check_device_status() == 0


def test_fp8_pv_buffers(attn):
    B, N, Hq, Hkv, d = 1, 300, 4, 2, 128
    q, k, v = _bf((B, N, Hq, d), 17), _bf((B, N, Hkv, d), 18), _bf((B, N, Hkv, d), 19)
    ld = (N + 15) // 16 * 16
    _rejects(attn.attn_quantize_fp8_v, v, vt8=torch.empty((B, Hkv, d, N), device=DEV, dtype=torch.uint8))
    _rejects(attn.attn_quantize_fp8_v, v, scales=torch.empty((B, Hkv, 1), device=DEV))
    _rejects(attn.attn_quantize_fp8_v, v.float())
    q8, qs = attn.attn_quantize_fp8(q)
    k8, ks = attn.attn_quantize_fp8(k)
    vt8, vs = attn.attn_quantize_fp8_v(v)
    assert tuple(vt8.shape) == (B, Hkv, d, ld)
    _rejects(attn.attn_fwd_fp8_pv, q8, k8, vt8[..., :N].contiguous(), qs, ks, vs, True)   # unpadded rows
    _rejects(attn.attn_fwd_fp8_pv, q8, k8, vt8, qs, ks, vs[:, :1].contiguous(), True)
    _rejects(attn.attn_fwd_fp8_pv, q8, k8, vt8, qs, ks, vs.double(), True)
    _rejects(attn.attn_fwd_fp8_pv, q8, k8, vt8.view(torch.int8), qs, ks, vs, True)
    _rejects(attn.attn_fwd_fp8_pv, q8, k8, vt8, qs, ks, vs, True, o=torch.empty((B, N, Hq, d), device=DEV))
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
    o, lse = attn.attn_fwd_fp8_pv(q8, k8, vt8, qs, ks, vs, True)
    torch.cuda.synchronize()
    assert torch.isfinite(lse).all() and attn.attn_check_device_status() == 0


def test_buffers_used_on_another_stream_are_recorded(attn):
    """A call on a stream other than the current one records its device
    tensors on that stream: a workspace the caller frees right after the
    call is not handed out again by torch's caching allocator while the
    stream (held back by a sleep queued on it) has not yet run the kernels
    that use it.  Without the record the same block comes straight back."""
    B, Hq, Hkv, Nk, d = 1, 8, 2, 4096, 128
    q, k, v = _bf((B, 1, Hq, d), 4), _bf((B, Nk, Hkv, d), 5), _bf((B, Nk, Hkv, d), 6)
    S = 8
    nbytes = attn.attn_decode_workspace_bytes(B, Hq, Hkv, Nk, d, S)
    ref_o, ref_l = attn.attn_decode_splitkv(q, k, v, 0.088, S)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        torch.cuda._sleep(50_000_000)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    ptr = ws.data_ptr()
    o, lse = attn.attn_decode_splitkv(q, k, v, 0.088, S, workspace=ws, stream=side)
    del ws
    again = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    assert again.data_ptr() != ptr
    again.fill_(0xFF)                     # NaN patterns, had the block been reused
    side.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)
    torch.cuda.synchronize()
    assert attn.attn_check_device_status() == 0
