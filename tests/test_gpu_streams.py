"""Concurrent use: calls on several CUDA streams, issued from several host
threads at once, give the same results as the same calls made one after
another.  This exercises what the calls share: the per-device launch
set-up caches (first use from several threads at once), the tensor-map
encoding, the per-thread event pools of attn_fwd_host and the device status
words.  Every kernel here is deterministic, so the comparison is bit for
bit."""
import math
import threading

import pytest
import torch

from exact_attention_62_gb300.inputs import make_paged, make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _jobs(attn):
    """(name, fn) pairs; each fn runs its calls on the current stream and
    returns its output tensors."""
    jobs = []
    for i, (B, Hq, Hkv, N, d, causal) in enumerate([(2, 8, 2, 700, 128, True), (3, 6, 3, 513, 64, False),
                                                    (1, 4, 1, 2000, 128, True)]):
        q, k, v = (x.to(DEV) for x in make_qkv(B, Hq, Hkv, N, N, d, 90 + i))
        jobs.append(("fwd%d" % i, lambda q=q, k=k, v=v, c=causal, d=d: attn.attn_fwd(q, k, v, c, 1 / math.sqrt(d))))
    for i, S in enumerate([1, 6, 40]):
        q, k, v = (x.to(DEV) for x in make_qkv(2, 16, 4, 1, 4000, 128, 95 + i))
        jobs.append(("dec%d" % i, lambda q=q, k=k, v=v, S=S: attn.attn_decode_splitkv(q, k, v, 0.088, S)))
    q, kp, vp, table, sl = (x.to(DEV) for x in make_paged(2, 8, 2, 128, 16, [900, 33], seed=98))
    jobs.append(("paged", lambda: attn.attn_decode_paged(q, kp, vp, table, sl, 900, 0.088)))
    qb, kb, vb = (x.to(DEV) for x in make_qkv(1, 4, 2, 300, 300, 128, 99))
    dout = torch.randn_like(qb)

    def bwd():
        o, lse = attn.attn_fwd(qb, kb, vb, True, 0.088)
        return (o, lse) + tuple(attn.attn_bwd(qb, kb, vb, o, lse, dout, True, 0.088))

    jobs.append(("bwd", bwd))
    q8, k8, v8 = (x.to(DEV) for x in make_qkv(1, 4, 2, 400, 400, 128, 100))

    def fp8():
        a, sa = attn.attn_quantize_fp8(q8)
        b, sb = attn.attn_quantize_fp8(k8)
        vt, sv = attn.attn_quantize_fp8_v(v8)
        return attn.attn_fwd_fp8_pv(a, b, vt, sa, sb, sv, True)

    jobs.append(("fp8", fp8))
    qh, kh, vh = make_qkv(1, 8, 2, 1024, 1024, 128, 101)
    qh, kh, vh = qh.pin_memory(), kh.pin_memory(), vh.pin_memory()
    jobs.append(("host", lambda: attn.attn_fwd_host(qh, kh, vh, True, 0.088, chunks=4)))
    return jobs


def test_concurrent_streams_and_threads_match_serial(attn):
    jobs = _jobs(attn)
    serial = {}
    for name, fn in jobs:
        outs = fn()
        # attn_fwd_host returns CPU tensors that its read-back copies fill
        # asynchronously: the results exist once the device is done
        torch.cuda.synchronize()
        serial[name] = [t.clone() for t in outs]
    assert attn.attn_check_device_status() == 0

    results, errors = {}, []

    def worker(name, fn):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                outs = [fn() for _ in range(3)]
            s.synchronize()
            results[name] = outs
        except Exception as e:  # reported below, on the main thread
            errors.append((name, repr(e)))

    threads = [threading.Thread(target=worker, args=job) for job in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert attn.attn_check_device_status() == 0
    for name, _ in jobs:
        for rep in results[name]:
            for a, b in zip(serial[name], rep):
                assert torch.equal(a.cpu(), b.cpu()), name
